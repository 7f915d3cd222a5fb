// gemv_hm.cu -- Q2_0 decode GEMV for 1..8 activation rows on the FP16 warp tensor cores.
//
// Source: init_q2.rs `set_packed_q2_qkvz` (decode runs `q2_0_gemv_vec`) and
// dense_ffn_decode_batch.rs `forward_km_q2` (`q2_0_gemv_vec_batchm` for gate/up/down).
//
// Design (GB300).  The packed weight (2.125 bits per weight) is the only large stream.  On
// sm_103a the legacy FP16 warp MMA (m16n8k16) runs at ~940 MAC/clk/SM while integer logic
// and FP16x2 arithmetic run at half rate, so the unpack of the 2-bit codes, not the MMA,
// sets the cost per weight.  Hence:
//
//  * Weights (A operand): one LOP3 per pair of codes ORs the code at bit position 2i of its
//    byte into the mantissa of the FP16 value 1024 in each 16-bit half (1024 + c 4^i; the
//    four positions of a byte's low half need no shift, the high bytes one shift per 32-bit
//    word), and one FP16 FMA by 4^-i minus (1024 4^-i + 2) turns that into c - 2, exactly.
//    A zero weight thus gives an exactly zero product: no large activation enters an MMA's
//    sums unless its weight is nonzero (an offset form such as c X - 2 X loses the small
//    products next to a large one inside the tensor core's sum).
//  * Activations (B operand): x is turned once per CTA into an FP16 table in fragment order,
//    X = x 2^s with one power of two 2^s per activation row (its maximum maps to
//    [2^14, 2^15)).  Every x within 22 binades of its row's maximum is exact in the table;
//    smaller ones are off by at most 2^-25 of the maximum.  Each 128-column block's fp32
//    sum of (c - 2) X is scaled by its BF16 d; the result is multiplied by 2^-s.
//  * Staging: the CTA's rows are a contiguous byte range of the code plane; chunks of 16 T
//    rows arrive by 1-D bulk copies into a ring (no tensor maps to encode per call), the
//    first ones requested before waiting on the previous kernel (programmatic dependent
//    launch: weights never depend on it), together with one bulk copy of the CTA's scales.
//    Waits suspend the warp in hardware (mbarrier.try_wait) and are bounded.
//  * Compute: WG groups of eight warps; group w takes the chunk's tiles w, w + WG, ..., and
//    warp j of a group the pack blocks j, j + 8, ... of its tiles, four at a time with
//    independent accumulators.  Every warp leaves its per-tile sums in a slot of its own;
//    the last warp to release a stage adds the slots in a fixed order (so results do not
//    depend on timing), stores the chunk's BF16 outputs (and the FFN's SiLU*mul) and
//    requests the next chunk into the stage.
//  * Work split: CTA c takes rows [c n / C, (c + 1) n / C), so every SM streams the same
//    number of bytes to within one row.
#include "common.cuh"

namespace bq8 {

constexpr int HM_MAX_STAGES = 8;
constexpr int HM_CHUNK_TARGET = 20480;     // code bytes per 8-warp group and chunk, about
constexpr int HM_SMEM_SHARE = 112 * 1024;  // one warp group: two CTAs per SM (the next launch's prologue)
constexpr int HM_SMEM_LIMIT = 225 * 1024;

static __device__ unsigned int g_hm_status;

unsigned int gemv_hm_status_take() {
    unsigned int v = 0, zero = 0;
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(&v, g_hm_status, sizeof v);
    cudaMemcpyToSymbol(g_hm_status, &zero, sizeof zero);
    return v;
}

struct HmParams {
    const uint8_t* codes;    // [n][k/4]
    const uint16_t* scales;  // [n][k/group] BF16
    const uint16_t* x;       // [m][k] BF16
    uint16_t* y;             // [m][n] BF16
    uint16_t* hgate;         // optional [m][n] BF16: replaced by BF16(SiLU(hgate) * y)
    int n, k, group;
    int rmax;                // rows of the largest CTA
    int tiles_per_chunk;     // T: a chunk is 16 T rows
    int nstages;
};

// Shared-memory carve-up, identical on host and device.
struct HmLayout {
    size_t ring, btab, scal, part, misc, total;
    __host__ __device__ HmLayout(int m, int k, int group, int T, int nstages, int rmax) {
        const size_t rowbytes = (size_t)k / 4;
        const size_t P = (size_t)k / 128, G = (size_t)k / group;
        const size_t rmax16 = ((size_t)rmax + 15) / 16 * 16;
        ring = 0;
        btab = ring + (size_t)nstages * 16 * T * rowbytes;                 // [P][8 MMAs][m][4 lanes][8 B]
        scal = btab + P * 8 * (size_t)m * 32;                               // CTA's scale rows (+ alignment)
        part = scal + ((rmax16 * G * 2 + 32 + 15) & ~size_t(15));           // [stage][T][8][16][m] fp32
        misc = part + (size_t)nstages * T * 8 * 16 * m * 4;                 // barriers, counters, row scales
        total = misc + HM_MAX_STAGES * 8 + 8 + HM_MAX_STAGES * 4 * 2 + 8 * 4 * 2 + 16;
    }
};

// Waits on phase `parity` of `bar` (suspending, bounded); the answer is the warp's, so the
// warp-synchronous MMAs that follow run with every lane or none.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
    const bool ok = mbar_wait_suspend(bar, parity);
    return __all_sync(0xffffffffu, ok) != 0;
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// c - 2 for the two codes at bit position I of the bytes picked by `w` (low bytes, or high
// bytes after a shift by 8), as an FP16 pair: (1024 + c 4^I) 4^-I - (1024 4^-I + 2).
template <int I>
__device__ __forceinline__ uint32_t codes_f16(uint32_t w) {
    constexpr uint32_t msk = 0x00030003u << (2 * I);
    constexpr uint32_t q4 = I == 0 ? 0x3C003C00u : I == 1 ? 0x34003400u : I == 2 ? 0x2C002C00u : 0x24002400u;
    constexpr uint32_t off = I == 0 ? 0xE402E402u : I == 1 ? 0xDC08DC08u : I == 2 ? 0xD420D420u : 0xCC80CC80u;
    return hfma2_bits(and_or(w, msk, 0x64006400u), q4, off);
}

template <int I>
__device__ __forceinline__ void mma_position(float (&acc)[4], uint32_t lo, uint32_t lo8, uint2 b) {
    mma_f16_16816(acc, codes_f16<I>(lo), codes_f16<I>(lo8), codes_f16<I>(lo >> 8), codes_f16<I>(lo8 >> 8), b.x, b.y);
}

// NB pack blocks (pb, pb + 8, ...) of one 16-row tile for lane (g, t): its code words 2t,
// 2t + 1 of rows g and g + 8 in each block, 8 MMAs per block (MMA 4s + i takes bit position
// i of word 2t + s: low bytes as fragment columns (k, k + 1), high bytes as (k + 8, k + 9)),
// then each block's sum scaled by its BF16 d into tot.  The NB accumulator chains are
// independent.  All lanes run the same instructions (the MMA is warp-synchronous); lanes
// past the activation rows keep zero B fragments.
template <int M, int NB>
__device__ __forceinline__ void hm_blocks(float (&tot)[4], const uint8_t* cg, const uint8_t* cg8, const uint8_t* bq,
                                          bool hasb, const uint16_t* sg, const uint16_t* sg8, int pb, int gsh) {
    uint2 w[NB], w8[NB];
#pragma unroll
    for (int q = 0; q < NB; q++) {
        w[q] = *reinterpret_cast<const uint2*>(cg + q * 8 * 32);
        w8[q] = *reinterpret_cast<const uint2*>(cg8 + q * 8 * 32);
    }
    float ac[NB][4];
#pragma unroll
    for (int q = 0; q < NB; q++) ac[q][0] = ac[q][1] = ac[q][2] = ac[q][3] = 0.f;
    constexpr int BBLK = 8 * M * 32;  // table bytes per pack block
#pragma unroll
    for (int s = 0; s < 2; s++) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
#pragma unroll
            for (int q = 0; q < NB; q++) {
                const uint32_t lo = s ? w[q].y : w[q].x, lo8 = s ? w8[q].y : w8[q].x;
                uint2 b = make_uint2(0u, 0u);
                if (hasb) b = *reinterpret_cast<const uint2*>(bq + q * 8 * BBLK + (4 * s + i) * M * 32);
                if (i == 0) mma_position<0>(ac[q], lo, lo8, b);
                if (i == 1) mma_position<1>(ac[q], lo, lo8, b);
                if (i == 2) mma_position<2>(ac[q], lo, lo8, b);
                if (i == 3) mma_position<3>(ac[q], lo, lo8, b);
            }
        }
    }
#pragma unroll
    for (int q = 0; q < NB; q++) {
        const int gi = (pb + q * 8) >> gsh;
        const float d0 = bf16_bits_to_f32(sg[gi]), d8 = bf16_bits_to_f32(sg8[gi]);
        tot[0] = fmaf(d0, ac[q][0], tot[0]);
        tot[1] = fmaf(d0, ac[q][1], tot[1]);
        tot[2] = fmaf(d8, ac[q][2], tot[2]);
        tot[3] = fmaf(d8, ac[q][3], tot[3]);
    }
}

template <int M, int WG>
__global__ void __launch_bounds__(256 * WG, WG == 1 ? 2 : 1) q2_gemv_hm_kernel(const HmParams p) {
    constexpr int NW = 8 * WG;  // warps
    constexpr int NT = 32 * NW;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int n = p.n, k = p.k;
    const HmLayout L(M, k, p.group, p.tiles_per_chunk, p.nstages, p.rmax);
    uint8_t* ring = smem_raw + L.ring;
    uint8_t* btab = smem_raw + L.btab;
    uint8_t* scal = smem_raw + L.scal;
    float* part = reinterpret_cast<float*>(smem_raw + L.part);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + L.misc);
    uint64_t* sbar = full + HM_MAX_STAGES;
    uint32_t* released = reinterpret_cast<uint32_t*>(sbar + 1);
    int* issued = reinterpret_cast<int*>(released + HM_MAX_STAGES);
    uint32_t* rowmax = reinterpret_cast<uint32_t*>(issued + HM_MAX_STAGES);
    float* rowback = reinterpret_cast<float*>(rowmax + 8);  // 2^-s per activation row

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wgrp = warp >> 3, ww = warp & 7;
    const int g = lane >> 2, t = lane & 3;
    const int r0 = (int)((int64_t)blockIdx.x * n / gridDim.x);
    const int R = (int)((int64_t)(blockIdx.x + 1) * n / gridDim.x) - r0;
    const size_t rowbytes = (size_t)k / 4;
    const int P = k >> 7, G = k / p.group;
    const int T = p.tiles_per_chunk, CR = 16 * T, NST = p.nstages;
    const int nch = (R + CR - 1) / CR;
    const int pre = nch < NST ? nch : NST;
    const uint8_t* src = p.codes + (size_t)r0 * rowbytes;
    const size_t stage_bytes = (size_t)CR * rowbytes;

    // the CTA's scales: bytes [s_lo, s_hi) of the plane by one bulk copy, the rest (at most
    // 14 bytes at the end of the plane) by plain loads
    const uint8_t* splane = reinterpret_cast<const uint8_t*>(p.scales);
    const int64_t s_lo = ((int64_t)r0 * G * 2) & ~int64_t(15);
    const int64_t s_end = (int64_t)(r0 + R) * G * 2;
    int64_t s_hi = (s_end + 15) & ~int64_t(15);
    const int64_t plane16 = ((int64_t)n * G * 2) & ~int64_t(15);
    if (s_hi > plane16) s_hi = plane16;
    if (s_hi < s_lo) s_hi = s_lo;
    const uint16_t* srow = reinterpret_cast<const uint16_t*>(scal + ((int64_t)r0 * G * 2 - s_lo));

    if (tid == 0) {
        for (int s = 0; s < NST; s++) {
            mbar_init(&full[s], 1);
            released[s] = 0;
            issued[s] = s < pre ? s : -1;
        }
        mbar_init(sbar, 1);
        fence_barrier_init();
        // weights first: they do not depend on the kernel launched before this one
        for (int c = 0; c < pre; c++) {
            const uint32_t bytes = (uint32_t)(min(CR, R - c * CR) * rowbytes);
            mbar_arrive_expect_tx(&full[c], bytes);
            bulk_load(ring + (size_t)c * stage_bytes, src + (size_t)c * stage_bytes, bytes, &full[c]);
        }
        mbar_arrive_expect_tx(sbar, (uint32_t)(s_hi - s_lo));
        if (s_hi > s_lo) bulk_load(scal, splane + s_lo, (uint32_t)(s_hi - s_lo), sbar);
    }
    if (tid == 32)
        for (int64_t o = s_hi; o < s_end; o += 2)
            *reinterpret_cast<uint16_t*>(scal + (o - s_lo)) = __ldg(reinterpret_cast<const uint16_t*>(splane + o));
    if (tid < 8) rowmax[tid] = 0u;
    __syncthreads();

    pdl_wait();
    pdl_launch_dependents();

    // ---- activations: per-row maximum, then the FP16 fragment table
    const int kv = k >> 3;  // 8-value vectors per row
    for (int j = 0; j < M; j++) {
        const uint4* xr = reinterpret_cast<const uint4*>(p.x + (size_t)j * k);
        float mx = 0.f;
        for (int v = tid; v < kv; v += NT) {
            const uint4 q = __ldg(xr + v);
            const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int h = 0; h < 4; h++)
                mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(u[h] << 16)), fabsf(__uint_as_float(u[h] & 0xFFFF0000u))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) atomicMax(&rowmax[j], __float_as_uint(mx));
    }
    __syncthreads();
    for (int j = 0; j < M; j++) {
        const uint32_t mb = rowmax[j];
        // 2^s with the row maximum in [2^14, 2^15); capped where 2^s and 2^-s stay normal floats
        int sh = mb ? 14 - (int)((mb >> 23) & 0xFF) + 127 : 0;
        sh = max(-113, min(sh, 120));
        const float p2s = __int_as_float((127 + sh) << 23);
        if (tid == 0) rowback[j] = __int_as_float((127 - sh) << 23);
        const uint4* xr = reinterpret_cast<const uint4*>(p.x + (size_t)j * k);
        for (int v = tid; v < kv; v += NT) {
            const uint4 q = __ldg(xr + v);
            const uint32_t u[4] = {q.x, q.y, q.z, q.w};
            float X[8];
#pragma unroll
            for (int h = 0; h < 4; h++) {
                X[2 * h] = __uint_as_float(u[h] << 16) * p2s;
                X[2 * h + 1] = __uint_as_float(u[h] & 0xFFFF0000u) * p2s;
            }
            const int col = v << 3;
            const int pb = col >> 7, i = (col >> 5) & 3, tt = (col >> 3) & 3;
#pragma unroll
            for (int s = 0; s < 2; s++) {
                const float* e = X + 4 * s;
                // entry of lane (j, tt) for MMA 4s + i: columns (0, 2) then (1, 3)
                const uint2 ent = make_uint2(f16x2_bits(e[0], e[2]), f16x2_bits(e[1], e[3]));
                *reinterpret_cast<uint2*>(btab + (((size_t)pb * 8 + 4 * s + i) * M + j) * 32 + tt * 8) = ent;
            }
        }
    }
    __syncthreads();

    // ---- main loop
    bool failed = !warp_wait(sbar, 0);
    const bool hasb = g < M;
    const uint8_t* blane = btab + (hasb ? g : 0) * 32 + t * 8;  // this lane's table entries
    const int gsh = __ffs(p.group) - 1 - 7;                       // group = 128 << gsh
    for (int c = 0; c < nch && !failed; c++) {
        const int s = c % NST;
        if (!warp_wait(&full[s], (uint32_t)(c / NST) & 1u)) {
            failed = true;
            break;
        }
        const uint8_t* st = ring + (size_t)s * stage_bytes;
        const int rows_in = min(CR, R - c * CR);
        const int ntiles = (rows_in + 15) >> 4;
        for (int tau = wgrp; tau < ntiles; tau += WG) {
            const int rt = c * CR + tau * 16;  // CTA row of the tile's first row
            const uint8_t* cg = st + (size_t)(tau * 16 + g) * rowbytes + t * 8;
            const uint8_t* cg8 = cg + 8 * rowbytes;
            const uint16_t* sg = srow + (size_t)(rt + g) * G;
            const uint16_t* sg8 = sg + 8 * G;
            float tot[4] = {0.f, 0.f, 0.f, 0.f};
            int pb = ww;
            for (; pb + 24 < P; pb += 32)
                hm_blocks<M, 4>(tot, cg + pb * 32, cg8 + pb * 32, blane + pb * 8 * M * 32, hasb, sg, sg8, pb, gsh);
            for (; pb < P; pb += 8)
                hm_blocks<M, 1>(tot, cg + pb * 32, cg8 + pb * 32, blane + pb * 8 * M * 32, hasb, sg, sg8, pb, gsh);
            // this warp's slot: [stage][tile][warp][row][activation row]
            float* slot = part + (((size_t)s * T + tau) * 8 + ww) * 16 * M;
            if (2 * t < M) {
                slot[g * M + 2 * t] = tot[0];
                slot[(g + 8) * M + 2 * t] = tot[2];
            }
            if (2 * t + 1 < M) {
                slot[g * M + 2 * t + 1] = tot[1];
                slot[(g + 8) * M + 2 * t + 1] = tot[3];
            }
        }
        // release the stage; the last warp to release it adds the slots, stores the chunk's
        // outputs and requests chunk c + NST into the stage
        __syncwarp();
        uint32_t before = 0;
        if (lane == 0) {
            __threadfence_block();
            before = atomicAdd(&released[s], 1u);
        }
        before = __shfl_sync(0xffffffffu, before, 0);
        if (before == (uint32_t)(NW * (c / NST + 1) - 1)) {
            __syncwarp();
            for (int o = lane; o < M * rows_in; o += 32) {
                const int j = o / rows_in, row = o - j * rows_in;
                const float* sl = part + (((size_t)s * T + (row >> 4)) * 8) * 16 * M + (row & 15) * M + j;
                float sum = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < 8; w8++) sum += sl[w8 * 16 * M];
                const __nv_bfloat16 bv = __float2bfloat16_rn(sum * rowback[j]);
                const uint16_t ub = *reinterpret_cast<const uint16_t*>(&bv);
                const size_t idx = (size_t)j * n + r0 + c * CR + row;
                p.y[idx] = ub;
                if (p.hgate) {
                    const __nv_bfloat16 hb =
                        __float2bfloat16_rn(silu_mul1(bf16_bits_to_f32(p.hgate[idx]), bf16_bits_to_f32(ub)));
                    p.hgate[idx] = *reinterpret_cast<const uint16_t*>(&hb);
                }
            }
            __syncwarp();
            const int cn = c + NST;
            if (lane == 0 && cn < nch) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issued[s] = cn;
                const uint32_t bytes = (uint32_t)(min(CR, R - cn * CR) * rowbytes);
                mbar_arrive_expect_tx(&full[s], bytes);
                bulk_load(ring + (size_t)s * stage_bytes, src + (size_t)cn * stage_bytes, bytes, &full[s]);
            }
        }
    }
    if (failed && lane == 0) atomicOr(&g_hm_status, 1u);
    __syncthreads();
    if (tid == 0) {  // wind down: every requested copy must have landed before the CTA exits
        for (int s = 0; s < NST; s++) {
            const int c = issued[s];
            if (c >= 0 && !mbar_wait_suspend(&full[s], (uint32_t)(c / NST) & 1u)) atomicOr(&g_hm_status, 1u);
        }
        if (!mbar_wait_suspend(sbar, 0)) atomicOr(&g_hm_status, 1u);
    }
}

// Launch plan: one CTA per SM (at most one per 16 rows), chunks of about HM_CHUNK_TARGET code
// bytes per warp group, as many ring stages as fit.  One warp group (256 threads) while two
// CTAs fit an SM's shared memory with three stages or more, so the next launch's CTA can
// start its weight copies early; two groups (512 threads, one CTA per SM) otherwise.
static int hm_plan(int m, int n, int k, int group, int sms, HmParams* prm, int* wg_out, size_t* smem_out) {
    const size_t rowbytes = (size_t)k / 4;
    int ncta = (n + 15) / 16;
    if (ncta > sms) ncta = sms;
    const int rmax = (n + ncta - 1) / ncta;
    const int tiles_max = (rmax + 15) / 16;
    size_t smem = 0;
    int T = 1, NST = 2, WG = 1;
    for (WG = 1; WG <= 2; WG++) {
        int per = (int)(HM_CHUNK_TARGET / (16 * rowbytes));
        if (per < 1) per = 1;
        T = per * WG;
        if (T > tiles_max) T = tiles_max;
        const int nch = (rmax + 16 * T - 1) / (16 * T);
        NST = HM_MAX_STAGES;
        if (NST > nch) NST = nch < 2 ? 2 : nch;
        const size_t cap = WG == 1 ? (size_t)HM_SMEM_SHARE : (size_t)HM_SMEM_LIMIT;
        while (NST > 2 && HmLayout(m, k, group, T, NST, rmax).total > cap) NST--;
        smem = HmLayout(m, k, group, T, NST, rmax).total;
        if (WG == 1 && smem <= (size_t)HM_SMEM_SHARE && (NST >= 3 || NST >= nch)) break;
        if (WG == 2) break;
    }
    prm->n = n;
    prm->k = k;
    prm->group = group;
    prm->rmax = rmax;
    prm->tiles_per_chunk = T;
    prm->nstages = NST;
    *wg_out = WG;
    *smem_out = smem;
    return ncta;
}

// Shapes this kernel takes: the activation table (2 m k bytes) and a two-stage ring fit one
// SM's shared memory.
bool gemv_hm_supported(const bq_q2_weight* w, uint32_t m) {
    if (w->k == 0 || w->n == 0 || m < 1 || m > 8) return false;
    HmParams prm;
    int wg = 1;
    size_t smem = 0;
    hm_plan((int)m, (int)w->n, (int)w->k, (int)w->group, 148, &prm, &wg, &smem);
    return smem <= (size_t)HM_SMEM_LIMIT;
}

typedef void (*HmKernel)(const HmParams);

template <int WG>
static HmKernel hm_kernel_for(uint32_t m) {
    switch (m) {
        case 1: return q2_gemv_hm_kernel<1, WG>;
        case 2: return q2_gemv_hm_kernel<2, WG>;
        case 3: return q2_gemv_hm_kernel<3, WG>;
        case 4: return q2_gemv_hm_kernel<4, WG>;
        case 5: return q2_gemv_hm_kernel<5, WG>;
        case 6: return q2_gemv_hm_kernel<6, WG>;
        case 7: return q2_gemv_hm_kernel<7, WG>;
        case 8: return q2_gemv_hm_kernel<8, WG>;
        default: return nullptr;
    }
}

int launch_q2_gemv_hm(const uint16_t* x, const bq_q2_weight* w, uint16_t* y, uint32_t m, uint16_t* hgate,
                      cudaStream_t stream, const char* who) {
    static int configured_smem[64][2][8] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64) dev = 63;
    if (m < 1 || m > 8) return fail(BQ_ERR_INVALID, "%s: m = %u, must be 1..8", who, m);
    HmParams prm;
    int WG = 1;
    size_t smem = 0;
    const int ncta = hm_plan((int)m, (int)w->n, (int)w->k, (int)w->group, sm_count(), &prm, &WG, &smem);
    if (smem > (size_t)HM_SMEM_LIMIT) return fail(BQ_ERR_INVALID, "%s: shape needs too much shared memory", who);
    const HmKernel kern = WG == 1 ? hm_kernel_for<1>(m) : hm_kernel_for<2>(m);
    if ((size_t)configured_smem[dev][WG - 1][m - 1] < smem) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: cannot reserve %zu bytes of shared memory", who, smem);
        configured_smem[dev][WG - 1][m - 1] = (int)smem;
    }
    prm.codes = (const uint8_t*)w->data;
    prm.scales = (const uint16_t*)((const uint8_t*)w->data + (size_t)w->n * (w->k / 4));
    prm.x = x;
    prm.y = y;
    prm.hgate = hgate;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ncta);
    cfg.blockDim = dim3(256u * WG);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) return check_launch(who);
    return check_launch(who);
}

}  // namespace bq8
