// gemv.cu -- Q2_0 decode GEMV for 1..8 activation rows, and the packed-Q2 FFN chain.
//
// Source: init_q2.rs `set_packed_q2_qkvz` (decode runs `q2_0_gemv_vec`) and
// dense_ffn_decode_batch.rs `forward_km_q2` (`q2_0_gemv_vec_batchm` for gate/up/down).
//
// Design (GB300).  The packed weight (2.125 bits per weight) is the only large stream; the
// kernel must keep the per-weight instruction count low and stay within the native legacy
// tensor pipe.  On sm_103a the warp-level BF16 MMA (m16n8k16, HMMA) is native; the e4m3 and
// int8 forms are not (they expand into conversions plus HMMAs), so:
//
//  * Weights (A operand, 16 rows x 16 columns per MMA): one lop3 per pair of codes drops a
//    2-bit code into the mantissa of BF16 1.0 in each 16-bit half, v = 1 + c*s with
//    s = 2^-7, 2^-5 or 2^-3 depending on the code's bit position (three of the four
//    positions need no shift).
//  * Activations (B operand, 16 columns x 8 rows): per pack block each warp builds its
//    fragment from the staged activations, each column pre-multiplied by 1/s (exact: a
//    power of two) and permuted to the lanes' code order, so sum(v*x/s) = sum(x/s) +
//    sum(c*x).
//  * sum((c - 2) x) = sum(v x/s) - sum((1/s + 2) x): the second sum, per activation row and
//    128-column block, is formed on the CUDA cores and seeds every tile's accumulator; each
//    128-column group is then scaled by its BF16 d.
//  * Staging: the CTA's rows stream through a shared-memory ring of up to four stages: per
//    chunk two TMA boxes of all the CTA's rows x 128 bytes (128-byte swizzle) for the codes
//    and 256-column boxes for the activations, mbarrier completion.  There is no producer
//    warp: the last warp to release a stage requests the next chunk into it.  Every wait
//    is bounded.
//  * Compute: eight warps; warp w takes pack block w of each 256-byte chunk for all of the
//    CTA's 16-row tiles.  MMAs are issued column-step outer, tile inner, so consecutive MMAs
//    are independent.
//  * Work split: CTA c takes a contiguous range of <= T row tiles (grid = SM count when
//    possible, so every SM streams the same number of rows); the warps' partial sums are
//    reduced through shared memory and stored as BF16.  When the rows are too few to give
//    every SM about seven tiles (the down projection: 320 tiles of a long k), a cluster of
//    S CTAs shares a row range, each streaming 1/S of the chunks, and the leader adds the
//    members' partial sums through distributed shared memory before the BF16 store.
#include "common.cuh"

namespace bq8 {

constexpr int GEMV_PBLK = 8;                          // pack blocks per chunk (256 bytes of a row)
constexpr int GEMV_CWARPS = 8;                        // warps: one per pack block
constexpr int GEMV_THREADS = GEMV_CWARPS * 32;
constexpr int GEMV_MAX_T = 8;                         // row tiles per CTA (128 rows)
constexpr int GEMV_MAX_STAGES = 4;
constexpr int GEMV_BOX = 16 * 128;                    // one codes box: 16 rows x 128 bytes
constexpr int GEMV_XBOX = 256;                        // activations per x box row (bf16)
constexpr int GEMV_SMEM_LIMIT = 225 * 1024;
constexpr int GEMV_SMEM_SHARE = 112 * 1024;            // two CTAs per SM

static __device__ unsigned int g_gemv_status;

unsigned int gemv_status_take() {
    unsigned int v = 0, zero = 0;
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(&v, g_gemv_status, sizeof v);
    cudaMemcpyToSymbol(g_gemv_status, &zero, sizeof zero);
    return v;
}

// Code pair SUB (0..7) of a packed 32-bit word: bytes (0,2) for SUB < 4, bytes (1,3)
// otherwise; sub-block i = SUB & 3 sits in bits 2i of each byte.  mask[i] holds the code
// mask of position i; `one` is bf16x2 (1.0, 1.0).
template <int SUB>
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w, const uint32_t (&mask)[3], uint32_t one) {
    if constexpr (SUB < 3) return and_or(w, mask[SUB], one);
    if constexpr (SUB == 3) return and_or(w >> 2, mask[2], one);
    if constexpr (SUB < 7) return and_or(w >> 8, mask[SUB - 4], one);
    return and_or(w >> 10, mask[2], one);
}

template <int RHO>
__device__ __forceinline__ uint32_t unpack_rho(uint2 w, const uint32_t (&mask)[3], uint32_t one) {
    return unpack_pair<RHO & 7>((RHO >> 3) ? w.y : w.x, mask, one);
}

// Column step MU (16 columns) of every tile of the warp: tile-inner, so the TQ MMAs in a
// row are independent.
template <int MU, int TQ>
__device__ __forceinline__ void gemv_step(float (&acc)[TQ][4], const uint2 (&wa)[TQ], const uint2 (&wb)[TQ],
                                          const uint32_t (&b)[16], const uint32_t (&mask)[3], uint32_t one) {
#pragma unroll
    for (int q = 0; q < TQ; q++)
        mma_bf16_16816(acc[q], unpack_rho<2 * MU>(wa[q], mask, one), unpack_rho<2 * MU>(wb[q], mask, one),
                       unpack_rho<2 * MU + 1>(wa[q], mask, one), unpack_rho<2 * MU + 1>(wb[q], mask, one),
                       b[2 * MU], b[2 * MU + 1], acc[q]);
}

// B fragment of lane (g, t) for one pack block, from activation row g's 128 columns (X[i]
// = columns 32i + 8t .. 32i + 8t + 7): register rho = 8w + sub pairs columns 4w + bo and
// 4w + bo + 2 of run i = sub & 3 (bo = sub >> 2), scaled by 1/s_i = 128, 32, 8, 8.  Also
// returns this lane's share of -sum((1/s + 2) x).
__device__ __forceinline__ float build_bfrag(uint32_t (&b)[16], const uint4 (&X)[4]) {
    const __nv_bfloat162 scl[4] = {__floats2bfloat162_rn(128.f, 128.f), __floats2bfloat162_rn(32.f, 32.f),
                                   __floats2bfloat162_rn(8.f, 8.f), __floats2bfloat162_rn(8.f, 8.f)};
    float off = 0.f;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float coef = i == 0 ? -130.f : (i == 1 ? -34.f : -10.f);
        const uint32_t wds[4] = {X[i].x, X[i].y, X[i].z, X[i].w};
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 4; j++) s += __uint_as_float(wds[j] << 16) + __uint_as_float(wds[j] & 0xFFFF0000u);
        off = fmaf(coef, s, off);
#pragma unroll
        for (int w = 0; w < 2; w++) {
#pragma unroll
            for (int bo = 0; bo < 2; bo++) {
                const uint32_t pr = __byte_perm(w ? X[i].z : X[i].x, w ? X[i].w : X[i].y, bo ? 0x7632 : 0x5410);
                b[8 * w + 4 * bo + i] = bf162_bits(__hmul2(bits_bf162(pr), scl[i]));
            }
        }
    }
    return off;
}

// Shared-memory layout of one stage: codes boxes [2 halves][T*16 rows][128 B] (128-byte
// swizzle), then the activation boxes [4][m rows][256 bf16].
template <int T>
struct GemvStage {
    static constexpr int CODES = 2 * T * GEMV_BOX;
    __host__ __device__ static int bytes(int m) { return CODES + 4 * m * GEMV_XBOX * 2; }
};

// Scale groups per row a CTA stages: all of them, or at most those touched by one K part.
__host__ __device__ inline int gemv_staged_groups(int k, int group, int ksplit) {
    const int G = k / group;
    if (ksplit <= 1) return G;
    const int nch_all = ((k >> 7) + GEMV_PBLK - 1) / GEMV_PBLK;
    const int maxch = (nch_all + ksplit - 1) / ksplit;
    const int gs = (maxch * GEMV_PBLK * 128 + group - 1) / group + 1;
    return gs < G ? gs : G;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// fp32 at the same shared-memory offset as `local` in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_cluster_f32(const void* local, uint32_t rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

// Requests chunk c into stage s: the codes of the CTA's rows (one box per 128-byte half;
// `tmap` has a box of exactly nt*16 rows) and the chunk's activation columns.
template <int T>
__device__ __forceinline__ void gemv_issue_codes(uint8_t* stages, int stage_bytes, uint64_t* full,
                                                 const CUtensorMap* tmap, int c, int s, int nt, int r0, int m) {
    uint8_t* dst = stages + s * stage_bytes;
    mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * nt * GEMV_BOX + 4 * m * GEMV_XBOX * 2));
    tma_load_2d(dst, tmap, c * 256, r0, &full[s]);
    tma_load_2d(dst + T * GEMV_BOX, tmap, c * 256 + 128, r0, &full[s]);
}

template <int T>
__device__ __forceinline__ void gemv_issue_x(uint8_t* stages, int stage_bytes, uint64_t* full, const CUtensorMap* xmap,
                                             int c, int s, int m) {
    uint8_t* dst = stages + s * stage_bytes;
    for (int j = 0; j < 4; j++)
        tma_load_2d(dst + GemvStage<T>::CODES + j * m * GEMV_XBOX * 2, xmap, c * (GEMV_PBLK * 128) + j * GEMV_XBOX, 0,
                    &full[s]);
}

template <int T>
__device__ __forceinline__ void gemv_issue(uint8_t* stages, int stage_bytes, uint64_t* full, const CUtensorMap* tmap,
                                           const CUtensorMap* xmap, int c, int s, int nt, int r0, int m) {
    gemv_issue_codes<T>(stages, stage_bytes, full, tmap, c, s, nt, r0, m);
    gemv_issue_x<T>(stages, stage_bytes, full, xmap, c, s, m);
}

// Stores output element idx = BF16(sum).  With `hgate` (the FFN chain's up projection) it
// also replaces hgate[idx] (the gate projection, whose value g was loaded earlier) by
// BF16(SiLU(g) * u), u the stored BF16.
__device__ __forceinline__ void gemv_store(uint16_t* y, uint16_t* hgate, size_t idx, float sum, uint16_t g) {
    const __nv_bfloat16 bv = __float2bfloat16_rn(sum);
    const uint16_t ub = *reinterpret_cast<const uint16_t*>(&bv);
    y[idx] = ub;
    if (hgate) {
        const __nv_bfloat16 hb = __float2bfloat16_rn(silu_mul1(bf16_bits_to_f32(g), bf16_bits_to_f32(ub)));
        hgate[idx] = *reinterpret_cast<const uint16_t*>(&hb);
    }
}

template <int T>
__global__ void __launch_bounds__(GEMV_THREADS, 1)
    q2_gemv_kernel(const __grid_constant__ CUtensorMap tmap_full, const __grid_constant__ CUtensorMap tmap_less,
                   const __grid_constant__ CUtensorMap xmap, const uint16_t* __restrict__ scales,
                   uint16_t* __restrict__ y, int m, int n, int k, int group, int ntiles, int nstages, int ksplit,
                   uint16_t* hgate) {
    constexpr int TQ = T;  // tiles per warp
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = align1024(smem_raw);
    const int stage_bytes = (GemvStage<T>::bytes(m) + 1023) & ~1023;
    const int G = k / group;
    // the CTA's scales (see below), then the barriers
    uint8_t* scs = stages + nstages * stage_bytes;
    uint64_t* full =
        reinterpret_cast<uint64_t*>(scs + (((size_t)32 * T * gemv_staged_groups(k, group, ksplit) + 32 + 15) & ~size_t(15)));
    uint64_t* sfull = full + GEMV_MAX_STAGES;                                   // scales landed
    uint32_t* released = reinterpret_cast<uint32_t*>(sfull + 1);               // per stage: warps done with it
    int* issued = reinterpret_cast<int*>(released + GEMV_MAX_STAGES);          // per stage: last chunk requested

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    // row group and K part (cluster rank) of this CTA
    const int rank = ksplit > 1 ? (int)cluster_rank() : 0;
    const int rg = blockIdx.x / ksplit, ngroups = gridDim.x / ksplit;
    const int tile0 = (int)((int64_t)rg * ntiles / ngroups);
    const int nt = (int)((int64_t)(rg + 1) * ntiles / ngroups) - tile0;
    const int r0 = tile0 * 16;
    const int P = k >> 7;
    const int nch_all = (P + GEMV_PBLK - 1) / GEMV_PBLK;
    const int c_lo = rank * nch_all / ksplit;                 // this CTA's chunks: [c_lo, c_lo + nch)
    const int nch = (rank + 1) * nch_all / ksplit - c_lo;
    const int pre = nch < nstages ? nch : nstages;
    const CUtensorMap* tmap = nt == T ? &tmap_full : &tmap_less;
    const int rows = min(16 * nt, n - r0);
    const uint8_t* splane = reinterpret_cast<const uint8_t*>(scales);
    // Scales in shared memory, [row][Gs] BF16 from group g_lo on.  Whole rows (ksplit == 1):
    // bytes [s_lo, s_hi) of the plane by one bulk copy, the rest (at most 14 bytes at the end
    // of the plane) by plain loads.  A K part (ksplit > 1): its groups only, by one bulk copy
    // per row when the row pieces are 16-byte aligned (G, g_lo, Gs multiples of 8), else by
    // plain loads.
    const int g_lo = ksplit > 1 ? (int)(((int64_t)c_lo * GEMV_PBLK * 128) / group) : 0;
    const int g_hi = ksplit > 1 ? min(G, (int)(((int64_t)(c_lo + nch) * GEMV_PBLK * 128 + group - 1) / group)) : G;
    const int Gs = g_hi - g_lo;
    int64_t s_lo = 0, s_hi = 0, s_end = 0;
    if (ksplit == 1) {
        s_lo = ((int64_t)r0 * G * 2) & ~int64_t(15);
        s_end = (int64_t)(r0 + rows) * G * 2;
        s_hi = (s_end + 15) & ~int64_t(15);
        const int64_t plane16 = ((int64_t)n * G * 2) & ~int64_t(15);
        if (s_hi > plane16) s_hi = plane16;
        if (s_hi < s_lo) s_hi = s_lo;
    }
    const uint16_t* sbase = ksplit == 1 ? reinterpret_cast<const uint16_t*>(scs + ((int64_t)r0 * G * 2 - s_lo))
                                        : reinterpret_cast<const uint16_t*>(scs);
    const bool srow_bulk = ksplit > 1 && (G & 7) == 0 && (g_lo & 7) == 0 && (Gs & 7) == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; s++) {
            mbar_init(&full[s], 1);
            released[s] = 0;
            issued[s] = s < pre ? s : -1;
        }
        mbar_init(sfull, 1);
        fence_barrier_init();
        // weights first: they do not depend on the kernel launched before this one
        // (programmatic dependent launch); the activations once that kernel has finished
        for (int c = 0; c < pre; c++) gemv_issue_codes<T>(stages, stage_bytes, full, tmap, c_lo + c, c, nt, r0, m);
        if (srow_bulk) {
            mbar_arrive_expect_tx(sfull, (uint32_t)(rows * Gs * 2));
            for (int rr = 0; rr < rows; rr++)
                bulk_load(scs + (size_t)rr * Gs * 2, scales + (size_t)(r0 + rr) * G + g_lo, (uint32_t)(Gs * 2), sfull);
        } else {
            mbar_arrive_expect_tx(sfull, (uint32_t)(s_hi - s_lo));
            if (s_hi > s_lo) bulk_load(scs, splane + s_lo, (uint32_t)(s_hi - s_lo), sfull);
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        for (int c = 0; c < pre; c++) gemv_issue_x<T>(stages, stage_bytes, full, &xmap, c_lo + c, c, m);
    }
    if (ksplit == 1) {
        if (threadIdx.x == 32)  // scale bytes past the bulk copy
            for (int64_t o = s_hi; o < s_end; o += 2)
                *reinterpret_cast<uint16_t*>(scs + (o - s_lo)) = __ldg(reinterpret_cast<const uint16_t*>(splane + o));
    } else if (!srow_bulk) {  // batches of eight loads in flight per thread
        uint16_t* sd = reinterpret_cast<uint16_t*>(scs);
        const int total = rows * Gs;
        for (int base = threadIdx.x; base < total; base += 8 * (int)blockDim.x) {
            uint16_t v[8];
#pragma unroll
            for (int e = 0; e < 8; e++) {
                const int i = base + e * (int)blockDim.x;
                const int rr = i / Gs, gg = i - rr * Gs;
                v[e] = i < total ? __ldg(scales + (size_t)(r0 + rr) * G + g_lo + gg) : (uint16_t)0;
            }
#pragma unroll
            for (int e = 0; e < 8; e++) {
                const int i = base + e * (int)blockDim.x;
                if (i < total) sd[i] = v[e];
            }
        }
    }
    __syncthreads();

    // Outputs of this thread in the store loops below: o = threadIdx.x + 256 i, i < 4 (at most
    // 8 x 128 outputs per CTA).  The fused epilogue's gate values are loaded now (the kernel
    // before this one has finished: thread 0 waited for it before the barrier above), so
    // their latency hides under the main loop.
    const int per_col = nt * 16;
    uint16_t hg[4] = {0, 0, 0, 0};
    if (hgate) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int o = threadIdx.x + GEMV_THREADS * i;
            if (o < per_col * m) {
                const int j = o / per_col, rem = o - j * per_col;
                if (r0 + rem < n) hg[i] = hgate[(size_t)j * n + r0 + rem];
            }
        }
    }

    bool failed = false;
    float tot[TQ][4];
#pragma unroll
    for (int q = 0; q < TQ; q++) tot[q][0] = tot[q][1] = tot[q][2] = tot[q][3] = 0.f;
    const int pb = warp;
    const int hb = pb >> 2;                                  // which 128-byte half of the chunk
    const int jch = ((pb & 3) << 1) | (t >> 1);              // 16-byte chunk holding bytes 8t..8t+7
    const int offw = ((jch ^ g) << 4) + ((t & 1) << 3);      // swizzled: (line & 7) == g
    const uint32_t mask[3] = {0x00030003u, 0x000C000Cu, 0x00300030u};
    const uint32_t one = 0x3F803F80u;
    for (int c = 0; c < nch; c++) {
        const int s = c % nstages;
        const int p = (c_lo + c) * GEMV_PBLK + pb;
        if (!mbar_wait(&full[s], (c / nstages) & 1)) {
            failed = true;
            break;
        }
        if (p < P) {
            const uint8_t* st = stages + s * stage_bytes;
            uint32_t b[16];
            float offp = 0.f;
            if (g < m) {
                const uint8_t* xs = st + GemvStage<T>::CODES + ((pb >> 1) * m + g) * (GEMV_XBOX * 2) +
                                    (((pb & 1) << 7) + (t << 3)) * 2;
                uint4 X[4];
#pragma unroll
                for (int i = 0; i < 4; i++) X[i] = *reinterpret_cast<const uint4*>(xs + 64 * i);
                offp = build_bfrag(b, X);
            } else {
#pragma unroll
                for (int r = 0; r < 16; r++) b[r] = 0u;
            }
            // -sum((1/s + 2) x) of activation rows 2t and 2t+1 (lanes 8t.. and 8t+4.. hold them)
            offp += __shfl_xor_sync(0xffffffffu, offp, 1);
            offp += __shfl_xor_sync(0xffffffffu, offp, 2);
            const float off0 = __shfl_sync(0xffffffffu, offp, 8 * t);
            const float off1 = __shfl_sync(0xffffffffu, offp, 8 * t + 4);
            uint2 wa[TQ], wb[TQ];
            const int gi = (p << 7) / group;
#pragma unroll
            for (int q = 0; q < TQ; q++) {
                const int tau = q;
                const bool v = tau < nt;
                const uint8_t* la = st + (hb * T * 16 + tau * 16 + g) * 128 + offw;
                wa[q] = v ? *reinterpret_cast<const uint2*>(la) : make_uint2(0, 0);
                wb[q] = v ? *reinterpret_cast<const uint2*>(la + 8 * 128) : make_uint2(0, 0);
            }
            float acc[TQ][4];
#pragma unroll
            for (int q = 0; q < TQ; q++) {
                acc[q][0] = off0; acc[q][1] = off1; acc[q][2] = off0; acc[q][3] = off1;
            }
            // tiles past nt hold zero codes: their (unused) sums cost an MMA but no branch
            gemv_step<0, TQ>(acc, wa, wb, b, mask, one);
            gemv_step<1, TQ>(acc, wa, wb, b, mask, one);
            gemv_step<2, TQ>(acc, wa, wb, b, mask, one);
            gemv_step<3, TQ>(acc, wa, wb, b, mask, one);
            gemv_step<4, TQ>(acc, wa, wb, b, mask, one);
            gemv_step<5, TQ>(acc, wa, wb, b, mask, one);
            gemv_step<6, TQ>(acc, wa, wb, b, mask, one);
            gemv_step<7, TQ>(acc, wa, wb, b, mask, one);
            if (c == 0 && !mbar_wait(sfull, 0)) {
                failed = true;
                break;
            }
            // scales of rows 16q + g and 16q + g + 8 (zero for tiles past nt)
            const uint16_t* sr = sbase + g * Gs + (gi - g_lo);
#pragma unroll
            for (int q = 0; q < TQ; q++) {
                const bool v = q < nt;
                const float da = v ? bf16_bits_to_f32(sr[(16 * q) * Gs]) : 0.f;
                const float db = v ? bf16_bits_to_f32(sr[(16 * q + 8) * Gs]) : 0.f;
                tot[q][0] = fmaf(da, acc[q][0], tot[q][0]);
                tot[q][1] = fmaf(da, acc[q][1], tot[q][1]);
                tot[q][2] = fmaf(db, acc[q][2], tot[q][2]);
                tot[q][3] = fmaf(db, acc[q][3], tot[q][3]);
            }
        }
        // release the stage; the last warp to release it requests chunk c + nstages into it
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            // counts only grow: use u of stage s is complete at 8 * (u + 1) releases
            const uint32_t before = atomicAdd(&released[s], 1u);
            if (before == (uint32_t)(GEMV_CWARPS * (c / nstages + 1) - 1)) {
                const int cn = c + nstages;
                if (cn < nch) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issued[s] = cn;
                    gemv_issue<T>(stages, stage_bytes, full, tmap, &xmap, c_lo + cn, s, nt, r0, m);
                }
            }
        }
    }
    if (failed) atomicOr(&g_gemv_status, 1u);
    __syncthreads();
    if (threadIdx.x == 0) {  // wind down: every requested chunk must have landed before the CTA exits
        for (int s = 0; s < nstages; s++) {
            const int c = issued[s];
            if (c >= 0 && !mbar_wait(&full[s], (c / nstages) & 1)) atomicOr(&g_gemv_status, 1u);
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- reduction + store
    // red[pb][tau][lane*5 + e]
    float* red = reinterpret_cast<float*>(stages);
#pragma unroll
    for (int q = 0; q < TQ; q++) {
#pragma unroll
        for (int e = 0; e < 4; e++) red[(pb * T + q) * 160 + lane * 5 + e] = tot[q][e];
    }
    __syncthreads();
    float* part = red + GEMV_PBLK * T * 160;  // [m][16 T]: this CTA's sums (K parts only)
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int o = threadIdx.x + GEMV_THREADS * i;
        if (o >= per_col * m) break;
        const int j = o / per_col, rem = o - j * per_col, tau = rem >> 4, r = rem & 15;
        const int row = r0 + rem;
        if (row >= n) continue;
        const int ln = (r & 7) * 4 + (j >> 1), e = (r >> 3) * 2 + (j & 1);
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < GEMV_PBLK; w++) sum += red[(w * T + tau) * 160 + ln * 5 + e];
        if (ksplit > 1) {
            part[j * 16 * T + rem] = sum;
        } else {
            gemv_store(y, hgate, (size_t)j * n + row, sum, hg[i]);
        }
    }
    if (ksplit > 1) {
        cluster_sync_all();  // every member's partial sums are in its shared memory
        if (rank == 0) {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int o = threadIdx.x + GEMV_THREADS * i;
                if (o >= per_col * m) break;
                const int j = o / per_col, rem = o - j * per_col;
                const int row = r0 + rem;
                if (row >= n) continue;
                // all members' values requested before any is added
                float v[8];
#pragma unroll
                for (int q = 1; q < 8; q++)
                    v[q] = q < ksplit ? ld_cluster_f32(&part[j * 16 * T + rem], (uint32_t)q) : 0.f;
                float sum = part[j * 16 * T + rem];
#pragma unroll
                for (int q = 1; q < 8; q++) sum += v[q];
                gemv_store(y, hgate, (size_t)j * n + row, sum, hg[i]);
            }
        }
        cluster_sync_all();  // members keep their shared memory until the leader has read it
    }
}

template <int T>
static int launch_t(const uint8_t* codes, const CUtensorMap& xmap, const uint16_t* scales, uint16_t* y, int m,
                    int n, int k, int group, int ntiles, int ncta, int ksplit, uint16_t* hgate, cudaStream_t stream,
                    const char* who) {
    static int configured_smem[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64) dev = 63;
    const int Gst = gemv_staged_groups(k, group, ksplit);
    const size_t stage = ((size_t)GemvStage<T>::bytes(m) + 1023) & ~size_t(1023);
    const size_t fixed = 1024 + (((size_t)32 * T * Gst + 32 + 15) & ~size_t(15)) + (GEMV_MAX_STAGES * 2 + 1) * 8 + 16;
    // At most ~112 KB where two stages allow it, so the CTA of the next launch (programmatic
    // dependent launch) can share the SM and start its weight copies before this one ends.
    int nstages = GEMV_MAX_STAGES;
    while (nstages > 2 && fixed + nstages * stage > (size_t)GEMV_SMEM_SHARE) nstages--;
    const size_t smem = fixed + nstages * stage;
    if (smem > (size_t)GEMV_SMEM_LIMIT) return fail(BQ_ERR_INVALID, "%s: shape needs too much shared memory", who);
    if ((size_t)configured_smem[dev] < smem) {
        if (cudaFuncSetAttribute(q2_gemv_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: cannot reserve %zu bytes of shared memory", who, smem);
        configured_smem[dev] = (int)smem;
    }
    // codes boxes of exactly T and T-1 tiles of rows (CTAs get one or the other)
    CUtensorMap map_full, map_less;
    int st = make_tmap_2d_u8(&map_full, codes, k / 4, n, k / 4, 128, 16 * T, true, who);
    if (st) return st;
    if ((st = make_tmap_2d_u8(&map_less, codes, k / 4, n, k / 4, 128, T > 1 ? 16 * (T - 1) : 16, true, who))) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ncta);
    cfg.blockDim = dim3(GEMV_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;  // the K parts of a row range
    attr[1].val.clusterDim.x = (unsigned)ksplit;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ksplit > 1 ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, q2_gemv_kernel<T>, map_full, map_less, xmap, scales, y, m, n, k, group, ntiles,
                           nstages, ksplit, hgate) != cudaSuccess)
        return check_launch(who);
    return BQ_OK;
}

// The warp-MMA GEMV: CTA c takes a contiguous range of T or T - 1 row tiles.
static int launch_q2_gemv_mma(const uint16_t* x, const bq_q2_weight* w, uint16_t* y, uint32_t m, uint16_t* hgate,
                              bool allow_split, cudaStream_t stream, const char* who) {
    const int G = (int)(w->k / w->group);
    const int ntiles = (int)((w->n + 15) / 16);
    int tmax = GEMV_MAX_T;
    while (tmax > 1 && (size_t)32 * tmax * G > 96 * 1024) tmax--;
    if ((size_t)32 * tmax * G > 96 * 1024)
        return fail(BQ_ERR_INVALID, "%s: k/group = %d groups per row is too many", who, G);
    const int sms = sm_count();
    int ncta = ntiles < sms ? ntiles : sms;
    int T = (ntiles + ncta - 1) / ncta;
    if (T > tmax) {
        ncta = (ntiles + tmax - 1) / tmax;
        T = (ntiles + ncta - 1) / ncta;  // every CTA then gets T or T - 1 tiles
    }
    // Too few rows for about seven tiles on every SM, but many chunks: split K over a cluster
    // of S CTAs per row range (S <= 8, at least three chunks per part).
    int ksplit = 1;
    const int T0 = tmax < 7 ? tmax : 7;
    const int nch_all = (int)(((w->k >> 7) + GEMV_PBLK - 1) / GEMV_PBLK);
    if (allow_split && ntiles < sms * (T0 - 1)) {
        const int ng = (ntiles + T0 - 1) / T0;
        int S = sms / ng;
        if (S > 8) S = 8;
        if (S > nch_all / 3) S = nch_all / 3;
        if (S >= 2) {
            ksplit = S;
            ncta = ng * S;
            T = (ntiles + ng - 1) / ng;
        }
    }
    const uint8_t* codes = (const uint8_t*)w->data;
    const uint16_t* scales = (const uint16_t*)(codes + (size_t)w->n * (w->k / 4));
    CUtensorMap xmap;
    // activations x [m][k] as 16-bit elements, boxes of 256 columns x m rows
    int st = make_tmap_2d(&xmap, x, 2, w->k, m, (uint64_t)w->k * 2, GEMV_XBOX, m, false, who);
    if (st) return st;
    const int mm = (int)m, n = (int)w->n, k = (int)w->k, gr = (int)w->group;
    switch (T) {
        case 1: st = launch_t<1>(codes, xmap, scales, y, mm, n, k, gr, ntiles, ncta, ksplit, hgate, stream, who); break;
        case 2: st = launch_t<2>(codes, xmap, scales, y, mm, n, k, gr, ntiles, ncta, ksplit, hgate, stream, who); break;
        case 3: st = launch_t<3>(codes, xmap, scales, y, mm, n, k, gr, ntiles, ncta, ksplit, hgate, stream, who); break;
        case 4: st = launch_t<4>(codes, xmap, scales, y, mm, n, k, gr, ntiles, ncta, ksplit, hgate, stream, who); break;
        case 5: st = launch_t<5>(codes, xmap, scales, y, mm, n, k, gr, ntiles, ncta, ksplit, hgate, stream, who); break;
        case 6: st = launch_t<6>(codes, xmap, scales, y, mm, n, k, gr, ntiles, ncta, ksplit, hgate, stream, who); break;
        case 7: st = launch_t<7>(codes, xmap, scales, y, mm, n, k, gr, ntiles, ncta, ksplit, hgate, stream, who); break;
        case 8: st = launch_t<8>(codes, xmap, scales, y, mm, n, k, gr, ntiles, ncta, ksplit, hgate, stream, who); break;
        default: return fail(BQ_ERR_INVALID, "%s: internal tile count %d", who, T);
    }
    if (st) return st;
    return check_launch(who);
}

// Launches the GEMV for an already validated weight.  With `hgate` (an [m][n] BF16 buffer
// holding the gate projection) the epilogue also turns hgate into BF16(SiLU(hgate) * y).
// `allow_split` permits the cluster K split.
int launch_q2_gemv(const uint16_t* x, const bq_q2_weight* w, uint16_t* y, uint32_t m, cudaStream_t stream,
                   const char* who, uint16_t* hgate = nullptr, bool allow_split = true) {
    if (m == 0 || w->n == 0) return ok();
    if (w->k == 0) {
        if (cudaMemsetAsync(y, 0, (size_t)m * w->n * 2, stream) != cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: memset failed", who);
        return ok();
    }
    if (gemv_hm_supported(w, m)) return launch_q2_gemv_hm(x, w, y, m, hgate, stream, who);
    return launch_q2_gemv_mma(x, w, y, m, hgate, allow_split, stream, who);
}

static int check_gemv_args(const uint16_t* x, const bq_q2_weight* w, const uint16_t* y, uint32_t m, const char* who) {
    int st = check_q2(w, who);
    if (st) return st;
    if (m < 1 || m > 8) return fail(BQ_ERR_INVALID, "%s: m = %u, must be 1..8", who, m);
    if (w->n >= (1u << 30) || (uint64_t)m * w->k >= (1ull << 31))
        return fail(BQ_ERR_INVALID, "%s: shape too large", who);
    if (w->n == 0) return BQ_OK;
    if (!y || !aligned16(y)) return fail(BQ_ERR_INVALID, "%s: y NULL or not 16-byte aligned", who);
    if (w->k > 0 && (!x || !aligned16(x))) return fail(BQ_ERR_INVALID, "%s: x NULL or not 16-byte aligned", who);
    return BQ_OK;
}

}  // namespace bq8

using namespace bq8;

extern "C" {

int q2_gemv(const uint16_t* x, const bq_q2_weight* w, uint16_t* y, bq_stream_t stream) {
    int st = check_gemv_args(x, w, y, 1, "q2_gemv");
    if (st) return st;
    return launch_q2_gemv(x, w, y, 1, (cudaStream_t)stream, "q2_gemv");
}

int q2_gemv_batchm(const uint16_t* x, const bq_q2_weight* w, uint16_t* y, uint32_t m, bq_stream_t stream) {
    if (m == 0) return ok();
    int st = check_gemv_args(x, w, y, m, "q2_gemv_batchm");
    if (st) return st;
    return launch_q2_gemv(x, w, y, m, (cudaStream_t)stream, "q2_gemv_batchm");
}

int ffn_q2_km(const uint16_t* x, const bq_q2_weight* gate, const bq_q2_weight* up, const bq_q2_weight* down,
              uint16_t* gate_scratch, uint16_t* up_scratch, uint16_t* out, uint32_t m, bq_stream_t stream) {
    const char* who = "ffn_q2_km";
    if (m == 0) return ok();
    int st;
    if ((st = check_gemv_args(x, gate, gate_scratch, m, who))) return st;
    if ((st = check_gemv_args(x, up, up_scratch, m, who))) return st;
    if ((st = check_gemv_args(gate_scratch, down, out, m, who))) return st;
    if (gate->n != up->n || gate->k != up->k || down->k != gate->n || down->n != gate->k)
        return fail(BQ_ERR_INVALID,
                    "%s: shapes must be gate/up [inter, hidden], down [hidden, inter] (gate %ux%u up %ux%u down %ux%u)",
                    who, gate->n, gate->k, up->n, up->k, down->n, down->k);
    const size_t inter_bytes = (size_t)m * gate->n * 2;
    const uintptr_t gs = reinterpret_cast<uintptr_t>(gate_scratch), us = reinterpret_cast<uintptr_t>(up_scratch);
    if (gs < us + inter_bytes && us < gs + inter_bytes)
        return fail(BQ_ERR_INVALID, "%s: gate_scratch and up_scratch overlap", who);
    cudaStream_t s = (cudaStream_t)stream;
    if (gate->n > 0 && gate->k > 0 && gate->group == up->group && gemv_hm_dual_supported(gate, m)) {
        // one launch streams the gate and up weights together: u into up_scratch and
        // h = SiLU(g) * u into gate_scratch, the same arithmetic as the two launches below
        if ((st = launch_q2_gemv_hm_dual(x, gate, up, gate_scratch, up_scratch, m, s, who))) return st;
    } else {
        if ((st = launch_q2_gemv(x, gate, gate_scratch, m, s, who))) return st;
        // the up projection's epilogue also forms h = SiLU(g) * u in gate_scratch
        if ((st = launch_q2_gemv(x, up, up_scratch, m, s, who, gate_scratch))) return st;
    }
    // The down projection: the FP16 warp-MMA kernel where its activation table fits one SM
    // (k = 17408: m <= 4), without the cluster K split of the older kernel (right after the
    // gate/up launch a cluster launch loses its early start: chain 42.8 against 36.7 us at
    // m = 2); where the table does not fit, the older kernel with its cluster K split (chain
    // 50.2 against 57.2 us unsplit at m = 8).
    if (gemv_hm_supported(down, m)) return launch_q2_gemv(gate_scratch, down, out, m, s, who, nullptr, false);
    return launch_q2_gemv_mma(gate_scratch, down, out, m, nullptr, true, s, who);
}

}  // extern "C"
