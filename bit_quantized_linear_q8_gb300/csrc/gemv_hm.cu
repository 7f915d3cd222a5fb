// gemv_hm.cu -- Q2_0 decode GEMV for 1..8 activation rows on the FP16 warp tensor cores.
//
// Source: init_q2.rs `set_packed_q2_qkvz` (decode runs `q2_0_gemv_vec`) and
// dense_ffn_decode_batch.rs `forward_km_q2` (`q2_0_gemv_vec_batchm` for gate/up/down).
//
// Design (GB300).  The packed weight (2.125 bits per weight) is the only large stream.  On
// sm_103a the legacy FP16 warp MMA (m16n8k16) and the integer / FP16x2 instructions that
// unpack its operands issue from the same warp schedulers, so the kernel is built to keep
// every scheduler issuing that work back to back:
//
//  * Weights (A operand): one LOP3 per pair of codes ORs the code at bit position 2i of its
//    byte into the mantissa of the FP16 value 1024 in each 16-bit half (1024 + c 4^i; the
//    four positions of a byte's low half need no shift, the high bytes one shift per 32-bit
//    word), and one FP16 add of -(1024 + 2 4^i) turns that into (c - 2) 4^i, exactly.  A zero
//    weight thus gives an exactly zero product: no large activation enters an MMA's sums
//    unless its weight is nonzero (an offset form such as c X - 2 X loses the small products
//    next to a large one inside the tensor core's sum).
//  * Activations (B operand): x is turned once per CTA into an FP16 table in fragment order,
//    X 4^-i with X = x 2^s, one power of two 2^s per activation row (its maximum maps to
//    [2^14, 2^15)) and 4^-i for the code position i of the column, so that A B = (c - 2) X.
//    Every x within 16 binades of its row's maximum is exact in the table; smaller ones are
//    off by at most 2^-25 of the maximum.  Each 128-column block's fp32 sum of (c - 2) X is
//    scaled by its BF16 d; the result is multiplied by 2^-s.
//  * Work split: the n rows form 16-row tiles; CTA c takes tiles [c T / C, (c + 1) T / C), a
//    contiguous byte range of the weight, so every SM streams the same bytes to within a tile.
//  * Staging: the CTA's tiles form row groups of up to eight; a chunk is one row group x 1024
//    columns (2048 for few long rows per CTA, see hm_plan), one TMA box of 128 bytes x 16
//    tiles-per-group rows per 512-column half, with
//    the 128-byte swizzle so that the eight rows a warp reads at once fall on distinct banks.
//    The boxes are tall on purpose: a TMA request costs an SM a roughly fixed time, so boxes
//    of 2 KB stream at a fifth of the rate of 16 KB ones.  Where K is a multiple of 512 the
//    weight is also described as a 3-D tensor (128-byte column block, row, block) so that
//    one request brings all halves of a chunk.  A producer warp requests the
//    chunks into a ring (mbarrier "full" per stage, transaction bytes) and refills a stage
//    once every consumer warp has arrived on its "empty" barrier; the ring usually holds the
//    CTA's whole slice.  The first chunk and the CTA's scales (one bulk copy) are requested at
//    once, the rest as soon as the activations have arrived (a deeper early prefetch queues
//    the activation loads, which every warp waits for, behind weight bytes).
//    The tensor maps come from a process-wide cache.  Every wait is bounded.
//  * Compute: sixteen consumer warps.  Warp w takes the tile pair w / P' of every row group
//    (two independent MMA chains) and pack blocks w % P', w % P' + P', ... of every chunk
//    (P' warps share a pair), so the B fragments of a block are loaded once for two tiles and
//    the running sums stay in registers over the whole K range.  When a warp takes two or four
//    blocks of a full chunk, a second instantiation runs them as an unrolled loop, so that the
//    next block's shared-memory loads issue under the current block's MMAs.  The launch
//    constants (shared-memory layout, the reciprocals that replace divisions) are computed
//    on the host.  At the end the P' partial
//    sums of each row meet in shared memory and are added in a fixed order (results do not
//    depend on timing), then stored as BF16 (with the FFN's SiLU*mul when asked).
#include <type_traits>

#include "common.cuh"

namespace bq8 {

constexpr int HM_CWARPS = 16;                     // consumer warps
constexpr int HM_MAX_PARTS = 8;                   // warps sharing a tile pair (each takes 1/parts of the blocks)
constexpr int HM_THREADS = (HM_CWARPS + 1) * 32;  // + the producer warp
constexpr int HM_MAX_STAGES = 8;
constexpr int HM_TG = 2;                          // tiles per MMA step (two chains per warp)
constexpr int HM_MAX_TGB = 8;                     // tiles per row group (one box height)
constexpr int HM_BOX = 16 * 128;                  // one box: 16 rows x 128 bytes
constexpr int HM_SMEM_LIMIT = 225 * 1024;
// Chunks requested before the activations have arrived: the SM's memory queue serves requests
// roughly in order, so a deep weight prefetch would hold back the activation loads that every
// warp waits for, while the weight stream has time to spare behind the table build.
constexpr int HM_EARLY_CHUNKS = 1;

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
    const uint8_t* codes2;   // dual form: the up weight (same shape)
    const uint16_t* scales2;
    const uint16_t* x;       // [m][k] BF16
    uint16_t* y;             // [m][n] BF16 (dual form: h = BF16(SiLU(g) * u))
    uint16_t* y2;            // dual form: [m][n] BF16 u
    uint16_t* hgate;         // optional [m][n] BF16: replaced by BF16(SiLU(hgate) * y)
    int n, k, group;
    int tmax;                // tiles of the largest CTA
    int tgb;                 // tiles per row group: each TMA box is 128 bytes x 16 tgb rows
    int nstages;
    // launch constants from the host, so that the CTA's prologue does no division
    uint32_t ring, btab, scal, scal_w, slot, misc;  // shared-memory offsets (HmLayout)
    int G;                   // scale groups per row, k / group
    int lw;                  // log2 of the warps per tile pair (hm_parts)
    uint32_t kmag;           // ceil(2^32 / (k / 8)): a vector's activation row by a multiply-high
    uint32_t cmag;           // ceil(2^32 / CTAs): the CTA's tile range by a multiply-high
    uint32_t gmag;           // ceil(2^32 / tgb): the CTA's row groups by a multiply-high
    int chunk3d;             // 1: the maps are 3-D chunk maps, one request per weight and chunk
    int hpc;                 // 512-column halves per chunk (the kernel's HPC; host side)
};

// x / d by a multiply-high with mag = ceil(2^32 / d) computed in 32 bits, which wraps to 0
// exactly when d = 1.
__device__ __forceinline__ uint32_t hm_div(uint32_t x, uint32_t mag) { return mag ? __umulhi(x, mag) : x; }

// Warps sharing a tile pair (each takes 1/parts of a chunk's pack blocks), from the tile
// pairs per row group: tgb / 2 rounded up, or tgb in the dual (nw = 2) form.
__host__ __device__ inline int hm_parts(int tgb, int nw) {
    const int np = nw == 2 ? tgb : (tgb + 1) >> 1;
    return np <= 2 ? HM_MAX_PARTS : np <= 4 ? 4 : 2;
}

// Shared-memory carve-up, identical on host and device (offsets from a 1024-aligned base);
// nw = 2 for the dual (gate and up) form.
struct HmLayout {
    size_t ring, btab, scal, scal_w, slot, misc, total;
    __host__ __device__ HmLayout(int m, int k, int group, int tgb, int nstages, int tmax, int nw, int hpc) {
        const size_t P = (size_t)k / 128, G = (size_t)k / group;
        ring = 0;                                                       // [stage][nw][hpc halves][16 tgb rows][128 B]
        btab = ring + (size_t)nstages * nw * hpc * tgb * HM_BOX;        // [P][4 quads][m][4 lanes][16 B]
        scal = btab + P * (size_t)m * 256;                              // [nw] CTA's scale rows (+ alignment)
        scal_w = ((size_t)tmax * 16 * G * 2 + 32 + 15) & ~size_t(15);
        slot = scal + nw * scal_w;                                      // [parts][nw][16 tmax rows][m] fp32
        misc = slot + (size_t)hm_parts(tgb, nw) * nw * 16 * tmax * m * 4;  // barriers, row maxima, row scales
        total = misc + 2 * HM_MAX_STAGES * 8 + 16 + 8 * 4 * 2 + 1024;   // + alignment
    }
};

// Shared-memory loads by 32-bit shared address (volatile: never moved across the barrier
// waits that publish the data).
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ float lds_bf16(uint32_t a) {  // one BF16 value as fp32
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return __uint_as_float((uint32_t)v << 16);
}

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

__device__ __forceinline__ uint32_t hadd2_bits(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// (c - 2) 4^I for the two codes at bit position I of the bytes picked by `w` (low bytes, or
// high bytes after a shift by 8), as an FP16 pair: (1024 + c 4^I) - (1024 + 2 4^I).
template <int I>
__device__ __forceinline__ uint32_t codes_f16(uint32_t w) {
    constexpr uint32_t msk = 0x00030003u << (2 * I);
    constexpr uint32_t neg = I == 0 ? 0xE402E402u : I == 1 ? 0xE408E408u : I == 2 ? 0xE420E420u : 0xE480E480u;
    return hadd2_bits(and_or(w, msk, 0x64006400u), neg);
}

// The 8 MMAs of one pack block for the first NT tiles (independent chains): lane (g, t)
// holds code words 2t, 2t + 1 of rows g (w) and g + 8 (w8) of each tile; MMA 4s + i takes
// bit position i of word 2t + s, low bytes as fragment columns (k, k + 1) and high bytes as
// (k + 8, k + 9); b[2 (4s + i)], b[2 (4s + i) + 1] are the lane's B fragment of that MMA.
template <int NT>
__device__ __forceinline__ void hm_tiles(float (&ac)[HM_TG][4], const uint2 (&w)[HM_TG], const uint2 (&w8)[HM_TG],
                                         const uint32_t (&b)[16]) {
    uint32_t hw[NT][2], hw8[NT][2];
#pragma unroll
    for (int q = 0; q < NT; q++) {
        hw[q][0] = w[q].x >> 8;
        hw[q][1] = w[q].y >> 8;
        hw8[q][0] = w8[q].x >> 8;
        hw8[q][1] = w8[q].y >> 8;
    }
#define HM_POS(S, I)                                                                                 \
    _Pragma("unroll") for (int q = 0; q < NT; q++) {                                                \
        const uint32_t lo = (S) ? w[q].y : w[q].x, lo8 = (S) ? w8[q].y : w8[q].x;                   \
        mma_f16_16816(ac[q], codes_f16<I>(lo), codes_f16<I>(lo8), codes_f16<I>(hw[q][S]),           \
                      codes_f16<I>(hw8[q][S]), b[2 * (4 * (S) + (I))], b[2 * (4 * (S) + (I)) + 1]); \
    }
    HM_POS(0, 0)
    HM_POS(0, 1)
    HM_POS(0, 2)
    HM_POS(0, 3)
    HM_POS(1, 0)
    HM_POS(1, 1)
    HM_POS(1, 2)
    HM_POS(1, 3)
#undef HM_POS
}

// Where a chunk sits: its stage and the stage's phase parity, its row group and column
// step.  Advanced by counting (no division in the loop).
struct HmCursor {
    int s, gi, kc;
    uint32_t ph;
    __device__ __forceinline__ void next(int nst, int nkc) {
        if (++kc == nkc) {
            kc = 0;
            gi++;
        }
        if (++s == nst) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// One block step of a warp: the 8 MMAs of pack block pb for the first NT tiles of its pair.
// c: the lane's code bytes of row g of the first tile (row g + 8 is 1024 bytes on, the
// second tile q1_off on); b: the lane's 64 bytes of B fragments (quads M * 64 bytes apart);
// s: the scale of row g of the first tile (row g + 8 at g8, the second tile at q1_s).
template <int NT, int M>
__device__ __forceinline__ void hm_block(float (&tot)[HM_TG][4], uint32_t c, uint32_t q1_off, uint32_t b, uint32_t s,
                                         uint32_t q1_s, uint32_t g8) {
    uint2 w[HM_TG], w8[HM_TG];
    w[0] = lds64(c);
    w8[0] = lds64(c + 8 * 128);
    w[1] = w8[1] = make_uint2(0u, 0u);
    if (NT == 2) {
        w[1] = lds64(c + q1_off);
        w8[1] = lds64(c + q1_off + 8 * 128);
    }
    uint32_t bf[16];
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const uint4 v = lds128(b + (uint32_t)e * (64u * M));
        bf[4 * e] = v.x;
        bf[4 * e + 1] = v.y;
        bf[4 * e + 2] = v.z;
        bf[4 * e + 3] = v.w;
    }
    float ac[HM_TG][4];
#pragma unroll
    for (int q = 0; q < HM_TG; q++) ac[q][0] = ac[q][1] = ac[q][2] = ac[q][3] = 0.f;
    hm_tiles<NT>(ac, w, w8, bf);
#pragma unroll
    for (int q = 0; q < NT; q++) {
        const float d0 = lds_bf16(s + q * q1_s), d8 = lds_bf16(s + q * q1_s + g8);
        tot[q][0] = fmaf(d0, ac[q][0], tot[q][0]);
        tot[q][1] = fmaf(d0, ac[q][1], tot[q][1]);
        tot[q][2] = fmaf(d8, ac[q][2], tot[q][2]);
        tot[q][3] = fmaf(d8, ac[q][3], tot[q][3]);
    }
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(HM_CWARPS * 32) : "memory");
}

// DUAL: one launch over the gate and up weights of an FFN (same shape), the warp's tile pair
// being gate tile t and up tile t; the store forms u and h = SiLU(g) * u.
// UNR: full chunks run a loop of constant trip count (two or four blocks a warp), a separate
// instantiation so that the other launches keep their own register allocation.
// HPC: 512-column halves per chunk, 2 (1024 columns) or 4 (2048 columns).
template <int M, bool DUAL, bool UNR, int HPC>
__global__ void __launch_bounds__(HM_THREADS, 1)
    q2_gemv_hm_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap2,
                      const HmParams p) {
    constexpr int NW = DUAL ? 2 : 1;  // weights streamed
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);  // the swizzled boxes need 1024-byte alignment
    const int n = p.n, k = p.k;
    const HmParams& L = p;  // the shared-memory offsets
    uint8_t* ring = smem + L.ring;
    uint8_t* btab = smem + L.btab;
    uint8_t* scal = smem + L.scal;
    float* slot = reinterpret_cast<float*>(smem + L.slot);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.misc);
    uint64_t* empty = full + HM_MAX_STAGES;
    uint64_t* sbar = empty + HM_MAX_STAGES;
    uint64_t* xready = sbar + 1;  // the activations have arrived (the first table pass is done)
    uint32_t* rowmax = reinterpret_cast<uint32_t*>(xready + 1);
    float* rowback = reinterpret_cast<float*>(rowmax + 8);  // 2^-s per activation row

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ntiles = (n + 15) >> 4;
    // tile range [c T / C, (c + 1) T / C) by multiply-highs (exact: the host keeps T C C below
    // 2^32, so c T (ceil(2^32 / C) C - 2^32) < 2^32)
    const int t0 = (int)hm_div(blockIdx.x * (uint32_t)ntiles, p.cmag);
    const int TC = (int)hm_div((blockIdx.x + 1) * (uint32_t)ntiles, p.cmag) - t0;  // the CTA's tiles
    const int r0 = 16 * t0;
    const int R = min(16 * TC, n - r0);  // the CTA's rows
    const int P = k >> 7, G = p.G;
    const int kb = k >> 2;  // code bytes per row
    const int NST = p.nstages, TGB = p.tgb;
    const int ngrp = (int)hm_div((uint32_t)(TC + TGB - 1), p.gmag);  // row groups
    constexpr int cbs = HPC == 4 ? 4 : 3;           // log2 pack blocks per chunk
    const int nkc = (P + (1 << cbs) - 1) >> cbs;    // chunks per row group
    const int nch = ngrp * nkc;
    const uint32_t box_bytes = (uint32_t)TGB * HM_BOX;
    const uint32_t stage_bytes = NW * HPC * box_bytes;  // [weight][half][box]

    // the CTA's scales: bytes [s_lo, s_hi) of the plane by one bulk copy, the rest (at most
    // 14 bytes at the end of the plane) by plain loads
    const uint8_t* splane = reinterpret_cast<const uint8_t*>(p.scales);
    const int64_t s_lo = ((int64_t)r0 * G * 2) & ~int64_t(15);
    const int64_t s_end = (int64_t)(r0 + R) * G * 2;
    int64_t s_hi = (s_end + 15) & ~int64_t(15);
    const int64_t plane16 = ((int64_t)n * G * 2) & ~int64_t(15);
    if (s_hi > plane16) s_hi = plane16;
    if (s_hi < s_lo) s_hi = s_lo;

    if (tid < NST) {
        mbar_init(&full[tid], 1);
        mbar_init(&empty[tid], HM_CWARPS);
        fence_barrier_init();
    }
    if (tid == 64) {
        mbar_init(sbar, 1);
        mbar_init(xready, 1);
        fence_barrier_init();
    }
    if (tid >= 96 && tid < 104) rowmax[tid - 96] = 0u;
    if (tid == 32)
        for (int w = 0; w < NW; w++) {
            const uint8_t* sp = w ? reinterpret_cast<const uint8_t*>(p.scales2) : splane;
            for (int64_t o = s_hi; o < s_end; o += 2)
                *reinterpret_cast<uint16_t*>(scal + w * L.scal_w + (o - s_lo)) =
                    __ldg(reinterpret_cast<const uint16_t*>(sp + o));
        }
    __syncthreads();  // the last barrier all 288 threads take

    if (warp == HM_CWARPS) {
        // ---- producer: weights need nothing from the previous kernel, so it starts at once
        if (lane == 0) {
            mbar_arrive_expect_tx(sbar, (uint32_t)(NW * (s_hi - s_lo)));
            if (s_hi > s_lo) {
                bulk_load(scal, splane + s_lo, (uint32_t)(s_hi - s_lo), sbar);
                if (DUAL)
                    bulk_load(scal + L.scal_w, reinterpret_cast<const uint8_t*>(p.scales2) + s_lo,
                              (uint32_t)(s_hi - s_lo), sbar);
            }
            bool ok = true;
            int nis = 0;  // chunks requested
            HmCursor cur = {0, 0, 0, 0u};
            for (int c = 0; c < nch; c++) {
                // the rest of the weight waits until the activations have arrived
                if (c == HM_EARLY_CHUNKS && !mbar_wait_suspend(xready, 0)) {
                    ok = false;
                    break;
                }
                // stage cur.s is free once every consumer released its previous chunk
                if (c >= NST && !mbar_wait_suspend(&empty[cur.s], cur.ph ^ 1u)) {
                    ok = false;
                    break;
                }
                uint8_t* dst = ring + (size_t)cur.s * stage_bytes;
                if (p.chunk3d) {
                    // one request per weight: the chunk's HPC 512-column halves (128-byte column
                    // blocks HPC kc ..) of 16 TGB rows, the layout of the 2-D boxes below (blocks
                    // past the row's end arrive as zeros and are never read)
                    mbar_arrive_expect_tx(&full[cur.s], (uint32_t)(NW * HPC) * box_bytes);
                    for (int w = 0; w < NW; w++)
                        tma_load_3d(dst + (size_t)(w * HPC) * box_bytes, w ? &tmap2 : &tmap, 0,
                                    r0 + 16 * cur.gi * TGB, HPC * cur.kc, &full[cur.s]);
                } else {
                    // one box of 128 bytes x 16 TGB rows per 512-column half that starts inside the row
                    int nh = 0;
                    while (nh < HPC && (cur.kc * HPC + nh) * 128 < kb) nh++;
                    mbar_arrive_expect_tx(&full[cur.s], (uint32_t)(NW * nh) * box_bytes);
                    for (int w = 0; w < NW; w++)
                        for (int h = 0; h < nh; h++)
                            tma_load_2d(dst + (size_t)(w * HPC + h) * box_bytes, w ? &tmap2 : &tmap,
                                        (cur.kc * HPC + h) * 128, r0 + 16 * cur.gi * TGB, &full[cur.s]);
                }
                nis++;
                if (c == (NST - 1 > HM_EARLY_CHUNKS ? NST - 1 : HM_EARLY_CHUNKS) && nch > NST) {
                    // the ring is full: the CTA's later row groups into L2, 64 KB per request
                    const size_t total = (size_t)R * kb;
                    for (int w = 0; w < NW; w++) {
                        const uint8_t* a = (w ? p.codes2 : p.codes) + (size_t)r0 * kb;
                        for (size_t o = (size_t)(NST / nkc) * TGB * 16 * kb; o < total; o += 65536) {
                            const uint32_t bytes = (uint32_t)(total - o < 65536 ? total - o : 65536);
                            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a + o), "r"(bytes) : "memory");
                        }
                    }
                }
                cur.next(NST, nkc);
            }
            if (!ok) atomicOr(&g_hm_status, 1u);
            // wind down: the last copy requested into each stage must land before the CTA exits
            // (the consumers wait for every one of them, unless one of their waits gave up)
            for (int c = nis > NST ? nis - NST : 0; c < nis; c++) {
                const int s = c % NST;
                if (!mbar_wait_suspend(&full[s], (uint32_t)(c / NST) & 1u)) atomicOr(&g_hm_status, 1u);
            }
        }
        return;
    }

    // ---- consumers
    const int g = lane >> 2, t = lane & 3;
    pdl_wait();
    pdl_launch_dependents();

    // activations: all M rows at once.  Pass 1 takes each row's maximum |x| (per thread and
    // row in registers, then one warp reduction per row); pass 2 writes the FP16 fragment table,
    // from registers when every vector fitted in one load batch, else reloading.  A vector's
    // row v / kv is a multiply-high by ceil(2^32 / kv): exact while v (ceil(2^32 / kv) kv -
    // 2^32) < 2^32, i.e. for every v < 8 kv when kv < 23170 (the host keeps k below that).
    // vectors of 8 values per thread and batch; the long-row (HPC = 4) form holds 2 * 17408
    // values in one batch at M = 2, and the single-weight form at M >= 7 holds M * 5120, so that
    // they are loaded once (m = 8, k = 5120: 15.9 -> 14.9 us; at M = 3 a batch of 13 vectors
    // measured slower than two batches of 8, and the dual form at M = 8 did not gain)
    constexpr int XV = HPC == 4 && M == 2 ? 9 : (HPC == 2 && M >= 7 && !DUAL ? 10 : 8);
    constexpr int NCT = HM_CWARPS * 32;
    const int kv = k >> 3;     // 8-value vectors per row
    const int tv = M * kv;     // vectors of x
    const uint32_t kmag = p.kmag;
    auto row_of = [&](int v) { return (int)__umulhi((uint32_t)v, kmag); };
    const uint4* xv = reinterpret_cast<const uint4*>(p.x);
    uint4 q[XV];
    float rmx[M];
#pragma unroll
    for (int jj = 0; jj < M; jj++) rmx[jj] = 0.f;
    for (int v0 = 0; v0 < tv; v0 += XV * NCT) {
#pragma unroll
        for (int e = 0; e < XV; e++) {
            const int v = v0 + e * NCT + tid;
            q[e] = v < tv ? __ldg(xv + v) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int e = 0; e < XV; e++) {
            const int v = v0 + e * NCT + tid;
            if (v >= tv) continue;
            const uint32_t u[4] = {q[e].x, q[e].y, q[e].z, q[e].w};
            float mx = 0.f;
#pragma unroll
            for (int h = 0; h < 4; h++)
                mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(u[h] << 16)), fabsf(__uint_as_float(u[h] & 0xFFFF0000u))));
            const int j = row_of(v);
#pragma unroll
            for (int jj = 0; jj < M; jj++) rmx[jj] = j == jj ? fmaxf(rmx[jj], mx) : rmx[jj];
        }
    }
#pragma unroll
    for (int jj = 0; jj < M; jj++) {
        float r = rmx[jj];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) r = fmaxf(r, __shfl_xor_sync(0xffffffffu, r, o));
        if (lane == 0 && r > 0.f) atomicMax(&rowmax[jj], __float_as_uint(r));
    }
    consumer_sync();
    if (tid == 0) mbar_arrive(xready);
    if (tid < M) {
        const uint32_t mb = rowmax[tid];
        int sh = mb ? 14 - (int)((mb >> 23) & 0xFF) + 127 : 0;
        sh = max(-113, min(sh, 120));
        rowback[tid] = __int_as_float((127 - sh) << 23);
    }
    for (int v0 = 0; v0 < tv; v0 += XV * NCT) {
        if (tv > XV * NCT) {  // more than one batch: reload this batch's vectors
#pragma unroll
            for (int e = 0; e < XV; e++) {
                const int v = v0 + e * NCT + tid;
                q[e] = v < tv ? __ldg(xv + v) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int e = 0; e < XV; e++) {
            const int v = v0 + e * NCT + tid;
            if (v >= tv) continue;
            const int j = row_of(v), col = (v - j * kv) << 3;
            const int pb = col >> 7, i = (col >> 5) & 3, tt = (col >> 3) & 3;
            // 2^s 4^-i, 2^s putting the row maximum in [2^14, 2^15) (capped where 2^s and 2^-s
            // stay normal): one exact power-of-two product per value
            const uint32_t mb = rowmax[j];
            int sh = mb ? 14 - (int)((mb >> 23) & 0xFF) + 127 : 0;
            sh = max(-113, min(sh, 120));
            const float sc = __int_as_float((127 + sh - 2 * i) << 23);
            const uint32_t u[4] = {q[e].x, q[e].y, q[e].z, q[e].w};
            float X[8];
#pragma unroll
            for (int h = 0; h < 4; h++) {
                X[2 * h] = __uint_as_float(u[h] << 16) * sc;
                X[2 * h + 1] = __uint_as_float(u[h] & 0xFFFF0000u) * sc;
            }
#pragma unroll
            for (int s = 0; s < 2; s++) {
                const float* e4 = X + 4 * s;
                // lane (j, tt)'s fragment for MMA 4s + i (columns 0, 2 then 1, 3 of the four),
                // in quad (4s + i) / 2 at half (4s + i) % 2
                const uint2 ent = make_uint2(f16x2_bits(e4[0], e4[2]), f16x2_bits(e4[1], e4[3]));
                const int quad = 2 * s + (i >> 1);
                *reinterpret_cast<uint2*>(btab + ((((size_t)pb * 4 + quad) * M + j) * 4 + tt) * 16 + (i & 1) * 8) = ent;
            }
        }
    }
    consumer_sync();

    // ---- main loop.  Warp w works on tile pair w / wpp of every row group (two MMA chains:
    // tiles 2 pair and 2 pair + 1, or in the dual form gate tile pair and up tile pair) and on
    // pack blocks part, part + wpp, ... (part = w % wpp) of every chunk, so its running sums
    // stay in registers over the whole K range.  A wait that gives up marks the status and
    // the remaining waits are skipped; the loop still runs to its end.
    bool failed = !warp_wait(sbar, 0);
    const int gsh = __ffs(p.group) - 1 - 7;  // group = 128 << gsh
    const uint16_t* srow = reinterpret_cast<const uint16_t*>(scal + ((int64_t)r0 * G * 2 - s_lo));
    const int tlast = TC - (ngrp - 1) * TGB;  // tiles of the last row group
    const int wpp = 1 << p.lw;  // warps per tile pair (a power of two, at most 8)
    const int pair = warp >> p.lw, part = warp & (wpp - 1);
    const int nbw = (1 << cbs) >> p.lw;  // pack blocks per chunk and warp
    const int jb = min(g, M - 1);  // activation row of the lane's B fragments (columns >= M are never stored)
    const size_t pstride = (size_t)16 * p.tmax * M;  // one part's (and weight's) partial sums
    // second tile of a pair: the next tile of the box, or the same tile of the up weight
    const uint32_t q1_off = DUAL ? HPC * box_bytes : HM_BOX;
    const uint32_t ring32 = smem_u32(ring), srow32 = smem_u32(srow);
    const uint32_t lane_c = (uint32_t)(g * 128 + ((t & 1) << 3));               // row g, 8-byte half of a chunk
    const uint32_t bbase = smem_u32(btab) + (uint32_t)(jb * 4 + t) * 16u;       // + pb * 256 m
    const uint32_t q1_s2 = DUAL ? (uint32_t)L.scal_w : 32u * (uint32_t)G;       // second tile's scales
    const uint32_t G8 = 16u * (uint32_t)G;                                       // 8 rows of scales
    // the 128-byte swizzle maps 16-byte chunk j of box row r to chunk j ^ (r & 7); rows g and
    // g + 8 share r & 7 = g
    auto swz = [&](int blk) { return (uint32_t)(((((blk & 3) << 1) | (t >> 1)) ^ g) << 4); };
    float tot[HM_TG][4];
#pragma unroll
    for (int q = 0; q < HM_TG; q++) tot[q][0] = tot[q][1] = tot[q][2] = tot[q][3] = 0.f;
    HmCursor ch = {0, 0, 0, 0u};
    for (int c = 0; c < nch; c++) {
        if (!failed && !warp_wait(&full[ch.s], ch.ph)) failed = true;
        const int ntg = ch.gi == ngrp - 1 ? tlast : TGB;
        // tiles of this warp's pair (<= 0: none) and its first tile in the CTA
        const int ntp = DUAL ? (pair < ntg ? 2 : 0) : min(HM_TG, ntg - HM_TG * pair);
        const int tile0 = ch.gi * TGB + (DUAL ? pair : HM_TG * pair);
        if (ntp > 0) {
            // 32-bit shared addresses: this warp's code bytes of the pair's first tile in the
            // stage (row g; the block's swizzled 16-byte chunk is added per block), its B
            // fragments (block pb at pb * 256 m bytes) and its scales (block pb at (pb >> gsh) * 2)
            const uint32_t cbase = ring32 + (uint32_t)ch.s * stage_bytes + (uint32_t)(tile0 - ch.gi * TGB) * HM_BOX + lane_c;
            const uint32_t sbase = srow32 + (uint32_t)(tile0 * 16 + g) * (uint32_t)G * 2u;
            const int pb0 = ch.kc << cbs;
            // the warp's blocks of the chunk: blk = part + bi wpp.  In the UNR instantiation a full
            // chunk (all its blocks inside the row) of two or four blocks a warp runs a loop of
            // constant trip count that the compiler unrolls, so the next block's loads can be
            // issued under the current block's MMAs; otherwise the counted loop.
            auto blocks = [&](auto nt, auto nb, int bi0) {
                constexpr int NT = decltype(nt)::value, NB = decltype(nb)::value;
#pragma unroll
                for (int bi = 0; bi < NB; bi++) {
                    const int blk = part + (bi0 + bi) * wpp;
                    const int pb = pb0 + blk;
                    hm_block<NT, M>(tot, cbase + (uint32_t)(blk >> 2) * box_bytes + swz(blk), q1_off,
                                    bbase + (uint32_t)pb * (256u * M), sbase + (uint32_t)(pb >> gsh) * 2u, q1_s2, G8);
                }
            };
            using I1 = std::integral_constant<int, 1>;
            using I2 = std::integral_constant<int, 2>;
            using I4 = std::integral_constant<int, 4>;
            const bool whole = UNR && pb0 + (1 << cbs) <= P;
            if (UNR && whole && nbw == 2) {
                if (ntp == 2) blocks(I2{}, I2{}, 0);
                else blocks(I1{}, I2{}, 0);
            } else if (UNR && whole && nbw == 4) {
                // the dual form unrolls two blocks at a time: its second weight's state leaves no
                // registers for four blocks in flight
                if (DUAL) {
                    blocks(I2{}, I2{}, 0);
                    blocks(I2{}, I2{}, 2);
                } else if (ntp == 2) {
                    blocks(I2{}, I4{}, 0);
                } else {
                    blocks(I1{}, I4{}, 0);
                }
            } else if (ntp == 2) {
                for (int bi = 0; bi < nbw; bi++) {
                    const int blk = part + bi * wpp;  // pack block within the chunk
                    const int pb = pb0 + blk;
                    if (pb >= P) break;
                    hm_block<2, M>(tot, cbase + (uint32_t)(blk >> 2) * box_bytes + swz(blk), q1_off,
                                   bbase + (uint32_t)pb * (256u * M), sbase + (uint32_t)(pb >> gsh) * 2u, q1_s2, G8);
                }
            } else {
                for (int bi = 0; bi < nbw; bi++) {
                    const int blk = part + bi * wpp;
                    const int pb = pb0 + blk;
                    if (pb >= P) break;
                    hm_block<1, M>(tot, cbase + (uint32_t)(blk >> 2) * box_bytes + swz(blk), q1_off,
                                   bbase + (uint32_t)pb * (256u * M), sbase + (uint32_t)(pb >> gsh) * 2u, q1_s2, G8);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[ch.s]);
        if (ch.kc == nkc - 1) {
            // end of a row group: the warp's sums for its pair's rows into its part's slots
            if (ntp > 0 && part < 8) {
                float* sl = slot + (size_t)part * NW * pstride;
#pragma unroll
                for (int q = 0; q < HM_TG; q++) {
                    if (q >= ntp) continue;
                    // slots [part][weight][row][m]: the dual form's second tile is the up weight's
                    float* s0 = sl + (DUAL ? q * pstride + (size_t)(tile0 * 16 + g) * M : (size_t)((tile0 + q) * 16 + g) * M);
                    float* s8 = s0 + 8 * M;
                    if (2 * t < M) {
                        s0[2 * t] = tot[q][0];
                        s8[2 * t] = tot[q][2];
                    }
                    if (2 * t + 1 < M) {
                        s0[2 * t + 1] = tot[q][1];
                        s8[2 * t + 1] = tot[q][3];
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < HM_TG; q++) tot[q][0] = tot[q][1] = tot[q][2] = tot[q][3] = 0.f;
        }
        ch.next(NST, nkc);
    }
    if (failed && lane == 0) atomicOr(&g_hm_status, 1u);
    consumer_sync();

    // ---- the parts' partial sums, added in a fixed order, stored as BF16 (the dual form: u,
    // and h = BF16(SiLU(BF16(g)) * BF16(u)), the arithmetic of the separate gate and up launches)
    for (int o = tid; o < M * R; o += NCT) {
        const int j = o / R, row = o - j * R;
        float sum = 0.f, sum2 = 0.f;
        for (int pp = 0; pp < wpp; pp++) {
            sum += slot[pp * NW * pstride + (size_t)row * M + j];
            if (DUAL) sum2 += slot[(pp * NW + 1) * pstride + (size_t)row * M + j];
        }
        const __nv_bfloat16 bv = __float2bfloat16_rn(sum * rowback[j]);
        const uint16_t ub = *reinterpret_cast<const uint16_t*>(&bv);
        const size_t idx = (size_t)j * n + r0 + row;
        if (DUAL) {
            const __nv_bfloat16 uv = __float2bfloat16_rn(sum2 * rowback[j]);
            const uint16_t uu = *reinterpret_cast<const uint16_t*>(&uv);
            p.y2[idx] = uu;
            const __nv_bfloat16 hb = __float2bfloat16_rn(silu_mul1(bf16_bits_to_f32(ub), bf16_bits_to_f32(uu)));
            p.y[idx] = *reinterpret_cast<const uint16_t*>(&hb);
            continue;
        }
        p.y[idx] = ub;
        if (p.hgate) {
            const __nv_bfloat16 hb = __float2bfloat16_rn(silu_mul1(bf16_bits_to_f32(p.hgate[idx]), bf16_bits_to_f32(ub)));
            p.hgate[idx] = *reinterpret_cast<const uint16_t*>(&hb);
        }
    }
}

// Launch plan: one CTA per SM (at most one per tile; sixteen consumer warps fill an SM's
// registers, so CTAs of consecutive launches never share one).  A row group is as many
// tiles as balance the CTA's tiles over the fewest groups of at most eight (TMA requests
// stream faster the larger they are: a box of 8 tiles is 16 KB); the ring gets as many
// stages as one SM holds, up to one per chunk, so a CTA's whole slice is usually requested
// at once.  A chunk spans 1024 columns, or 2048 where each tile pair of a single weight has
// eight warps (one or two pairs per row group, as in an FFN's down projection: few rows, long
// rows) and three such stages fit: each warp then takes two pack blocks per chunk, which halves the
// per-chunk waits, releases and requests and lets the unrolled block loop run.  nw = 2: the
// dual (gate and up) form.
static int hm_plan(int m, int n, int k, int group, int nw, int sms, HmParams* prm, size_t* smem_out) {
    const int ntiles = (n + 15) / 16;
    const int ncta = ntiles < sms ? ntiles : sms;
    const int tmax = (ntiles + ncta - 1) / ncta;
    // the fewest row groups whose two-stage ring fits, then as many stages as fit
    int ngrp = (tmax + HM_MAX_TGB - 1) / HM_MAX_TGB, tgb = (tmax + ngrp - 1) / ngrp;
    while (tgb > 1 && HmLayout(m, k, group, tgb, 2, tmax, nw, 2).total > (size_t)HM_SMEM_LIMIT) {
        ngrp++;
        tgb = (tmax + ngrp - 1) / ngrp;
    }
    const int hpc = nw == 1 && hm_parts(tgb, nw) == HM_MAX_PARTS && k / 128 >= 16 &&
                            HmLayout(m, k, group, tgb, 3, tmax, nw, 4).total <= (size_t)HM_SMEM_LIMIT
                        ? 4
                        : 2;
    const int nkc = (k / 128 + 4 * hpc - 1) / (4 * hpc);
    const int nch = ngrp * nkc;
    int NST = HM_MAX_STAGES < nch ? HM_MAX_STAGES : nch;
    if (NST < 2) NST = 2;
    while (NST > 2 && HmLayout(m, k, group, tgb, NST, tmax, nw, hpc).total > (size_t)HM_SMEM_LIMIT) NST--;
    prm->n = n;
    prm->k = k;
    prm->group = group;
    prm->tmax = tmax;
    prm->tgb = tgb;
    prm->nstages = NST;
    prm->hpc = hpc;
    *smem_out = HmLayout(m, k, group, tgb, NST, tmax, nw, hpc).total;
    return ncta;
}

// Shapes this kernel takes: its shared-memory carve-up fits one SM.
bool gemv_hm_supported(const bq_q2_weight* w, uint32_t m) {
    if (w->k == 0 || w->n == 0 || m < 1 || m > 8 || w->k / 8 >= 23170) return false;
    if ((uint64_t)((w->n + 15) / 16) * (uint64_t)sm_count() * (uint64_t)sm_count() >= (1ull << 32)) return false;
    HmParams prm;
    size_t smem = 0;
    hm_plan((int)m, (int)w->n, (int)w->k, (int)w->group, 1, sm_count(), &prm, &smem);
    return smem <= (size_t)HM_SMEM_LIMIT;
}

// The dual form for an FFN's gate and up weights (the caller has checked that they match).
bool gemv_hm_dual_supported(const bq_q2_weight* gate, uint32_t m) {
    if (gate->k == 0 || gate->n == 0 || m < 1 || m > 8 || gate->k / 8 >= 23170) return false;
    if ((uint64_t)((gate->n + 15) / 16) * (uint64_t)sm_count() * (uint64_t)sm_count() >= (1ull << 32)) return false;
    HmParams prm;
    size_t smem = 0;
    hm_plan((int)m, (int)gate->n, (int)gate->k, (int)gate->group, 2, sm_count(), &prm, &smem);
    return smem <= (size_t)HM_SMEM_LIMIT;
}

typedef void (*HmKernel)(const CUtensorMap, const CUtensorMap, const HmParams);

template <bool DUAL, bool UNR, int HPC>
static HmKernel hm_kernel_for(uint32_t m) {
    switch (m) {
        case 1: return q2_gemv_hm_kernel<1, DUAL, UNR, HPC>;
        case 2: return q2_gemv_hm_kernel<2, DUAL, UNR, HPC>;
        case 3: return q2_gemv_hm_kernel<3, DUAL, UNR, HPC>;
        case 4: return q2_gemv_hm_kernel<4, DUAL, UNR, HPC>;
        case 5: return q2_gemv_hm_kernel<5, DUAL, UNR, HPC>;
        case 6: return q2_gemv_hm_kernel<6, DUAL, UNR, HPC>;
        case 7: return q2_gemv_hm_kernel<7, DUAL, UNR, HPC>;
        case 8: return q2_gemv_hm_kernel<8, DUAL, UNR, HPC>;
        default: return nullptr;
    }
}

// Shared launch path: w2 / y2 non-null selects the dual form (w = gate, w2 = up; y gets h,
// y2 gets u).
static int launch_hm(const uint16_t* x, const bq_q2_weight* w, const bq_q2_weight* w2, uint16_t* y, uint16_t* y2,
                     uint32_t m, uint16_t* hgate, cudaStream_t stream, const char* who) {
    static int configured_smem[64][5][8] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64) dev = 63;
    if (m < 1 || m > 8) return fail(BQ_ERR_INVALID, "%s: m = %u, must be 1..8", who, m);
    const bool dual = w2 != nullptr;
    HmParams prm;
    size_t smem = 0;
    const int ncta = hm_plan((int)m, (int)w->n, (int)w->k, (int)w->group, dual ? 2 : 1, sm_count(), &prm, &smem);
    if (smem > (size_t)HM_SMEM_LIMIT) return fail(BQ_ERR_INVALID, "%s: shape needs too much shared memory", who);
    // two or four blocks a warp per chunk: the unrolled instantiation
    const int nbw = 4 * prm.hpc / hm_parts(prm.tgb, dual ? 2 : 1);
    const bool unr = nbw == 2 || nbw == 4;
    // (hm_plan gives 2048-column chunks only to the single-weight form with eight warps per
    // tile pair, i.e. always with two blocks a warp: the one HPC = 4 instantiation)
    const int kind = prm.hpc == 4 ? 4 : (dual ? 1 : 0) + (unr ? 2 : 0);
    const HmKernel kern = prm.hpc == 4 ? hm_kernel_for<false, true, 4>(m)
                          : dual ? (unr ? hm_kernel_for<true, true, 2>(m) : hm_kernel_for<true, false, 2>(m))
                                 : (unr ? hm_kernel_for<false, true, 2>(m) : hm_kernel_for<false, false, 2>(m));
    if ((size_t)configured_smem[dev][kind][m - 1] < smem) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: cannot reserve %zu bytes of shared memory", who, smem);
        configured_smem[dev][kind][m - 1] = (int)smem;
    }
    // rows of a whole number of 128-byte column blocks (k % 512 == 0): one 3-D request brings a chunk's
    // column blocks; otherwise one 2-D box per 512-column half
    CUtensorMap tmap, tmap2;
    int st;
    prm.chunk3d = (w->k % 512 == 0) ? 1 : 0;
    if (prm.chunk3d) {
        if ((st = cached_tmap_chunks_u8(&tmap, w->data, w->k / 4, w->n, 16 * prm.tgb, prm.hpc, who))) return st;
        tmap2 = tmap;
        if (dual && (st = cached_tmap_chunks_u8(&tmap2, w2->data, w2->k / 4, w2->n, 16 * prm.tgb, prm.hpc, who)))
            return st;
    } else {
        if ((st = cached_tmap_2d_u8(&tmap, w->data, w->k / 4, w->n, w->k / 4, 128, 16 * prm.tgb, true, who))) return st;
        tmap2 = tmap;
        if (dual &&
            (st = cached_tmap_2d_u8(&tmap2, w2->data, w2->k / 4, w2->n, w2->k / 4, 128, 16 * prm.tgb, true, who)))
            return st;
    }
    {
        const HmLayout L(m, (int)w->k, (int)w->group, prm.tgb, prm.nstages, prm.tmax, dual ? 2 : 1, prm.hpc);
        prm.ring = (uint32_t)L.ring;
        prm.btab = (uint32_t)L.btab;
        prm.scal = (uint32_t)L.scal;
        prm.scal_w = (uint32_t)L.scal_w;
        prm.slot = (uint32_t)L.slot;
        prm.misc = (uint32_t)L.misc;
        prm.G = (int)(w->k / w->group);
        const int wpp = hm_parts(prm.tgb, dual ? 2 : 1);
        prm.lw = wpp == 8 ? 3 : wpp == 4 ? 2 : wpp == 2 ? 1 : 0;
        prm.kmag = 0xFFFFFFFFu / (w->k / 8) + 1u;
        prm.cmag = 0xFFFFFFFFu / (uint32_t)ncta + 1u;
        prm.gmag = 0xFFFFFFFFu / (uint32_t)prm.tgb + 1u;
    }
    prm.codes = (const uint8_t*)w->data;
    prm.scales = (const uint16_t*)((const uint8_t*)w->data + (size_t)w->n * (w->k / 4));
    prm.codes2 = dual ? (const uint8_t*)w2->data : nullptr;
    prm.scales2 = dual ? (const uint16_t*)((const uint8_t*)w2->data + (size_t)w2->n * (w2->k / 4)) : nullptr;
    prm.x = x;
    prm.y = y;
    prm.y2 = y2;
    prm.hgate = hgate;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ncta);
    cfg.blockDim = dim3(HM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tmap, tmap2, prm) != cudaSuccess) return check_launch(who);
    return check_launch(who);
}

int launch_q2_gemv_hm(const uint16_t* x, const bq_q2_weight* w, uint16_t* y, uint32_t m, uint16_t* hgate,
                      cudaStream_t stream, const char* who) {
    return launch_hm(x, w, nullptr, y, nullptr, m, hgate, stream, who);
}

int launch_q2_gemv_hm_dual(const uint16_t* x, const bq_q2_weight* gate, const bq_q2_weight* up, uint16_t* h,
                           uint16_t* u, uint32_t m, cudaStream_t stream, const char* who) {
    return launch_hm(x, gate, up, h, u, m, nullptr, stream, who);
}

}  // namespace bq8
