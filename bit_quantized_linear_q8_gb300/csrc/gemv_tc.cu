// gemv_tc.cu -- Q2_0 decode GEMV for 1..8 activation rows on the tcgen05 tensor cores.
//
// Source: init_q2.rs `set_packed_q2_qkvz` (decode runs `q2_0_gemv_vec`) and
// dense_ffn_decode_batch.rs `forward_km_q2` (`q2_0_gemv_vec_batchm` for gate/up/down).
//
// The packed weight (2.125 bits per weight) is the only large stream, so the kernel has to
// consume ~176 K weights per microsecond per SM.  Design (GB300, sm_103a):
//
//  * One tcgen05.mma of kind f8f6f4 (M = 128 rows, N = 16, K = 32) per 32 columns.  Weights
//    are its A operand, held in tensor memory as e4m3 bytes with exponent field 0: the
//    2-bit code c in the low mantissa bits is the subnormal c * 2^-9, so one AND (and a
//    shift) turns four codes into four operands.  Sixteen "unpack" warps write them into
//    TMEM with tcgen05.st (lane = row), a pair of 128-column groups at a time, six pairs in
//    flight.  The tensor cores take e4m3 subnormals exactly.
//  * Activations are the B operand, K-major in shared memory, built by the same sixteen
//    warps as each stage lands: per 128-column group and activation row j, a power-of-two
//    scale S puts max |x| in [128, 256); x * S is split exactly into hi + lo, both e4m3 (hi
//    keeps 4 significant bits, lo the at most 4 bits left), in B rows j and 8 + j.  Every
//    product is exact.
//  * The wanted sum_k (c - 2) x is (row - row of a virtual weight with every code 2) summed
//    over hi and lo, times 2^9 / S.  TMEM lane 31 of each 32-lane quadrant is that row (so a
//    CTA holds 4 x 31 = 124 weight rows); four epilogue warps take the difference with one
//    shuffle and apply the group's BF16 scale d in fp32.
//  * Issuing a tcgen05.mma costs the issuing thread about 54 cycles, so five issuing warps
//    take the groups round robin and commit to per-accumulator mbarriers; the epilogue
//    warps drain the eight accumulators four groups (one TMA stage) at a time, so the fixed
//    cost of every wait, fence and arrival is paid once per pair or per stage.  B tiles
//    live in a 16-tile ring.
//  * A producer warp streams the CTA's rows through a 5-stage TMA ring (512 columns per
//    stage, 128-byte swizzle) plus the stage's activation columns, and bulk-copies the
//    rows' group scales.  The weights do not depend on the previous kernel, so their
//    copies are issued before griddepcontrol.wait (programmatic dependent launch); the
//    activations after it.
//  * Shapes with few rows split K over a thread-block cluster of up to 8 CTAs; the partial
//    sums meet in the leader CTA through distributed shared memory.
//  * Every mbarrier wait is bounded; on a timeout the kernel records it in the status word
//    and winds down (tensor memory is always released).
#include "common.cuh"

namespace bq8 {

constexpr int TC_UW = 16;                            // unpack warps 0..15 (four per TMEM lane quadrant)
constexpr int TC_EW = 4;                             // epilogue / B-tile warps 16..19 (one per quadrant)
constexpr int TC_IW = 5;                             // MMA-issuing warps 20..24
constexpr int TC_EW0 = TC_UW;
constexpr int TC_IW0 = TC_UW + TC_EW;
constexpr int TC_PRODUCER = TC_IW0 + TC_IW;          // warp 25: TMA producer
constexpr int TC_THREADS = (TC_PRODUCER + 1) * 32;
constexpr int TC_NAB = 5;                            // A blocks of two groups (64 TMEM columns)
// D accumulators.  An unpack warp waits for the MMAs of the pair TC_NAB back before reusing
// its A block; the slot's next phase must still be ahead of it: TC_ND >= 2 * TC_NAB.
constexpr int TC_ND = 10;
constexpr int TC_NB = 16;                            // B tiles
// 2^9 / S per group and activation row.  A group's entry is rewritten 32 groups later; the
// MMA gating keeps the builders at most 2 + 2 * TC_NAB + TC_ND = 22 groups ahead of the
// last drained group.
constexpr int TC_NE = 32;
constexpr int TC_NS = 5;                             // TMA stages, 4 groups (512 columns) each
constexpr int TC_RQ = 31;                            // weight rows per TMEM lane quadrant
constexpr int TC_ROWS = 4 * TC_RQ;                   // 124 weight rows per CTA
constexpr int TC_CODES = 16384;                      // stage codes: <= 124 rows x 128 B
constexpr int TC_XB = 8192;                          // stage activations: 2 boxes x m x 256 bf16
constexpr int TC_STAGE = TC_CODES + TC_XB;
constexpr int TC_LBO = 272;                          // B core matrices (8 rows x 16 B) along K, padded
constexpr int TC_SBO = 128;                          // B rows 8..15 (the lo parts)
constexpr int TC_BT = 8 * TC_LBO;                    // B tile: 16 rows x 128 e4m3 (K-major)
constexpr int TC_TMEM_COLS = 512;
constexpr int TC_ACOL = 0;                           // A block b: TMEM columns 64b .. 64b + 63
constexpr int TC_DCOL = 64 * TC_NAB;                 // D accumulator d: TMEM columns 320 + 16d ..
static_assert(TC_ND >= 2 * TC_NAB && 64 * TC_NAB + 16 * TC_ND <= TC_TMEM_COLS, "TMEM ring sizes");
static_assert(2 + 2 * TC_NAB + TC_ND < TC_NE, "scale ring");
constexpr int TC_NBAR = 2 * TC_NS + TC_NAB + TC_NB + 2 * TC_ND + TC_NE + 1;
constexpr int TC_SMEM_LIMIT = 225 * 1024;

static __device__ unsigned int g_gemv_tc_status;

unsigned int gemv_tc_status_take() {
    unsigned int v = 0, zero = 0;
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(&v, g_gemv_tc_status, sizeof v);
    cudaMemcpyToSymbol(g_gemv_tc_status, &zero, sizeof zero);
    return v;
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4: D fp32, A and B e4m3, both K-major,
// N = 16, M = 128.
constexpr uint32_t TC_IDESC = (1u << 4) | (0u << 7) | (0u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// Shared-memory matrix descriptor, no swizzle: 8-row x 16-byte core matrices, `lbo` bytes
// apart along K, `sbo` bytes apart along M/N.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %3, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %4, p;\n}\n"
        ::"r"(d), "r"(a), "l"(bdesc), "r"(accumulate), "r"(TC_IDESC));
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
        "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tc_ld4(uint32_t taddr, float (&v)[4]) {
    uint32_t r0, r1, r2, r3;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    v[0] = __uint_as_float(r0);
    v[1] = __uint_as_float(r1);
    v[2] = __uint_as_float(r2);
    v[3] = __uint_as_float(r3);
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float ld_cluster_f32(const void* local, uint32_t rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

// Two words of packed codes of one row (word w holds bytes 4w..4w+3 of the row's 32-byte
// pack block, byte l carrying columns 32i + l of sub-blocks i = 0..3 in bits 2i) -> 8 TMEM
// columns of four e4m3 operands: column 4w' + i holds columns 32i + 4w + 0..3, each code c
// as the subnormal c * 2^-9.
__device__ __forceinline__ void unpack_words(const uint2& cw, uint32_t (&r)[8]) {
    const uint32_t wds[2] = {cw.x, cw.y};
#pragma unroll
    for (int q = 0; q < 2; q++) {
        const uint32_t w = wds[q];
        r[4 * q + 0] = w & 0x03030303u;
        r[4 * q + 1] = (w >> 2) & 0x03030303u;
        r[4 * q + 2] = (w >> 4) & 0x03030303u;
        r[4 * q + 3] = (w >> 6) & 0x03030303u;
    }
}

__device__ __forceinline__ void tc_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// W (4 or 8) consecutive accumulator columns of this warp's lane quadrant.
template <int W>
__device__ __forceinline__ void tc_ldw(uint32_t taddr, float* v) {
    if constexpr (W == 8)
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
                     : "r"(taddr)
                     : "memory");
    else
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                     : "r"(taddr)
                     : "memory");
}

// Two e4m3 bytes (RN) of a pair of fp32 values, in the low 16 bits.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(lo), "f"(hi));
    return r;
}

template <int MV>  // activation rows m
__global__ void __launch_bounds__(TC_THREADS, 1)
    q2_gemv_tc_kernel(const __grid_constant__ CUtensorMap cmap_hi, const __grid_constant__ CUtensorMap cmap_lo,
                      const __grid_constant__ CUtensorMap xmap, const uint8_t* __restrict__ splane,
                      uint16_t* __restrict__ y, int n, int k, int group, int nclus, int csplit, int rows_hi,
                      int sc_cap) {
    constexpr int m = MV;
    constexpr int DW = MV > 4 ? 8 : 4;  // accumulator columns read per part (hi, lo)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = align1024(smem_raw);
    uint8_t* btile = stages + TC_NS * TC_STAGE;
    float* red = reinterpret_cast<float*>(btile + TC_NB * TC_BT);  // [8][124] partial sums
    float* escl = red + 8 * TC_ROWS;                                // [32 groups][8 rows]: 2^9 / S
    uint8_t* scs = reinterpret_cast<uint8_t*>(escl + TC_NE * 8);    // the rows' scale bytes
    uint64_t* full = reinterpret_cast<uint64_t*>(scs + sc_cap);     // TMA stage landed
    uint64_t* empty = full + TC_NS;                                  // stage consumed
    uint64_t* afull = empty + TC_NS;                                 // A block written
    uint64_t* bfull = afull + TC_NAB;                                // B tile written
    uint64_t* mdone = bfull + TC_NB;                                 // accumulator's MMAs complete
    uint64_t* dfree = mdone + TC_ND;                                 // accumulator read by the epilogue
    uint64_t* eready = dfree + TC_ND;                                // a group's 2^9 / S written
    uint64_t* sfull = eready + TC_NE;                                // scales landed
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sfull + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NG = k >> 7;
    const int clus = blockIdx.x / csplit;
    const uint32_t rank = csplit > 1 ? cluster_rank() : 0u;
    const int r0 = (int)((int64_t)clus * n / nclus);
    const int R = (int)((int64_t)(clus + 1) * n / nclus) - r0;
    const int gb = (int)((int64_t)rank * NG / csplit);
    const int NGc = (int)((int64_t)(rank + 1) * NG / csplit) - gb;
    const int nst = (NGc + 3) >> 2;
    const int G = k / group;
    const uint32_t xbytes = 1024u * (uint32_t)m;  // two boxes of m rows x 256 BF16
    const CUtensorMap* cmap = R == rows_hi ? &cmap_hi : &cmap_lo;
    // scale bytes of the CTA's rows: [s_lo, s_hi) arrive by one bulk copy, the rest (at most
    // 14 bytes at the end of the plane) is copied by the threads that own those rows
    const int64_t s_lo = ((int64_t)r0 * G * 2) & ~int64_t(15);
    int64_t s_hi = ((int64_t)(r0 + R) * G * 2 + 15) & ~int64_t(15);
    const int64_t plane16 = ((int64_t)n * G * 2) & ~int64_t(15);
    if (s_hi > plane16) s_hi = plane16;
    if (s_hi < s_lo) s_hi = s_lo;
    const uint32_t sbytes = (uint32_t)(s_hi - s_lo);
    bool failed = false;
    float tot[MV];
#pragma unroll
    for (int j = 0; j < MV; j++) tot[j] = 0.f;

    if (warp == TC_PRODUCER && lane == 0) {
        for (int s = 0; s < TC_NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], TC_UW);
        }
        for (int b = 0; b < TC_NAB; b++) mbar_init(&afull[b], TC_UW);
        for (int t = 0; t < TC_NB; t++) mbar_init(&bfull[t], TC_UW);
        for (int d = 0; d < TC_ND; d++) {
            mbar_init(&mdone[d], 1);
            mbar_init(&dfree[d], TC_EW);
        }
        for (int g = 0; g < TC_NE; g++) mbar_init(&eready[g], TC_UW);
        mbar_init(sfull, 1);
        fence_barrier_init();
        // weights first: they do not depend on the kernel before this one
        mbar_arrive_expect_tx(sfull, sbytes);
        if (sbytes) bulk_load(scs, splane + s_lo, sbytes, sfull);
        for (int st = 0; st < TC_NS && st < nst; st++) {
            mbar_arrive_expect_tx(&full[st], (uint32_t)R * 128u + xbytes);
            tma_load_2d(stages + st * TC_STAGE, cmap, (gb + 4 * st) * 32, r0, &full[st]);
        }
    }
    if (warp == TC_IW0) {  // tensor memory for the A blocks and the accumulators
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "n"(TC_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

    if (warp == TC_PRODUCER) {
        if (lane == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            for (int st = 0; st < nst; st++) {
                const int s = st % TC_NS;
                if (st >= TC_NS) {
                    if (!mbar_wait(&empty[s], ((st / TC_NS) - 1) & 1)) {
                        failed = true;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], (uint32_t)R * 128u + xbytes);
                    tma_load_2d(stages + s * TC_STAGE, cmap, (gb + 4 * st) * 32, r0, &full[s]);
                }
                uint8_t* xs = stages + s * TC_STAGE + TC_CODES;
                tma_load_2d(xs, &xmap, (gb + 4 * st) * 128, 0, &full[s]);
                tma_load_2d(xs + m * 512, &xmap, (gb + 4 * st) * 128 + 256, 0, &full[s]);
            }
        }
    } else if (warp >= TC_IW0) {  // MMA issuers: issuer i takes groups i, i + 5, ...
        const int iw = warp - TC_IW0;
        if (lane == 0) {
            int last = -1;
            for (int gi = iw; gi < NGc; gi += TC_IW) {
                const int d = gi % TC_ND, t = gi % TC_NB, pr = gi >> 1, b = pr % TC_NAB;
                if (!mbar_wait(&afull[b], (pr / TC_NAB) & 1) || !mbar_wait(&bfull[t], (gi / TC_NB) & 1) ||
                    (gi >= TC_ND && !mbar_wait(&dfree[d], ((gi - TC_ND) / TC_ND) & 1))) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t bb = smem_u32(btile + t * TC_BT), dcol = tbase + TC_DCOL + 16 * d;
                const uint32_t acol = tbase + TC_ACOL + 64 * b + 32 * (gi & 1);
#pragma unroll
                for (int kk = 0; kk < 4; kk++)
                    tc_mma(dcol, acol + 8 * kk, smem_desc(bb + 2 * TC_LBO * kk, TC_LBO, TC_SBO), kk > 0);
                tc_commit(&mdone[d]);
                last = gi;
            }
            // the last commit must land before the tensor memory is released
            if (last >= 0 && !mbar_wait(&mdone[last % TC_ND], (last / TC_ND) & 1)) failed = true;
        }
    } else if (warp >= TC_EW0) {  // epilogue warps: per stage, B tiles out, accumulators of two stages back in
        const int qd = warp & 3;
        const int rho = TC_RQ * qd + lane;
        const bool rowok = lane < TC_RQ && rho < R;
        const int64_t srow = (int64_t)(r0 + (rowok ? rho : 0)) * G * 2;  // the row's scales in the plane
        const uint32_t tq = tbase + ((uint32_t)(32 * qd) << 16);
        if (rowok) {  // scale bytes past the bulk copy: this thread's own row only
            for (int64_t o = srow > s_hi ? srow : s_hi; o < srow + (int64_t)G * 2; o += 2)
                *reinterpret_cast<uint16_t*>(scs + (o - s_lo)) = __ldg(reinterpret_cast<const uint16_t*>(splane + o));
        }
        const uint16_t* myscale = reinterpret_cast<const uint16_t*>(scs + (srow - s_lo));
        const int gpr = group >> 7;  // 128-column groups per scale
        int sidx = gb / gpr, ssub = gb - (gb / gpr) * gpr;
        for (int st = 2; st < nst + 2; st++) {
            // accumulators of stage st - 2
            const int e0 = 4 * (st - 2), ne = st >= 2 ? (NGc - e0 < 4 ? NGc - e0 : 4) : 0;
            if (ne > 0) {
                if (st == 2 && !mbar_wait(sfull, 0)) {
                    failed = true;
                    break;
                }
                bool ok = true;
                for (int u = 0; u < ne && ok; u++) {
                    ok = mbar_wait(&mdone[(e0 + u) % TC_ND], ((e0 + u) / TC_ND) & 1) &&
                         mbar_wait(&eready[(e0 + u) % TC_NE], ((e0 + u) / TC_NE) & 1);
                }
                if (!ok) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                // two accumulators at a time (a slot past the last group holds stale sums, unused):
                // the hi columns 0.. and the lo columns 8.. of each
#pragma unroll
                for (int hf = 0; hf < 2; hf++) {
                    float dv[2][2 * DW];
#pragma unroll
                    for (int uu = 0; uu < 2; uu++) {
                        const uint32_t dcol = tq + TC_DCOL + 16 * ((e0 + 2 * hf + uu) % TC_ND);
                        tc_ldw<DW>(dcol, dv[uu]);
                        tc_ldw<DW>(dcol + 8, dv[uu] + DW);
                    }
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    // (row minus the all-codes-2 row, lane 31) over hi + lo, times d * 2^9 / S
#pragma unroll
                    for (int uu = 0; uu < 2; uu++) {
                        const int u = 2 * hf + uu;
                        const bool live = u < ne;  // warp-uniform; no branch around the shuffles
                        const float ds = rowok && live ? bf16_bits_to_f32(myscale[sidx]) : 0.f;
                        if (live && ++ssub == gpr) {
                            ssub = 0;
                            sidx++;
                        }
                        const float* es = escl + ((e0 + u) % TC_NE) * 8;
#pragma unroll
                        for (int j = 0; j < MV; j++) {
                            const float v = dv[uu][j] + dv[uu][DW + j];
                            const float off = __shfl_sync(0xffffffffu, v, 31);
                            const float t = fmaf(ds * es[j], v - off, tot[j]);
                            tot[j] = live ? t : tot[j];
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    for (int u = 0; u < ne; u++) mbar_arrive(&dfree[(e0 + u) % TC_ND]);
            }
        }
        tc_fence_before();
    } else {  // unpack warps: four per lane quadrant, each a quarter of a row's 32 code bytes, a pair of groups at a time
        const int qd = warp & 3, part = warp >> 2;
        const int rho = TC_RQ * qd + lane;
        const uint32_t tq = tbase + ((uint32_t)(32 * qd) << 16);
        const int npr = (NGc + 1) >> 1;
        for (int pr = 0; pr < npr; pr++) {
            const int b = pr % TC_NAB, st = pr >> 1, s = st % TC_NS, g0 = 2 * pr;
            if (!(pr & 1)) {
                if (!mbar_wait(&full[s], (st / TC_NS) & 1)) {
                    failed = true;
                    break;
                }
                // this warp's share of the stage's B tiles: items (group gl, row j), 4m of them.
                // Tile t was last read by the MMAs of group 4st + gl - 16, complete since this
                // warp waited for pair pr - 6.
                const int gs0 = 4 * st, nb = NGc - gs0 < 4 ? NGc - gs0 : 4;
                const uint8_t* xs = stages + s * TC_STAGE + TC_CODES;
                const int i = lane >> 3, w = lane & 7;
#pragma unroll
                for (int it = 0; it < 2; it++) {
                    const int item = warp + TC_UW * it, gl = item / MV, j = item - gl * MV;
                    if (item < 4 * MV && gl < nb) {  // warp-uniform
                        const int col = 128 * gl + 32 * i + 4 * w;  // columns 32i + 4w .. + 3 of the group
                        const uint2 v =
                            *reinterpret_cast<const uint2*>(xs + (((col >> 8) * m + j) * 256 + (col & 255)) * 2);
                        const float xv[4] = {__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                                             __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u)};
                        // S = 2^(134 - e), e the biased exponent of the group's max |x|: max |x| S in [128, 256)
                        uint32_t mb = max(max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu),
                                          max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu));
                        mb = __reduce_max_sync(0xffffffffu, mb);
                        int e = (int)(mb >> 7);
                        e = e < 8 ? 8 : (e > 252 ? 252 : e);
                        const float S = __uint_as_float((uint32_t)(261 - e) << 23);
                        float hi[4], lo[4];
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            const float yq = xv[q] * S;
                            // hi: 4 significant bits (zero below the e4m3 normal range); lo: the rest
                            const float h = __uint_as_float(__float_as_uint(yq) & 0xFFF00000u);
                            hi[q] = fabsf(yq) < 0x1p-6f ? 0.f : h;
                            lo[q] = yq - hi[q];
                        }
                        const int tile = (gs0 + gl) % TC_NB;
                        uint8_t* bt = btile + tile * TC_BT + w * TC_LBO + 4 * i + j * 16;
                        *reinterpret_cast<uint32_t*>(bt) = e4m3x2(hi[0], hi[1]) | (e4m3x2(hi[2], hi[3]) << 16);
                        *reinterpret_cast<uint32_t*>(bt + TC_SBO) = e4m3x2(lo[0], lo[1]) | (e4m3x2(lo[2], lo[3]) << 16);
                        if (lane == 0)  // 2^9 / S
                            escl[((gs0 + gl) % TC_NE) * 8 + j] = __uint_as_float((uint32_t)(e + 2) << 23);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    for (int gl = 0; gl < nb; gl++) {
                        mbar_arrive(&bfull[(gs0 + gl) % TC_NB]);
                        mbar_arrive(&eready[(gs0 + gl) % TC_NE]);
                    }
                }
            }
            uint2 c0, c1;
            if (lane < TC_RQ) {
                const uint8_t* row = stages + s * TC_STAGE + rho * 128 + 8 * (part & 1);
                const int gl = g0 & 3;
                c0 = *reinterpret_cast<const uint2*>(row + (((2 * gl + (part >> 1)) ^ (rho & 7)) << 4));
                c1 = *reinterpret_cast<const uint2*>(row + (((2 * gl + 2 + (part >> 1)) ^ (rho & 7)) << 4));
            } else {
                c0 = c1 = make_uint2(0xAAAAAAAAu, 0xAAAAAAAAu);  // every code 2
            }
            uint32_t r0v[8], r1v[8];
            unpack_words(c0, r0v);
            unpack_words(c1, r1v);
            if (pr >= TC_NAB) {  // A block b is free once the MMAs of pair pr - 3 are complete
                const int gp = 2 * (pr - TC_NAB);
                if (!mbar_wait(&mdone[gp % TC_ND], (gp / TC_ND) & 1) ||
                    !mbar_wait(&mdone[(gp + 1) % TC_ND], ((gp + 1) / TC_ND) & 1)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
            }
            const uint32_t ta = tq + TC_ACOL + 64 * b + 8 * part;
            tc_st8(ta, r0v);
            tc_st8(ta + 32, r1v);  // past the last group: an unused half of the block
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&afull[b]);
                if ((pr & 1) || pr == npr - 1) mbar_arrive(&empty[s]);
            }
        }
        tc_fence_before();
    }
    if (failed) atomicOr(&g_gemv_tc_status, 1u);

    // ------------------------------------------------------------------ partial sums -> y
    const int orow = TC_RQ * (warp & 3) + lane;
    const bool owner = warp >= TC_EW0 && warp < TC_IW0 && lane < TC_RQ && orow < R;
    __syncwarp();
    if (csplit > 1) {
        if (owner) {
#pragma unroll
            for (int j = 0; j < MV; j++) red[j * TC_ROWS + orow] = tot[j];
        }
        cluster_sync_all();
        if (rank == 0 && owner) {
            for (int q = 1; q < csplit; q++) {
#pragma unroll
                for (int j = 0; j < MV; j++) tot[j] += ld_cluster_f32(&red[j * TC_ROWS + orow], (uint32_t)q);
            }
        }
    }
    if (rank == 0 && owner) {
#pragma unroll
        for (int j = 0; j < MV; j++) {
            const __nv_bfloat16 bv = __float2bfloat16_rn(tot[j]);
            y[(size_t)j * n + r0 + orow] = *reinterpret_cast<const uint16_t*>(&bv);
        }
    }
    if (csplit > 1) cluster_sync_all();  // peers keep their shared memory until the leader has read it
    __syncthreads();
    if (warp == TC_IW0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "n"(TC_TMEM_COLS));
    }
}

// Launches the tcgen05 GEMV for an already validated weight (k > 0, n > 0, 1 <= m <= 8).
int launch_q2_gemv_tc(const uint16_t* x, const bq_q2_weight* w, uint16_t* y, uint32_t m, cudaStream_t stream,
                      const char* who) {
    const int n = (int)w->n, k = (int)w->k, group = (int)w->group;
    const int NG = k / 128, G = k / group;
    const int nsm = sm_count();
    // clusters of `csplit` CTAs split K; every cluster owns <= 124 rows
    const int g0 = (n + TC_ROWS - 1) / TC_ROWS;
    int csplit = 1, nclus = g0;
    if (g0 < nsm) {
        csplit = nsm / g0;
        if (csplit > 8) csplit = 8;
        if (csplit > NG) csplit = NG;
        if (csplit < 1) csplit = 1;
        nclus = nsm / csplit;
        if (nclus < g0) nclus = g0;
        if (nclus > n) nclus = n;
    }
    const int rows_hi = (n + nclus - 1) / nclus;
    const int sc_cap = (rows_hi * G * 2 + 32 + 15) & ~15;
    const size_t smem =
        1024 + (size_t)TC_NS * TC_STAGE + TC_NB * TC_BT + 8 * TC_ROWS * 4 + TC_NE * 8 * 4 + sc_cap + TC_NBAR * 8 + 16;
    if (smem > (size_t)TC_SMEM_LIMIT)
        return fail(BQ_ERR_INVALID, "%s: k/group = %d scales per row need %zu bytes of shared memory", who, G, smem);

    static int configured[64][8] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 63;
    void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, const uint8_t*, uint16_t*, int, int, int, int, int, int,
                 int) = nullptr;
    switch (m) {
        case 1: kern = q2_gemv_tc_kernel<1>; break;
        case 2: kern = q2_gemv_tc_kernel<2>; break;
        case 3: kern = q2_gemv_tc_kernel<3>; break;
        case 4: kern = q2_gemv_tc_kernel<4>; break;
        case 5: kern = q2_gemv_tc_kernel<5>; break;
        case 6: kern = q2_gemv_tc_kernel<6>; break;
        case 7: kern = q2_gemv_tc_kernel<7>; break;
        case 8: kern = q2_gemv_tc_kernel<8>; break;
        default: return fail(BQ_ERR_INVALID, "%s: m = %u, must be 1..8", who, m);
    }
    if ((size_t)configured[dev][m - 1] < smem) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: cannot reserve %zu bytes of shared memory", who, smem);
        configured[dev][m - 1] = (int)smem;
    }

    const uint8_t* codes = static_cast<const uint8_t*>(w->data);
    const uint8_t* splane = codes + (size_t)n * (k / 4);
    CUtensorMap cmap_hi, cmap_lo, xmap;
    int st = make_tmap_2d_u8(&cmap_hi, codes, k / 4, n, k / 4, 128, rows_hi, true, who);
    if (st) return st;
    if ((st = make_tmap_2d_u8(&cmap_lo, codes, k / 4, n, k / 4, 128, rows_hi > 1 ? rows_hi - 1 : 1, true, who)))
        return st;
    if ((st = make_tmap_2d(&xmap, x, 2, k, m, (uint64_t)k * 2, 256, m, false, who))) return st;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nclus * csplit));
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    na++;
    if (csplit > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)csplit;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        na++;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    const cudaError_t e =
        cudaLaunchKernelEx(&cfg, kern, cmap_hi, cmap_lo, xmap, splane, y, n, k, group, nclus, csplit, rows_hi, sc_cap);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction ? BQ_ERR_UNSUPPORTED
                                                                                                : BQ_ERR_LAUNCH,
                    "%s: launch failed: %s", who, cudaGetErrorString(e));
    }
    return BQ_OK;
}

}  // namespace bq8
