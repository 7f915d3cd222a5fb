// gemv_tc.cu -- Q2_0 decode GEMV for 1..8 activation rows on the tcgen05 tensor cores.
//
// Source: init_q2.rs `set_packed_q2_qkvz` (decode runs `q2_0_gemv_vec`) and
// dense_ffn_decode_batch.rs `forward_km_q2` (`q2_0_gemv_vec_batchm` for gate/up/down).
//
// The packed weight (2.125 bits per weight) is the only large stream, so the kernel has to
// consume ~176 K weights per microsecond per SM.  Design (GB300, sm_103a):
//
//  * Weights are the MMA's A operand (M = 128 rows), held in tensor memory.  Eight
//    "unpack" warps turn each 2-bit code into the mantissa of BF16 1.0 with one lop3 per
//    pair of codes, v = 1 + c*s (s = 2^-7, 2^-5, 2^-3, 2^-3 by the code's bit position),
//    and store the rows into TMEM with tcgen05.st (lane = row).
//  * Activations are the B operand (N = 16; only rows 0..m-1 matter, the descriptor's
//    row-group stride of 0 repeats rows 0..7 for 8..15): per 128-column group the unpack
//    warps write a K-major tile of x/s, permuted into the order of the TMEM columns.
//  * sum_k (1 + c s) x/s = sum x/s + sum c x, so the wanted sum_k (c - 2) x is the MMA row
//    minus the row of a virtual weight with every code 2.  TMEM lane 31 of each 32-lane
//    quadrant is that row (so a CTA holds 4 x 31 = 124 weight rows); the epilogue takes
//    the difference with one shuffle and applies the group's BF16 scale d in fp32.
//  * One tcgen05.mma (128 x 16 x 16) per 16 columns.  Its issue costs the issuing thread
//    about 54 cycles, so four issuing warps take the 128-column groups round robin, each
//    with its own A/B/D buffer, and commit to an mbarrier the epilogue waits on.
//  * A producer warp streams the CTA's rows through a 5-stage TMA ring (512 columns per
//    stage, 128-byte swizzle) plus the stage's activation columns.  The weights do not
//    depend on the previous kernel, so their copies are issued before
//    griddepcontrol.wait (programmatic dependent launch); the activations after it.
//  * Shapes with few rows split K over a thread-block cluster of up to 8 CTAs; the partial
//    sums meet in the leader CTA through distributed shared memory.
//  * Every mbarrier wait is bounded; on a timeout the kernel records it in the status word
//    and winds down (tensor memory is always released).
#include "common.cuh"

namespace bq8 {

constexpr int TC_UW = 8;                              // unpack / B-tile / epilogue warps
constexpr int TC_IW = 4;                              // MMA-issuing warps
constexpr int TC_THREADS = (TC_UW + TC_IW + 1) * 32;  // + one TMA producer warp
constexpr int TC_PRODUCER = TC_UW + TC_IW;            // warp index of the producer
constexpr int TC_NA = TC_IW;                          // A/B/D buffers: issuer i owns buffer i
constexpr int TC_NS = 5;                              // TMA stages, 4 groups (512 columns) each
constexpr int TC_RQ = 31;                             // weight rows per TMEM lane quadrant
constexpr int TC_ROWS = 4 * TC_RQ;                    // 124 weight rows per CTA
constexpr int TC_CODES = 16384;                       // stage codes: <= 124 rows x 128 B
constexpr int TC_XB = 8192;                           // stage activations: 2 boxes x m x 256 bf16
constexpr int TC_STAGE = TC_CODES + TC_XB;
constexpr int TC_BT = 2048;                           // B tile: 8 rows x 128 bf16 (K-major)
constexpr int TC_TMEM_COLS = 512;
constexpr int TC_ACOL = 0;                            // A buffer a: TMEM columns 64a .. 64a + 63
constexpr int TC_DCOL = 256;                          // D buffer a: TMEM columns 256 + 16a ..
constexpr int TC_SMEM_LIMIT = 225 * 1024;

static __device__ unsigned int g_gemv_tc_status;

unsigned int gemv_tc_status_take() {
    unsigned int v = 0, zero = 0;
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(&v, g_gemv_tc_status, sizeof v);
    cudaMemcpyToSymbol(g_gemv_tc_status, &zero, sizeof zero);
    return v;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32, A and B BF16, both K-major,
// N = 16, M = 128.
constexpr uint32_t TC_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// Shared-memory matrix descriptor, no swizzle: 8-row x 16-byte core matrices, `lbo` bytes
// apart along K, `sbo` bytes apart along M/N.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %3, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n}\n"
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

// The 32 TMEM columns (64 weights) of one unpack thread for one group: four 32-bit words
// of packed codes (word w holds bytes 4w..4w+3 of the row's 32-byte pack block, byte l
// carrying columns 32i + l of sub-blocks i = 0..3 in bits 2i).  Column 8w' + 2i + h holds
// the pair (columns 32i + 4w + h, 32i + 4w + h + 2) for h = 0, 1.
__device__ __forceinline__ void unpack_group(const uint4& cw, uint32_t (&r)[32]) {
    const uint32_t one = 0x3F803F80u, m0 = 0x00030003u, m1 = 0x000C000Cu, m2 = 0x00300030u;
    const uint32_t wds[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const uint32_t w = wds[q], s2 = w >> 2, s8 = w >> 8, s10 = w >> 10;
        r[8 * q + 0] = and_or(w, m0, one);
        r[8 * q + 1] = and_or(s8, m0, one);
        r[8 * q + 2] = and_or(w, m1, one);
        r[8 * q + 3] = and_or(s8, m1, one);
        r[8 * q + 4] = and_or(w, m2, one);
        r[8 * q + 5] = and_or(s8, m2, one);
        r[8 * q + 6] = and_or(s2, m2, one);
        r[8 * q + 7] = and_or(s10, m2, one);
    }
}

__global__ void __launch_bounds__(TC_THREADS, 1)
    q2_gemv_tc_kernel(const __grid_constant__ CUtensorMap cmap_hi, const __grid_constant__ CUtensorMap cmap_lo,
                      const __grid_constant__ CUtensorMap xmap, const uint16_t* __restrict__ scales,
                      uint16_t* __restrict__ y, int m, int n, int k, int group, int nclus, int csplit, int rows_hi,
                      int ngmax) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = align1024(smem_raw);
    uint8_t* btile = stages + TC_NS * TC_STAGE;
    float* red = reinterpret_cast<float*>(btile + TC_NA * TC_BT);   // [8][124] partial sums
    uint16_t* sc = reinterpret_cast<uint16_t*>(red + 8 * TC_ROWS);  // [ngmax][124] scales
    uint64_t* bars = reinterpret_cast<uint64_t*>(sc + ((ngmax * TC_ROWS + 7) & ~7));
    uint64_t* full = bars;               // TMA stage landed (1 arrival + bytes)
    uint64_t* empty = bars + TC_NS;      // stage consumed (one arrival per unpack warp)
    uint64_t* afull = bars + 2 * TC_NS;  // A/B buffer written (one arrival per unpack warp)
    uint64_t* mdone = afull + TC_NA;     // MMAs of the buffer's group complete (commit)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mdone + TC_NA);

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
    const uint32_t xbytes = 2u * (uint32_t)m * 256u * 2u;
    const CUtensorMap* cmap = R == rows_hi ? &cmap_hi : &cmap_lo;
    bool failed = false;

    if (warp == TC_PRODUCER && lane == 0) {
        for (int s = 0; s < TC_NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], TC_UW);
        }
        for (int a = 0; a < TC_NA; a++) {
            mbar_init(&afull[a], TC_UW);
            mbar_init(&mdone[a], 1);
        }
        fence_barrier_init();
        // weights first: they do not depend on the kernel before this one
        for (int st = 0; st < TC_NS && st < nst; st++) {
            mbar_arrive_expect_tx(&full[st], (uint32_t)R * 128u + xbytes);
            tma_load_2d(stages + st * TC_STAGE, cmap, (gb + 4 * st) * 32, r0, &full[st]);
        }
    }
    if (warp == TC_UW) {  // tensor memory for the A and D buffers
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "n"(TC_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (warp < TC_UW) {  // this CTA's group scales, sc[group][row]; eight loads in flight per thread
        const int total = R * NGc;
        for (int base = threadIdx.x; base < total; base += 8 * TC_UW * 32) {
            uint16_t v[8];
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int e = base + u * TC_UW * 32;
                const int row = e / NGc, gl = e - row * NGc;
                v[u] = e < total ? __ldg(scales + (size_t)(r0 + row) * G + ((gb + gl) * 128) / group) : (uint16_t)0;
            }
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int e = base + u * TC_UW * 32;
                const int row = e / NGc, gl = e - row * NGc;
                if (e < total) sc[gl * TC_ROWS + row] = v[u];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

    float tot[4] = {0.f, 0.f, 0.f, 0.f};
    const int qd = warp & 3, hh = (warp >> 2) & 1;
    const int rho = TC_RQ * qd + lane;  // weight row of an unpack thread (lane < 31)
    const uint32_t tq = tbase + ((uint32_t)(32 * qd) << 16);

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
    } else if (warp >= TC_UW) {  // MMA issuers: issuer i owns buffer i and groups i, i + 4, ...
        const int iw = warp - TC_UW;
        if (lane == 0) {
            const uint32_t bbase = smem_u32(btile + iw * TC_BT);
            const uint32_t dcol = tbase + TC_DCOL + 16 * iw, acol = tbase + TC_ACOL + 64 * iw;
            int last = -1;
            for (int gi = iw; gi < NGc; gi += TC_IW) {
                if (!mbar_wait(&afull[iw], (gi / TC_NA) & 1)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; kk++) tc_mma(dcol, acol + 8 * kk, smem_desc(bbase + 256 * kk, 128, 0), kk > 0);
                tc_commit(&mdone[iw]);
                last = gi;
            }
            // the buffer's last commit must land before the tensor memory is released
            if (last >= 0 && !mbar_wait(&mdone[iw], (last / TC_NA) & 1)) failed = true;
        }
    } else {  // unpack warps
        auto epilogue = [&](int ge) {
            const int a = ge % TC_NA;
            if (4 * hh < m) {  // warp-uniform
                float d4[4];
                tc_ld4(tq + TC_DCOL + 16 * a + 4 * hh, d4);
                const float d = bf16_bits_to_f32(sc[ge * TC_ROWS + (lane < TC_RQ ? rho : 0)]);
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const float off = __shfl_sync(0xffffffffu, d4[j], 31);
                    tot[j] = fmaf(d, d4[j] - off, tot[j]);
                }
            }
        };
        for (int gi = 0; gi < NGc; gi++) {
            const int a = gi % TC_NA, st = gi >> 2, s = st % TC_NS, gl = gi & 3;
            if (gl == 0 && !mbar_wait(&full[s], (st / TC_NS) & 1)) {
                failed = true;
                break;
            }
            if (gi >= TC_NA) {  // the buffer's previous group: its sums, then the buffer is free
                if (!mbar_wait(&mdone[a], ((gi - TC_NA) / TC_NA) & 1)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                epilogue(gi - TC_NA);
            }
            const uint8_t* stg = stages + s * TC_STAGE;
            if (warp < m) {  // B tile row j = warp: x/s for the group's 128 columns, TMEM column order
                const int col = 128 * gl + 4 * lane, b = col >> 8, c = col & 255;
                const uint2 v = *reinterpret_cast<const uint2*>(stg + TC_CODES + ((b * m + warp) * 256 + c) * 2);
                const int i = lane >> 3, w = lane & 7;
                const float sv = i == 0 ? 128.f : (i == 1 ? 32.f : 8.f);  // 1/s of sub-block i
                const __nv_bfloat162 f = __floats2bfloat162_rn(sv, sv);
                const uint32_t lo = bf162_bits(__hmul2(bits_bf162(__byte_perm(v.x, v.y, 0x5410)), f));
                const uint32_t hi = bf162_bits(__hmul2(bits_bf162(__byte_perm(v.x, v.y, 0x7632)), f));
                *reinterpret_cast<uint2*>(btile + a * TC_BT + (2 * w + (i >> 1)) * 128 + warp * 16 + (i & 1) * 8) =
                    make_uint2(lo, hi);
            }
            uint4 cw;
            if (lane < TC_RQ)
                cw = *reinterpret_cast<const uint4*>(stg + rho * 128 + (((2 * gl + hh) ^ (rho & 7)) << 4));
            else
                cw = make_uint4(0xAAAAAAAAu, 0xAAAAAAAAu, 0xAAAAAAAAu, 0xAAAAAAAAu);  // every code 2
            uint32_t r[32];
            unpack_group(cw, r);
            tc_st32(tq + TC_ACOL + 64 * a + 32 * hh, r);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&afull[a]);
                if (gl == 3 || gi == NGc - 1) mbar_arrive(&empty[s]);
            }
        }
        if (!failed) {
            for (int ge = NGc - TC_NA > 0 ? NGc - TC_NA : 0; ge < NGc; ge++) {
                if (!mbar_wait(&mdone[ge % TC_NA], (ge / TC_NA) & 1)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                epilogue(ge);
            }
        }
        tc_fence_before();
    }
    if (failed) atomicOr(&g_gemv_tc_status, 1u);

    // ------------------------------------------------------------------ partial sums -> y
    const bool owner = warp < TC_UW && lane < TC_RQ && rho < R;
    __syncwarp();
    if (csplit > 1) {
        if (owner) {
#pragma unroll
            for (int j = 0; j < 4; j++)
                if (4 * hh + j < m) red[(4 * hh + j) * TC_ROWS + rho] = tot[j];
        }
        cluster_sync_all();
        if (rank == 0 && owner) {
            for (int q = 1; q < csplit; q++) {
#pragma unroll
                for (int j = 0; j < 4; j++)
                    if (4 * hh + j < m) tot[j] += ld_cluster_f32(&red[(4 * hh + j) * TC_ROWS + rho], (uint32_t)q);
            }
        }
    }
    if (rank == 0 && owner) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if (4 * hh + j < m) {
                const __nv_bfloat16 bv = __float2bfloat16_rn(tot[j]);
                y[(size_t)(4 * hh + j) * n + r0 + rho] = *reinterpret_cast<const uint16_t*>(&bv);
            }
        }
    }
    if (csplit > 1) cluster_sync_all();  // peers keep their shared memory until the leader has read it
    __syncthreads();
    if (warp == TC_UW) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "n"(TC_TMEM_COLS));
    }
}

// Launches the tcgen05 GEMV for an already validated weight (k > 0, n > 0, 1 <= m <= 8).
int launch_q2_gemv_tc(const uint16_t* x, const bq_q2_weight* w, uint16_t* y, uint32_t m, cudaStream_t stream,
                      const char* who) {
    const int n = (int)w->n, k = (int)w->k, group = (int)w->group;
    const int NG = k / 128;
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
    const int ngmax = (NG + csplit - 1) / csplit;
    const size_t smem = 1024 + (size_t)TC_NS * TC_STAGE + TC_NA * TC_BT + 8 * TC_ROWS * 4 +
                        (((size_t)ngmax * TC_ROWS + 7) & ~size_t(7)) * 2 + (2 * TC_NS + 2 * TC_NA) * 8 + 16;
    if (smem > (size_t)TC_SMEM_LIMIT)
        return fail(BQ_ERR_INVALID, "%s: k = %d needs %zu bytes of shared memory for its scales", who, k, smem);

    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 63;
    if ((size_t)configured[dev] < smem) {
        if (cudaFuncSetAttribute(q2_gemv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: cannot reserve %zu bytes of shared memory", who, smem);
        configured[dev] = (int)smem;
    }

    const uint8_t* codes = static_cast<const uint8_t*>(w->data);
    const uint16_t* scales = reinterpret_cast<const uint16_t*>(codes + (size_t)n * (k / 4));
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
    const cudaError_t e = cudaLaunchKernelEx(&cfg, q2_gemv_tc_kernel, cmap_hi, cmap_lo, xmap, scales, y, (int)m, n, k,
                                             group, nclus, csplit, rows_hi, ngmax);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction ? BQ_ERR_UNSUPPORTED
                                                                                                : BQ_ERR_LAUNCH,
                    "%s: launch failed: %s", who, cudaGetErrorString(e));
    }
    return BQ_OK;
}

}  // namespace bq8
