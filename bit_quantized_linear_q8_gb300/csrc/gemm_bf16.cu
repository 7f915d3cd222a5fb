// gemm_bf16.cu -- dense BF16 GEMM on the tcgen05 tensor cores: out[m, n] = a[m, k] @ w[n, k]^T.
//
// Source: init_q2.rs `qkvz_q2_prefill_gemm`, the fallback branch: `dequant_q2_0_gn_to_bf16`
// writes the weight as BF16 and `dense_gemm_bf16_pipelined` multiplies it with the BF16
// activations (fp32 accumulation, BF16 store).
//
// Design (GB300, sm_103a).  A plain tiled GEMM on the fifth-generation tensor cores:
//  * Tile 128 (m) x 256 (n), K step 64.  Both operands are K-major BF16 in global memory and
//    arrive by TMA with the 128-byte swizzle (a box row is 64 values = 128 bytes), four
//    stages of 16 KB (a) + 32 KB (w) in shared memory; the MMAs read them through
//    shared-memory descriptors (swizzle 128B, 8-row groups 1024 bytes apart, each K16 slice
//    32 bytes further into the swizzle atom).
//  * Persistent grid: one CTA per SM (at most one per tile) walks the tiles id = blockIdx.x,
//    + gridDim.x, ..., m tiles varying fastest.
//  * Two accumulators (128 lanes x 256 fp32 columns each, all 512 tensor-memory columns):
//    tile i of a CTA accumulates into buffer i % 2, so the epilogue of one tile overlaps the
//    MMAs of the next.
//  * Warp 1 (one lane) streams the K steps of all the CTA's tiles through the stage ring
//    without a break at tile boundaries; warp 0 allocates tensor memory and one lane issues
//    the M128 N256 K16 MMAs (four per K step), committing each step to the stage's `empty`
//    barrier and each tile's last step to the buffer's `full` barrier; warps 4-7 (one
//    tensor-memory lane quadrant each, one output row per thread) read a finished buffer
//    with tcgen05.ld, store BF16 and hand the buffer back through its `empty` barrier.
//  * Every wait is bounded; a wait that gives up raises the CTA's abort flag and the status
//    word, and the kernel winds down (the MMA warp still waits for its own MMAs before the
//    tensor memory is freed).
#include "common.cuh"

namespace bq8 {

static __device__ unsigned int g_gemm_status;

unsigned int gemm_bf16_status_take() {
    unsigned int v = 0, zero = 0;
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof v);
    cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof zero);
    return v;
}

constexpr int GB_BM = 128;
constexpr int GB_BN = 256;
constexpr int GB_BK = 64;
constexpr int GB_NS = 4;                               // pipeline stages
constexpr uint32_t GB_ASTAGE = GB_BM * GB_BK * 2;      // 16 KB
constexpr uint32_t GB_BSTAGE = GB_BN * GB_BK * 2;      // 32 KB
constexpr uint32_t GB_STAGE = GB_ASTAGE + GB_BSTAGE;
constexpr int GB_THREADS = 8 * 32;
constexpr uint32_t GB_TMEM_COLS = 512;                 // two 256-column accumulators
constexpr uint32_t GB_WAIT_LIMIT = 1u << 20;           // try_waits before a wait gives up
constexpr size_t GB_SMEM = 1024 + (size_t)GB_NS * GB_STAGE + (2 * GB_NS + 5) * 8 + 16;
static_assert(GB_SMEM <= 227 * 1024, "shared memory budget");

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bit 4), A and B BF16 (bits 7-9,
// 10-12), both K-major (bits 15, 16 clear), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t GB_IDESC =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(GB_BN >> 3) << 17) | ((uint32_t)(GB_BM >> 4) << 24);

// Shared-memory matrix descriptor for a K-major tile with the 128-byte swizzle: start address,
// leading byte offset 16 (unused by this layout), stride byte offset 1024 (one 8-row group of
// 128-byte rows), descriptor version bit 46, swizzle mode 2 (128 bytes) at bits 61-63.
__device__ __forceinline__ uint64_t gb_desc(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// D[tmem] (+)= A[smem] * B[smem]^T, M128 N256 K16, BF16 in, fp32 accumulate.
__device__ __forceinline__ void gb_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %3, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n}\n" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(accumulate), "r"(GB_IDESC));
}

__device__ __forceinline__ void gb_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool gb_try(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait that also gives up as soon as another thread of the CTA has raised `abort`.
__device__ __forceinline__ bool gb_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    for (uint32_t it = 0; it < GB_WAIT_LIMIT; it++) {
        if (gb_try(bar, parity)) return true;
        if (*abort) return false;
    }
    *abort = 1;
    atomicOr(&g_gemm_status, 1u);
    return false;
}

__device__ __forceinline__ void gb_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// (Launch bounds of 256 threads: eight warps, two per SM sub-partition.)
__global__ void __launch_bounds__(GB_THREADS, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapW,
                        uint16_t* __restrict__ out, int m, int n, int k, int ntm, int ntiles) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = align1024(smem_raw);  // [stage][a 128 x 64 | w 256 x 64] BF16, 128-byte swizzle
    uint64_t* full = reinterpret_cast<uint64_t*>(stages + GB_NS * GB_STAGE);
    uint64_t* empty = full + GB_NS;
    uint64_t* accf = empty + GB_NS;  // [2] accumulator buffer holds a finished tile
    uint64_t* acce = accf + 2;       // [2] accumulator buffer read out by the epilogue
    uint64_t* done = acce + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int S = k / GB_BK;
    const int G = gridDim.x;
    // tile id -> (m0, n0) with m tiles varying fastest: the tiles in flight at once (ids
    // i G .. (i + 1) G - 1) share few weight tiles, and the activations stay in L2
    auto tile_m0 = [&](int id) { return (id % ntm) * GB_BM; };
    auto tile_n0 = [&](int id) { return (id / ntm) * GB_BN; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < GB_NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 4);  // one arrival per epilogue warp
        }
        mbar_init(done, 1);
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "n"(GB_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tbase = *tslot;

    if (warp == 1) {
        // ---------------------------------------------------------------- TMA producer
        // one continuous stream of K steps over the CTA's tiles
        if (lane == 0) {
            int64_t it = 0;
            bool ok = true;
            for (int id = blockIdx.x; id < ntiles && ok; id += G) {
                const int m0 = tile_m0(id), n0 = tile_n0(id);
                for (int ks = 0; ks < S; ks++, it++) {
                    const int st = (int)(it % GB_NS);
                    if (it >= GB_NS && !gb_wait(&empty[st], (uint32_t)((it / GB_NS) - 1) & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = stages + (size_t)st * GB_STAGE;
                    mbar_arrive_expect_tx(&full[st], GB_STAGE);
                    tma_load_2d(dst, &mapA, ks * GB_BK * 2, m0, &full[st]);
                    tma_load_2d(dst + GB_ASTAGE, &mapW, ks * GB_BK * 2, n0, &full[st]);
                }
            }
            // wind down: every copy requested must have landed before the CTA exits
            for (int64_t j = it > GB_NS ? it - GB_NS : 0; j < it; j++)
                if (!mbar_wait_suspend(&full[j % GB_NS], (uint32_t)(j / GB_NS) & 1u)) atomicOr(&g_gemm_status, 2u);
        }
        __syncwarp();
    } else if (warp == 0) {
        // ---------------------------------------------------------------- MMA issuer
        // tile i of the CTA accumulates into buffer i % 2 (columns 256 (i % 2) ..) once the
        // epilogue has read out tile i - 2
        if (lane == 0) {
            int64_t it = 0;
            bool ok = true;
            int ti = 0;
            for (int id = blockIdx.x; id < ntiles && ok; id += G, ti++) {
                const int buf = ti & 1;
                if (ti >= 2 && !gb_wait(&acce[buf], (uint32_t)((ti >> 1) - 1) & 1u, abort)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tbase + (uint32_t)(buf * GB_BN);
                for (int ks = 0; ks < S; ks++, it++) {
                    const int st = (int)(it % GB_NS);
                    if (!gb_wait(&full[st], (uint32_t)(it / GB_NS) & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t abase = smem_u32(stages + (size_t)st * GB_STAGE);
                    const uint32_t bbase = abase + GB_ASTAGE;
#pragma unroll
                    for (int kk = 0; kk < GB_BK / 16; kk++)
                        gb_mma(d, gb_desc(abase + 32u * kk), gb_desc(bbase + 32u * kk), (ks | kk) != 0);
                    gb_commit(&empty[st]);  // the stage is free once these MMAs have read it
                }
                gb_commit(&accf[buf]);  // the tile's accumulator is complete once its MMAs are
            }
            gb_commit(done);  // completes once every MMA issued above has finished
            if (!mbar_wait_suspend(done, 0)) atomicOr(&g_gemm_status, 2u);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- epilogue
        // warp w reads tensor-memory lanes 32 (w % 4) .. + 31: output rows m0 + 32 (w % 4) + lane
        const int qd = warp & 3;
        const bool vec = (n & 7) == 0;
        int ti = 0;
        for (int id = blockIdx.x; id < ntiles; id += G, ti++) {
            const int buf = ti & 1;
            bool ok = gb_wait(&accf[buf], (uint32_t)(ti >> 1) & 1u, abort);
            ok = __all_sync(0xffffffffu, ok && !*abort) != 0;
            if (!ok) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int m0 = tile_m0(id), n0 = tile_n0(id);
            const int row = m0 + 32 * qd + lane;
            const uint32_t tq = tbase + ((uint32_t)(32 * qd) << 16) + (uint32_t)(buf * GB_BN);
#pragma unroll 1
            for (int c = 0; c < GB_BN / 32; c++) {
                const int col0 = n0 + 32 * c;
                if (col0 >= n) break;  // warp-uniform
                uint32_t v[32];
                gb_ld32(tq + 32u * c, v);
                if (row >= m) continue;
                uint16_t* dst = out + (size_t)row * n + col0;
                if (vec && col0 + 32 <= n) {
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        uint4 o;
                        o.x = bf162_bits(__floats2bfloat162_rn(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])));
                        o.y = bf162_bits(__floats2bfloat162_rn(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])));
                        o.z = bf162_bits(__floats2bfloat162_rn(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])));
                        o.w = bf162_bits(__floats2bfloat162_rn(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                        *reinterpret_cast<uint4*>(dst + 8 * q) = o;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e++) {
                        if (col0 + e < n) {
                            const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[e]));
                            dst[e] = *reinterpret_cast<const uint16_t*>(&b);
                        }
                    }
                }
            }
            // the buffer's reads are complete (tcgen05.ld waited): hand it back to the MMA warp
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[buf]);
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "n"(GB_TMEM_COLS));
    }
}

}  // namespace bq8

using namespace bq8;

// ---------------------------------------------------------------------------------------
// The CTA-pair form (m > 128): a cluster of two CTAs computes a 256 x 256 NB output tile (NB = 1
// or 2) with tcgen05.mma.cta_group::2 M256 N256 K16, NB MMAs per K16 step sharing the
// activation operand, issued by the even CTA.  CTA r of the pair holds rows 128 r .. 128 r + 127
// of the tile's activations and, for MMA h, weight rows 256 h + 128 r .. + 127 (the MMA's B
// operand is split along N across the pair), all at the same shared-memory offsets in both
// CTAs, and receives its 128 output rows x 256 NB columns in its own tensor memory.  Per K step
// each CTA stages 16 KB + 16 NB KB instead of 16 + 32 KB for a 128 x 256 tile, so the operand
// traffic through each SM's shared memory per MMA is a third lower (NB = 1) or half (NB = 2).
//  * Each CTA's producer lane streams its own halves through a ring (six stages, four at
//    NB = 2); both CTAs' copies complete their bytes on the even CTA's `full` barrier (the
//    cta_group::2 form of the TMA load), whose one arrival expects the pair's bytes per stage.
//  * NB = 1 keeps two accumulator buffers in tensor memory, so a tile's epilogue overlaps the
//    next tile's main loop; at NB = 2 the one 512-column accumulator is read out between tiles.
//  * The even CTA's MMA lane commits each K step to the `empty` barriers of both CTAs and each
//    tile's last step to both CTAs' accumulator barriers (multicast commits); both CTAs'
//    epilogue warps read their lanes and arrive (the odd CTA's remotely) on the even CTA's
//    accumulator-empty barrier, which counts eight warps.
//  * Tensor memory is allocated and freed for the pair (cta_group::2, one warp in each CTA).
//  * Every wait is bounded; both CTAs reach the final cluster barrier on every path.
constexpr int GP_BM = 128;                              // rows per CTA (256 per pair)
constexpr int GP_BN = 256;                              // output columns per MMA (N)
constexpr uint32_t GP_ASTAGE = GP_BM * GB_BK * 2;      // 16 KB
constexpr uint32_t GP_BSTAGE = (GP_BN / 2) * GB_BK * 2;  // 16 KB: this CTA's half of one MMA's weight rows
// D fp32, A and B BF16, both K-major, N = 256, M = 256 (the pair)
constexpr uint32_t GP_IDESC =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(GP_BN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
// A pair tile is 256 x 256 NB: NB MMAs of N = 256 per K16 step share the activation operand.
// NB = 1: six stages of 32 KB and two accumulator buffers (the epilogue of one tile overlaps
// the next tile's main loop).  NB = 2: four stages of 48 KB and one 512-column accumulator;
// a quarter fewer operand bytes per MMA, the epilogue not overlapped.
template <int NB>
struct GpCfg {
    static constexpr int NS = NB == 1 ? 6 : 4;
    static constexpr int NBUF = NB == 1 ? 2 : 1;  // accumulator buffers of 256 NB columns
    static constexpr uint32_t STAGE = GP_ASTAGE + NB * GP_BSTAGE;
    static constexpr size_t SMEM = 1024 + (size_t)NS * STAGE + (2 * NS + 5) * 8 + 16;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(NBUF * NB * GP_BN <= GB_TMEM_COLS, "tensor memory budget");
};

__device__ __forceinline__ uint32_t gp_cluster_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void gp_arrive_cluster(uint32_t addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
// 2-D TMA tile load into this CTA's shared memory whose bytes complete on `bar_cluster`, a
// barrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void gp_tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void gp_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void gp_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((uint16_t)3)
        : "memory");
}
__device__ __forceinline__ bool gp_try_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, "
        "p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Bounded wait with cluster-scope acquire (for barriers that receive remote arrivals).
__device__ __forceinline__ bool gp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    for (uint32_t it = 0; it < GB_WAIT_LIMIT; it++) {
        if (gp_try_cluster(bar, parity)) return true;
        if (*abort) return false;
    }
    *abort = 1;
    atomicOr(&g_gemm_status, 1u);
    return false;
}

template <int NB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GB_THREADS, 1)
    gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapW,
                          uint16_t* __restrict__ out, int m, int n, int k, int ntm, int ntiles) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int GP_NS = GpCfg<NB>::NS, NBUF = GpCfg<NB>::NBUF;
    constexpr uint32_t GP_STAGE = GpCfg<NB>::STAGE;
    uint8_t* stages = align1024(smem_raw);  // [stage][a 128 x 64 | NB x w 128 x 64] BF16, 128-byte swizzle
    uint64_t* full = reinterpret_cast<uint64_t*>(stages + GP_NS * GP_STAGE);
    uint64_t* empty = full + GP_NS;
    uint64_t* accf = empty + GP_NS;  // [2] accumulator buffer holds a finished tile (both CTAs)
    uint64_t* acce = accf + 2;       // [2] both CTAs' epilogues have read the buffer (even CTA)
    uint64_t* done = acce + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);

    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int S = k / GB_BK;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    auto tile_m0 = [&](int id) { return (id % ntm) * (2 * GP_BM); };
    auto tile_n0 = [&](int id) { return (id / ntm) * (GP_BN * NB); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < GP_NS; s++) {
            mbar_init(&full[s], 1);  // the even CTA's: one arrival expecting both CTAs' bytes
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 8);  // four epilogue warps in each CTA (used on the even CTA)
        }
        mbar_init(done, 1);
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "n"(GB_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    gp_cluster_sync();  // both CTAs' barriers exist before any remote arrive or MMA
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tbase = *tslot;

    if (warp == 1) {
        // ---------------------------------------------------------------- TMA producer (each CTA)
        if (lane == 0) {
            int64_t it = 0;
            bool ok = true;
            for (int id = pair; id < ntiles && ok; id += npairs) {
                const int ma0 = tile_m0(id) + GP_BM * (int)rank, nb0 = tile_n0(id) + (GP_BN / 2) * (int)rank;
                for (int ks = 0; ks < S; ks++, it++) {
                    const int st = (int)(it % GP_NS);
                    // the stage is free in both CTAs once the pair's MMAs of step it - NS have read it
                    if (it >= GP_NS && !gb_wait(&empty[st], (uint32_t)((it / GP_NS) - 1) & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = stages + (size_t)st * GP_STAGE;
                    const uint32_t bar = gp_cluster_addr(&full[st], 0);
                    if (rank == 0) mbar_arrive_expect_tx(&full[st], 2 * GP_STAGE);
                    gp_tma_load_2d(dst, &mapA, ks * GB_BK * 2, ma0, bar);
#pragma unroll
                    for (int h = 0; h < NB; h++)  // MMA h's weight rows: output columns n0 + 256 h ..
                        gp_tma_load_2d(dst + GP_ASTAGE + h * GP_BSTAGE, &mapW, ks * GB_BK * 2, nb0 + GP_BN * h, bar);
                }
            }
            // wind down (even CTA): the last copies of both CTAs land before the pair passes its
            // final cluster barrier
            if (rank == 0)
                for (int64_t j = it > GP_NS ? it - GP_NS : 0; j < it; j++)
                    if (!mbar_wait_suspend(&full[j % GP_NS], (uint32_t)(j / GP_NS) & 1u)) atomicOr(&g_gemm_status, 2u);
        }
        __syncwarp();
    } else if (warp == 0 && rank == 0) {
        // ---------------------------------------------------------------- MMA issuer (even CTA)
        if (lane == 0) {
            int64_t it = 0;
            bool ok = true;
            int ti = 0;
            for (int id = pair; id < ntiles && ok; id += npairs, ti++) {
                const int buf = ti % NBUF;
                if (ti >= NBUF && !gp_wait(&acce[buf], (uint32_t)((ti / NBUF) - 1) & 1u, abort)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tbase + (uint32_t)(buf * GP_BN * NB);
                for (int ks = 0; ks < S; ks++, it++) {
                    const int st = (int)(it % GP_NS);
                    if (!gb_wait(&full[st], (uint32_t)(it / GP_NS) & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t abase = smem_u32(stages + (size_t)st * GP_STAGE);
                    const uint32_t bbase = abase + GP_ASTAGE;
#pragma unroll
                    for (int kk = 0; kk < GB_BK / 16; kk++)
#pragma unroll
                        for (int h = 0; h < NB; h++)
                            asm volatile(
                                "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
                                "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d + GP_BN * h),
                                "l"(gb_desc(abase + 32u * kk)), "l"(gb_desc(bbase + GP_BSTAGE * h + 32u * kk)),
                                "r"(GP_IDESC), "r"((uint32_t)(ks | kk)));
                    gp_commit_pair(&empty[st]);  // both CTAs' stage is free once these MMAs have read it
                }
                gp_commit_pair(&accf[buf]);  // both CTAs' accumulator rows are complete
            }
            gp_commit_pair(done);  // completes once every MMA issued above has finished
            if (!mbar_wait_suspend(done, 0)) atomicOr(&g_gemm_status, 2u);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- epilogue (each CTA)
        // warp w reads tensor-memory lanes 32 (w % 4) .. + 31: output rows m0 + 128 rank + 32 (w % 4) + lane
        const int qd = warp & 3;
        const bool vec = (n & 7) == 0;
        const uint32_t acce_addr0 = gp_cluster_addr(&acce[0], 0), acce_addr1 = gp_cluster_addr(&acce[1], 0);
        int ti = 0;
        for (int id = pair; id < ntiles; id += npairs, ti++) {
            const int buf = ti % NBUF;
            bool ok = gb_wait(&accf[buf], (uint32_t)(ti / NBUF) & 1u, abort);
            ok = __all_sync(0xffffffffu, ok && !*abort) != 0;
            if (!ok) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int m0 = tile_m0(id) + GP_BM * (int)rank, n0 = tile_n0(id);
            const int row = m0 + 32 * qd + lane;
            const uint32_t tq = tbase + ((uint32_t)(32 * qd) << 16) + (uint32_t)(buf * GP_BN * NB);
#pragma unroll 1
            for (int c = 0; c < GP_BN * NB / 32; c++) {
                const int col0 = n0 + 32 * c;
                if (col0 >= n) break;  // warp-uniform
                uint32_t v[32];
                gb_ld32(tq + 32u * c, v);
                if (row >= m) continue;
                uint16_t* dst = out + (size_t)row * n + col0;
                if (vec && col0 + 32 <= n) {
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        uint4 o;
                        o.x = bf162_bits(__floats2bfloat162_rn(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])));
                        o.y = bf162_bits(__floats2bfloat162_rn(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])));
                        o.z = bf162_bits(__floats2bfloat162_rn(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])));
                        o.w = bf162_bits(__floats2bfloat162_rn(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                        *reinterpret_cast<uint4*>(dst + 8 * q) = o;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e++) {
                        if (col0 + e < n) {
                            const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[e]));
                            dst[e] = *reinterpret_cast<const uint16_t*>(&b);
                        }
                    }
                }
            }
            // this warp's reads of the buffer are complete: tell the even CTA's MMA lane
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) gp_arrive_cluster(buf ? acce_addr1 : acce_addr0);
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    gp_cluster_sync();  // no remote arrive or MMA of the pair is outstanding past this point
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tbase), "n"(GB_TMEM_COLS));
    }
}

// The CTA-pair form for m > 128: one pair per two SMs walks the 256 x 256 NB tiles.
template <int NB>
static int launch_pair_nb(const uint16_t* a, const uint16_t* w, uint16_t* out, uint32_t m, uint32_t n, uint32_t k,
                          cudaStream_t stream, int dev, const char* who) {
    static int configured[64] = {};
    constexpr size_t smem = GpCfg<NB>::SMEM;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(gemm_bf16_pair_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: cannot reserve %zu bytes of shared memory", who, smem);
        configured[dev] = 1;
    }
    CUtensorMap ma, mw;
    int st = cached_tmap_2d_u8(&ma, a, (uint64_t)k * 2, m, (uint64_t)k * 2, 128, GP_BM, true, who);
    if (st) return st;
    if ((st = cached_tmap_2d_u8(&mw, w, (uint64_t)k * 2, n, (uint64_t)k * 2, 128, GP_BN / 2, true, who))) return st;
    const uint64_t ntiles64 = (uint64_t)((m + 2 * GP_BM - 1) / (2 * GP_BM)) * ((n + GP_BN * NB - 1) / (GP_BN * NB));
    if (ntiles64 >= (1ull << 31)) return fail(BQ_ERR_INVALID, "%s: too many output tiles", who);
    const int ntm = (int)((m + 2 * GP_BM - 1) / (2 * GP_BM));
    const int ntiles = (int)ntiles64;
    const int pairs_max = sm_count() / 2;
    const int npairs = ntiles < pairs_max ? ntiles : pairs_max;
    gemm_bf16_pair_kernel<NB><<<(unsigned)(2 * npairs), GB_THREADS, smem, stream>>>(ma, mw, out, (int)m, (int)n, (int)k,
                                                                                   ntm, ntiles);
    return check_launch(who);
}

// Both forms run a tile near the tensor pipe's rate, so the time is about rounds of tiles x
// tile width: the 512-wide form where its rounds x 2 do not exceed the 256-wide form's rounds
// (n = 16384: m = 512 and 4096 take it, m = 2048, 4 rounds against 7, does not).
static int launch_pair(const uint16_t* a, const uint16_t* w, uint16_t* out, uint32_t m, uint32_t n, uint32_t k,
                       cudaStream_t stream, int dev, const char* who) {
    const uint64_t ntm = (m + 2 * GP_BM - 1) / (2 * GP_BM), pairs = (uint64_t)(sm_count() / 2);
    auto rounds = [&](uint64_t bn) { return (ntm * ((n + bn - 1) / bn) + pairs - 1) / pairs; };
    if (2 * rounds(2 * GP_BN) <= rounds(GP_BN)) return launch_pair_nb<2>(a, w, out, m, n, k, stream, dev, who);
    return launch_pair_nb<1>(a, w, out, m, n, k, stream, dev, who);
}

extern "C" int dense_gemm_bf16(const uint16_t* a, const uint16_t* w, uint16_t* out, uint32_t m, uint32_t n,
                               uint32_t k, bq_stream_t stream) {
    const char* who = "dense_gemm_bf16";
    if (m == 0 || n == 0) return ok();
    if (k == 0) {
        if (!out) return fail(BQ_ERR_INVALID, "%s: out is NULL", who);
        if (cudaMemsetAsync(out, 0, (size_t)m * n * 2, (cudaStream_t)stream) != cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: memset failed", who);
        return ok();
    }
    if (k % GB_BK != 0) return fail(BQ_ERR_INVALID, "%s: k = %u, must be a multiple of %d", who, k, GB_BK);
    if (m >= (1u << 30) || n >= (1u << 30) || (uint64_t)k * 2 >= (1ull << 32))
        return fail(BQ_ERR_INVALID, "%s: shape too large", who);
    if (!a || !w || !out || !aligned16(a) || !aligned16(w) || !aligned16(out))
        return fail(BQ_ERR_INVALID, "%s: a, w and out must be non-NULL and 16-byte aligned", who);
    static int configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64) dev = 63;
    if (m > (uint32_t)GB_BM) return launch_pair(a, w, out, m, n, k, (cudaStream_t)stream, dev, who);
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(gemm_bf16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GB_SMEM) !=
            cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: cannot reserve %zu bytes of shared memory", who, GB_SMEM);
        configured[dev] = 1;
    }
    // both operands as byte matrices with 128-byte (64-value) box rows
    CUtensorMap ma, mw;
    int st = cached_tmap_2d_u8(&ma, a, (uint64_t)k * 2, m, (uint64_t)k * 2, 128, GB_BM, true, who);
    if (st) return st;
    if ((st = cached_tmap_2d_u8(&mw, w, (uint64_t)k * 2, n, (uint64_t)k * 2, 128, GB_BN, true, who))) return st;
    const uint64_t ntiles64 = (uint64_t)((m + GB_BM - 1) / GB_BM) * ((n + GB_BN - 1) / GB_BN);
    if (ntiles64 >= (1ull << 31)) return fail(BQ_ERR_INVALID, "%s: too many output tiles", who);
    const int ntm = (int)((m + GB_BM - 1) / GB_BM);
    const int ntiles = (int)ntiles64;
    const int grid = ntiles < sm_count() ? ntiles : sm_count();  // persistent: one CTA per SM
    gemm_bf16_tc_kernel<<<(unsigned)grid, GB_THREADS, GB_SMEM, (cudaStream_t)stream>>>(ma, mw, out, (int)m, (int)n,
                                                                                       (int)k, ntm, ntiles);
    return check_launch(who);
}
