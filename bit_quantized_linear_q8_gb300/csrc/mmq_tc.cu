// mmq_tc.cu -- Q2_0 MMQ on the tcgen05 tensor cores: q8_1 activations x Q2_0 weights, BF16 store.
//
// Source: init_q2.rs `qkvz_q2_prefill_gemm` (MMQ route, group 128):
//     out[m, n] = sum_k (d_a q)[m, k] * (d_w (c - 2))[n, k]
// with q8_1 activation values d_a * q (one fp32 d_a per 32 values) and Q2_0 weights
// d_w * (c - 2) (one BF16 d_w per 128 values).
//
// Design (GB300, sm_103a).  The tcgen05 tensor cores of sm_103a have no int8 kind, so the
// contraction runs on the BF16 kind (kind::f16, fp32 accumulation in tensor memory) with
// operands that carry the quantised values:
//  * Weights: d_w * (c - 2) is exact in BF16 (a BF16 scale times -2, -1, 0 or 1), so the group
//    scale and the code offset are part of the operand and nothing per group is left over.
//  * Activations: v = d_a * q (fp32) is split into hi = bf16(v) and lo = bf16(v - hi); hi + lo
//    equals v to 2^-17 relative.  Each K step multiplies both halves with the same weight
//    operand into the same accumulator (two MMAs per K16), so the per-32 activation scale is
//    inside the operand too and the accumulator is read only once, at the end.
//  Every product of two BF16 values is exact in fp32; the sums are the tensor cores' fp32.
//
//  * Tile 128 (m) x 256 (n), K step 64.  Tensor memory holds the accumulator (256 columns)
//    and four stages of the activation operand (A from tensor memory: lane = row, column j =
//    K elements 2j, 2j+1; 32 columns hi + 32 columns lo per stage).  Shared memory holds four
//    stages of the weight operand (256 x 64 BF16, no-swizzle K-major 8 x 16-byte core
//    matrices) and a five-step ring of the packed inputs.  No global scratch.
//  * Warp 13 streams the packed inputs of each K step into the ring with TMA: the q8_1 codes
//    (a [run][row][16 B] box, so that a warp reads 32 consecutive rows), the q8_1 (d, s)
//    pairs and the 2-bit weight codes.  The group scales (one BF16 per 128 columns) are read
//    one pack block ahead with plain loads.
//  * Warp 0 allocates tensor memory; one lane issues M128 N256 K16 MMAs (8 per K step) and
//    commits each step to the stage's `empty` barrier.
//  * Warps 1-8 (two per tensor-memory lane quadrant, one activation row per thread, each
//    warp two of the step's four 16-byte code runs) expand the q8_1 codes into the hi/lo
//    operand with tcgen05.st, then run the epilogue (tcgen05.ld -> BF16 -> global).
//  * Warps 9-12 (two weight rows per thread) expand the 2-bit codes into shared memory.
//  * K order inside a step: the 64 columns of step s are those of pack block s/2 with
//    in-block offsets 32i + 16(s%2) + l (i = 0..3, l = 0..15), and 32-bit operand word
//    q = 16(i/2) + 4u + 2(i%2) + j holds offsets (l = 4u + j, l = 4u + j + 2).  In the Q2
//    layout (byte l of a pack block holds the codes of offsets 32i + l in bits 2i) those two
//    codes sit 16 bits apart in one 32-bit word of packed codes, so a mask and one LOP3 place
//    a pair of codes into a BF16 pair; the activation warp that owns runs i = 2hf, 2hf + 1
//    writes the contiguous words 16hf .. 16hf + 15.  Both operands use this order, so the
//    contraction is unchanged.
//  * Every wait is bounded; a wait that gives up raises the CTA's abort flag and the status
//    word, and the kernel winds down (it still waits for its own MMAs before freeing tensor
//    memory).
#include "common.cuh"

namespace bq8 {

static __device__ unsigned int g_mmq_tc_status;

unsigned int mmq_tc_status_take() {
    unsigned int v = 0, zero = 0;
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(&v, g_mmq_tc_status, sizeof v);
    cudaMemcpyToSymbol(g_mmq_tc_status, &zero, sizeof zero);
    return v;
}

constexpr int QT_BM = 128;
constexpr int QT_BN = 256;
constexpr int QT_NS = 4;                         // operand stages (tensor memory and shared memory)
constexpr int QT_NR = 5;                         // ring stages of packed inputs
constexpr int QT_AWARP0 = 1;                     // warps 1..8: activation operand, epilogue
constexpr int QT_BWARP0 = 9;                     // warps 9..12: weight operand, two rows a thread
constexpr int QT_PWARP = 13;                     // TMA producer
constexpr int QT_THREADS = 14 * 32;
constexpr uint32_t QT_BSTAGE = QT_BN * 64 * 2;   // 32 KB of weight operand per stage
constexpr uint32_t QT_R_A = 0;                   // ring stage: q8_1 codes [4 runs][128 rows][16 B]
constexpr uint32_t QT_R_D = 8192;                // (d, s) pairs [2][128 rows][16 B]
constexpr uint32_t QT_R_B = 12288;               // weight codes [256 rows][16 B]
constexpr uint32_t QT_RSTAGE = 16384;
constexpr uint32_t QT_TMEM_COLS = 512;
constexpr uint32_t QT_ACOL = 256;                // first column of the activation stages
constexpr uint32_t QT_WAIT_LIMIT = 1u << 20;     // try_waits before a wait gives up (0.05-4 s)
static_assert(QT_ACOL + 64 * QT_NS <= QT_TMEM_COLS, "tensor memory budget");
static_assert(QT_BWARP0 == QT_AWARP0 + 8 && QT_PWARP == QT_BWARP0 + QT_BN / 64 && QT_THREADS == (QT_PWARP + 1) * 32,
              "warp roles");
constexpr size_t QT_SMEM = 1024 + (size_t)QT_NS * QT_BSTAGE + (size_t)QT_NR * QT_RSTAGE + (3 * QT_NS + 2 * QT_NR + 1) * 8 + 16;
static_assert(QT_SMEM <= 227 * 1024, "shared memory budget");

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bit 4), A and B BF16 (bits 7-9,
// 10-12), both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t QT_IDESC =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(QT_BN >> 3) << 17) | ((uint32_t)(QT_BM >> 4) << 24);

// Shared-memory matrix descriptor, no swizzle: 8-row x 16-byte core matrices, `lbo` bytes
// apart along K, `sbo` bytes apart along N; bit 46 is the descriptor version.
__device__ __forceinline__ uint64_t qt_smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// D[tmem] (+)= A[tmem] * B[smem]^T, M128 N256 K16, BF16 in, fp32 accumulate.
__device__ __forceinline__ void qt_mma(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %3, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n}\n" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(accumulate), "r"(QT_IDESC));
}

__device__ __forceinline__ void qt_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void qt_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void qt_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void qt_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void qt_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void qt_ld32(uint32_t taddr, uint32_t (&r)[32]) {
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

// One mbarrier.try_wait: the warp may be suspended in hardware until the phase completes or
// a system-dependent time limit (microseconds) passes; true once phase `parity` completed.
__device__ __forceinline__ bool qt_try(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait that also gives up as soon as another thread of the CTA has raised `abort`.
// (Every step's waits here last microseconds, so a suspending try_wait costs the pipeline
// nothing and frees issue slots that polling would take.)
__device__ __forceinline__ bool qt_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    for (uint32_t it = 0; it < QT_WAIT_LIMIT; it++) {
        if (qt_try(bar, parity)) return true;
        if (*abort) return false;
    }
    *abort = 1;
    atomicOr(&g_mmq_tc_status, 1u);
    return false;
}

// The same for a whole warp, with a warp-uniform answer (the callers go on to .sync.aligned
// tensor-memory instructions).
__device__ __forceinline__ bool qt_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort) {
    const bool ok = qt_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok) != 0;
}

// Two signed int8 codes (bytes b0 and b1 of `w`, biased by 0x80) times d, as fp32, split into
// a BF16 pair hi and a BF16 pair lo with hi + lo = d * q to 2^-17.
__device__ __forceinline__ void qt_split_pair(uint32_t wb, uint32_t sel0, uint32_t sel1, float d, uint32_t& hi,
                                              uint32_t& lo) {
    // 0x4B0000xx is the float 2^23 + xx; subtracting 2^23 + 128 leaves the signed code exactly.
    const float f0 = __uint_as_float(__byte_perm(wb, 0x4B000000u, sel0));
    const float f1 = __uint_as_float(__byte_perm(wb, 0x4B000000u, sel1));
    const float2 v = __fmul2_rn(__fadd2_rn(make_float2(f0, f1), make_float2(-8388736.0f, -8388736.0f)),
                                make_float2(d, d));
    hi = bf162_bits(__floats2bfloat162_rn(v.x, v.y));
    const float2 h = make_float2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xFFFF0000u));
    const float2 r = __fadd2_rn(v, make_float2(-h.x, -h.y));
    lo = bf162_bits(__floats2bfloat162_rn(r.x, r.y));
}

// -(128 + 2 * 4^f) as a BF16 pair: -130, -136, -160.
__device__ __forceinline__ __nv_bfloat162 qt_m_off(int f) {
    return bits_bf162(f == 0 ? 0xC302C302u : f == 1 ? 0xC308C308u : 0xC320C320u);
}

__device__ __forceinline__ uint32_t u4_get(const uint4& v, int u) {
    return u == 0 ? v.x : u == 1 ? v.y : u == 2 ? v.z : v.w;
}

// Epilogue of one activation row: accumulator columns 32c .. 32c + 31 for c in [c0, c1)
// (tensor-memory lane quadrant base tA) -> BF16 -> out[row][n0 + ...], guarding the m and n
// tails.  All lanes of the warp call it (tcgen05.ld is warp-wide); `ok` is warp-uniform.
__device__ __forceinline__ void qt_epilogue(uint32_t tA, int c0, int c1, int row, int m, int n, int n0, bool ok,
                                            uint16_t* __restrict__ out) {
    if (!ok) return;
    const bool vec = (n & 7) == 0;
#pragma unroll 1
    for (int c = c0; c < c1; c++) {
        const int col0 = n0 + 32 * c;
        if (col0 >= n) break;  // warp-uniform
        uint32_t v[32];
        qt_ld32(tA + 32u * c, v);
        if (row < m) {
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
    }
}

// (Launch bounds of 512 threads keep ptxas at <= 128 registers: 14 warps put four warps on
// one SM sub-partition, whose register file holds 16 K registers.)
__global__ void __launch_bounds__(512, 1)
    q2_mmq_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapD,
                     const __grid_constant__ CUtensorMap mapB, const uint16_t* __restrict__ wsc,
                     uint16_t* __restrict__ out, int m, int n, int k, int ntm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* bst = align1024(smem_raw);
    uint8_t* ring = bst + QT_NS * QT_BSTAGE;
    uint64_t* afull = reinterpret_cast<uint64_t*>(ring + QT_NR * QT_RSTAGE);
    uint64_t* bfull = afull + QT_NS;
    uint64_t* sempty = bfull + QT_NS;
    uint64_t* rfull = sempty + QT_NS;
    uint64_t* rempty = rfull + QT_NR;
    uint64_t* accfull = rempty + QT_NR;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(accfull + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // m tiles vary fastest: the CTAs resident at once share few weight tiles, each weight tile
    // is read from HBM once while the activations stay in L2
    const int m0 = (blockIdx.x % ntm) * QT_BM, n0 = (blockIdx.x / ntm) * QT_BN;
    const int S = k >> 6;  // K steps of 64
    const int G = k >> 7;  // groups of 128 (one BF16 scale each)

    if (threadIdx.x == 0) {
        for (int s = 0; s < QT_NS; s++) {
            mbar_init(&afull[s], 8 * 32);
            mbar_init(&bfull[s], 4 * 32);
            mbar_init(&sempty[s], 1);
        }
        for (int r = 0; r < QT_NR; r++) {
            mbar_init(&rfull[r], 1);
            mbar_init(&rempty[r], 12);  // one arrival per consuming warp
        }
        mbar_init(accfull, 1);
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "n"(QT_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    qt_fence_before();
    __syncthreads();
    qt_fence_after();
    const uint32_t tbase = *tslot;

    if (warp == QT_PWARP) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            for (int s = 0; s < S; s++) {
                const int r = s % QT_NR;
                if (s >= QT_NR && !qt_wait(&rempty[r], (uint32_t)((s / QT_NR) - 1) & 1u, abort)) break;
                const int pb = s >> 1, h = s & 1;
                uint8_t* dst = ring + r * QT_RSTAGE;
                mbar_arrive_expect_tx(&rfull[r], QT_RSTAGE);
                tma_load_3d(dst + QT_R_A, &mapA, 16 * h, m0, 4 * pb, &rfull[r]);
                tma_load_3d(dst + QT_R_D, &mapD, 0, m0, 2 * pb, &rfull[r]);
                tma_load_2d(dst + QT_R_B, &mapB, 32 * pb + 16 * h, n0, &rfull[r]);
            }
        }
        __syncwarp();
    } else if (warp == 0) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            for (int s = 0; s < S; s++) {
                const int st = s % QT_NS;
                const uint32_t par = (uint32_t)(s / QT_NS) & 1u;
                if (!qt_wait(&afull[st], par, abort) || !qt_wait(&bfull[st], par, abort)) break;
                qt_fence_after();
                const uint32_t bbase = smem_u32(bst + st * QT_BSTAGE);
                const uint32_t abase = tbase + QT_ACOL + 64u * st;
#pragma unroll
                for (int kk = 0; kk < 4; kk++) {
                    const uint64_t bd = qt_smem_desc(bbase + 256u * kk, 128u, 1024u);
                    qt_mma(tbase, abase + 8u * kk, bd, (s | kk) != 0);
                    qt_mma(tbase, abase + 32u + 8u * kk, bd, 1u);
                }
                qt_commit(&sempty[st]);
            }
            qt_commit(accfull);  // completes once every MMA issued above has finished
            if (!mbar_wait(accfull, 0)) atomicOr(&g_mmq_tc_status, 2u);
        }
        __syncwarp();
    } else if (warp < QT_BWARP0) {
        // ---------------------------------------------------------------- activation operand
        // Two warps per tensor-memory lane quadrant; warp half `hf` expands code runs
        // i = 2hf, 2hf + 1 (operand words 16hf .. 16hf + 15) of each step and later stores
        // output columns 128hf .. 128hf + 127.
        const int qd = warp & 3;  // tensor-memory lane quadrant this warp may access
        const int hf = (warp - QT_AWARP0) >> 2;
        const int lrow = 32 * qd + lane;  // row within the tile
        const uint32_t tA = tbase + ((uint32_t)(32 * qd) << 16);
        for (int s = 0; s < S; s++) {
            const int st = s % QT_NS, r = s % QT_NR;
            if (!qt_wait_warp(&rfull[r], (uint32_t)(s / QT_NR) & 1u, abort)) break;
            const uint8_t* rs = ring + r * QT_RSTAGE;
            uint4 cr[2];
#pragma unroll
            for (int ii = 0; ii < 2; ii++)
                cr[ii] = *reinterpret_cast<const uint4*>(rs + QT_R_A + (2 * hf + ii) * 2048 + lrow * 16);
            const float4 dp = *reinterpret_cast<const float4*>(rs + QT_R_D + hf * 2048 + lrow * 16);
            const float cd[2] = {dp.x, dp.z};  // d of q8_1 blocks 4(s/2) + 2hf, + 1
            __syncwarp();
            if (lane == 0) mbar_arrive(&rempty[r]);
            if (s >= QT_NS) {
                if (!qt_wait_warp(&sempty[st], (uint32_t)((s / QT_NS) - 1) & 1u, abort)) break;
                qt_fence_after();
            }
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int u = 0; u < 4; u++) {
#pragma unroll
                for (int ii = 0; ii < 2; ii++) {
                    const uint32_t wb = u4_get(cr[ii], u) ^ 0x80808080u;
                    // word 16hf + 4u + 2ii + j: offsets 4u + j (low half) and 4u + j + 2 (high half)
                    qt_split_pair(wb, 0x7540u, 0x7542u, cd[ii], hw[4 * u + 2 * ii], lw[4 * u + 2 * ii]);
                    qt_split_pair(wb, 0x7541u, 0x7543u, cd[ii], hw[4 * u + 2 * ii + 1], lw[4 * u + 2 * ii + 1]);
                }
            }
            const uint32_t tcol = tA + QT_ACOL + 64u * st + 16u * hf;
            qt_st16(tcol, hw);
            qt_st16(tcol + 32u, lw);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            qt_fence_before();
            mbar_arrive(&afull[st]);
        }
        // ---------------------------------------------------------------- epilogue
        bool ok = mbar_wait(accfull, 0);
        ok = __all_sync(0xffffffffu, ok && !*abort) != 0;
        qt_fence_after();
        qt_epilogue(tA, 4 * hf, 4 * hf + 4, m0 + lrow, m, n, n0, ok, out);
    } else {
        // ---------------------------------------------------------------- weight operand
        // Thread t expands weight rows t and t + 128 of the tile.
        const int bt = 32 * (warp - QT_BWARP0) + lane;
        const uint16_t* srow[2];
        bool nv[2];
        uint32_t cs[2], ns[2];
#pragma unroll
        for (int r = 0; r < 2; r++) {
            const int nr = n0 + bt + 128 * r;
            nv[r] = nr < n;
            srow[r] = wsc + (size_t)(nv[r] ? nr : 0) * G;
            cs[r] = nv[r] ? srow[r][0] : 0u;
            ns[r] = (nv[r] && G > 1) ? srow[r][1] : 0u;
        }
        for (int s = 0; s < S; s++) {
            const int st = s % QT_NS, rr = s % QT_NR;
            const int pb = s >> 1;
            if (s > 0 && (s & 1) == 0) {  // new pack block: its scale was loaded one block ago
#pragma unroll
                for (int r = 0; r < 2; r++) {
                    cs[r] = ns[r];
                    if (nv[r] && pb + 1 < G) ns[r] = srow[r][pb + 1];
                }
            }
            if (!qt_wait_warp(&rfull[rr], (uint32_t)(s / QT_NR) & 1u, abort)) break;
            const uint8_t* rs = ring + rr * QT_RSTAGE + QT_R_B;
            uint4 cp[2];
#pragma unroll
            for (int r = 0; r < 2; r++) cp[r] = *reinterpret_cast<const uint4*>(rs + (bt + 128 * r) * 16);
            __syncwarp();
            if (lane == 0) mbar_arrive(&rempty[rr]);
            if (s >= QT_NS) {
                if (!qt_wait_warp(&sempty[st], (uint32_t)((s / QT_NS) - 1) & 1u, abort)) break;
            }
#pragma unroll
            for (int r = 0; r < 2; r++) {
                const int row = bt + 128 * r;
                // Field i of a code byte (bits 2i, 2i + 1; i = 0..2 in place, i = 3 shifted to
                // i = 2) masked into the mantissa of 128 gives 128 + c 4^i; subtracting
                // 128 + 2 4^i and multiplying by d 4^-i gives d (c - 2), every step exact.
                const __nv_bfloat162 d0 = bits_bf162(cs[r] | (cs[r] << 16));
                const __nv_bfloat162 dsc[3] = {d0, __hmul2(d0, bits_bf162(0x3E803E80u)),   // d / 4
                                               __hmul2(d0, bits_bf162(0x3D803D80u))};      // d / 16
                uint8_t* dst = bst + st * QT_BSTAGE + (row >> 3) * 1024 + (row & 7) * 16;
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const uint32_t w0 = u4_get(cp[r], u);
                    const uint32_t w1 = __byte_perm(w0, 0u, 0x4341u);  // bytes 1, 3 -> 0, 2
                    uint32_t o[8];
#pragma unroll
                    for (int i = 0; i < 4; i++) {
#pragma unroll
                        for (int j = 0; j < 2; j++) {
                            // codes of offsets 4u + j and 4u + j + 2
                            const uint32_t wj = j ? w1 : w0;
                            const int f = i < 3 ? i : 2;
                            const uint32_t x = and_or(i < 3 ? wj : wj >> 2, 0x00030003u << (2 * f), 0x43004300u);
                            o[2 * i + j] = bf162_bits(__hmul2(__hadd2(bits_bf162(x), qt_m_off(f)), dsc[f]));
                        }
                    }
                    // words 4u + 2(i%2) + j of core matrix u (i < 2) and 4 + u (i >= 2)
                    *reinterpret_cast<uint4*>(dst + u * 128) = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4*>(dst + (4 + u) * 128) = make_uint4(o[4], o[5], o[6], o[7]);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&bfull[st]);
        }
    }

    qt_fence_before();
    __syncthreads();
    if (warp == 0) {
        qt_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "n"(QT_TMEM_COLS));
    }
}

// =====================================================================================
// Q4_K.  Source: q4k_mmq.rs `q4k_mmq_gemm` (C[m, n] = A[m, k] x W[n, k], BF16 store) with
// block_q4_K weights w = d sc_j q - dmin m_j (256 values, 144 bytes: fp16 d, fp16 dmin, 12
// bytes of 6-bit sc_j / m_j, 128 bytes of 4-bit codes; byte 32c + l holds value l of
// sub-block 2c in its low nibble and of sub-block 2c + 1 in its high nibble).
//
// The weight w (fp32: d sc_j q is exact, the difference rounds once) is not exact in BF16,
// so it is split like the activations: wh = bf16(w), wl = bf16(w - wh).  Three MMAs per
// K16 slice, A_hi B_hi + A_lo B_hi + A_hi B_lo, into one fp32 accumulator; the dropped
// A_lo B_lo term is below 2^-17 of each product.  The dmin m_j term is inside the operand.
//  * Tile 128 (m) x 256 (n), K step 64 (a quarter super-block: sub-blocks 2t, 2t + 1 whose
//    codes are the 32 bytes 16 + 32t of the block).  Natural K order within a step.
//  * Tensor memory: accumulator (256 columns) + four activation stages (hi, lo: 64 columns).
//    Shared memory: two weight stages (hi and lo halves, 2 x 32 KB) + a three-step TMA ring
//    (q8_1 codes, (d, s) pairs, the weight codes and the 16-byte block headers).
//  * Warp 0 issues the MMAs; warps 1-4 expand activations (one row per thread) and run the
//    epilogue; warps 5-12 expand weights (one row per thread); warp 13 is the TMA producer.
// =====================================================================================
constexpr int Q4T_NSA = 4;                       // activation stages (tensor memory)
constexpr int Q4T_NSB = 2;                       // weight stages (shared memory)
constexpr int Q4T_NR = 3;                        // ring stages
constexpr int Q4T_AWARP0 = 1, Q4T_BWARP0 = 5, Q4T_PWARP = 13;
constexpr int Q4T_THREADS = 14 * 32;
constexpr uint32_t Q4T_BHALF = QT_BN * 64 * 2;   // 32 KB: the hi or the lo half of a stage
constexpr uint32_t Q4T_BSTAGE = 2 * Q4T_BHALF;
constexpr uint32_t Q4T_R_A = 0;                  // q8_1 codes [4 runs][128 rows][16 B]
constexpr uint32_t Q4T_R_D = 8192;               // (d, s) pairs [128 rows][16 B]
constexpr uint32_t Q4T_R_Q = 10240;              // weight codes [2][256 rows][16 B]
constexpr uint32_t Q4T_R_H = 18432;              // block headers [256 rows][16 B]
constexpr uint32_t Q4T_RSTAGE = 22528;
static_assert(QT_ACOL + 64 * Q4T_NSA <= QT_TMEM_COLS, "tensor memory budget");
static_assert(Q4T_BWARP0 == Q4T_AWARP0 + 4 && Q4T_PWARP == Q4T_BWARP0 + QT_BN / 32 && Q4T_THREADS == (Q4T_PWARP + 1) * 32,
              "warp roles");
constexpr size_t Q4T_SMEM = 1024 + (size_t)Q4T_NSB * Q4T_BSTAGE + (size_t)Q4T_NR * Q4T_RSTAGE +
                            (2 * Q4T_NSA + 2 * Q4T_NSB + 2 * Q4T_NR + 1) * 8 + 16;
static_assert(Q4T_SMEM <= 227 * 1024, "shared memory budget");

// Byte i (0..11) of the 12 scale bytes held in the words a, b, c.
__device__ __forceinline__ int q4t_sbyte(uint32_t a, uint32_t b, uint32_t c, int i) {
    const uint32_t w = i < 4 ? a : (i < 8 ? b : c);
    return (int)((w >> (8 * (i & 3))) & 0xFFu);
}

// 6-bit scale and min of sub-block j from the 12 scale bytes (the block_q4_K packing).
__device__ __forceinline__ void q4t_scale_min(uint32_t a, uint32_t b, uint32_t c, int j, int& sc, int& mn) {
    if (j < 4) {
        sc = q4t_sbyte(a, b, c, j) & 63;
        mn = q4t_sbyte(a, b, c, j + 4) & 63;
    } else {
        sc = (q4t_sbyte(a, b, c, j + 4) & 15) | ((q4t_sbyte(a, b, c, j - 4) >> 6) << 4);
        mn = (q4t_sbyte(a, b, c, j + 4) >> 4) | ((q4t_sbyte(a, b, c, j) >> 6) << 4);
    }
}

// Two 4-bit codes (bytes b0, b0 + 1 of nib, each 0..15) -> w = q D - M (fp32), split into
// a BF16 pair hi and a BF16 pair lo.
__device__ __forceinline__ void q4t_split_pair(uint32_t nib, uint32_t sel0, uint32_t sel1, float D, float M,
                                               uint32_t& hi, uint32_t& lo) {
    const float f0 = __uint_as_float(__byte_perm(nib, 0x4B000000u, sel0));  // 2^23 + q
    const float f1 = __uint_as_float(__byte_perm(nib, 0x4B000000u, sel1));
    const float2 q = __fadd2_rn(make_float2(f0, f1), make_float2(-8388608.0f, -8388608.0f));
    const float2 w = __ffma2_rn(q, make_float2(D, D), make_float2(-M, -M));
    hi = bf162_bits(__floats2bfloat162_rn(w.x, w.y));
    const float2 h = make_float2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xFFFF0000u));
    const float2 r = __fadd2_rn(w, make_float2(-h.x, -h.y));
    lo = bf162_bits(__floats2bfloat162_rn(r.x, r.y));
}

__global__ void __launch_bounds__(512, 1)
    q4k_mmq_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapD,
                      const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapH,
                      uint16_t* __restrict__ out, int m, int n, int k, int ntm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* bst = align1024(smem_raw);
    uint8_t* ring = bst + Q4T_NSB * Q4T_BSTAGE;
    uint64_t* afull = reinterpret_cast<uint64_t*>(ring + Q4T_NR * Q4T_RSTAGE);
    uint64_t* aempty = afull + Q4T_NSA;
    uint64_t* bfull = aempty + Q4T_NSA;
    uint64_t* bempty = bfull + Q4T_NSB;
    uint64_t* rfull = bempty + Q4T_NSB;
    uint64_t* rempty = rfull + Q4T_NR;
    uint64_t* accfull = rempty + Q4T_NR;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(accfull + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // m tiles vary fastest: the CTAs resident at once share few weight tiles, each weight tile
    // is read from HBM once while the activations stay in L2
    const int m0 = (blockIdx.x % ntm) * QT_BM, n0 = (blockIdx.x / ntm) * QT_BN;
    const int S = k >> 6;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Q4T_NSA; s++) {
            mbar_init(&afull[s], 4 * 32);
            mbar_init(&aempty[s], 1);
        }
        for (int s = 0; s < Q4T_NSB; s++) {
            mbar_init(&bfull[s], 8 * 32);
            mbar_init(&bempty[s], 1);
        }
        for (int r = 0; r < Q4T_NR; r++) {
            mbar_init(&rfull[r], 1);
            mbar_init(&rempty[r], 12);  // one arrival per consuming warp
        }
        mbar_init(accfull, 1);
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "n"(QT_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    qt_fence_before();
    __syncthreads();
    qt_fence_after();
    const uint32_t tbase = *tslot;

    if (warp == Q4T_PWARP) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            for (int s = 0; s < S; s++) {
                const int r = s % Q4T_NR;
                if (s >= Q4T_NR && !qt_wait(&rempty[r], (uint32_t)((s / Q4T_NR) - 1) & 1u, abort)) break;
                const int sb = s >> 2, t = s & 3;
                uint8_t* dst = ring + r * Q4T_RSTAGE;
                mbar_arrive_expect_tx(&rfull[r], Q4T_RSTAGE);
                tma_load_3d(dst + Q4T_R_A, &mapA, 0, m0, 4 * s, &rfull[r]);
                tma_load_2d(dst + Q4T_R_D, &mapD, 16 * s, m0, &rfull[r]);
                tma_load_3d(dst + Q4T_R_Q, &mapQ, 0, n0, 9 * sb + 1 + 2 * t, &rfull[r]);
                tma_load_3d(dst + Q4T_R_H, &mapH, 0, n0, 9 * sb, &rfull[r]);
            }
        }
        __syncwarp();
    } else if (warp == 0) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            for (int s = 0; s < S; s++) {
                const int sa = s % Q4T_NSA, sbi = s % Q4T_NSB;
                if (!qt_wait(&afull[sa], (uint32_t)(s / Q4T_NSA) & 1u, abort) ||
                    !qt_wait(&bfull[sbi], (uint32_t)(s / Q4T_NSB) & 1u, abort))
                    break;
                qt_fence_after();
                const uint32_t bhi = smem_u32(bst + sbi * Q4T_BSTAGE), blo = bhi + Q4T_BHALF;
                const uint32_t abase = tbase + QT_ACOL + 64u * sa;
#pragma unroll
                for (int kk = 0; kk < 4; kk++) {
                    const uint64_t dh = qt_smem_desc(bhi + 256u * kk, 128u, 1024u);
                    const uint64_t dl = qt_smem_desc(blo + 256u * kk, 128u, 1024u);
                    qt_mma(tbase, abase + 8u * kk, dh, (s | kk) != 0);   // A_hi B_hi
                    qt_mma(tbase, abase + 32u + 8u * kk, dh, 1u);        // A_lo B_hi
                    qt_mma(tbase, abase + 8u * kk, dl, 1u);              // A_hi B_lo
                }
                qt_commit(&aempty[sa]);
                qt_commit(&bempty[sbi]);
            }
            qt_commit(accfull);  // completes once every MMA issued above has finished
            if (!mbar_wait(accfull, 0)) atomicOr(&g_mmq_tc_status, 2u);
        }
        __syncwarp();
    } else if (warp < Q4T_BWARP0) {
        // ---------------------------------------------------------------- activation operand
        const int qd = warp & 3;
        const int lrow = 32 * qd + lane;
        const uint32_t tA = tbase + ((uint32_t)(32 * qd) << 16);
        for (int s = 0; s < S; s++) {
            const int sa = s % Q4T_NSA, r = s % Q4T_NR;
            if (!qt_wait_warp(&rfull[r], (uint32_t)(s / Q4T_NR) & 1u, abort)) break;
            const uint8_t* rs = ring + r * Q4T_RSTAGE;
            uint4 cr[4];
#pragma unroll
            for (int i = 0; i < 4; i++) cr[i] = *reinterpret_cast<const uint4*>(rs + Q4T_R_A + i * 2048 + lrow * 16);
            const float4 dp = *reinterpret_cast<const float4*>(rs + Q4T_R_D + lrow * 16);
            __syncwarp();
            if (lane == 0) mbar_arrive(&rempty[r]);
            if (s >= Q4T_NSA) {
                if (!qt_wait_warp(&aempty[sa], (uint32_t)((s / Q4T_NSA) - 1) & 1u, abort)) break;
                qt_fence_after();
            }
            const uint32_t tcol = tA + QT_ACOL + 64u * sa;
#pragma unroll
            for (int i = 0; i < 4; i++) {  // run i: columns 16i .. 16i + 15, q8_1 block i / 2
                const float d = i < 2 ? dp.x : dp.z;
                uint32_t hw[8], lw[8];
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const uint32_t wb = u4_get(cr[i], u) ^ 0x80808080u;
                    // words 8i + 2u + p: columns 16i + 4u + 2p, + 1
                    qt_split_pair(wb, 0x7540u, 0x7541u, d, hw[2 * u], lw[2 * u]);
                    qt_split_pair(wb, 0x7542u, 0x7543u, d, hw[2 * u + 1], lw[2 * u + 1]);
                }
                qt_st8(tcol + 8u * i, hw);
                qt_st8(tcol + 32u + 8u * i, lw);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            qt_fence_before();
            mbar_arrive(&afull[sa]);
        }
        bool ok = mbar_wait(accfull, 0);
        ok = __all_sync(0xffffffffu, ok && !*abort) != 0;
        qt_fence_after();
        qt_epilogue(tA, 0, QT_BN / 32, m0 + lrow, m, n, n0, ok, out);
    } else {
        // ---------------------------------------------------------------- weight operand
        const int bt = 32 * (warp - Q4T_BWARP0) + lane;  // weight row within the tile
        for (int s = 0; s < S; s++) {
            const int sbi = s % Q4T_NSB, r = s % Q4T_NR, t = s & 3;
            if (!qt_wait_warp(&rfull[r], (uint32_t)(s / Q4T_NR) & 1u, abort)) break;
            const uint8_t* rs = ring + r * Q4T_RSTAGE;
            const uint4 hdr = *reinterpret_cast<const uint4*>(rs + Q4T_R_H + bt * 16);
            const uint4 q0 = *reinterpret_cast<const uint4*>(rs + Q4T_R_Q + bt * 16);
            const uint4 q1 = *reinterpret_cast<const uint4*>(rs + Q4T_R_Q + 4096 + bt * 16);
            __syncwarp();
            if (lane == 0) mbar_arrive(&rempty[r]);
            // D_j = d sc_j, M_j = dmin m_j of sub-blocks 2t (low nibbles) and 2t + 1 (high)
            const float dd = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xFFFFu)));
            const float dm = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
            int sc0, mn0, sc1, mn1;
            q4t_scale_min(hdr.y, hdr.z, hdr.w, 2 * t, sc0, mn0);
            q4t_scale_min(hdr.y, hdr.z, hdr.w, 2 * t + 1, sc1, mn1);
            const float D0 = dd * (float)sc0, M0 = dm * (float)mn0;
            const float D1 = dd * (float)sc1, M1 = dm * (float)mn1;
            if (s >= Q4T_NSB) {
                if (!qt_wait_warp(&bempty[sbi], (uint32_t)((s / Q4T_NSB) - 1) & 1u, abort)) break;
            }
            uint8_t* dsth = bst + sbi * Q4T_BSTAGE + (bt >> 3) * 1024 + (bt & 7) * 16;
            uint8_t* dstl = dsth + Q4T_BHALF;
#pragma unroll
            for (int v = 0; v < 4; v++) {  // code bytes 8v .. 8v + 7: columns 8v .. (low), 32 + 8v .. (high)
                const uint32_t w0 = u4_get(v < 2 ? q0 : q1, (2 * v) & 3);
                const uint32_t w1 = u4_get(v < 2 ? q0 : q1, (2 * v + 1) & 3);
                uint32_t hl[4], ll[4], hh[4], lh[4];
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    const uint32_t w = e ? w1 : w0;
                    const uint32_t nl = w & 0x0F0F0F0Fu, nh = (w >> 4) & 0x0F0F0F0Fu;
                    q4t_split_pair(nl, 0x7540u, 0x7541u, D0, M0, hl[2 * e], ll[2 * e]);
                    q4t_split_pair(nl, 0x7542u, 0x7543u, D0, M0, hl[2 * e + 1], ll[2 * e + 1]);
                    q4t_split_pair(nh, 0x7540u, 0x7541u, D1, M1, hh[2 * e], lh[2 * e]);
                    q4t_split_pair(nh, 0x7542u, 0x7543u, D1, M1, hh[2 * e + 1], lh[2 * e + 1]);
                }
                // words 4v .. 4v + 3 (core matrix v) and 16 + 4v .. (core matrix 4 + v)
                *reinterpret_cast<uint4*>(dsth + v * 128) = make_uint4(hl[0], hl[1], hl[2], hl[3]);
                *reinterpret_cast<uint4*>(dstl + v * 128) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
                *reinterpret_cast<uint4*>(dsth + (4 + v) * 128) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                *reinterpret_cast<uint4*>(dstl + (4 + v) * 128) = make_uint4(lh[0], lh[1], lh[2], lh[3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&bfull[sbi]);
        }
    }

    qt_fence_before();
    __syncthreads();
    if (warp == 0) {
        qt_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "n"(QT_TMEM_COLS));
    }
}

static int qt_reserve_smem(const void* fn, int* cache, size_t bytes, const char* who) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64) dev = 63;
    if ((size_t)cache[dev] < bytes) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: cannot reserve %zu bytes of shared memory", who, bytes);
        cache[dev] = (int)bytes;
    }
    return BQ_OK;
}

}  // namespace bq8

using namespace bq8;

extern "C" int q2_mmq_gemm(const void* act_q8, const bq_q2_weight* w, uint16_t* out, uint32_t m,
                           bq_stream_t stream) {
    const char* who = "q2_mmq_gemm";
    int st = check_q2(w, who);
    if (st) return st;
    if (w->group != 128) return fail(BQ_ERR_INVALID, "%s: the MMQ route needs group size 128 (got %u)", who, w->group);
    if (m == 0 || w->n == 0) return ok();
    if (!out || !aligned16(out)) return fail(BQ_ERR_INVALID, "%s: out NULL or not 16-byte aligned", who);
    if (w->k == 0) {
        if (cudaMemsetAsync(out, 0, (size_t)m * w->n * 2, (cudaStream_t)stream) != cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: memset failed", who);
        return ok();
    }
    if (!act_q8 || !aligned16(act_q8)) return fail(BQ_ERR_INVALID, "%s: act_q8 NULL or not 16-byte aligned", who);
    if (m > (1u << 24) || w->n > (1u << 24) || w->k > (1u << 24))
        return fail(BQ_ERR_INVALID, "%s: shape too large", who);
    const uint64_t kp = ((uint64_t)w->k + 255) / 256 * 256;
    const uint64_t k = w->k, n = w->n;
    const uint8_t* codes = (const uint8_t*)act_q8;
    const uint8_t* ds = codes + (uint64_t)m * kp;
    const uint8_t* wcodes = (const uint8_t*)w->data;
    const uint16_t* wsc = (const uint16_t*)(wcodes + (size_t)n * (k / 4));
    CUtensorMap mA, mD, mB;
    // q8_1 codes as [kp/32 chunks][m rows][32 B]: box {16 B, 128 rows, 4 chunks}
    if ((st = make_tmap_3d_u8(&mA, codes, {32, m, kp / 32}, {kp, 32}, {16, QT_BM, 4}, who))) return st;
    // (d, s) pairs as [kp/64 pair-pairs][m rows][16 B]: box {16 B, 128 rows, 2}
    if ((st = make_tmap_3d_u8(&mD, ds, {16, m, kp / 64}, {kp / 4, 16}, {16, QT_BM, 2}, who))) return st;
    // weight codes [n rows][k/4 B]: box {16 B, 256 rows}
    if ((st = make_tmap_2d_u8(&mB, wcodes, k / 4, n, k / 4, 16, QT_BN, false, who))) return st;
    static int cache[64] = {0};
    if ((st = qt_reserve_smem((const void*)q2_mmq_tc_kernel, cache, QT_SMEM, who))) return st;
    const int ntm = (int)((m + QT_BM - 1) / QT_BM);
    const uint64_t tiles = (uint64_t)ntm * ((n + QT_BN - 1) / QT_BN);
    if (tiles > 0x7FFFFFFFull) return fail(BQ_ERR_INVALID, "%s: shape too large", who);
    q2_mmq_tc_kernel<<<(unsigned)tiles, QT_THREADS, QT_SMEM, (cudaStream_t)stream>>>(mA, mD, mB, wsc, out, (int)m,
                                                                                   (int)n, (int)k, ntm);
    return check_launch(who);
}

extern "C" int q4k_mmq_gemm(const void* act_q8, const void* w_q4k, uint16_t* out, uint32_t m, uint32_t n, uint32_t k,
                            bq_stream_t stream) {
    const char* who = "q4k_mmq_gemm";
    if (k % 256 != 0) return fail(BQ_ERR_INVALID, "%s: k = %u must be a multiple of 256", who, k);
    if (m == 0 || n == 0) return ok();
    if (!out || !aligned16(out)) return fail(BQ_ERR_INVALID, "%s: out NULL or not 16-byte aligned", who);
    if (k == 0) {
        if (cudaMemsetAsync(out, 0, (size_t)m * n * 2, (cudaStream_t)stream) != cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: memset failed", who);
        return ok();
    }
    if (!act_q8 || !aligned16(act_q8) || !w_q4k || !aligned16(w_q4k))
        return fail(BQ_ERR_INVALID, "%s: act_q8 / w_q4k NULL or not 16-byte aligned", who);
    if (m > (1u << 24) || n > (1u << 24) || k > (1u << 24)) return fail(BQ_ERR_INVALID, "%s: shape too large", who);
    const uint64_t kp = k;  // k % 256 == 0: no padding
    const uint8_t* codes = (const uint8_t*)act_q8;
    const uint8_t* ds = codes + (uint64_t)m * kp;
    const uint64_t wrow = (uint64_t)(k / 256) * 144;  // bytes per weight row, a multiple of 16
    int st;
    CUtensorMap mA, mD, mQ, mH;
    // q8_1 codes as [kp/16 runs][m rows][16 B]: box {16 B, 128 rows, 4 runs}
    if ((st = make_tmap_3d_u8(&mA, codes, {16, m, kp / 16}, {kp, 16}, {16, QT_BM, 4}, who))) return st;
    // (d, s) pairs [m rows][kp/4 B]: box {16 B (two pairs), 128 rows}
    if ((st = make_tmap_2d_u8(&mD, ds, kp / 4, m, kp / 4, 16, QT_BM, false, who))) return st;
    // weight blocks as [wrow/16 pieces][n rows][16 B]: codes box {16, 256, 2}, header box {16, 256, 1}
    if ((st = make_tmap_3d_u8(&mQ, w_q4k, {16, n, wrow / 16}, {wrow, 16}, {16, QT_BN, 2}, who))) return st;
    if ((st = make_tmap_3d_u8(&mH, w_q4k, {16, n, wrow / 16}, {wrow, 16}, {16, QT_BN, 1}, who))) return st;
    static int cache[64] = {0};
    if ((st = qt_reserve_smem((const void*)q4k_mmq_tc_kernel, cache, Q4T_SMEM, who))) return st;
    const int ntm = (int)((m + QT_BM - 1) / QT_BM);
    const uint64_t tiles = (uint64_t)ntm * ((n + QT_BN - 1) / QT_BN);
    if (tiles > 0x7FFFFFFFull) return fail(BQ_ERR_INVALID, "%s: shape too large", who);
    q4k_mmq_tc_kernel<<<(unsigned)tiles, Q4T_THREADS, Q4T_SMEM, (cudaStream_t)stream>>>(mA, mD, mQ, mH, out, (int)m,
                                                                                      (int)n, (int)k, ntm);
    return check_launch(who);
}
