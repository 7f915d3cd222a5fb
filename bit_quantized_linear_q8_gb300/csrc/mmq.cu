// mmq.cu -- integer MMQ GEMMs: q8_1 activations x Q2_0 / block_q4_K weights, BF16 store.
//
// Sources: init_q2.rs `qkvz_q2_prefill_gemm` (MMQ route, group 128) and q4k_mmq.rs
// `q4k_mmq_gemm` (C[m, n] = A[m, k] x W[n, k], 128 x 128 tiles, BF16 store).
//
// Design (GB300, sm_103a).  The tcgen05 tensor cores of sm_103a have no int8 kind, and
// q8_1's per-32 activation scale has to be applied to every 32-wide partial product, so the
// contraction runs on the warp-level integer MMA (mma.sync m16n8k32, s8 x u8 -> s32), one
// instruction per 32-value block, which gives the exact integer partial P_b of each block:
//
//  * Staging: a producer warp streams, per 128-column K step, the CTA's q8_1 code tile
//    (128 rows x 128 bytes, 128-byte swizzle), its (d, s) pairs and the weight tile through
//    a 4-stage TMA / mbarrier ring.  Bounded waits throughout.
//  * Compute: eight consumer warps, each a 64 (m) x 32 (n) warp tile = 4 x 4 MMAs per
//    block.  A fragments come from ldmatrix on the swizzled tile; B fragments are built in
//    registers straight from the packed codes (Q2_0: one shift + AND per 4 codes, because
//    byte l of a pack block holds column 32i + l of each sub-block i).
//  * Exact conversion: each MMA starts from the int32 bit pattern of 1.5 * 2^23, so its
//    result reinterpreted as fp32 is exactly 1.5*2^23 + P_b; one packed fp32 add removes
//    the offset, one packed FMA applies the activation scale d_a.  Per 128-column group
//    the Q2 scale d_w and the code offset (-2 * sum of s) are applied.
#include "common.cuh"

namespace bq8 {

static __device__ unsigned int g_mmq_status;

unsigned int mmq_status_take() {
    unsigned int v = 0, zero = 0;
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(&v, g_mmq_status, sizeof v);
    cudaMemcpyToSymbol(g_mmq_status, &zero, sizeof zero);
    return v;
}

constexpr int MMQ_CWARPS = 8;
constexpr int MMQ_THREADS = (MMQ_CWARPS + 1) * 32;
constexpr int MMQ_STAGES = 4;
constexpr int MMQ_TILE = 128;                  // BM = BN = 128, K step 128
constexpr int Q2S_A = 0;                       // q8_1 codes, 128 x 128 B, swizzled
constexpr int Q2S_D = 16384;                   // (d, s) pairs, 128 x 32 B
constexpr int Q2S_B = 20480;                   // Q2 codes, 128 x 32 B
constexpr int Q2S_STAGE = 24576;
constexpr int MAGIC_I = 0x4B400000;            // bits of 1.5 * 2^23
constexpr float MAGIC_F = 12582912.0f;

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

__device__ __forceinline__ float2 i2f_magic(int a, int b) {
    return __fadd2_rn(make_float2(__int_as_float(a), __int_as_float(b)), make_float2(-MAGIC_F, -MAGIC_F));
}

// Stores a warp's 64 x 32 tile of fp32 results as BF16 (row-major out[m][n]), guarding
// the m and n tails; pairs of columns go out as one 4-byte store when n is even.
__device__ __forceinline__ void store_tile(const float2 (&acc)[4][4][2], uint16_t* __restrict__ out, int m, int n,
                                           int row0, int col0, int g, int t) {
    const bool pair_ok = (n & 1) == 0;
#pragma unroll
    for (int mt = 0; mt < 4; mt++) {
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int row = row0 + mt * 16 + g + 8 * h;
            if (row >= m) continue;
#pragma unroll
            for (int nt = 0; nt < 4; nt++) {
                const int col = col0 + nt * 8 + 2 * t;
                const float2 v = acc[mt][nt][h];
                uint16_t* dst = out + (size_t)row * n + col;
                if (pair_ok && col + 1 < n) {
                    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(v.x, v.y);
                } else {
                    if (col < n) {
                        const __nv_bfloat16 b = __float2bfloat16_rn(v.x);
                        dst[0] = *reinterpret_cast<const uint16_t*>(&b);
                    }
                    if (col + 1 < n) {
                        const __nv_bfloat16 b = __float2bfloat16_rn(v.y);
                        dst[1] = *reinterpret_cast<const uint16_t*>(&b);
                    }
                }
            }
        }
    }
}

__global__ void __launch_bounds__(MMQ_THREADS, 1)
    q2_mmq_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapD,
                  const __grid_constant__ CUtensorMap mapB, const uint16_t* __restrict__ wscales,
                  uint16_t* __restrict__ out, int m, int n, int k) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = align1024(smem_raw);
    const int G = k >> 7;
    uint16_t* sc_s = reinterpret_cast<uint16_t*>(stages + MMQ_STAGES * Q2S_STAGE);
    uint64_t* bars =
        reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(sc_s + MMQ_TILE * G) + 7) & ~uintptr_t(7));
    uint64_t* full = bars;
    uint64_t* empty = bars + MMQ_STAGES;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int n0 = blockIdx.x * MMQ_TILE, m0 = blockIdx.y * MMQ_TILE;

    if (threadIdx.x == 0) {
        for (int s = 0; s < MMQ_STAGES; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], MMQ_CWARPS);
        }
        fence_barrier_init();
    }
    {   // the weight tile's group scales (contiguous rows of the scale plane)
        const int rows = min(MMQ_TILE, n - n0);
        copy_to_smem(sc_s, wscales + (size_t)n0 * G, rows * G * 2, threadIdx.x, blockDim.x);
        for (int idx = rows * G + threadIdx.x; idx < MMQ_TILE * G; idx += blockDim.x) sc_s[idx] = 0;
    }
    __syncthreads();

    bool failed = false;
    float2 acc[4][4][2];
#pragma unroll
    for (int a = 0; a < 4; a++)
#pragma unroll
        for (int b = 0; b < 4; b++) acc[a][b][0] = acc[a][b][1] = make_float2(0.f, 0.f);
    const int wm = warp & 1, wn = warp >> 1;

    if (warp == MMQ_CWARPS) {
        if (lane == 0) {
            for (int c = 0; c < G; c++) {
                const int s = c % MMQ_STAGES;
                if (c >= MMQ_STAGES && !mbar_wait(&empty[s], ((c / MMQ_STAGES) - 1) & 1)) {
                    failed = true;
                    break;
                }
                uint8_t* dst = stages + s * Q2S_STAGE;
                mbar_arrive_expect_tx(&full[s], Q2S_STAGE);
                tma_load_2d(dst + Q2S_A, &mapA, c * 128, m0, &full[s]);
                tma_load_2d(dst + Q2S_D, &mapD, c * 32, m0, &full[s]);
                tma_load_2d(dst + Q2S_B, &mapB, c * 32, n0, &full[s]);
            }
            const int first = G > MMQ_STAGES ? G - MMQ_STAGES : 0;
            for (int c = first; c < G && !failed; c++)
                if (!mbar_wait(&full[c % MMQ_STAGES], (c / MMQ_STAGES) & 1)) failed = true;
        }
    } else {
        const int cmagic[4] = {MAGIC_I, MAGIC_I, MAGIC_I, MAGIC_I};
        for (int c = 0; c < G; c++) {
            const int s = c % MMQ_STAGES;
            if (!mbar_wait(&full[s], (c / MMQ_STAGES) & 1)) {
                failed = true;
                break;
            }
            const uint8_t* A = stages + s * Q2S_STAGE + Q2S_A;
            const uint8_t* D = stages + s * Q2S_STAGE + Q2S_D;
            const uint8_t* Bt = stages + s * Q2S_STAGE + Q2S_B;
            uint32_t w0[4], w1[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int row = wn * 32 + j * 8 + g;
                w0[j] = *reinterpret_cast<const uint32_t*>(Bt + row * 32 + 4 * t);
                w1[j] = *reinterpret_cast<const uint32_t*>(Bt + row * 32 + 16 + 4 * t);
            }
            float2 ag[4][4][2];
#pragma unroll
            for (int a = 0; a < 4; a++)
#pragma unroll
                for (int b = 0; b < 4; b++) ag[a][b][0] = ag[a][b][1] = make_float2(0.f, 0.f);
            float ssum[4][2];
#pragma unroll
            for (int a = 0; a < 4; a++) ssum[a][0] = ssum[a][1] = 0.f;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                float da[4][2];
                uint32_t af[4][4];
#pragma unroll
                for (int mt = 0; mt < 4; mt++) {
                    const int rlo = wm * 64 + mt * 16 + g;
                    const float2 vlo = *reinterpret_cast<const float2*>(D + rlo * 32 + 8 * i);
                    const float2 vhi = *reinterpret_cast<const float2*>(D + (rlo + 8) * 32 + 8 * i);
                    da[mt][0] = vlo.x;
                    da[mt][1] = vhi.x;
                    ssum[mt][0] += vlo.y;
                    ssum[mt][1] += vhi.y;
                    const int rl = wm * 64 + mt * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
                    const int ch = 2 * i + (lane >> 4);
                    ldmatrix_x4(af[mt], A + rl * 128 + ((ch ^ (rl & 7)) << 4));
                }
#pragma unroll
                for (int nt = 0; nt < 4; nt++) {
                    const uint32_t b0 = (w0[nt] >> (2 * i)) & 0x03030303u;
                    const uint32_t b1 = (w1[nt] >> (2 * i)) & 0x03030303u;
#pragma unroll
                    for (int mt = 0; mt < 4; mt++) {
                        int d[4];
                        mma_s8u8_16832(d, af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1, cmagic);
                        ag[mt][nt][0] = __ffma2_rn(i2f_magic(d[0], d[1]), make_float2(da[mt][0], da[mt][0]),
                                                   ag[mt][nt][0]);
                        ag[mt][nt][1] = __ffma2_rn(i2f_magic(d[2], d[3]), make_float2(da[mt][1], da[mt][1]),
                                                   ag[mt][nt][1]);
                    }
                }
            }
            // group epilogue: out += d_w * (sum_b d_a P_b - 2 sum_b s_b)
#pragma unroll
            for (int nt = 0; nt < 4; nt++) {
                const int col = wn * 32 + nt * 8 + 2 * t;
                const float2 dw = make_float2(bf16_bits_to_f32(sc_s[col * G + c]), bf16_bits_to_f32(sc_s[(col + 1) * G + c]));
#pragma unroll
                for (int mt = 0; mt < 4; mt++) {
                    const float2 o0 = make_float2(-2.f * ssum[mt][0], -2.f * ssum[mt][0]);
                    const float2 o1 = make_float2(-2.f * ssum[mt][1], -2.f * ssum[mt][1]);
                    acc[mt][nt][0] = __ffma2_rn(__fadd2_rn(ag[mt][nt][0], o0), dw, acc[mt][nt][0]);
                    acc[mt][nt][1] = __ffma2_rn(__fadd2_rn(ag[mt][nt][1], o1), dw, acc[mt][nt][1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
    if (failed) atomicOr(&g_mmq_status, 2u);

    if (warp < MMQ_CWARPS) store_tile(acc, out, m, n, m0 + wm * 64, n0 + wn * 32, g, t);
}

// ------------------------------------------------------------------------------------
// Q4_K.  K step = one 256-value superblock.  Stage: q8_1 codes [2][128][128] (swizzled),
// (d, s) pairs [128][8], the weight blocks [128][144], and a table the consumers fill
// with d*sc_j and dmin*m_j per (sub-block j, weight row).
// Per 32-value block j:  out += d_a * (d*sc_j) * P_j  -  s_a * (dmin*m_j).
// ------------------------------------------------------------------------------------
constexpr int Q4S_A = 0;
constexpr int Q4S_D = 32768;
constexpr int Q4S_B = 40960;
constexpr int Q4S_TAB = 59392;            // [2][8][128] floats: d*sc_j, dmin*m_j
constexpr int Q4S_STAGE = 68608;          // 67 KB, multiple of 1024
constexpr int Q4S_TX = 59392;             // bytes delivered by TMA per stage
constexpr int Q4_STAGES = 3;

__device__ __forceinline__ void q4k_scale_min(const uint8_t* s, int j, int& sc, int& mn) {
    if (j < 4) {
        sc = s[j] & 63;
        mn = s[j + 4] & 63;
    } else {
        sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

__global__ void __launch_bounds__(MMQ_THREADS, 1)
    q4k_mmq_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapD,
                   const __grid_constant__ CUtensorMap mapB, uint16_t* __restrict__ out, int m, int n, int k) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = align1024(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(stages + Q4_STAGES * Q4S_STAGE);
    uint64_t* full = bars;
    uint64_t* empty = bars + Q4_STAGES;
    const int nsb = k >> 8;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int n0 = blockIdx.x * MMQ_TILE, m0 = blockIdx.y * MMQ_TILE;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Q4_STAGES; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], MMQ_CWARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();

    bool failed = false;
    float2 acc[4][4][2];
#pragma unroll
    for (int a = 0; a < 4; a++)
#pragma unroll
        for (int b = 0; b < 4; b++) acc[a][b][0] = acc[a][b][1] = make_float2(0.f, 0.f);
    const int wm = warp & 1, wn = warp >> 1;

    if (warp == MMQ_CWARPS) {
        if (lane == 0) {
            for (int c = 0; c < nsb; c++) {
                const int s = c % Q4_STAGES;
                if (c >= Q4_STAGES && !mbar_wait(&empty[s], ((c / Q4_STAGES) - 1) & 1)) {
                    failed = true;
                    break;
                }
                uint8_t* dst = stages + s * Q4S_STAGE;
                mbar_arrive_expect_tx(&full[s], Q4S_TX);
                tma_load_2d(dst + Q4S_A, &mapA, c * 256, m0, &full[s]);
                tma_load_2d(dst + Q4S_A + 16384, &mapA, c * 256 + 128, m0, &full[s]);
                tma_load_2d(dst + Q4S_D, &mapD, c * 64, m0, &full[s]);
                tma_load_2d(dst + Q4S_B, &mapB, c * 144, n0, &full[s]);
            }
            const int first = nsb > Q4_STAGES ? nsb - Q4_STAGES : 0;
            for (int c = first; c < nsb && !failed; c++)
                if (!mbar_wait(&full[c % Q4_STAGES], (c / Q4_STAGES) & 1)) failed = true;
        }
    } else {
        const int cmagic[4] = {MAGIC_I, MAGIC_I, MAGIC_I, MAGIC_I};
        const int ctid = threadIdx.x;  // 0..255 among the consumer warps
        for (int c = 0; c < nsb; c++) {
            const int s = c % Q4_STAGES;
            if (!mbar_wait(&full[s], (c / Q4_STAGES) & 1)) {
                failed = true;
                break;
            }
            uint8_t* st = stages + s * Q4S_STAGE;
            const uint8_t* A = st + Q4S_A;
            const uint8_t* D = st + Q4S_D;
            const uint8_t* Bt = st + Q4S_B;
            float* tab = reinterpret_cast<float*>(st + Q4S_TAB);
            {   // d*sc_j and dmin*m_j of every weight row of the tile (exact in fp32)
                const int r = ctid & 127, jh = ctid >> 7;
                const uint8_t* blk = Bt + r * 144;
                const float d = __half2float(*reinterpret_cast<const __half*>(blk));
                const float dm = __half2float(*reinterpret_cast<const __half*>(blk + 2));
#pragma unroll
                for (int jj = 0; jj < 4; jj++) {
                    const int j = jh * 4 + jj;
                    int sc, mn;
                    q4k_scale_min(blk + 4, j, sc, mn);
                    tab[j * 128 + r] = d * (float)sc;
                    tab[1024 + j * 128 + r] = dm * (float)mn;
                }
            }
            asm volatile("bar.sync 1, %0;" ::"n"(MMQ_CWARPS * 32) : "memory");
#pragma unroll 1
            for (int ch = 0; ch < 4; ch++) {  // 64-value chunk: sub-blocks 2ch (low nibbles), 2ch+1 (high)
                uint32_t w0[4], w1[4];
#pragma unroll
                for (int nt = 0; nt < 4; nt++) {
                    const uint8_t* q = Bt + (wn * 32 + nt * 8 + g) * 144 + 16 + 32 * ch;
                    w0[nt] = *reinterpret_cast<const uint32_t*>(q + 4 * t);
                    w1[nt] = *reinterpret_cast<const uint32_t*>(q + 16 + 4 * t);
                }
#pragma unroll
                for (int hn = 0; hn < 2; hn++) {
                    const int j = 2 * ch + hn;
                    float2 da2[4][2], sa2[4][2];
                    uint32_t af[4][4];
#pragma unroll
                    for (int mt = 0; mt < 4; mt++) {
                        const int rlo = wm * 64 + mt * 16 + g;
                        const float2 vlo = *reinterpret_cast<const float2*>(D + rlo * 64 + 8 * j);
                        const float2 vhi = *reinterpret_cast<const float2*>(D + (rlo + 8) * 64 + 8 * j);
                        da2[mt][0] = make_float2(vlo.x, vlo.x);
                        da2[mt][1] = make_float2(vhi.x, vhi.x);
                        sa2[mt][0] = make_float2(-vlo.y, -vlo.y);
                        sa2[mt][1] = make_float2(-vhi.y, -vhi.y);
                        const int rl = wm * 64 + mt * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
                        const int chunk16 = 2 * (j & 3) + (lane >> 4);
                        ldmatrix_x4(af[mt], A + (j >> 2) * 16384 + rl * 128 + ((chunk16 ^ (rl & 7)) << 4));
                    }
#pragma unroll
                    for (int nt = 0; nt < 4; nt++) {
                        const uint32_t b0 = (w0[nt] >> (4 * hn)) & 0x0F0F0F0Fu;
                        const uint32_t b1 = (w1[nt] >> (4 * hn)) & 0x0F0F0F0Fu;
                        const int col = wn * 32 + nt * 8 + 2 * t;
                        const float2 dsc = *reinterpret_cast<const float2*>(tab + j * 128 + col);
                        const float2 dmn = *reinterpret_cast<const float2*>(tab + 1024 + j * 128 + col);
#pragma unroll
                        for (int mt = 0; mt < 4; mt++) {
                            int d[4];
                            mma_s8u8_16832(d, af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1, cmagic);
                            float2 a0 = __ffma2_rn(i2f_magic(d[0], d[1]), __fmul2_rn(da2[mt][0], dsc), acc[mt][nt][0]);
                            float2 a1 = __ffma2_rn(i2f_magic(d[2], d[3]), __fmul2_rn(da2[mt][1], dsc), acc[mt][nt][1]);
                            acc[mt][nt][0] = __ffma2_rn(sa2[mt][0], dmn, a0);
                            acc[mt][nt][1] = __ffma2_rn(sa2[mt][1], dmn, a1);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
    if (failed) atomicOr(&g_mmq_status, 4u);

    if (warp < MMQ_CWARPS) store_tile(acc, out, m, n, m0 + wm * 64, n0 + wn * 32, g, t);
}

static int reserve_smem(const void* fn, size_t bytes, int* cache, const char* who) {
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

extern "C" {

int q2_mmq_gemm(const void* act_q8, const bq_q2_weight* w, uint16_t* out, uint32_t m, bq_stream_t stream) {
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
    if (m > (1u << 24) || w->n > (1u << 24)) return fail(BQ_ERR_INVALID, "%s: shape too large", who);
    const uint64_t kp = ((uint64_t)w->k + 255) / 256 * 256;
    const uint8_t* codes = (const uint8_t*)act_q8;
    const uint8_t* ds = codes + (uint64_t)m * kp;
    const uint8_t* wcodes = (const uint8_t*)w->data;
    const uint16_t* wsc = (const uint16_t*)(wcodes + (size_t)w->n * (w->k / 4));
    CUtensorMap mA, mD, mB;
    if ((st = make_tmap_2d_u8(&mA, codes, kp, m, kp, 128, 128, true, who))) return st;
    if ((st = make_tmap_2d_u8(&mD, ds, kp / 4, m, kp / 4, 32, 128, false, who))) return st;
    if ((st = make_tmap_2d_u8(&mB, wcodes, w->k / 4, w->n, w->k / 4, 32, 128, false, who))) return st;
    const int G = (int)(w->k / 128);
    const size_t smem = 1024 + (size_t)MMQ_STAGES * Q2S_STAGE + (size_t)MMQ_TILE * G * 2 + 8 + 2 * MMQ_STAGES * 8;
    if (smem > 227 * 1024) return fail(BQ_ERR_INVALID, "%s: k = %u too large for the scale buffer", who, w->k);
    static int cache[64] = {0};
    if ((st = reserve_smem((const void*)q2_mmq_kernel, smem, cache, who))) return st;
    const dim3 grid((w->n + MMQ_TILE - 1) / MMQ_TILE, (m + MMQ_TILE - 1) / MMQ_TILE);
    q2_mmq_kernel<<<grid, MMQ_THREADS, smem, (cudaStream_t)stream>>>(mA, mD, mB, wsc, out, (int)m, (int)w->n,
                                                                      (int)w->k);
    return check_launch(who);
}

int q4k_mmq_gemm(const void* act_q8, const void* w_q4k, uint16_t* out, uint32_t m, uint32_t n, uint32_t k,
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
    if (m > (1u << 24) || n > (1u << 24)) return fail(BQ_ERR_INVALID, "%s: shape too large", who);
    const uint64_t kp = k;  // k % 256 == 0: no padding
    const uint8_t* codes = (const uint8_t*)act_q8;
    const uint8_t* ds = codes + (uint64_t)m * kp;
    const uint64_t wrow = (uint64_t)(k / 256) * 144;
    CUtensorMap mA, mD, mB;
    int st;
    if ((st = make_tmap_2d_u8(&mA, codes, kp, m, kp, 128, 128, true, who))) return st;
    if ((st = make_tmap_2d_u8(&mD, ds, kp / 4, m, kp / 4, 64, 128, false, who))) return st;
    if ((st = make_tmap_2d_u8(&mB, w_q4k, wrow, n, wrow, 144, 128, false, who))) return st;
    const size_t smem = 1024 + (size_t)Q4_STAGES * Q4S_STAGE + 2 * Q4_STAGES * 8;
    static int cache[64] = {0};
    if ((st = reserve_smem((const void*)q4k_mmq_kernel, smem, cache, who))) return st;
    const dim3 grid((n + MMQ_TILE - 1) / MMQ_TILE, (m + MMQ_TILE - 1) / MMQ_TILE);
    q4k_mmq_kernel<<<grid, MMQ_THREADS, smem, (cudaStream_t)stream>>>(mA, mD, mB, out, (int)m, (int)n, (int)k);
    return check_launch(who);
}

}  // extern "C"
