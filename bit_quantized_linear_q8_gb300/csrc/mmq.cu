// mmq.cu -- Q4_K MMQ GEMM: q8_1 activations x block_q4_K weights, BF16 store.
//
// Source: q4k_mmq.rs `q4k_mmq_gemm` (C[m, n] = A[m, k] x W[n, k], 128 x 128 tiles, BF16
// store).  (The Q2_0 MMQ is in mmq_tc.cu.)
//
// Design (GB300, sm_103a).  The tcgen05 tensor cores of sm_103a have no int8 kind, and
// q8_1's per-32 activation scale and Q4_K's per-32 sub-block scale have to be applied to
// every 32-wide partial product, so the contraction runs on the warp-level integer MMA
// (mma.sync m16n8k32, s8 x u8 -> s32), one instruction per 32-value block, which gives the
// exact integer partial P_j of each block:
//
//  * Staging: a producer warp streams, per 256-column K step (one super-block), the CTA's
//    q8_1 code tile (128-byte swizzle), its (d, s) pairs and the weight blocks through a
//    3-stage TMA / mbarrier ring.  Bounded waits throughout.
//  * Compute: eight consumer warps, each a 64 (m) x 32 (n) warp tile = 4 x 4 MMAs per
//    block.  A fragments come from ldmatrix on the swizzled tile; B fragments are built in
//    registers from the 4-bit codes.
//  * Exact conversion: each MMA starts from the int32 bit pattern of 1.5 * 2^23, so its
//    result reinterpreted as fp32 is exactly 1.5*2^23 + P_j; one packed fp32 add removes
//    the offset, one packed FMA applies the scales.
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
