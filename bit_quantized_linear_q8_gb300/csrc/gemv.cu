// gemv.cu -- Q2_0 decode GEMV for 1..8 activation rows, and the packed-Q2 FFN chain.
//
// Source: init_q2.rs `set_packed_q2_qkvz` (decode runs `q2_0_gemv_vec`) and
// dense_ffn_decode_batch.rs `forward_km_q2` (`q2_0_gemv_vec_batchm` for gate/up/down).
//
// Design (GB300).  The packed weight (2.125 bits per weight) is the only large stream, so
// the kernel is built to keep HBM busy:
//
//  * Staging: one producer warp streams the CTA's rows through a 4-stage shared-memory
//    ring with TMA (cp.async.bulk.tensor, 16 rows x 128 bytes per box, 128-byte swizzle,
//    mbarrier completion).  A stage is a 256-byte chunk of every row of the CTA (8 pack
//    blocks of 128 codes); up to four chunks are in flight per SM without costing
//    registers.  Every wait is bounded.
//  * Compute: eight consumer warps; warp w takes pack block w of each chunk for all of
//    the CTA's row tiles (16 rows each).  The multiply-accumulates for all m <= 8 rows go
//    to the tensor cores through the warp-level MMA m16n8k16 (A = 16 weight rows x 16
//    columns, B = 16 columns x 8 activation rows), so the CUDA cores only unpack:
//      - one AND/OR (lop3) per pair of codes drops a 2-bit code into the mantissa of BF16
//        1.0 in each 16-bit half, v = 1 + c*s with s = 2^-7, 2^-5 or 2^-3 depending on
//        the code's bit position (three of the four positions need no shift);
//      - the activation fragment is built once per pack block per warp, each column
//        pre-multiplied by 1/s (exact, a power of two) and permuted to the lanes' code
//        order, so sum(v*x/s) = sum(x/s) + sum(c*x);
//      - sum((c-2)*x) = sum(v*x/s) - sum((1/s + 2)*x); the correction comes from eight
//        extra MMAs per pack block with a constant A of -(1 + 2s) and seeds every tile's
//        accumulator, so it costs nothing per row tile;
//      - each 128-column group is scaled by its BF16 scale d (held in shared memory).
//  * Work split: CTA c takes a contiguous range of <= T row tiles (grid = SM count when
//    possible, so every SM streams the same number of rows); the warps' partial sums are
//    reduced through shared memory and stored as BF16.
#include "common.cuh"

namespace bq8 {

constexpr int GEMV_CWARPS = 8;                        // consumer warps = pack blocks per chunk
constexpr int GEMV_THREADS = (GEMV_CWARPS + 1) * 32;  // + one producer warp
constexpr int GEMV_MAX_T = 8;                         // row tiles per CTA (128 rows)
constexpr int GEMV_STAGES = 4;
constexpr int GEMV_BOX = 16 * 128;                    // one TMA box: 16 rows x 128 bytes
constexpr int GEMV_MAX_SCALE_BYTES = 64 * 1024;

static __device__ unsigned int g_gemv_status;

unsigned int gemv_status_take() {
    unsigned int v = 0, zero = 0;
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(&v, g_gemv_status, sizeof v);
    cudaMemcpyToSymbol(g_gemv_status, &zero, sizeof zero);
    return v;
}

// Code pair `SUB` (0..7) of a packed 32-bit word: bytes (0,2) for SUB < 4, bytes (1,3)
// otherwise; sub-block i = SUB & 3 sits in bits 2i of each byte.
template <int SUB>
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w) {
    constexpr uint32_t ONE = 0x3F803F80u;  // bf16x2 (1.0, 1.0)
    if constexpr (SUB == 0) return (w & 0x00030003u) | ONE;
    if constexpr (SUB == 1) return (w & 0x000C000Cu) | ONE;
    if constexpr (SUB == 2) return (w & 0x00300030u) | ONE;
    if constexpr (SUB == 3) return ((w >> 2) & 0x00300030u) | ONE;
    if constexpr (SUB == 4) return ((w >> 8) & 0x00030003u) | ONE;
    if constexpr (SUB == 5) return ((w >> 8) & 0x000C000Cu) | ONE;
    if constexpr (SUB == 6) return ((w >> 8) & 0x00300030u) | ONE;
    return ((w >> 10) & 0x00300030u) | ONE;
}

template <int RHO>
__device__ __forceinline__ uint32_t unpack_rho(uint2 w) {
    return unpack_pair<RHO & 7>((RHO >> 3) ? w.y : w.x);
}

// -(1 + 2s) for sub-block i (s = 2^-7, 2^-5, 2^-3, 2^-3), as bf16x2.
__device__ __forceinline__ uint32_t neg_offset_coef(int i) {
    return i == 0 ? 0xBF82BF82u : (i == 1 ? 0xBF88BF88u : 0xBFA0BFA0u);
}

// B-fragment registers of lane (g, t) for one pack block: activation row g, columns
// 32i + 8t + {0..7} of the block, paired as the codes are and scaled by 1/s.
__device__ __forceinline__ void build_bfrag(uint32_t (&b)[16], const uint4 (&X)[4]) {
    const __nv_bfloat162 scl[4] = {__floats2bfloat162_rn(128.f, 128.f), __floats2bfloat162_rn(32.f, 32.f),
                                   __floats2bfloat162_rn(8.f, 8.f), __floats2bfloat162_rn(8.f, 8.f)};
#pragma unroll
    for (int rho = 0; rho < 16; rho++) {
        const int w = rho >> 3, sub = rho & 7, i = sub & 3, hi = sub >> 2;
        const uint32_t a = w ? X[i].z : X[i].x;
        const uint32_t c = w ? X[i].w : X[i].y;
        const uint32_t pr = __byte_perm(a, c, hi ? 0x7632 : 0x5410);
        b[rho] = bf162_bits(__hmul2(bits_bf162(pr), scl[i]));
    }
}

__device__ __forceinline__ void load_x(uint4 (&X)[4], const uint16_t* __restrict__ x, int k, int p, int g, int t,
                                       bool valid) {
    if (valid) {
        const uint16_t* xr = x + (size_t)g * k + (p << 7) + (t << 3);
#pragma unroll
        for (int i = 0; i < 4; i++) X[i] = ldg_nc128(xr + 32 * i);
    } else {
#pragma unroll
        for (int i = 0; i < 4; i++) X[i] = make_uint4(0, 0, 0, 0);
    }
}

template <int T>
__global__ void __launch_bounds__(GEMV_THREADS, 1)
    q2_gemv_kernel(const __grid_constant__ CUtensorMap tmap, const uint16_t* __restrict__ x,
                   const uint16_t* __restrict__ scales, uint16_t* __restrict__ y, int m, int n, int k, int group,
                   int ntiles) {
    constexpr int STAGE_BYTES = 2 * T * GEMV_BOX;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = align1024(smem_raw);
    const int G = k / group;
    uint16_t* sc_s = reinterpret_cast<uint16_t*>(stages + GEMV_STAGES * STAGE_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(sc_s + 16 * T * G) + 7) & ~uintptr_t(7));
    uint64_t* full = bars;
    uint64_t* empty = bars + GEMV_STAGES;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int tile0 = (int)((int64_t)blockIdx.x * ntiles / gridDim.x);
    const int nt = (int)((int64_t)(blockIdx.x + 1) * ntiles / gridDim.x) - tile0;
    const int r0 = tile0 * 16;
    const int P = k >> 7;
    const int nch = (P + GEMV_CWARPS - 1) / GEMV_CWARPS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < GEMV_STAGES; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], GEMV_CWARPS);
        }
        fence_barrier_init();
    }
    for (int idx = threadIdx.x; idx < nt * 16 * G; idx += blockDim.x) {
        const int row = r0 + idx / G;
        sc_s[idx] = row < n ? scales[(size_t)row * G + idx % G] : (uint16_t)0;
    }
    __syncthreads();

    bool failed = false;
    float tot[T][4];
#pragma unroll
    for (int tau = 0; tau < T; tau++) tot[tau][0] = tot[tau][1] = tot[tau][2] = tot[tau][3] = 0.f;

    if (warp == GEMV_CWARPS) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            for (int c = 0; c < nch; c++) {
                const int s = c % GEMV_STAGES;
                if (c >= GEMV_STAGES && !mbar_wait(&empty[s], ((c / GEMV_STAGES) - 1) & 1)) {
                    failed = true;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], 2 * nt * GEMV_BOX);
                uint8_t* dst = stages + s * STAGE_BYTES;
                for (int h = 0; h < 2; h++)
                    for (int tau = 0; tau < nt; tau++)
                        tma_load_2d(dst + (h * T + tau) * GEMV_BOX, &tmap, c * 256 + h * 128, r0 + 16 * tau, &full[s]);
            }
            // wind down: every issued chunk must have landed before the CTA may exit
            const int first = nch > GEMV_STAGES ? nch - GEMV_STAGES : 0;
            for (int c = first; c < nch && !failed; c++)
                if (!mbar_wait(&full[c % GEMV_STAGES], (c / GEMV_STAGES) & 1)) failed = true;
        }
    } else {
        // ---------------------------------------------------------------- consumers
        const int pb = warp;
        const int half = pb >> 2;
        const int jchunk = ((pb & 3) << 1) | (t >> 1);   // 16-byte chunk within the 128-byte line
        const int inner = (t & 1) << 3;
        uint4 xc[4], xn[4];
        load_x(xc, x, k, pb, g, t, g < m && pb < P);
        for (int c = 0; c < nch; c++) {
            const int s = c % GEMV_STAGES;
            const int p = c * GEMV_CWARPS + pb;
            const int pnext = p + GEMV_CWARPS;
            load_x(xn, x, k, pnext, g, t, g < m && pnext < P && c + 1 < nch);
            if (!mbar_wait(&full[s], (c / GEMV_STAGES) & 1)) {
                failed = true;
                break;
            }
            if (p < P) {
                uint32_t b[16];
                build_bfrag(b, xc);
                float neg[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int mu = 0; mu < 8; mu++) {
                    const uint32_t c0 = neg_offset_coef((2 * mu) & 3), c1 = neg_offset_coef((2 * mu + 1) & 3);
                    mma_bf16_16816(neg, c0, c0, c1, c1, b[2 * mu], b[2 * mu + 1], neg);
                }
                const int gi = (p << 7) / group;
                const uint8_t* st = stages + s * STAGE_BYTES;
                const int off = ((jchunk ^ g) << 4) + inner;   // swizzled: (line & 7) == g
#pragma unroll
                for (int tau = 0; tau < T; tau++) {
                    if (tau < nt) {
                        const int line = (half * T + tau) * 16 + g;
                        const uint2 wa = *reinterpret_cast<const uint2*>(st + line * 128 + off);
                        const uint2 wb = *reinterpret_cast<const uint2*>(st + (line + 8) * 128 + off);
                        const float da = bf16_bits_to_f32(sc_s[(tau * 16 + g) * G + gi]);
                        const float db = bf16_bits_to_f32(sc_s[(tau * 16 + g + 8) * G + gi]);
                        float acc[4] = {neg[0], neg[1], neg[2], neg[3]};
#define BQ8_MMA(MU)                                                                                     \
    mma_bf16_16816(acc, unpack_rho<2 * MU>(wa), unpack_rho<2 * MU>(wb), unpack_rho<2 * MU + 1>(wa),    \
                   unpack_rho<2 * MU + 1>(wb), b[2 * MU], b[2 * MU + 1], acc);
                        BQ8_MMA(0) BQ8_MMA(1) BQ8_MMA(2) BQ8_MMA(3) BQ8_MMA(4) BQ8_MMA(5) BQ8_MMA(6) BQ8_MMA(7)
#undef BQ8_MMA
                        tot[tau][0] = fmaf(da, acc[0], tot[tau][0]);
                        tot[tau][1] = fmaf(da, acc[1], tot[tau][1]);
                        tot[tau][2] = fmaf(db, acc[2], tot[tau][2]);
                        tot[tau][3] = fmaf(db, acc[3], tot[tau][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
            for (int i = 0; i < 4; i++) xc[i] = xn[i];
        }
    }
    if (failed) atomicOr(&g_gemv_status, 1u);
    __syncthreads();

    // ---------------------------------------------------------------- reduction + store
    float* red = reinterpret_cast<float*>(stages);  // [CWARPS][T][32 lanes * 5]
    if (warp < GEMV_CWARPS) {
#pragma unroll
        for (int tau = 0; tau < T; tau++)
#pragma unroll
            for (int e = 0; e < 4; e++) red[(warp * T + tau) * 160 + lane * 5 + e] = tot[tau][e];
    }
    __syncthreads();
    const int per_col = nt * 16;
    for (int o = threadIdx.x; o < per_col * m; o += blockDim.x) {
        const int j = o / per_col, rem = o % per_col, tau = rem >> 4, r = rem & 15;
        const int row = r0 + tau * 16 + r;
        if (row >= n) continue;
        const int ln = (r & 7) * 4 + (j >> 1), e = (r >> 3) * 2 + (j & 1);
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < GEMV_CWARPS; w++) sum += red[(w * T + tau) * 160 + ln * 5 + e];
        const __nv_bfloat16 bv = __float2bfloat16_rn(sum);
        y[(size_t)j * n + row] = *reinterpret_cast<const uint16_t*>(&bv);
    }
}

template <int T>
static size_t gemv_smem_bytes(int G) {
    return 1024 + (size_t)GEMV_STAGES * 2 * T * GEMV_BOX + (size_t)16 * T * G * 2 + 8 + 2 * GEMV_STAGES * 8;
}

template <int T>
static int launch_t(const CUtensorMap& map, const uint16_t* x, const uint16_t* scales, uint16_t* y, int m, int n,
                    int k, int group, int ntiles, int ncta, cudaStream_t stream) {
    static int configured_smem[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = gemv_smem_bytes<T>(k / group);
    if (dev < 64 && (size_t)configured_smem[dev] < smem) {
        if (cudaFuncSetAttribute(q2_gemv_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "q2 gemv: cannot reserve %zu bytes of shared memory", smem);
        configured_smem[dev] = (int)smem;
    }
    q2_gemv_kernel<T><<<ncta, GEMV_THREADS, smem, stream>>>(map, x, scales, y, m, n, k, group, ntiles);
    return BQ_OK;
}

// Launches the GEMV for an already validated weight.
int launch_q2_gemv(const uint16_t* x, const bq_q2_weight* w, uint16_t* y, uint32_t m, cudaStream_t stream,
                   const char* who) {
    if (m == 0 || w->n == 0) return ok();
    if (w->k == 0) {
        if (cudaMemsetAsync(y, 0, (size_t)m * w->n * 2, stream) != cudaSuccess)
            return fail(BQ_ERR_LAUNCH, "%s: memset failed", who);
        return ok();
    }
    const int G = (int)(w->k / w->group);
    const int ntiles = (int)((w->n + 15) / 16);
    int tmax = GEMV_MAX_T;
    while (tmax > 1 && (size_t)16 * tmax * G * 2 > (size_t)GEMV_MAX_SCALE_BYTES) tmax--;
    if ((size_t)16 * tmax * G * 2 > (size_t)GEMV_MAX_SCALE_BYTES)
        return fail(BQ_ERR_INVALID, "%s: k/group = %d groups per row is too many", who, G);
    int ncta = ntiles < sm_count() ? ntiles : sm_count();
    int T = (ntiles + ncta - 1) / ncta;
    if (T > tmax) {
        T = tmax;
        ncta = (ntiles + T - 1) / T;
    }
    const uint8_t* codes = (const uint8_t*)w->data;
    const uint16_t* scales = (const uint16_t*)(codes + (size_t)w->n * (w->k / 4));
    CUtensorMap map;
    int st = make_tmap_2d_u8(&map, codes, w->k / 4, w->n, w->k / 4, 128, 16, true, who);
    if (st) return st;
    const int mm = (int)m, n = (int)w->n, k = (int)w->k, gr = (int)w->group;
    switch (T) {
        case 1: st = launch_t<1>(map, x, scales, y, mm, n, k, gr, ntiles, ncta, stream); break;
        case 2: st = launch_t<2>(map, x, scales, y, mm, n, k, gr, ntiles, ncta, stream); break;
        case 3: st = launch_t<3>(map, x, scales, y, mm, n, k, gr, ntiles, ncta, stream); break;
        case 4: st = launch_t<4>(map, x, scales, y, mm, n, k, gr, ntiles, ncta, stream); break;
        case 5: st = launch_t<5>(map, x, scales, y, mm, n, k, gr, ntiles, ncta, stream); break;
        case 6: st = launch_t<6>(map, x, scales, y, mm, n, k, gr, ntiles, ncta, stream); break;
        case 7: st = launch_t<7>(map, x, scales, y, mm, n, k, gr, ntiles, ncta, stream); break;
        case 8: st = launch_t<8>(map, x, scales, y, mm, n, k, gr, ntiles, ncta, stream); break;
        default: return fail(BQ_ERR_INVALID, "%s: internal tile count %d", who, T);
    }
    if (st) return st;
    return check_launch(who);
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
    cudaStream_t s = (cudaStream_t)stream;
    if ((st = launch_q2_gemv(x, gate, gate_scratch, m, s, who))) return st;
    if ((st = launch_q2_gemv(x, up, up_scratch, m, s, who))) return st;
    if ((st = silu_mul_bf16(gate_scratch, up_scratch, gate_scratch, (size_t)m * gate->n, stream))) return st;
    return launch_q2_gemv(gate_scratch, down, out, m, s, who);
}

}  // extern "C"
