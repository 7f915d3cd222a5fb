// formats.cu -- weight packing, dequantisation (Q2_0 and NVFP4 to BF16), activation
// quantisation (q8_1), the Q4_K weight quantiser and SiLU*mul.
//
// All of these are streaming kernels without shared memory: coalesced 8/16-byte accesses,
// grids sized as a multiple of the SM count (the NVFP4 dequant keeps the page's one CTA per
// row), except the q8_1 quantiser for k % 256 == 0, which stages its input through shared
// memory with bulk copies and replaces the IEEE division per value by an exact FMA form.
#include "common.cuh"

namespace bq8 {

// =====================================================================================
// Q2_0 pack: codes [n][k] (one per byte) + scales [n][k/group] -> packed buffer.
// Thread -> 4 output bytes (l0..l0+3 of one 32-byte pack block): byte l of pack block p
// holds the codes of columns 128p + 32i + l in bits 2i (i = 0..3).
// Source: init_q2.rs, `set_packed_q2_qkvz` (the packed weight it installs).
// =====================================================================================
__global__ void q2_pack_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                               uint8_t* __restrict__ out, int64_t n, int64_t k, int64_t nsc) {
    const int64_t words_per_row = k / 16;  // 4 output bytes per thread, k/4 bytes per row
    const int64_t total = n * words_per_row;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; id < total; id += stride) {
        const int64_t r = id / words_per_row, wi = id % words_per_row;
        const int64_t p = wi / 8, l0 = (wi % 8) * 4;
        const uint8_t* src = codes + r * k + p * 128 + l0;
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t c4 = *reinterpret_cast<const uint32_t*>(src + 32 * i);
            word |= (c4 & 0x03030303u) << (2 * i);
        }
        *reinterpret_cast<uint32_t*>(out + r * (k / 4) + p * 32 + l0) = word;
    }
    uint16_t* sc_out = reinterpret_cast<uint16_t*>(out + n * (k / 4));
    for (int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; id < nsc; id += stride) sc_out[id] = scales[id];
}

// =====================================================================================
// Q2_0 -> BF16: w = d * (c - 2), exact.
// Thread -> 8 packed bytes (32 codes) = 4 runs of 8 consecutive columns.  Each code is
// moved into mantissa bits 5..6 of a bf16 1.0 (value 1 + c/4), then (v - 1.5) * 4d gives
// d*(c-2) exactly (both steps are exact in BF16).
// Source: init_q2.rs, `qkvz_q2_prefill_gemm` fallback (`dequant_q2_0_gn_to_bf16`).
// =====================================================================================
// One 8-byte quarter of a pack block (32 codes: 4 runs of 8 consecutive columns) to BF16.
__device__ __forceinline__ void q2_dequant_quarter(uint2 w, float d, uint16_t* __restrict__ dst) {
    const __nv_bfloat162 c15 = __floats2bfloat162_rn(1.5f, 1.5f);
    const __nv_bfloat162 d4 = __floats2bfloat162_rn(4.0f * d, 4.0f * d);
    // bytes (b, b+1) into the low byte of each 16-bit half
    const uint32_t e[4] = {__byte_perm(w.x, 0, 0x4140), __byte_perm(w.x, 0, 0x4342), __byte_perm(w.y, 0, 0x4140),
                           __byte_perm(w.y, 0, 0x4342)};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const uint32_t s = (i < 3) ? (e[j] << (5 - 2 * i)) : (e[j] >> 1);
            const uint32_t v = (s & 0x00600060u) | 0x3F803F80u;
            o[j] = bf162_bits(__hmul2(__hsub2(bits_bf162(v), c15), d4));
        }
        *reinterpret_cast<uint4*>(dst + 32 * i) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Two quarters a thread per step (id and id + stride), both quarters' loads issued first.
// Quarter id is row id / (k/32), quarter id % (k/32) of the row (32-bit division when every
// index fits).
__global__ void __launch_bounds__(256) q2_dequant_kernel(const uint8_t* __restrict__ packed, uint16_t* __restrict__ out,
                                                         int64_t n, int64_t k, int group) {
    const int64_t q_per_row = k / 32;  // 8-byte quarters of pack blocks per row
    const int64_t total = n * q_per_row;
    const int64_t groups = k / group;
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(packed + n * (k / 4));
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const bool idx32 = total + 2 * stride <= 0xFFFFFFFFll;
    auto split = [&](int64_t id, int64_t& r, int64_t& qi) {
        if (idx32) {
            const uint32_t u = (uint32_t)id, qpr = (uint32_t)q_per_row;
            r = u / qpr;
            qi = u - (uint32_t)r * qpr;
        } else {
            r = id / q_per_row;
            qi = id - r * q_per_row;
        }
    };
    for (int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; id < total; id += 2 * stride) {
        const int64_t id2 = id + stride;
        int64_t r1, q1, r2 = 0, q2 = 0;
        split(id, r1, q1);
        const uint2 w1 = ldg_stream64(packed + r1 * (k / 4) + (q1 >> 2) * 32 + (q1 & 3) * 8);
        const uint16_t s1 = sc[r1 * groups + ((uint32_t)(q1 >> 2) * 128u) / (uint32_t)group];
        uint2 w2 = make_uint2(0u, 0u);
        uint16_t s2 = 0;
        if (id2 < total) {
            split(id2, r2, q2);
            w2 = ldg_stream64(packed + r2 * (k / 4) + (q2 >> 2) * 32 + (q2 & 3) * 8);
            s2 = sc[r2 * groups + ((uint32_t)(q2 >> 2) * 128u) / (uint32_t)group];
        }
        q2_dequant_quarter(w1, bf16_bits_to_f32(s1), out + r1 * k + (q1 >> 2) * 128 + (q1 & 3) * 8);
        if (id2 < total) q2_dequant_quarter(w2, bf16_bits_to_f32(s2), out + r2 * k + (q2 >> 2) * 128 + (q2 & 3) * 8);
    }
}

// =====================================================================================
// q8_1 arithmetic.  q8_1 (q4k_mmq.rs, `quantize_act_q8_1`) takes per 32-value block
// d = RN(amax / 127), code = round-half-away(RN(x / d)) clamped to [-127, 127] and
// s = RN(d * sum(code)), each an IEEE fp32 operation.
// The kernels compute the same codes without a division per value:
//  * RN(a / d) for a = |x| is Markstein's correction of y0 = RN(a r) with r = RN(1/d):
//    RN(y0 + r RN(a - d y0)), two FMAs (P. Markstein, "Computation of elementary functions on
//    the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990: with a correctly
//    rounded reciprocal and a quotient within an ulp, one correction rounds correctly).
//  * round-half-away of that y >= 0 is floor(RZ(y + 1/2)) (the integers are representable,
//    so rounding the sum toward zero never crosses one), and a second round-toward-zero add
//    of 2^23 leaves it in the low mantissa byte.
//  * d = RN(amax / 127) from q0 = RN(amax c), c = RN(1/127), and one FMA correction of the
//    exact residual amax - 127 q0.
// Both forms are checked on the host against the IEEE divisions for every BF16 pair
// |x| <= amax of several binades (tests/test_q8_1_arith.py); the quotient can differ only
// where the residual underflows, for quotients below 2^-100 whose code is 0.  Scaling by
// powers of two keeps all of it exact while d is normal, so blocks with amax >= 2^-94 take
// this path and smaller ones the IEEE divisions.  The four code bytes of a word are gathered
// with byte permutes and the signs applied to all four at once.
// =====================================================================================
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Four codes with magnitudes c (0..127, the low byte of each of m0..m3) and the signs of the
// BF16 values in bytes 1 and 3 of w0 and w1, as one word of int8 codes.  Each sign byte is
// 0x00 or 0xFF (prmt's sign-replicating selector); -c per byte is ((c ^ 0xFF) & 0x7F) + 1
// with the top bit flipped, which never carries into the next byte (c = 0 gives 0x80 ^ 0x80).
__device__ __forceinline__ uint32_t q8_pack4(uint32_t m0, uint32_t m1, uint32_t m2, uint32_t m3, uint32_t w0,
                                             uint32_t w1) {
    const uint32_t mag = prmt(prmt(m0, m1, 0x0040u), prmt(m2, m3, 0x0040u), 0x5410u);
    const uint32_t sgn = prmt(w0, w1, 0xFDB9u);
    const uint32_t low = ((mag ^ sgn) & 0x7F7F7F7Fu) + (sgn & 0x01010101u);
    return low ^ (sgn & 0x80808080u);
}

// 2^23 + |code| as float bits, by IEEE division (any d > 0): floor(RZ(|y| + 1/2)) equals
// floor(|y| + 1/2) because the integers are representable; clamped to 127.
__device__ __forceinline__ uint32_t q8_mag_div(float v, float d) {
    const float a = fminf(__fadd_rz(fabsf(__fdiv_rn(v, d)), 0.5f), 127.0f);
    return __float_as_uint(__fadd_rz(a, 8388608.0f));
}

// The same bits without a division per value (d normal, r = RN(1/d)).
__device__ __forceinline__ uint32_t q8_mag_fast(float v, float d, float r) {
    const float a = fabsf(v);
    const float y0 = __fmul_rn(a, r);
    const float y = __fmaf_rn(__fmaf_rn(-d, y0, a), r, y0);  // RN(a / d)
    return __float_as_uint(__fadd_rz(__fadd_rz(y, 0.5f), 8388608.0f));
}

// RN(amax / 127) for a BF16 amax >= 2^-94.
__device__ __forceinline__ float q8_scale(float amax) {
    constexpr float c127 = 1.0f / 127.0f;
    const float q0 = __fmul_rn(amax, c127);
    return __fmaf_rn(__fmaf_rn(-q0, 127.0f, amax), c127, q0);
}

// =====================================================================================
// q8_1 quantisation.  Thread -> 8 values; a quad of 4 threads owns one 32-value block.
// d = RN(amax/127), q = round-half-away(RN(x/d)), s = RN(d*sum(q)), with the division-free
// exact form above (IEEE divisions for blocks with amax < 2^-94).  This form takes any k
// (zero padding to kp); k % 256 == 0 goes to q8_1_block_kernel below.
// Source: q4k_mmq.rs, `quantize_act_q8_1`.
// =====================================================================================
template <bool VEC>
__global__ void __launch_bounds__(256) q8_1_kernel(const uint16_t* __restrict__ x, int8_t* __restrict__ codes,
                                                   float2* __restrict__ ds, int64_t m, int64_t k, int64_t kp) {
    const int64_t per_row = kp / 8;
    const int64_t total = m * per_row;  // multiple of 32: kp % 256 == 0
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; id < total; id += stride) {
        const int64_t r = id / per_row, c0 = (id % per_row) * 8;
        float v[8];
        if (VEC && c0 + 8 <= k) {
            const uint4 u = *reinterpret_cast<const uint4*>(x + r * k + c0);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; j++) {
                v[2 * j] = __uint_as_float(w[j] << 16);
                v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; j++) v[j] = (c0 + j < k) ? bf16_bits_to_f32(x[r * k + c0 + j]) : 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; j++) amax = fmaxf(amax, fabsf(v[j]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        // the BF16 bit patterns of the eight values (their signs for the packing)
        uint32_t wb[4];
#pragma unroll
        for (int j = 0; j < 4; j++) wb[j] = (__float_as_uint(v[2 * j]) >> 16) | (__float_as_uint(v[2 * j + 1]) & 0xFFFF0000u);
        float d;
        uint32_t lo = 0, hi = 0;
        if (amax >= 0x1p-94f) {
            d = q8_scale(amax);
            const float rc = __frcp_rn(d);
            lo = q8_pack4(q8_mag_fast(v[0], d, rc), q8_mag_fast(v[1], d, rc), q8_mag_fast(v[2], d, rc),
                          q8_mag_fast(v[3], d, rc), wb[0], wb[1]);
            hi = q8_pack4(q8_mag_fast(v[4], d, rc), q8_mag_fast(v[5], d, rc), q8_mag_fast(v[6], d, rc),
                          q8_mag_fast(v[7], d, rc), wb[2], wb[3]);
        } else {
            d = __fdiv_rn(amax, 127.0f);
            if (amax != 0.0f) {
                lo = q8_pack4(q8_mag_div(v[0], d), q8_mag_div(v[1], d), q8_mag_div(v[2], d), q8_mag_div(v[3], d),
                              wb[0], wb[1]);
                hi = q8_pack4(q8_mag_div(v[4], d), q8_mag_div(v[5], d), q8_mag_div(v[6], d), q8_mag_div(v[7], d),
                              wb[2], wb[3]);
            }
        }
        int sum = __dp4a((int)hi, 0x01010101, __dp4a((int)lo, 0x01010101, 0));
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        *reinterpret_cast<uint2*>(codes + r * kp + c0) = make_uint2(lo, hi);
        if ((threadIdx.x & 3) == 0) ds[r * (kp / 32) + c0 / 32] = make_float2(d, __fmul_rn(d, (float)sum));
    }
}

// -------------------------------------------------------------------------------------
// q8_1 for k % 256 == 0 (then kp == k and the rows of x, of the codes and of the (d, s)
// pairs are each one flat array): the flat value range is cut into units of Q8U values,
// copied into shared memory by one bulk copy each (a ring of Q8S stages per CTA, refilled by
// a producer warp), so that the bytes in flight do not depend on the consumers' registers.
// Units are 16 KB because a bulk request costs the SM a roughly fixed time (4 KB ones held
// the whole GPU near 2.7 TB/s).  One consumer thread takes one 32-value block: its amax
// from BF16 pair maxima, its codes (the exact arithmetic above), the sum of its codes by
// dp4a, and its (d, s) pair.
// -------------------------------------------------------------------------------------
static __device__ unsigned int g_q8_status;

unsigned int q8_status_take() {
    unsigned int v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_q8_status, sizeof v);
    cudaMemcpyToSymbol(g_q8_status, &zero, sizeof zero);
    return v;
}

constexpr int Q8U = 8192;                // values per unit (16 KB of BF16 in)
constexpr int Q8S = 3;                   // ring stages per CTA
constexpr int Q8C = Q8U / 32;           // consumer threads (one 32-value block each)
constexpr int Q8T = Q8C + 32;            // plus one producer warp
constexpr int Q8_CTAS_PER_SM = 4;
constexpr int Q8_SMEM = Q8S * Q8U * 2 + 2 * Q8S * 8;

// Producer warp of the flat q8_1 kernels: one bulk copy per unit into the ring.
__device__ __forceinline__ void q8_produce(const uint16_t* __restrict__ x, uint8_t (*stage)[Q8U * 2], uint64_t* full,
                                           uint64_t* empty, int64_t total) {
    const int64_t units = (total + Q8U - 1) / Q8U;
    int64_t i = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x, i++) {
        const int s = (int)(i % Q8S);
        if (i >= Q8S && !mbar_wait_suspend(&empty[s], (uint32_t)((i / Q8S - 1) & 1))) {
            ok = false;
            break;
        }
        const int64_t len = min((int64_t)Q8U, total - u * Q8U);
        mbar_arrive_expect_tx(&full[s], (uint32_t)(len * 2));
        bulk_load(stage[s], x + u * Q8U, (uint32_t)(len * 2), &full[s]);
    }
    // every copy issued has landed before the CTA ends (the consumers waited for all of them
    // unless one gave up)
    for (int64_t j = (i > Q8S ? i - Q8S : 0); j < i; j++)
        if (!mbar_wait_suspend(&full[j % Q8S], (uint32_t)((j / Q8S) & 1))) ok = false;
    if (!ok) atomicOr(&g_q8_status, 1u);
}

// One consumer thread per 32-value block: the block's four 16-byte chunks are read in an
// order rotated by (thread / 2) % 4, which puts the eight threads of each shared-memory
// phase on distinct banks, and its codes are stored in that order.
__global__ void __launch_bounds__(Q8T, Q8_CTAS_PER_SM)
    q8_1_block_kernel(const uint16_t* __restrict__ x, int8_t* __restrict__ codes, float2* __restrict__ ds,
                      int64_t total) {
    extern __shared__ __align__(128) uint8_t q8_smem[];
    uint8_t(*stage)[Q8U * 2] = reinterpret_cast<uint8_t(*)[Q8U * 2]>(q8_smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(q8_smem + Q8S * Q8U * 2);
    uint64_t* empty = full + Q8S;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t units = (total + Q8U - 1) / Q8U;
    if (tid < Q8S) {
        mbar_init(&full[tid], 1);
        mbar_init(&empty[tid], Q8C / 32);
    }
    fence_barrier_init();
    __syncthreads();
    // programmatic dependent launch: the set-up above may overlap the previous kernel on the
    // stream; x and the output are touched only once that kernel has completed
    pdl_wait();
    pdl_launch_dependents();
    if (warp == Q8C / 32) {
        if (lane == 0) q8_produce(x, stage, full, empty, total);
        return;
    }
    const int rot = (tid >> 1) & 3;
    int64_t i = 0;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x, i++) {
        const int s = (int)(i % Q8S);
        const bool ok = mbar_wait_suspend(&full[s], (uint32_t)((i / Q8S) & 1));
        if (__any_sync(0xffffffffu, !ok)) {
            if (lane == 0) atomicOr(&g_q8_status, 2u);
            break;
        }
        const int64_t len = min((int64_t)Q8U, total - u * Q8U);  // a multiple of 256
        if (32 * tid < len) {
            uint4 c[4];
#pragma unroll
            for (int j = 0; j < 4; j++)
                c[j] = *reinterpret_cast<const uint4*>(stage[s] + 64 * tid + 16 * ((j + rot) & 3));
            __nv_bfloat162 m2 = bits_bf162(c[0].x & 0x7FFF7FFFu);
#pragma unroll
            for (int j = 0; j < 4; j++) {
                if (j) m2 = __hmax2(m2, bits_bf162(c[j].x & 0x7FFF7FFFu));
                m2 = __hmax2(m2, bits_bf162(c[j].y & 0x7FFF7FFFu));
                m2 = __hmax2(m2, bits_bf162(c[j].z & 0x7FFF7FFFu));
                m2 = __hmax2(m2, bits_bf162(c[j].w & 0x7FFF7FFFu));
            }
            const uint32_t mb = bf162_bits(m2);
            const float amax = fmaxf(__uint_as_float(mb << 16), __uint_as_float(mb & 0xFFFF0000u));
            float d;
            uint32_t pk[8];
#pragma unroll
            for (int j = 0; j < 8; j++) pk[j] = 0;
            if (amax >= 0x1p-94f) {
                d = q8_scale(amax);
                const float r = __frcp_rn(d);
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const uint4 w = c[j];
                    pk[2 * j] = q8_pack4(q8_mag_fast(__uint_as_float(w.x << 16), d, r),
                                         q8_mag_fast(__uint_as_float(w.x & 0xFFFF0000u), d, r),
                                         q8_mag_fast(__uint_as_float(w.y << 16), d, r),
                                         q8_mag_fast(__uint_as_float(w.y & 0xFFFF0000u), d, r), w.x, w.y);
                    pk[2 * j + 1] = q8_pack4(q8_mag_fast(__uint_as_float(w.z << 16), d, r),
                                             q8_mag_fast(__uint_as_float(w.z & 0xFFFF0000u), d, r),
                                             q8_mag_fast(__uint_as_float(w.w << 16), d, r),
                                             q8_mag_fast(__uint_as_float(w.w & 0xFFFF0000u), d, r), w.z, w.w);
                }
            } else {
                d = __fdiv_rn(amax, 127.0f);
                if (amax != 0.0f) {
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const uint4 w = c[j];
                        pk[2 * j] = q8_pack4(q8_mag_div(__uint_as_float(w.x << 16), d),
                                             q8_mag_div(__uint_as_float(w.x & 0xFFFF0000u), d),
                                             q8_mag_div(__uint_as_float(w.y << 16), d),
                                             q8_mag_div(__uint_as_float(w.y & 0xFFFF0000u), d), w.x, w.y);
                        pk[2 * j + 1] = q8_pack4(q8_mag_div(__uint_as_float(w.z << 16), d),
                                                 q8_mag_div(__uint_as_float(w.z & 0xFFFF0000u), d),
                                                 q8_mag_div(__uint_as_float(w.w << 16), d),
                                                 q8_mag_div(__uint_as_float(w.w & 0xFFFF0000u), d), w.z, w.w);
                    }
                }
            }
            int sum = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) sum = __dp4a((int)pk[j], 0x01010101, sum);
            int8_t* dst = codes + u * Q8U + 32 * tid;
#pragma unroll
            for (int j = 0; j < 4; j++)
                *reinterpret_cast<uint2*>(dst + 8 * ((j + rot) & 3)) = make_uint2(pk[2 * j], pk[2 * j + 1]);
            ds[u * (Q8U / 32) + tid] = make_float2(d, __fmul_rn(d, (float)sum));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

// =====================================================================================
// NVFP4 -> BF16: w = e2m1(code) * e4m3(scale) * scale2, the exact product rounded once to
// BF16.  Layout: codes [n][k/2] bytes (value 2j in the low nibble of byte j), one E4M3
// scale byte per 16 values [n][k/16].  (The page launches one CTA of 256 threads per row;
// here one thread takes one 16-value group of the flattened weight, see below.)
// e2m1 * e4m3 is exact in fp32; the product with scale2 is taken with round-to-odd in
// fp32 (truncate, then set the last bit if the FMA residual is nonzero), and rounding
// that to BF16 to nearest equals rounding the exact product once, because fp32 carries
// more than two extra bits (Boldo and Melquiond, "When double rounding is odd", 2005).
// Nonzero magnitudes below 2^-120 (near the BF16 subnormal range, where the residual may be
// inexact) take the exact fp64 product instead.  (A zero code gives an exact signed zero on
// the fast path; a product that underflows fp32 to zero rounds to the same signed zero in
// BF16.)
// Source: q4k_mmq.rs, `dequant_nvfp4_to_bf16`.
// =====================================================================================
__device__ __forceinline__ float nv_e2m1(uint32_t c) {  // OCP FP4 E2M1
    const uint32_t e = (c >> 1) & 3u, m = c & 1u;
    const float mag = e == 0 ? 0.5f * (float)m : __uint_as_float(((e + 126u) << 23) | (m << 22));
    return (c & 8u) ? -mag : mag;
}

__device__ __forceinline__ float nv_e4m3(uint32_t b) {  // OCP FP8 E4M3 (0x7F / 0xFF: NaN)
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    float mag = e == 0 ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
    if (e == 15u && m == 7u) mag = __uint_as_float(0x7FC00000u);
    return (b & 0x80u) ? -mag : mag;
}

// Fast path: BF16 bits of the product, and whether it needs the exact path instead.
__device__ __forceinline__ uint32_t nv_bf16_fast(float a, float s2, uint32_t& tiny) {
    const float p = __fmul_rz(a, s2);
    const float r = __fmaf_rn(a, s2, -p);  // exact residual of the truncated product
    tiny = (p != 0.0f && fabsf(p) < 0x1p-120f) ? 1u : 0u;
    const __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(__float_as_uint(p) | (r != 0.0f ? 1u : 0u)));
    return *reinterpret_cast<const uint16_t*>(&h);
}

__device__ __forceinline__ uint32_t nv_bf16_exact(float a, float s2) {
    const __nv_bfloat16 h = __double2bfloat16((double)a * (double)s2);  // exact product (<= 30 bits)
    return *reinterpret_cast<const uint16_t*>(&h);
}

// One 32-bit word of codes (8 values) through the group's table: lo / hi hold the low and
// high bytes of T[0..7], T[i] the BF16 of e2m1 magnitude i (0, .5, 1, 1.5, 2, 3, 4, 6) times
// sc * scale2; each nibble's low three bits index T by byte permutes, its bit 3 flips the
// sign.  o[0..3] receive values (0, 1) .. (6, 7) of the word.
__device__ __forceinline__ void nv_word_lookup(uint32_t w, uint32_t lo0, uint32_t lo1, uint32_t hi0, uint32_t hi1,
                                               uint32_t* o) {
    const uint32_t v = w << 4;  // byte k of v carries the sign of byte k's low nibble in bit 7
#pragma unroll
    for (int p = 0; p < 2; p++) {
        const uint32_t sel = (w >> (16 * p)) & 0x7777u;  // magnitude indices of four values
        const uint32_t a = __byte_perm(lo0, lo1, sel), b = __byte_perm(hi0, hi1, sel);
        const uint32_t s0 = __byte_perm(w, v, p ? 0x2060u : 0x0040u);  // signs of values 4p, 4p + 1
        const uint32_t s1 = __byte_perm(w, v, p ? 0x3070u : 0x1050u);  // and 4p + 2, 4p + 3
        o[2 * p] = __byte_perm(a, b, 0x5140u) ^ (s0 & 0x80008000u);
        o[2 * p + 1] = __byte_perm(a, b, 0x7362u) ^ (s1 & 0x80008000u);
    }
}

// The [n][k] weight is a flat sequence of n k / 16 groups of 16 values (8 code bytes, one
// scale byte, 32 output bytes), contiguous across rows; a full-occupancy grid strides over
// them, so a warp reads 256 contiguous code bytes and writes 1 KB per step.
// Per group the sixteen products are power-of-two multiples of Q = sc * scale2 or of 1.5 Q,
// so two exactly rounded values b1 = BF16(Q) and b3 = BF16(1.5 Q) give all eight magnitudes
// by exponent adds (exact while the results stay normal BF16 numbers); groups where they
// would not (zero, huge or tiny Q, a NaN scale) take the per-value path.
// One group: 16 values from their 8 code bytes c and E4M3 scale byte, stored as 32 bytes.
__device__ __forceinline__ void nvfp4_group(uint2 c, uint32_t sbyte, float scale2, uint16_t* __restrict__ out) {
    const float sc = nv_e4m3(sbyte);
    uint32_t o[8];
    uint32_t t1, t3;
    const uint32_t b1 = nv_bf16_fast(sc, scale2, t1);
    const uint32_t b3 = nv_bf16_fast(1.5f * sc, scale2, t3);  // 1.5 sc is exact
    const uint32_t e1 = (b1 >> 7) & 0xFFu, e3 = (b3 >> 7) & 0xFFu;
    if ((t1 | t3) == 0u && e1 >= 2u && e1 <= 252u && e3 >= 1u && e3 <= 252u) {
        // T = (+-0, Q/2, Q, 1.5Q, 2Q, 3Q, 4Q, 6Q) as BF16, the zero with Q's sign
        const uint32_t p01 = (b1 & 0x8000u) | ((b1 - 128u) << 16), p23 = b1 | (b3 << 16);
        const uint32_t p45 = (b1 + 128u) | ((b3 + 128u) << 16), p67 = (b1 + 256u) | ((b3 + 256u) << 16);
        const uint32_t lo0 = __byte_perm(p01, p23, 0x6420u), hi0 = __byte_perm(p01, p23, 0x7531u);
        const uint32_t lo1 = __byte_perm(p45, p67, 0x6420u), hi1 = __byte_perm(p45, p67, 0x7531u);
        nv_word_lookup(c.x, lo0, lo1, hi0, hi1, o);
        nv_word_lookup(c.y, lo0, lo1, hi0, hi1, o + 4);
    } else {
        float a[16];
        uint32_t tiny = 0;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const uint32_t byte = ((j < 4 ? c.x : c.y) >> (8 * (j & 3))) & 0xFFu;
            a[2 * j] = nv_e2m1(byte & 15u) * sc;  // exact
            a[2 * j + 1] = nv_e2m1(byte >> 4) * sc;
            uint32_t u0, u1;
            o[j] = nv_bf16_fast(a[2 * j], scale2, u0) | (nv_bf16_fast(a[2 * j + 1], scale2, u1) << 16);
            tiny |= (u0 << (2 * j)) | (u1 << (2 * j + 1));
        }
#pragma unroll
        for (int e = 0; e < 16; e++) {  // products near the BF16 subnormal range, exactly
            if ((tiny >> e) & 1u) {
                const uint32_t v = nv_bf16_exact(a[e], scale2);
                o[e >> 1] = (e & 1) ? ((o[e >> 1] & 0xFFFFu) | (v << 16)) : ((o[e >> 1] & 0xFFFF0000u) | v);
            }
        }
    }
    uint4* dst = reinterpret_cast<uint4*>(out);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// Two groups a thread per step (g and g + stride), both groups' loads issued first.
__global__ void __launch_bounds__(256) nvfp4_dequant_kernel(const uint8_t* __restrict__ packed,
                                                            const uint8_t* __restrict__ scales,
                                                            uint16_t* __restrict__ out, float scale2,
                                                            int64_t ngroups) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < ngroups; g += 2 * stride) {
        const int64_t g2 = g + stride;
        const uint2 c1 = __ldg(reinterpret_cast<const uint2*>(packed + 8 * g));
        const uint32_t s1 = __ldg(scales + g);
        uint2 c2 = make_uint2(0u, 0u);
        uint32_t s2 = 0;
        if (g2 < ngroups) {
            c2 = __ldg(reinterpret_cast<const uint2*>(packed + 8 * g2));
            s2 = __ldg(scales + g2);
        }
        nvfp4_group(c1, s1, scale2, out + 16 * g);
        if (g2 < ngroups) nvfp4_group(c2, s2, scale2, out + 16 * g2);
    }
}

// =====================================================================================
// SiLU(gate) * up -> BF16 (silu_mul1 in common.cuh).
// Source: dense_ffn_decode_batch.rs, `forward_km_q2` (`silu_mul`).
// =====================================================================================
template <bool VEC>
__global__ void __launch_bounds__(256) silu_mul_kernel(const uint16_t* __restrict__ gate, const uint16_t* __restrict__ up,
                                                       uint16_t* out, int64_t count) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if (VEC) {
        for (int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; id < count / 8; id += stride) {
            const uint4 g = *reinterpret_cast<const uint4*>(gate + 8 * id);
            const uint4 u = *reinterpret_cast<const uint4*>(up + 8 * id);
            const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const float a = silu_mul1(__uint_as_float(gw[j] << 16), __uint_as_float(uw[j] << 16));
                const float b = silu_mul1(__uint_as_float(gw[j] & 0xFFFF0000u), __uint_as_float(uw[j] & 0xFFFF0000u));
                o[j] = bf162_bits(__floats2bfloat162_rn(a, b));
            }
            *reinterpret_cast<uint4*>(out + 8 * id) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    } else {
        for (int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; id < count; id += stride) {
            const float h = silu_mul1(bf16_bits_to_f32(gate[id]), bf16_bits_to_f32(up[id]));
            const __nv_bfloat16 b = __float2bfloat16_rn(h);
            out[id] = *reinterpret_cast<const uint16_t*>(&b);
        }
    }
}

// =====================================================================================
// BF16 -> block_q4_K, one thread per 256-value block (the page's launch: block 128).
// Min/max quantiser; every decision is one IEEE fp32 operation (explicit _rn intrinsics)
// and fp16 conversions round to nearest even.
// Source: q4k_mmq.rs, `quantize_weight_q4k`.
// =====================================================================================
__global__ void __launch_bounds__(128) q4k_quant_kernel(const uint16_t* __restrict__ w, uint8_t* __restrict__ out,
                                                        int64_t n, int64_t k) {
    const int64_t nsb = k / 256;
    const int64_t total = n * nsb;
    const int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (id >= total) return;
    const int64_t r = id / nsb, sb = id % nsb;
    const uint16_t* src = w + r * k + sb * 256;
    uint8_t* blk = out + id * 144;

    float scale[8], negmin[8], max_scale = 0.0f, max_min = 0.0f;
    for (int j = 0; j < 8; j++) {
        float lo = bf16_bits_to_f32(src[32 * j]), hi = lo;
        for (int l = 1; l < 32; l++) {
            const float v = bf16_bits_to_f32(src[32 * j + l]);
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        if (lo > 0.0f) lo = 0.0f;
        scale[j] = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
        negmin[j] = -lo;
        if (scale[j] > max_scale) max_scale = scale[j];
        if (negmin[j] > max_min) max_min = negmin[j];
    }
    const __half dh = __float2half_rn(__fdiv_rn(max_scale, 63.0f));
    const __half mh = __float2half_rn(__fdiv_rn(max_min, 63.0f));
    const float d = __half2float(dh), dmin = __half2float(mh);
    int sc[8], mn[8];
    for (int j = 0; j < 8; j++) {
        sc[j] = d > 0.0f ? max(0, min(63, (int)roundf(__fdiv_rn(scale[j], d)))) : 0;
        mn[j] = dmin > 0.0f ? max(0, min(63, (int)roundf(__fdiv_rn(negmin[j], dmin)))) : 0;
    }
    const uint16_t dbits = *reinterpret_cast<const uint16_t*>(&dh), mbits = *reinterpret_cast<const uint16_t*>(&mh);
    uint32_t head = (uint32_t)dbits | ((uint32_t)mbits << 16);
    uint8_t s12[12];
    for (int j = 0; j < 4; j++) {
        s12[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        s12[j + 4] = (uint8_t)((mn[j] & 63) | ((mn[j + 4] >> 4) << 6));
    }
    for (int j = 4; j < 8; j++) s12[j + 4] = (uint8_t)((sc[j] & 15) | ((mn[j] & 15) << 4));
    // 144-byte blocks are 16-byte aligned (144 = 9 * 16) when the output base is.
    uint32_t words[36];
    words[0] = head;
    for (int i = 0; i < 3; i++)
        words[1 + i] = (uint32_t)s12[4 * i] | ((uint32_t)s12[4 * i + 1] << 8) | ((uint32_t)s12[4 * i + 2] << 16) |
                       ((uint32_t)s12[4 * i + 3] << 24);
    for (int c = 0; c < 4; c++) {
        const int j0 = 2 * c, j1 = 2 * c + 1;
        const float ds0 = __fmul_rn(d, (float)sc[j0]), dm0 = __fmul_rn(dmin, (float)mn[j0]);
        const float ds1 = __fmul_rn(d, (float)sc[j1]), dm1 = __fmul_rn(dmin, (float)mn[j1]);
        for (int l4 = 0; l4 < 8; l4++) {
            uint32_t word = 0;
            for (int b = 0; b < 4; b++) {
                const int l = 4 * l4 + b;
                int q0 = 0, q1 = 0;
                if (ds0 > 0.0f)
                    q0 = max(0, min(15, (int)roundf(__fdiv_rn(__fadd_rn(bf16_bits_to_f32(src[32 * j0 + l]), dm0), ds0))));
                if (ds1 > 0.0f)
                    q1 = max(0, min(15, (int)roundf(__fdiv_rn(__fadd_rn(bf16_bits_to_f32(src[32 * j1 + l]), dm1), ds1))));
                word |= (uint32_t)(q0 | (q1 << 4)) << (8 * b);
            }
            words[4 + 8 * c + l4] = word;
        }
    }
    uint4* dst = reinterpret_cast<uint4*>(blk);
    for (int i = 0; i < 9; i++) dst[i] = make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]);
}

static int grid_for(int64_t work_items, int threads) {
    const int64_t want = (work_items + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count() * 16;  // grid-stride beyond 16 CTAs per SM
    return (int)(want < 1 ? 1 : (want > cap ? cap : want));
}

}  // namespace bq8

using namespace bq8;

extern "C" {

int bq_q2_pack(const uint8_t* codes, const uint16_t* scales, void* out, uint32_t n, uint32_t k, uint32_t group,
               bq_stream_t stream) {
    if (group == 0 || group % 128 != 0 || k % 128 != 0 || k % group != 0)
        return fail(BQ_ERR_INVALID, "bq_q2_pack: need k %% 128 == 0, group %% 128 == 0, k %% group == 0 (k=%u group=%u)",
                    k, group);
    if (n == 0 || k == 0) return ok();
    if (!codes || !scales || !out) return fail(BQ_ERR_INVALID, "bq_q2_pack: NULL pointer");
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(out))
        return fail(BQ_ERR_INVALID, "bq_q2_pack: pointers must be 16-byte aligned");
    const int64_t nsc = (int64_t)n * (k / group);
    const int64_t work = (int64_t)n * (k / 16) > nsc ? (int64_t)n * (k / 16) : nsc;
    q2_pack_kernel<<<grid_for(work, 256), 256, 0, (cudaStream_t)stream>>>(codes, scales, (uint8_t*)out, n, k, nsc);
    return check_launch("bq_q2_pack");
}

int dequant_q2_to_bf16(const bq_q2_weight* w, uint16_t* out, bq_stream_t stream) {
    int st = check_q2(w, "dequant_q2_to_bf16");
    if (st) return st;
    if (w->n == 0 || w->k == 0) return ok();
    if (!out || !aligned16(out)) return fail(BQ_ERR_INVALID, "dequant_q2_to_bf16: out NULL or not 16-byte aligned");
    const int64_t work = (int64_t)w->n * (w->k / 32);
    q2_dequant_kernel<<<grid_for(work, 256), 256, 0, (cudaStream_t)stream>>>((const uint8_t*)w->data, out, w->n, w->k,
                                                                            (int)w->group);
    return check_launch("dequant_q2_to_bf16");
}

int quantize_act_q8_1(const uint16_t* x, void* act_q8, uint32_t m, uint32_t k, bq_stream_t stream) {
    if (m == 0 || k == 0) return ok();
    if (!x || !act_q8) return fail(BQ_ERR_INVALID, "quantize_act_q8_1: NULL pointer");
    if (!aligned16(x) || !aligned16(act_q8))
        return fail(BQ_ERR_INVALID, "quantize_act_q8_1: pointers must be 16-byte aligned");
    const int64_t kp = ((int64_t)k + 255) / 256 * 256;
    int8_t* codes = (int8_t*)act_q8;
    float2* ds = (float2*)((uint8_t*)act_q8 + (int64_t)m * kp);
    if (k % 256 == 0) {
        const int64_t total = (int64_t)m * k;
        const int64_t units = (total + Q8U - 1) / Q8U;
        const int64_t cap = (int64_t)sm_count() * Q8_CTAS_PER_SM;
        static int configured[64] = {};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
            return fail(BQ_ERR_LAUNCH, "quantize_act_q8_1: no current CUDA device");
        if (!configured[dev]) {
            if (cudaFuncSetAttribute(q8_1_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Q8_SMEM) !=
                cudaSuccess)
                return fail(BQ_ERR_LAUNCH, "quantize_act_q8_1: cannot reserve %d bytes of shared memory", Q8_SMEM);
            configured[dev] = 1;
        }
        // launched with programmatic stream serialization: its CTAs may start while the previous
        // kernel drains and wait (griddepcontrol) before they touch memory
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(units < cap ? units : cap));
        cfg.blockDim = dim3(Q8T);
        cfg.dynamicSmemBytes = Q8_SMEM;
        cfg.stream = (cudaStream_t)stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t le = cudaLaunchKernelEx(&cfg, q8_1_block_kernel, x, codes, ds, (int64_t)total);
        if (le != cudaSuccess) {
            (void)cudaGetLastError();  // clear it: the failure is reported here
            return fail(le == cudaErrorNoKernelImageForDevice || le == cudaErrorInvalidDeviceFunction
                            ? BQ_ERR_UNSUPPORTED
                            : BQ_ERR_LAUNCH,
                        "quantize_act_q8_1: launch failed: %s", cudaGetErrorString(le));
        }
        return check_launch("quantize_act_q8_1");
    }
    const int64_t work = (int64_t)m * kp / 8;
    if (k % 8 == 0)
        q8_1_kernel<true><<<grid_for(work, 256), 256, 0, (cudaStream_t)stream>>>(x, codes, ds, m, k, kp);
    else
        q8_1_kernel<false><<<grid_for(work, 256), 256, 0, (cudaStream_t)stream>>>(x, codes, ds, m, k, kp);
    return check_launch("quantize_act_q8_1");
}

int dequant_nvfp4_to_bf16(const void* packed, const void* scales, uint16_t* out, float scale2, uint32_t n,
                          uint32_t k, bq_stream_t stream) {
    const char* who = "dequant_nvfp4_to_bf16";
    if (k % 16 != 0) return fail(BQ_ERR_INVALID, "%s: k = %u must be a multiple of 16", who, k);
    if (n == 0 || k == 0) return ok();
    if (!packed || !scales || !out) return fail(BQ_ERR_INVALID, "%s: NULL pointer", who);
    if (!aligned16(packed) || !aligned16(out))
        return fail(BQ_ERR_INVALID, "%s: packed and out must be 16-byte aligned", who);
    if (n > 0x7FFFFFFFu || k > (1u << 30)) return fail(BQ_ERR_INVALID, "%s: shape too large", who);
    const int64_t ngroups = (int64_t)n * (k / 16);
    nvfp4_dequant_kernel<<<grid_for(ngroups, 256), 256, 0, (cudaStream_t)stream>>>(
        (const uint8_t*)packed, (const uint8_t*)scales, out, scale2, ngroups);
    return check_launch(who);
}

int silu_mul_bf16(const uint16_t* gate, const uint16_t* up, uint16_t* out, size_t count, bq_stream_t stream) {
    if (count == 0) return ok();
    if (!gate || !up || !out) return fail(BQ_ERR_INVALID, "silu_mul_bf16: NULL pointer");
    const bool vec = aligned16(gate) && aligned16(up) && aligned16(out) && count % 8 == 0;
    if (vec)
        silu_mul_kernel<true><<<grid_for((int64_t)count / 8, 256), 256, 0, (cudaStream_t)stream>>>(gate, up, out, count);
    else
        silu_mul_kernel<false><<<grid_for((int64_t)count, 256), 256, 0, (cudaStream_t)stream>>>(gate, up, out, count);
    return check_launch("silu_mul_bf16");
}

int quantize_weight_q4k(const uint16_t* w, void* out_q4k, uint32_t n, uint32_t k, bq_stream_t stream) {
    if (k % 256 != 0) return fail(BQ_ERR_INVALID, "quantize_weight_q4k: k %u must be a multiple of 256", k);
    if (n == 0 || k == 0) return ok();
    if (!w || !out_q4k || !aligned16(w) || !aligned16(out_q4k))
        return fail(BQ_ERR_INVALID, "quantize_weight_q4k: pointers must be non-NULL and 16-byte aligned");
    const int64_t total = (int64_t)n * (k / 256);
    const int64_t blocks = (total + 127) / 128;
    if (blocks > 0x7fffffff) return fail(BQ_ERR_INVALID, "quantize_weight_q4k: weight too large");
    q4k_quant_kernel<<<(unsigned)blocks, 128, 0, (cudaStream_t)stream>>>(w, (uint8_t*)out_q4k, n, k);
    return check_launch("quantize_weight_q4k");
}

}  // extern "C"
