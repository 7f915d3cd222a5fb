/*
 * bq8_oracle.c -- plain, slow CPU oracle for the quantized-weight linear projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or calls
 * this file; only the tests, the package's smoke check and the bench's CPU-baseline
 * leg use it.  It shares no code, header, table or constant generator with the CUDA
 * path.
 *
 * Every floating-point result that is not fixed by a format is computed in fp64 with
 * plain loops, in the order of the definition.  Where a floating-point step decides an
 * integer (a q8_1 code, a Q4_K scale or code) the step is taken in fp32, the precision
 * the formats store, and the file is compiled with -ffp-contract=off so that no
 * multiply-add is fused behind our back.
 *
 * Sources (page title, section):
 *  - metrale_model_layers/layers/qwen3_ssm/init_q2.rs, `qkvz_q2_prefill_gemm`:
 *    out[m, n] = input[m, k] @ W^T; packed Q2_0 weight with group size 128; the
 *    dequantise-to-BF16 fallback and the q8_1 + MMQ route compute the same product.
 *  - metrale_model_layers/layers/ops/q4k_mmq.rs, `QK_K`, `Q4K_BLOCK_BYTES`,
 *    `q4k_weight_bytes`, `quantize_act_q8_1`, `q4k_mmq_gemm`: 256-value / 144-byte
 *    blocks, k padded to 256 for q8_1, C[m, n] = A[m, k] x W[n, k] with a BF16 store.
 *  - metrale_model_layers/layers/dense_ffn_decode_batch.rs, `forward_km_q2`:
 *    gate and up GEMV, SiLU(gate) * up written over the gate buffer, then down GEMV.
 *
 * The pages do not print the Q2_0 byte layout, the q8_1 rounding rules or the Q4_K
 * quantiser; the readings taken here are stated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define Q2_PACK 128         /* codes per 32-byte pack block of a Q2_0 row */
#define Q8_BLOCK 32         /* values per q8_1 block */
#define KPAD_UNIT 256       /* q8_1 rows are padded to a multiple of QK_K = 256 */
#define QK_K 256            /* values per block_q4_K */
#define Q4K_BYTES 144       /* sizeof(block_q4_K) */

/* ------------------------------------------------------------------------------ */
/* number formats                                                                 */
/* ------------------------------------------------------------------------------ */

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* BF16 is the top half of an IEEE binary32. */
float orc_bf16_to_f32(uint16_t h) { return bits_to_f32((uint32_t)h << 16); }

/* Round a real (held exactly in a double) to the nearest value with `prec` significant
 * bits, ties to even, with the smallest quantum 2^qmin (subnormal range).  Returns the
 * rounded value; the caller encodes it. */
static double round_to_precision(double a, int prec, int qmin) {
    int e;
    frexp(a, &e);                 /* a in [2^(e-1), 2^e) */
    int q = (e - 1) - (prec - 1); /* spacing of the binade that holds a */
    if (q < qmin) q = qmin;
    return ldexp(nearbyint(ldexp(a, -q)), q); /* nearbyint: current mode, ties-to-even */
}

/* Real -> bfloat16, round to nearest even.  8 significant bits, emin -126. */
uint16_t orc_f64_to_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    double r = round_to_precision(a, 8, -133);
    if (r >= 0x1p128) return sign | 0x7F80;
    return sign | (uint16_t)(f32_to_bits((float)r) >> 16);
}

/* Real -> IEEE binary16, round to nearest even.  11 significant bits, emin -14. */
uint16_t orc_f64_to_f16(double v) {
    if (isnan(v)) return 0x7E00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    double r = round_to_precision(a, 11, -24);
    if (r > 65504.0) return sign | 0x7C00;
    if (r < 0x1p-14) return sign | (uint16_t)ldexp(r, 24); /* subnormal: r / 2^-24 */
    int e;
    frexp(r, &e); /* r in [2^(e-1), 2^e) */
    int ue = e - 1;
    uint16_t mant = (uint16_t)(ldexp(r, 10 - ue) - 1024.0);
    return sign | (uint16_t)((ue + 15) << 10) | mant;
}

float orc_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1, ex = (h >> 10) & 31, mant = h & 1023;
    double v;
    if (ex == 0) v = ldexp((double)mant, -24);
    else if (ex == 31) v = mant ? NAN : INFINITY;
    else v = ldexp(1024.0 + mant, ex - 25);
    return (float)(sign ? -v : v);
}

/* ------------------------------------------------------------------------------ */
/* sizes                                                                          */
/* ------------------------------------------------------------------------------ */

int64_t orc_kpad(int64_t k) { return (k + KPAD_UNIT - 1) / KPAD_UNIT * KPAD_UNIT; }

/* Q2_0: n*k/4 bytes of codes, then n*(k/group) BF16 scales. */
int64_t orc_q2_bytes(int64_t n, int64_t k, int64_t group) { return n * k / 4 + n * (k / group) * 2; }

/* q8_1: m*kp int8 codes, then m*kp/32 (d, s) float pairs. */
int64_t orc_q8_1_bytes(int64_t m, int64_t k) { int64_t kp = orc_kpad(k); return m * kp + m * (kp / Q8_BLOCK) * 8; }

/* q4k_mmq.rs, `q4k_weight_bytes`: nrows * (n_per_row / 256) * 144. */
int64_t orc_q4k_bytes(int64_t n, int64_t k) { return n * (k / QK_K) * Q4K_BYTES; }

/* ------------------------------------------------------------------------------ */
/* Q2_0 layout (fixed here; the pages name the format and group 128 only)         */
/*                                                                                */
/* A row of k codes is cut into pack blocks of 128 consecutive codes, 32 bytes    */
/* each.  Byte l (0..31) of pack block p holds the codes of columns               */
/* 128p + 32i + l for i = 0..3, the code of sub-block i in bits 2i..2i+1.  The     */
/* codes plane is [n][k/4] bytes; the BF16 scale plane [n][k/group] follows it.   */
/* Decode (affine, offset 2 = 2^(bits-1)): w = d * (c - 2).                        */
/* ------------------------------------------------------------------------------ */

static int q2_code_at(const uint8_t* row_codes, int64_t col) {
    int64_t p = col / Q2_PACK, r = col % Q2_PACK;
    int64_t i = r / 32, l = r % 32;
    return (row_codes[p * 32 + l] >> (2 * i)) & 3;
}

void orc_q2_pack(const uint8_t* codes, const uint16_t* scales, int64_t n, int64_t k, int64_t group,
                 uint8_t* out) {
    uint8_t* plane = out;
    uint16_t* sc = (uint16_t*)(out + n * k / 4);
    for (int64_t r = 0; r < n; r++) {
        for (int64_t p = 0; p < k / Q2_PACK; p++) {
            for (int64_t l = 0; l < 32; l++) {
                uint8_t b = 0;
                for (int i = 0; i < 4; i++) b |= (uint8_t)((codes[r * k + p * Q2_PACK + 32 * i + l] & 3) << (2 * i));
                plane[r * (k / 4) + p * 32 + l] = b;
            }
        }
    }
    memcpy(sc, scales, (size_t)(n * (k / group)) * 2);
}

void orc_q2_unpack(const uint8_t* packed, int64_t n, int64_t k, int64_t group, uint8_t* codes,
                   uint16_t* scales) {
    for (int64_t r = 0; r < n; r++)
        for (int64_t c = 0; c < k; c++) codes[r * k + c] = (uint8_t)q2_code_at(packed + r * (k / 4), c);
    memcpy(scales, packed + n * k / 4, (size_t)(n * (k / group)) * 2);
}

/* The dequantised weight as an exact real: d * (c - 2). */
static double q2_weight(const uint8_t* packed, int64_t n, int64_t k, int64_t group, int64_t r, int64_t c) {
    const uint16_t* sc = (const uint16_t*)(packed + n * k / 4);
    double d = orc_bf16_to_f32(sc[r * (k / group) + c / group]);
    return d * (double)(q2_code_at(packed + r * (k / 4), c) - 2);
}

/* init_q2.rs, `qkvz_q2_prefill_gemm` fallback: dequantise to BF16.  d*(c-2) is d times
 * one of {-2,-1,0,1}, always exactly a BF16 value, so the conversion never rounds. */
void orc_q2_dequant_bf16(const uint8_t* packed, int64_t n, int64_t k, int64_t group, uint16_t* out) {
    for (int64_t r = 0; r < n; r++)
        for (int64_t c = 0; c < k; c++) out[r * k + c] = orc_f64_to_bf16(q2_weight(packed, n, k, group, r, c));
}

/* out[m, n] = input[m, k] @ Wdq^T in fp64 (the decode GEMV for m = 1..8). */
void orc_q2_gemv(const uint16_t* x, const uint8_t* packed, int64_t m, int64_t n, int64_t k, int64_t group,
                 double* y) {
#pragma omp parallel
    {
        double* wrow = (double*)malloc((size_t)k * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t r = 0; r < n; r++) {
            for (int64_t c = 0; c < k; c++) wrow[c] = q2_weight(packed, n, k, group, r, c);
            for (int64_t i = 0; i < m; i++) {
                double acc = 0.0;
                for (int64_t c = 0; c < k; c++) acc += (double)orc_bf16_to_f32(x[i * k + c]) * wrow[c];
                y[i * n + r] = acc;
            }
        }
        free(wrow);
    }
}

/* Dense BF16 GEMM of the fallback prefill route (init_q2.rs, `qkvz_q2_prefill_gemm`:
 * `dense_gemm_bf16_pipelined` after `dequant_q2_0_gn_to_bf16`): out[i][j] = sum over c of
 * a[i][c] * w[j][c], the BF16 operands taken exactly, summed in fp64 in column order. */
void orc_gemm_bf16(const uint16_t* a, const uint16_t* w, int64_t m, int64_t n, int64_t k, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < m; i++)
        for (int64_t j = 0; j < n; j++) {
            double acc = 0.0;
            for (int64_t c = 0; c < k; c++)
                acc += (double)orc_bf16_to_f32(a[i * k + c]) * (double)orc_bf16_to_f32(w[j * k + c]);
            out[i * n + j] = acc;
        }
}

/* dense_ffn_decode_batch.rs, `forward_km_q2`: SiLU(gate) * up, rounded once to BF16.
 * SiLU(z) = z * sigmoid(z) = z / (1 + e^-z). */
void orc_silu_mul_bf16(const uint16_t* gate, const uint16_t* up, int64_t count, uint16_t* out) {
    for (int64_t i = 0; i < count; i++) {
        double g = orc_bf16_to_f32(gate[i]), u = orc_bf16_to_f32(up[i]);
        out[i] = orc_f64_to_bf16(g / (1.0 + exp(-g)) * u);
    }
}

static void round_all_bf16(const double* v, int64_t count, uint16_t* out) {
    for (int64_t i = 0; i < count; i++) out[i] = orc_f64_to_bf16(v[i]);
}

/* dense_ffn_decode_batch.rs, `forward_km_q2`: the packed-Q2 FFN chain for m rows.
 * The gate/up/hidden buffers are BF16 (they are shared with the BF16 paths), so g, u and
 * h are rounded to BF16 between stages; y is returned unrounded (fp64). */
void orc_ffn_q2(const uint16_t* x, const uint8_t* gate_w, const uint8_t* up_w, const uint8_t* down_w,
                int64_t m, int64_t hidden, int64_t inter, int64_t group, uint16_t* g, uint16_t* u,
                uint16_t* h, double* y) {
    double* t = (double*)malloc((size_t)(m * inter) * sizeof(double));
    orc_q2_gemv(x, gate_w, m, inter, hidden, group, t);
    round_all_bf16(t, m * inter, g);
    orc_q2_gemv(x, up_w, m, inter, hidden, group, t);
    round_all_bf16(t, m * inter, u);
    free(t);
    orc_silu_mul_bf16(g, u, m * inter, h);
    orc_q2_gemv(h, down_w, m, hidden, inter, group, y);
}

/* ------------------------------------------------------------------------------ */
/* q8_1 activation quantisation                                                   */
/*                                                                                */
/* q4k_mmq.rs, `quantize_act_q8_1`: BF16 [m, k] -> q8_1 with k padded to 256.     */
/* Per row and 32-value block (values beyond k are 0):                            */
/*   amax = max |x|;  d = amax / 127;  q = round(x / d) (0 when amax = 0);         */
/*   s = d * sum(q).                                                              */
/* Readings: fp32 division and product, each rounded to nearest even; round()     */
/* rounds half away from zero; q clamped to [-127, 127]; d and s stored as fp32.  */
/* Layout: int8 codes [m][kp], then (d, s) float pairs [m][kp/32] at byte         */
/* offset m*kp.                                                                   */
/* ------------------------------------------------------------------------------ */

void orc_quantize_q8_1(const uint16_t* x, int64_t m, int64_t k, uint8_t* out) {
    int64_t kp = orc_kpad(k), nb = kp / Q8_BLOCK;
    int8_t* codes = (int8_t*)out;
    float* ds = (float*)(out + m * kp);
    for (int64_t r = 0; r < m; r++) {
        for (int64_t b = 0; b < nb; b++) {
            float v[Q8_BLOCK];
            float amax = 0.0f;
            for (int j = 0; j < Q8_BLOCK; j++) {
                int64_t c = b * Q8_BLOCK + j;
                v[j] = c < k ? orc_bf16_to_f32(x[r * k + c]) : 0.0f;
                float a = fabsf(v[j]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            int sum = 0;
            for (int j = 0; j < Q8_BLOCK; j++) {
                int q = 0;
                if (amax != 0.0f) {
                    float t = v[j] / d;
                    q = (int)roundf(t);
                    if (q > 127) q = 127;
                    if (q < -127) q = -127;
                }
                codes[r * kp + b * Q8_BLOCK + j] = (int8_t)q;
                sum += q;
            }
            ds[(r * nb + b) * 2 + 0] = d;
            ds[(r * nb + b) * 2 + 1] = d * (float)sum;
        }
    }
}

/* The dequantised activation d * q as an exact real. */
static double q8_value(const uint8_t* act, int64_t m, int64_t k, int64_t r, int64_t c) {
    int64_t kp = orc_kpad(k);
    const int8_t* codes = (const int8_t*)act;
    const float* ds = (const float*)(act + m * kp);
    return (double)ds[(r * (kp / Q8_BLOCK) + c / Q8_BLOCK) * 2] * (double)codes[r * kp + c];
}

/* init_q2.rs, `qkvz_q2_prefill_gemm` MMQ route: out[m, n] = q8_1(x) @ Wdq^T, the fp64 sum
 * of products of the dequantised operands.  rows[] selects which of the m activation rows
 * are computed (nrows of them); out is [nrows, n]. */
void orc_q2_mmq(const uint8_t* act, const uint8_t* packed, int64_t m, int64_t n, int64_t k, int64_t group,
                const int64_t* rows, int64_t nrows, double* out) {
#pragma omp parallel
    {
        double* wrow = (double*)malloc((size_t)k * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t r = 0; r < n; r++) {
            for (int64_t c = 0; c < k; c++) wrow[c] = q2_weight(packed, n, k, group, r, c);
            for (int64_t ii = 0; ii < nrows; ii++) {
                double acc = 0.0;
                for (int64_t c = 0; c < k; c++) acc += q8_value(act, m, k, rows[ii], c) * wrow[c];
                out[ii * n + r] = acc;
            }
        }
        free(wrow);
    }
}

/* ------------------------------------------------------------------------------ */
/* block_q4_K (q4k_mmq.rs: 256 values, 144 bytes)                                 */
/*                                                                                */
/* Bytes 0-1 fp16 d, 2-3 fp16 dmin, 4-15 the 6-bit scale sc_j and min m_j of the  */
/* eight 32-value sub-blocks, 16-143 the 4-bit codes.                              */
/* Scale bytes s[0..11]: for j < 4, sc_j = s[j] & 63 and m_j = s[j+4] & 63; for    */
/* j >= 4, sc_j = (s[j+4] & 15) | (s[j-4] >> 6) << 4 and                            */
/* m_j = (s[j+4] >> 4) | (s[j] >> 6) << 4.                                          */
/* Codes: byte 32c + l holds value l of sub-block 2c in its low nibble and value l */
/* of sub-block 2c+1 in its high nibble.                                           */
/* Decode: w = d * sc_j * q - dmin * m_j.                                           */
/* ------------------------------------------------------------------------------ */

static void q4k_get_scale_min(const uint8_t* s, int j, int* sc, int* mn) {
    if (j < 4) {
        *sc = s[j] & 63;
        *mn = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

static void q4k_put_scale_min(uint8_t* s, const int* sc, const int* mn) {
    memset(s, 0, 12);
    for (int j = 0; j < 4; j++) {
        s[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        s[j + 4] = (uint8_t)((mn[j] & 63) | ((mn[j + 4] >> 4) << 6));
    }
    for (int j = 4; j < 8; j++) s[j + 4] = (uint8_t)((sc[j] & 15) | ((mn[j] & 15) << 4));
}

void orc_q4k_pack_scales(const int32_t* sc, const int32_t* mn, uint8_t* s12) { q4k_put_scale_min(s12, sc, mn); }

void orc_q4k_unpack_scales(const uint8_t* s12, int32_t* sc, int32_t* mn) {
    for (int j = 0; j < 8; j++) {
        int a, b;
        q4k_get_scale_min(s12, j, &a, &b);
        sc[j] = a;
        mn[j] = b;
    }
}

static int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* q4k_mmq.rs, `quantize_weight_q4k` (the kernel exists on the page; its algorithm is not
 * printed).  Reading: the plain min/max quantiser, every decision in fp32:
 *   per sub-block j: mn_j = min(0, min x), scale_j = (max x - mn_j) / 15;
 *   d = fp16(max_j scale_j / 63), dmin = fp16(max_j (-mn_j) / 63);
 *   sc_j = clamp(round(scale_j / d), 0, 63)    (0 when d == 0);
 *   m_j  = clamp(round(-mn_j / dmin), 0, 63)   (0 when dmin == 0);
 *   q = clamp(round((x + dmin*m_j) / (d*sc_j)), 0, 15)   (0 when d*sc_j == 0).
 * round() is half away from zero; fp16() rounds to nearest even. */
void orc_quantize_q4k(const uint16_t* w, int64_t n, int64_t k, uint8_t* out) {
    int64_t nsb = k / QK_K;
    for (int64_t r = 0; r < n; r++) {
        for (int64_t sb = 0; sb < nsb; sb++) {
            const uint16_t* src = w + r * k + sb * QK_K;
            uint8_t* blk = out + (r * nsb + sb) * Q4K_BYTES;
            float x[QK_K];
            for (int i = 0; i < QK_K; i++) x[i] = orc_bf16_to_f32(src[i]);
            float scale[8], negmin[8], max_scale = 0.0f, max_min = 0.0f;
            for (int j = 0; j < 8; j++) {
                float lo = x[32 * j], hi = x[32 * j];
                for (int l = 1; l < 32; l++) {
                    if (x[32 * j + l] < lo) lo = x[32 * j + l];
                    if (x[32 * j + l] > hi) hi = x[32 * j + l];
                }
                if (lo > 0.0f) lo = 0.0f;
                scale[j] = (hi - lo) / 15.0f;
                negmin[j] = -lo;
                if (scale[j] > max_scale) max_scale = scale[j];
                if (negmin[j] > max_min) max_min = negmin[j];
            }
            uint16_t dh = orc_f64_to_f16((double)(max_scale / 63.0f));
            uint16_t mh = orc_f64_to_f16((double)(max_min / 63.0f));
            float d = orc_f16_to_f32(dh), dmin = orc_f16_to_f32(mh);
            int sc[8], mn[8];
            for (int j = 0; j < 8; j++) {
                sc[j] = d > 0.0f ? clampi((int)roundf(scale[j] / d), 0, 63) : 0;
                mn[j] = dmin > 0.0f ? clampi((int)roundf(negmin[j] / dmin), 0, 63) : 0;
            }
            uint8_t q[QK_K];
            for (int j = 0; j < 8; j++) {
                float dsc = d * (float)sc[j];
                float dm = dmin * (float)mn[j];
                for (int l = 0; l < 32; l++) {
                    int v = 0;
                    if (dsc > 0.0f) {
                        float t = (x[32 * j + l] + dm) / dsc;
                        v = clampi((int)roundf(t), 0, 15);
                    }
                    q[32 * j + l] = (uint8_t)v;
                }
            }
            blk[0] = (uint8_t)(dh & 0xFF);
            blk[1] = (uint8_t)(dh >> 8);
            blk[2] = (uint8_t)(mh & 0xFF);
            blk[3] = (uint8_t)(mh >> 8);
            q4k_put_scale_min(blk + 4, sc, mn);
            for (int c = 0; c < 4; c++)
                for (int l = 0; l < 32; l++)
                    blk[16 + 32 * c + l] = (uint8_t)(q[64 * c + l] | (q[64 * c + 32 + l] << 4));
        }
    }
}

/* One Q4_K weight as an exact real: d * sc_j * q - dmin * m_j. */
static double q4k_weight(const uint8_t* w, int64_t k, int64_t r, int64_t c) {
    int64_t nsb = k / QK_K;
    const uint8_t* blk = w + (r * nsb + c / QK_K) * Q4K_BYTES;
    int64_t e = c % QK_K;
    int j = (int)(e / 32), l = (int)(e % 32), ch = (int)(e / 64);
    double d = orc_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    double dmin = orc_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
    int sc, mn;
    q4k_get_scale_min(blk + 4, j, &sc, &mn);
    uint8_t byte = blk[16 + 32 * ch + l];
    int q = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
    return d * sc * q - dmin * mn;
}

void orc_dequant_q4k(const uint8_t* w, int64_t n, int64_t k, double* out) {
    for (int64_t r = 0; r < n; r++)
        for (int64_t c = 0; c < k; c++) out[r * k + c] = q4k_weight(w, k, r, c);
}

/* q4k_mmq.rs, `q4k_mmq_gemm`: C[m, n] = A[m, k] x W[n, k], fp64 sum over the dequantised
 * operands, for the selected activation rows. */
void orc_q4k_mmq(const uint8_t* act, const uint8_t* w, int64_t m, int64_t n, int64_t k, const int64_t* rows,
                 int64_t nrows, double* out) {
#pragma omp parallel
    {
        double* wrow = (double*)malloc((size_t)k * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t r = 0; r < n; r++) {
            for (int64_t c = 0; c < k; c++) wrow[c] = q4k_weight(w, k, r, c);
            for (int64_t ii = 0; ii < nrows; ii++) {
                double acc = 0.0;
                for (int64_t c = 0; c < k; c++) acc += q8_value(act, m, k, rows[ii], c) * wrow[c];
                out[ii * n + r] = acc;
            }
        }
        free(wrow);
    }
}

/* ------------------------------------------------------------------------------ */
/* NVFP4 weights (q4k_mmq.rs, `dequant_nvfp4_to_bf16`: "packed E2M1, E4M3 group      */
/* scales and the per-tensor scale2" -> BF16 [n, k], one block per row).  The page    */
/* prints the launch contract only; the readings taken here:                          */
/*  - packed [n][k/2] bytes: value 2j of a row in the low nibble of byte j, value     */
/*    2j + 1 in the high nibble;                                                      */
/*  - scales [n][k/16] E4M3 bytes, one per 16 consecutive values of a row;            */
/*  - w = e2m1(code) * e4m3(scale) * scale2, the exact real product rounded once to    */
/*    BF16 (round to nearest even).                                                   */
/* ------------------------------------------------------------------------------ */

/* FP4 E2M1 (OCP microscaling formats): bit 3 sign, bits 1-2 exponent (bias 1), bit 0 */
/* mantissa; exponent 0 is subnormal (0 or 0.5).  Magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_value(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* FP8 E4M3 (OCP 8-bit floating point): bit 7 sign, bits 3-6 exponent (bias 7), bits  */
/* 0-2 mantissa; exponent 0 is subnormal (m * 2^-9); exponent 15 with mantissa 7 is  */
/* NaN and there are no infinities, so the largest value is 448.                      */
double orc_e4m3_value(int b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

void orc_dequant_nvfp4(const uint8_t* packed, const uint8_t* scales, float scale2, int64_t n, int64_t k,
                       uint16_t* out) {
    for (int64_t r = 0; r < n; r++)
        for (int64_t c = 0; c < k; c++) {
            uint8_t byte = packed[r * (k / 2) + c / 2];
            int code = (c % 2 == 0) ? (byte & 15) : (byte >> 4);
            double w = orc_e2m1_value(code) * orc_e4m3_value(scales[r * (k / 16) + c / 16]) * (double)scale2;
            out[r * k + c] = orc_f64_to_bf16(w); /* the product has <= 30 bits: exact in fp64 */
        }
}

/* Threads the oracle's parallel loops use from now on (timing on one core). */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
