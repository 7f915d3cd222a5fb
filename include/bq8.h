/*
 * bq8.h -- C ABI of libbq8, the GB300 (sm_103a) quantized-weight linear projection.
 *
 * Every entry point follows the projection contract of the serving stack's layers,
 *     out[m, n] = input[m, k] @ W^T
 * (metrale_model_layers/layers/qwen3_ssm/init_q2.rs, `qkvz_q2_prefill_gemm`;
 *  metrale_model_layers/layers/ops/q4k_mmq.rs, `q4k_mmq_gemm`: C[m, n] = A[m, k] x W[n, k]).
 *
 * Conventions shared by all calls
 *  - All data pointers are DEVICE pointers, 16-byte aligned, rows contiguous (row-major).
 *  - BF16 and FP16 values are passed as their 16-bit patterns (uint16_t).
 *  - The caller owns every buffer; the library allocates and frees nothing (the layer
 *    method "allocates nothing", init_q2.rs `qkvz_q2_prefill_gemm`).  Scratch buffers
 *    are passed in.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream) and never synchronises.
 *  - Every call returns a status code (below).  On a nonzero status nothing was launched
 *    unless the code is BQ_ERR_LAUNCH; bq_last_error() then describes the failure (the
 *    message is per host thread and stays valid until that thread's next call).
 *  - m = 0 or n = 0 launches nothing and returns BQ_OK.  k = 0 writes zeros to `out`.
 *
 * Formats (the pages name them; where a byte layout is not printed it is fixed here)
 *  Q2_0 (bq_q2_weight, one buffer): codes plane [n][k/4] bytes, then the BF16 scale plane
 *    [n][k/group] at byte offset n*k/4.  A row is cut into pack blocks of 128 codes (32
 *    bytes); byte l of pack block p holds the 2-bit codes of columns 128p + 32i + l,
 *    i = 0..3, in bits 2i..2i+1.  Decode: w = d * (c - 2), d the scale of the column's
 *    group.  k % 128 == 0 and group % 128 == 0 and k % group == 0.
 *  q8_1 (activations): int8 codes [m][kp], kp = k rounded up to 256 (zero padded), then
 *    (d, s) float pairs [m][kp/32] at byte offset m*kp.  Per 32-value block:
 *    d = amax/127, q = round-half-away(x/d), s = d * sum(q)  (fp32, round to nearest).
 *  block_q4_K (Q4_K weights): 144 bytes per 256 values along k: fp16 d, fp16 dmin, 12
 *    bytes of 6-bit sub-block scales/mins, 128 bytes of 4-bit codes (the GGUF layout);
 *    w = d * sc_j * q - dmin * m_j for sub-block j.
 */
#ifndef BQ8_H
#define BQ8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream, declared without the CUDA headers. */
typedef struct CUstream_st* bq_stream_t;

/* Status codes. */
enum {
    BQ_OK = 0,
    BQ_ERR_INVALID = 1,     /* null/misaligned pointer, size or shape out of range      */
    BQ_ERR_UNSUPPORTED = 2, /* no kernel image for this device (the library is sm_103a) */
    BQ_ERR_LAUNCH = 3,      /* the CUDA launch itself failed                            */
    BQ_ERR_DEVICE = 4       /* a device-side check or bounded wait reported failure     */
};

/* A packed Q2_0 weight: codes plane followed by the scale plane in one device buffer.
 * (init_q2.rs, `set_packed_q2_qkvz`: PackedQ2Weight { weight, n, k, group }.) */
typedef struct bq_q2_weight {
    const void* data;
    uint32_t n, k, group;
} bq_q2_weight;

/* ---------------------------------------------------------------- sizes (host only) */

/* Bytes of a Q2_0 weight: n*k/4 codes + n*(k/group)*2 scale bytes; 0 if the shape is
 * invalid. */
size_t bq_q2_weight_bytes(uint32_t n, uint32_t k, uint32_t group);

/* Bytes of a q8_1 activation buffer: m*kp codes + m*(kp/32)*8 (d, s) bytes, kp = k
 * rounded up to 256.  Always within the page's budget m*kp*4 + 1 MiB
 * (q4k_mmq.rs, `q8_1_scratch_bytes`). */
size_t bq_q8_1_bytes(uint32_t m, uint32_t k);

/* Bytes of a Q4_K weight [n, k]: n*(k/256)*144 (q4k_mmq.rs, `q4k_weight_bytes`); 0 if
 * k % 256 != 0. */
size_t bq_q4k_weight_bytes(uint32_t n, uint32_t k);

/* ---------------------------------------------------------------- weight preparation */

/* Packs 2-bit codes and group scales into the Q2_0 layout above.
 * codes:  [n][k] uint8, one code per byte (only the low 2 bits are used).
 * scales: [n][k/group] BF16.
 * out:    bq_q2_weight_bytes(n, k, group) bytes.
 * Source: init_q2.rs, `set_packed_q2_qkvz` (the packed weight it installs). */
int bq_q2_pack(const uint8_t* codes, const uint16_t* scales, void* out, uint32_t n, uint32_t k,
               uint32_t group, bq_stream_t stream);

/* Quantises BF16 weights [n][k] to block_q4_K, one 144-byte block per 256 values along
 * k (k % 256 == 0).  The quantiser: per 32-value sub-block, min clipped to 0 and
 * scale = (max - min)/15; d = fp16(max scale / 63), dmin = fp16(max -min / 63); 6-bit
 * sc and m by rounding; 4-bit codes by rounding (x + dmin*m)/(d*sc), all in fp32.
 * Source: q4k_mmq.rs, `quantize_weight_q4k` (BF16 -> block_q4_K). */
int quantize_weight_q4k(const uint16_t* w, void* out_q4k, uint32_t n, uint32_t k, bq_stream_t stream);

/* ---------------------------------------------------------------- the hot path */

/* q8_1 activation quantisation: BF16 x [m][k] -> act_q8 (bq_q8_1_bytes(m, k) bytes).
 * Bit-exact, fp32 decisions as described in the format section.  For k % 256 == 0 the
 * kernel is launched with programmatic stream serialization: its set-up may overlap the
 * previous kernel on the stream, but it reads x and writes act_q8 only after that kernel
 * has completed, so stream order holds as for any launch.
 * Source: q4k_mmq.rs, `quantize_act_q8_1` (k padded to 256). */
int quantize_act_q8_1(const uint16_t* x, void* act_q8, uint32_t m, uint32_t k, bq_stream_t stream);

/* Decode GEMV, one activation row: y[1][n] = x[1][k] @ Wdq^T, fp32 accumulation, BF16
 * store.  Source: init_q2.rs, `set_packed_q2_qkvz` (decode runs `q2_0_gemv_vec`). */
int q2_gemv(const uint16_t* x, const bq_q2_weight* w, uint16_t* y, bq_stream_t stream);

/* Batched decode GEMV for 1 <= m <= 8 rows: y[m][n] = x[m][k] @ Wdq^T.  The weight is
 * streamed once for all m rows.
 * Source: dense_ffn_decode_batch.rs, `forward_km_q2` (`q2_0_gemv_vec_batchm`). */
int q2_gemv_batchm(const uint16_t* x, const bq_q2_weight* w, uint16_t* y, uint32_t m, bq_stream_t stream);

/* out[i] = BF16(SiLU(gate[i]) * up[i]) for i < count; out may alias gate.
 * Source: dense_ffn_decode_batch.rs, `forward_km_q2` (`silu_mul` in place into the gate
 * buffer). */
int silu_mul_bf16(const uint16_t* gate, const uint16_t* up, uint16_t* out, size_t count, bq_stream_t stream);

/* Packed-Q2 dense-FFN decode for 1 <= m <= 8 rows (SiLU only):
 *   gate_scratch = x @ gate^T; up_scratch = x @ up^T (both [m][inter] BF16);
 *   gate_scratch = SiLU(gate_scratch) * up_scratch; out = gate_scratch @ down^T ([m][hidden]).
 * Shapes: gate, up: n = inter, k = hidden; down: n = hidden, k = inter.  On return (after
 * the stream drains) gate_scratch holds h and up_scratch holds u, as on the page; the two
 * must not overlap (BQ_ERR_INVALID).  Two launches: one streams the gate and up weights
 * together and forms u and h (the SiLU*mul with the same arithmetic as silu_mul_bf16 on
 * the BF16 g and u), then the down projection; where the two weights' tile pairs do not fit
 * one SM (large k at m near 8) the gate and up projections run as two launches instead.
 * Source: dense_ffn_decode_batch.rs, `forward_km_q2`. */
int ffn_q2_km(const uint16_t* x, const bq_q2_weight* gate, const bq_q2_weight* up, const bq_q2_weight* down,
              uint16_t* gate_scratch, uint16_t* up_scratch, uint16_t* out, uint32_t m, bq_stream_t stream);

/* Largest m * inter that ffn_q2_km_noalloc accepts (values per intermediate buffer). */
#define BQ_FFN_NOALLOC_MAX_ELEMS 262144u

/* ffn_q2_km for callers that cannot allocate device memory (no counterpart on the pages:
 * it exists for this library's users).  A host framework that hands a plugin only its
 * inputs and outputs, a runtime whose pool owns all device memory, or C code linked
 * without an allocator has nowhere to put ffn_q2_km's two [m][inter] intermediates; this
 * entry point keeps them in a fixed 1 MiB array inside the library's device image and calls
 * no allocator at all.  Same arguments and result as ffn_q2_km without the two scratch
 * pointers; out = SiLU(x @ gate^T) * (x @ up^T) @ down^T, [m][hidden] BF16.
 *  - m * inter must not exceed BQ_FFN_NOALLOC_MAX_ELEMS (else BQ_ERR_INVALID, nothing
 *    launched); every other check is ffn_q2_km's.
 *  - The first call on each device looks up the array's device address with that device
 *    current (cudaGetSymbolAddress) and caches it; make that first call before any stream
 *    capture on the device.  If the device's context is replaced (cudaDeviceReset), the
 *    next call looks the address up again, so make that call before any capture too.
 *  - The array is shared by every call in the process and keeps the last call's contents;
 *    calls that overlap on the GPU (other streams or host threads) race on it.  Calls on
 *    one stream are ordered and safe.  The array stays allocated on every GPU that loaded
 *    the library until the process exits. */
int ffn_q2_km_noalloc(const uint16_t* x, const bq_q2_weight* gate, const bq_q2_weight* up, const bq_q2_weight* down,
                      uint16_t* out, uint32_t m, bq_stream_t stream);

/* Q2_0 MMQ: out[m][n] = q8_1(act) @ Wdq^T, i.e. sum_k (d_a q)[m][k] * (d_w (c - 2))[n][k],
 * fp32 accumulation, BF16 store.  act_q8 is quantize_act_q8_1's output for [m][w->k];
 * w->group must be 128 (the page's MMQ condition).  Any m >= 1 and any n.
 * Computed on the BF16 tensor cores: the weight operand d_w (c - 2) is exact in BF16 and
 * each activation value d_a q enters as a pair of BF16 values whose sum equals it to
 * 2^-17 relative.
 * Source: init_q2.rs, `qkvz_q2_prefill_gemm` (MMQ route, `q2_0_mmq_gemm`). */
int q2_mmq_gemm(const void* act_q8, const bq_q2_weight* w, uint16_t* out, uint32_t m, bq_stream_t stream);

/* Q4_K MMQ: out[m][n] = q8_1(act) @ W_q4k^T, i.e. sum_k (d_a q)[m][k] * w[n][k] with
 * w = d sc_j q - dmin m_j, fp32 accumulation, BF16 store.  k % 256 == 0.  Computed on the
 * BF16 tensor cores: each activation value and each weight enters as a pair of BF16 values
 * whose sum equals it to 2^-17 relative (three products per pair of pairs; the product of
 * the two small halves is dropped).
 * Source: q4k_mmq.rs, `q4k_mmq_gemm` (C[m, n] = A[m, k] x W[n, k], BF16 store). */
int q4k_mmq_gemm(const void* act_q8, const void* w_q4k, uint16_t* out, uint32_t m, uint32_t n, uint32_t k,
                 bq_stream_t stream);

/* Dequantise a Q2_0 weight to dense BF16 out[n][k] (exact: d * (c - 2) is a BF16 value).
 * Source: init_q2.rs, `qkvz_q2_prefill_gemm` fallback (`dequant_q2_0_gn_to_bf16` into the
 * caller's scratch, then a dense BF16 GEMM). */
int dequant_q2_to_bf16(const bq_q2_weight* w, uint16_t* out, bq_stream_t stream);

/* Dense BF16 GEMM, the second half of the fallback prefill route: out[m, n] = a[m, k] @
 * w[n, k]^T with fp32 accumulation and one BF16 rounding per output (round to nearest even).
 * a: [m][k] BF16 row-major (the activations), w: [n][k] BF16 row-major (a dequantised
 * weight, as dequant_q2_to_bf16 writes it), out: [m][n] BF16 row-major; all three device
 * pointers, 16-byte aligned, owned by the caller.  k must be a multiple of 64 (else
 * BQ_ERR_INVALID); m = 0 or n = 0 is a no-op, k = 0 writes zeros.  Tensor-core (tcgen05)
 * kernel of this library, not a vendor GEMM.  A failed internal wait is reported by
 * bq_device_status.
 * Source: init_q2.rs, `qkvz_q2_prefill_gemm` (the fallback: `dequant_q2_0_gn_to_bf16`, then
 * `dense_gemm_bf16_pipelined`). */
int dense_gemm_bf16(const uint16_t* a, const uint16_t* w, uint16_t* out, uint32_t m, uint32_t n, uint32_t k,
                    bq_stream_t stream);

/* Dequantise an NVFP4 weight [n][k] to BF16 out[n][k] (the weight-preparation step before
 * quantize_weight_q4k):  w = e2m1(code) * e4m3(scale) * scale2, the exact product rounded
 * once to BF16 (round to nearest even).
 *   packed: [n][k/2] bytes of OCP FP4 E2M1 codes, value 2j of a row in the low nibble of
 *           byte j, value 2j + 1 in the high nibble (16-byte aligned);
 *   scales: [n][k/16] OCP FP8 E4M3 bytes, one per 16 consecutive values of a row;
 *   scale2: the per-tensor fp32 scale;  out: 16-byte aligned.  k % 16 == 0.
 * A NaN scale byte (0x7F, 0xFF) gives a NaN output whose bit pattern is not specified.
 * Source: q4k_mmq.rs, `dequant_nvfp4_to_bf16` (grid [n], block 256). */
int dequant_nvfp4_to_bf16(const void* packed, const void* scales, uint16_t* out, float scale2, uint32_t n, uint32_t k,
                          bq_stream_t stream);

/* ---------------------------------------------------------------- diagnostics */

/* Message for the calling thread's last failed call ("" after a successful call). */
const char* bq_last_error(void);

/* Synchronises the current device, then reads and clears the library's device status:
 * BQ_ERR_DEVICE if any kernel gave up on a bounded wait (each wait is limited to about a
 * second, after which the kernel records the failure and returns instead of hanging),
 * BQ_OK otherwise. */
int bq_device_status(void);

/* Library build string: version and target architecture. */
const char* bq_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* BQ8_H */
