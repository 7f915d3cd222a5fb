// api.cu -- status handling, size helpers and shared host checks of the libbq8 C ABI.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"

namespace bq8 {

static thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int ok() {
    g_err[0] = 0;
    return BQ_OK;
}

int check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return ok();
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
        return fail(BQ_ERR_UNSUPPORTED, "%s: no kernel image for this device (built for sm_103a): %s", what,
                    cudaGetErrorString(e));
    return fail(BQ_ERR_LAUNCH, "%s: launch failed: %s", what, cudaGetErrorString(e));
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    if (dev < 64 && cached[dev]) return cached[dev];
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    if (dev < 64) cached[dev] = v;
    return v;
}

int check_q2(const bq_q2_weight* w, const char* who) {
    if (!w) return fail(BQ_ERR_INVALID, "%s: weight descriptor is NULL", who);
    if (w->group == 0 || w->group % 128 != 0)
        return fail(BQ_ERR_INVALID, "%s: group %u must be a positive multiple of 128", who, w->group);
    if (w->k % 128 != 0 || w->k % w->group != 0)
        return fail(BQ_ERR_INVALID, "%s: k %u must be a multiple of 128 and of group %u", who, w->k, w->group);
    if (w->n > 0 && w->k > 0) {
        if (!w->data) return fail(BQ_ERR_INVALID, "%s: weight data is NULL", who);
        if (!aligned16(w->data)) return fail(BQ_ERR_INVALID, "%s: weight data must be 16-byte aligned", who);
    }
    return BQ_OK;
}

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled encode_fn() {
    static PFN_encodeTiled fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_encodeTiled>(p);
    }
    return fn;
}

int make_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t stride_bytes,
                    uint32_t box_bytes, uint32_t box_rows, bool swizzle128, const char* who) {
    return make_tmap_2d(map, base, 1, row_bytes, rows, stride_bytes, box_bytes, box_rows, swizzle128, who);
}

int make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t row_elems, uint64_t rows,
                 uint64_t stride_bytes, uint32_t box_elems, uint32_t box_rows, bool swizzle128, const char* who) {
    PFN_encodeTiled fn = encode_fn();
    if (!fn) return fail(BQ_ERR_UNSUPPORTED, "%s: cuTensorMapEncodeTiled unavailable from the driver", who);
    const cuuint64_t dims[2] = {row_elems, rows};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {box_elems, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(BQ_ERR_INVALID, "%s: tensor map encoding failed (CUresult %d)", who, (int)r);
    return BQ_OK;
}

// Encoded 2-D byte tensor maps, keyed by everything the encoding depends on (base address,
// shape, stride, box, swizzle, device), so repeated calls on the same weight encode nothing.
// The map describes only addresses and shapes, never contents, so a cached entry stays valid
// for any data later placed at that address.  128 entries, replaced round-robin.
int cached_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t stride_bytes,
                      uint32_t box_bytes, uint32_t box_rows, bool swizzle128, const char* who) {
    struct Entry {
        const void* base;
        uint64_t row_bytes, rows, stride;
        uint32_t box_bytes, box_rows;
        int swz, dev;
        bool used;
        CUtensorMap map;
    };
    constexpr int N = 128;
    static Entry table[N];
    static int next = 0;
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < N; i++) {
            const Entry& e = table[i];
            if (e.used && e.base == base && e.row_bytes == row_bytes && e.rows == rows && e.stride == stride_bytes &&
                e.box_bytes == box_bytes && e.box_rows == box_rows && e.swz == (int)swizzle128 && e.dev == dev) {
                *map = e.map;
                return BQ_OK;
            }
        }
    }
    CUtensorMap fresh;
    const int st = make_tmap_2d_u8(&fresh, base, row_bytes, rows, stride_bytes, box_bytes, box_rows, swizzle128, who);
    if (st) return st;
    std::lock_guard<std::mutex> lock(mu);
    Entry& e = table[next];
    next = (next + 1) % N;
    e.base = base;
    e.row_bytes = row_bytes;
    e.rows = rows;
    e.stride = stride_bytes;
    e.box_bytes = box_bytes;
    e.box_rows = box_rows;
    e.swz = (int)swizzle128;
    e.dev = dev;
    e.map = fresh;
    e.used = true;
    *map = fresh;
    return BQ_OK;
}

// A byte matrix [rows][row_bytes] (row_bytes a multiple of 128) seen as 128-byte column blocks:
// dims (128, rows, row_bytes / 128), strides (row_bytes, 128), box (128, box_rows, nblk), 128-byte
// swizzle.  One request brings nblk column blocks of box_rows rows, laid out [block][row][128 B]
// in shared memory, the layout of nblk separate 2-D boxes.  Cached like cached_tmap_2d_u8.
int cached_tmap_chunks_u8(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows,
                          uint32_t nblk, const char* who) {
    struct Entry {
        const void* base;
        uint64_t row_bytes, rows;
        uint32_t box_rows, nblk;
        int dev;
        bool used;
        CUtensorMap map;
    };
    constexpr int N = 64;
    static Entry table[N];
    static int next = 0;
    static std::mutex mu;
    if (row_bytes % 128 != 0 || nblk == 0) return fail(BQ_ERR_INVALID, "%s: internal chunk map shape", who);
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < N; i++) {
            const Entry& e = table[i];
            if (e.used && e.base == base && e.row_bytes == row_bytes && e.rows == rows && e.box_rows == box_rows &&
                e.nblk == nblk && e.dev == dev) {
                *map = e.map;
                return BQ_OK;
            }
        }
    }
    PFN_encodeTiled fn = encode_fn();
    if (!fn) return fail(BQ_ERR_UNSUPPORTED, "%s: cuTensorMapEncodeTiled unavailable from the driver", who);
    const cuuint64_t gd[3] = {128, rows, row_bytes / 128};
    const cuuint64_t gs[2] = {row_bytes, 128};
    const cuuint32_t bx[3] = {128, box_rows, nblk};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUtensorMap fresh;
    CUresult r = fn(&fresh, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), gd, gs, bx, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(BQ_ERR_INVALID, "%s: tensor map encoding failed (CUresult %d)", who, (int)r);
    std::lock_guard<std::mutex> lock(mu);
    Entry& e = table[next];
    next = (next + 1) % N;
    e.base = base;
    e.row_bytes = row_bytes;
    e.rows = rows;
    e.box_rows = box_rows;
    e.nblk = nblk;
    e.dev = dev;
    e.map = fresh;
    e.used = true;
    *map = fresh;
    return BQ_OK;
}

int make_tmap_3d_u8(CUtensorMap* map, const void* base, const uint64_t (&dims)[3], const uint64_t (&strides)[2],
                    const uint32_t (&box)[3], const char* who) {
    PFN_encodeTiled fn = encode_fn();
    if (!fn) return fail(BQ_ERR_UNSUPPORTED, "%s: cuTensorMapEncodeTiled unavailable from the driver", who);
    const cuuint64_t gd[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t gs[2] = {strides[0], strides[1]};
    const cuuint32_t bx[3] = {box[0], box[1], box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), gd, gs, bx, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(BQ_ERR_INVALID, "%s: tensor map encoding failed (CUresult %d)", who, (int)r);
    return BQ_OK;
}

}  // namespace bq8

extern "C" {

int bq_device_status(void) {
    const unsigned int s = bq8::gemv_status_take() | bq8::gemv_hm_status_take() | bq8::mmq_tc_status_take() |
                           bq8::gemm_bf16_status_take() | bq8::q8_status_take();
    if (s) return bq8::fail(BQ_ERR_DEVICE, "a kernel gave up on a bounded wait (status bits 0x%x)", s);
    return bq8::ok();
}

size_t bq_q2_weight_bytes(uint32_t n, uint32_t k, uint32_t group) {
    if (group == 0 || group % 128 != 0 || k % group != 0) return 0;
    return (size_t)n * (k / 4) + (size_t)n * (k / group) * 2;
}

size_t bq_q8_1_bytes(uint32_t m, uint32_t k) {
    size_t kp = ((size_t)k + 255) / 256 * 256;
    return (size_t)m * kp + (size_t)m * (kp / 32) * 8;
}

size_t bq_q4k_weight_bytes(uint32_t n, uint32_t k) {
    if (k % 256 != 0) return 0;
    return (size_t)n * (k / 256) * 144;
}

const char* bq_last_error(void) { return bq8::g_err; }

const char* bq_build_info(void) { return "libbq8 0.1 (sm_103a; C ABI: include/bq8.h)"; }

}  // extern "C"
