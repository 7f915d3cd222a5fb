// common.cuh -- internals shared by the libbq8 translation units (not installed).
#pragma once

#include <cuda.h>  // CUtensorMap (types only; the driver entry point is fetched at run time)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bq8.h"

namespace bq8 {

// ------------------------------------------------------------------ host-side status
// Records `msg` as the calling thread's last error and returns `code`.
int fail(int code, const char* fmt, ...);
// Clears the calling thread's last error and returns BQ_OK.
int ok();
// Maps the launch error of the most recent kernel launch to a status code.
int check_launch(const char* what);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Number of SMs of the current device (cached per device).
int sm_count();

// Validates a Q2_0 weight descriptor; returns BQ_OK or an error status.
int check_q2(const bq_q2_weight* w, const char* who);

// Encodes a 2-D tiled TMA descriptor over a row-major byte matrix [rows][row_bytes]
// (row stride `stride_bytes`), box [box_rows][box_bytes], optional 128-byte swizzle.
int make_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows,
                    uint64_t stride_bytes, uint32_t box_bytes, uint32_t box_rows, bool swizzle128,
                    const char* who);
// Same for 1- or 2-byte elements: matrix [rows][row_elems], box [box_rows][box_elems]
// (box_elems <= 256).
int make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t row_elems, uint64_t rows,
                 uint64_t stride_bytes, uint32_t box_elems, uint32_t box_rows, bool swizzle128, const char* who);

// make_tmap_2d_u8 through a small process-wide cache (no encoding on a hit).
int cached_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t stride_bytes,
                      uint32_t box_bytes, uint32_t box_rows, bool swizzle128, const char* who);

// 3-D tiled TMA descriptor over bytes: dims {d0, d1, d2}, byte strides of d1 and d2 (any
// order, multiples of 16), box {b0, b1, b2} (b0 a multiple of 16), no swizzle.
// A byte matrix [rows][row_bytes] (row_bytes a multiple of 128) as 128-byte column blocks: one
// request brings nblk blocks of box_rows rows, laid out [block][row][128 B] (api.cu).
int cached_tmap_chunks_u8(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows,
                          uint32_t nblk, const char* who);
int make_tmap_3d_u8(CUtensorMap* map, const void* base, const uint64_t (&dims)[3], const uint64_t (&strides)[2],
                    const uint32_t (&box)[3], const char* who);

// Reads and clears each translation unit's device status word (nonzero after a bounded
// wait gave up).
unsigned int gemv_status_take();
unsigned int gemv_hm_status_take();
unsigned int mmq_tc_status_take();
unsigned int gemm_bf16_status_take();
unsigned int q8_status_take();

// The FP16 warp-MMA GEMV (gemv_hm.cu) and the shapes it takes.
bool gemv_hm_supported(const bq_q2_weight* w, uint32_t m);
int launch_q2_gemv_hm(const uint16_t* x, const bq_q2_weight* w, uint16_t* y, uint32_t m, uint16_t* hgate,
                      cudaStream_t stream, const char* who);
// The dual form for an FFN's gate and up weights of the same shape: h = BF16(SiLU(g) * u)
// into h and u into u, in one launch (gemv_hm.cu).
bool gemv_hm_dual_supported(const bq_q2_weight* gate, uint32_t m);
int launch_q2_gemv_hm_dual(const uint16_t* x, const bq_q2_weight* gate, const bq_q2_weight* up, uint16_t* h,
                           uint16_t* u, uint32_t m, cudaStream_t stream, const char* who);

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// 64-bit streaming load of weight bytes: not kept in L1, L2 prefetches the 256-byte
// window around the access (the rest of the row's codes are read right after).
__device__ __forceinline__ uint2 ldg_stream64(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0, %1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ldg_nc128(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + C, fp32 accumulate (legacy warp MMA).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1, const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// D = A(16x32 s8, row) * B(32x8 u8, col) + C, int32 accumulate (legacy warp MMA).
__device__ __forceinline__ void mma_s8u8_16832(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1, const int (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.u8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%10, %11, %12, %13};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]));
}

// ------------------------------------------------------------------ mbarrier / TMA
// Every wait is bounded: after over a second of polling the caller gets `false`, records
// the failure in its status word and winds down instead of hanging the GPU.

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n"
                 ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(smem_u32(bar)) : "memory");
}

// Non-blocking probe of phase `parity` of `bar`.  (mbarrier.try_wait may park the warp for
// microseconds before it returns false, which the short stages of these kernels cannot
// afford, so waits poll test_wait with a short sleep instead.)
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for phase `parity` of `bar` to complete.  Polls with a short sleep; gives up (false)
// after ~2^26 polls (well over a second), so a wait that can never complete ends the kernel
// instead of hanging the GPU.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    for (uint32_t it = 0; it < (1u << 26); it++) {
        __nanosleep(32);
        if (mbar_test(bar, parity)) return true;
    }
    return false;
}

// Waits for phase `parity` of `bar` with mbarrier.try_wait, which suspends the warp in
// hardware until the phase completes (or a system time limit of microseconds passes), so a
// waiting warp takes no issue slots.  Gives up (false) once 20 ms have passed on the global
// timer (a copy of a few kilobytes takes microseconds), or after 2^22 tries.
__device__ __forceinline__ bool mbar_wait_suspend(uint64_t* bar, uint32_t parity) {
    uint64_t start = 0;
    for (uint32_t it = 0; it < (1u << 22); it++) {
        uint32_t done;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (done) return true;
        if ((it & 63) == 63) {
            uint64_t now;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
            if (start == 0) start = now;
            else if (now - start > 20000000ull) return false;
        }
    }
    return false;
}

// (a & b) | c in one LOP3 with all three operands in registers.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// 2-D TMA tile load global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 3-D TMA tile load global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// Cooperative copy of `bytes` contiguous bytes global -> shared (both 16-byte aligned,
// bytes % 2 == 0): 16-byte vectors, every load of a thread issued before its stores so a
// thread pays one memory latency, not one per element.
__device__ __forceinline__ void copy_to_smem(void* dst, const void* src, int bytes, int tid, int nthreads) {
    const int nvec = bytes >> 4;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    constexpr int B = 8;
    for (int base = tid; base < nvec; base += B * nthreads) {
        uint4 v[B];
#pragma unroll
        for (int j = 0; j < B; j++) {
            const int i = base + j * nthreads;
            if (i < nvec) v[j] = __ldg(s4 + i);
        }
#pragma unroll
        for (int j = 0; j < B; j++) {
            const int i = base + j * nthreads;
            if (i < nvec) d4[i] = v[j];
        }
    }
    const uint16_t* s2 = reinterpret_cast<const uint16_t*>(src);
    uint16_t* d2 = reinterpret_cast<uint16_t*>(dst);
    for (int i = (nvec << 3) + tid; i < (bytes >> 1); i += nthreads) d2[i] = s2[i];
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// D = A(16x32 e4m3, row) * B(32x8 e4m3, col) + C, fp32 accumulate (legacy warp MMA).
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 1-D bulk copy global -> shared (16-byte aligned, size % 16 == 0), completion on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Programmatic dependent launch: let the next grid start / wait for the previous grid.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// SiLU(g) * u in fp32: SiLU(z) = z * sigmoid(z), sigmoid from e = exp(-|z|) so that neither
// branch overflows.  (The SiLU*mul kernel and the FFN chain's fused epilogue share it, so
// both give the same bits.)
__device__ __forceinline__ float silu_mul1(float g, float u) {
    const float e = expf(-fabsf(g));
    const float sig = (g >= 0.0f) ? 1.0f / (1.0f + e) : e / (1.0f + e);
    return g * sig * u;
}

__device__ __forceinline__ uint32_t bf162_bits(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __nv_bfloat162 bits_bf162(uint32_t u) { return *reinterpret_cast<__nv_bfloat162*>(&u); }

}  // namespace bq8
