// ffn_noalloc.cu -- the packed-Q2 FFN decode chain for callers that cannot allocate device
// memory.
//
// ffn_q2_km needs two [m][inter] BF16 intermediates (the gate and up outputs) and takes
// them from its caller.  Some callers have no way to obtain them: a plugin that only ever
// receives its inputs and outputs from a host framework, code that runs where cudaMalloc
// is forbidden (inside a memory-pool-managed runtime that owns all device memory), or a C
// program linked without an allocator.  ffn_q2_km_noalloc gives them the same chain with the
// intermediates placed in a fixed array inside this library's device image instead.
//
// The array lives as long as the library is loaded, on every GPU that loads it, and every
// call shares it: two calls that overlap on the GPU (different streams, different host
// threads) race on it and give undefined results.  Calls on one stream are ordered and
// safe.  Nothing in the array needs to start at zero: the gate and up GEMVs overwrite every
// element the later steps read.
#include <mutex>

#include "common.cuh"

namespace bq8 {

// Two buffers of BQ_FFN_NOALLOC_MAX_ELEMS BF16 values each (gate, then up): 1 MiB in all.
static __device__ __align__(256) uint16_t g_ffn_scratch[2 * BQ_FFN_NOALLOC_MAX_ELEMS];

constexpr int FFN_NOALLOC_MAX_DEVICES = 64;

typedef CUresult (*PFN_ctxGetCurrent)(CUcontext*);
typedef CUresult (*PFN_ctxGetId)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 if the driver cannot say).  A
// context created after cudaDeviceReset gets a new id, so an address cached for the old one
// is looked up again.
static unsigned long long current_context_id() {
    static PFN_ctxGetCurrent get_current = nullptr;
    static PFN_ctxGetId get_id = nullptr;
    static bool tried = false;
    if (!tried) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_ctxGetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_ctxGetId>(p);
        tried = true;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

// Device address of g_ffn_scratch on the current device.  In host code the array's name
// is only a host-side shadow, so the address is looked up with that device current the
// first time a device is used (and again if its context was replaced) and cached; later
// calls do no CUDA runtime work here beyond reading the context id.
static int scratch_address(uint16_t** out, const char* who) {
    static std::mutex mu;
    static uint16_t* addr[FFN_NOALLOC_MAX_DEVICES] = {};
    static unsigned long long ctx_id[FFN_NOALLOC_MAX_DEVICES] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return fail(BQ_ERR_DEVICE, "%s: no current CUDA device", who);
    if (dev >= FFN_NOALLOC_MAX_DEVICES)
        return fail(BQ_ERR_UNSUPPORTED, "%s: device ordinal %d is beyond the %d this entry point tracks", who, dev,
                    FFN_NOALLOC_MAX_DEVICES);
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = addr[dev] ? current_context_id() : 0;
    if (!addr[dev] || (id != 0 && id != ctx_id[dev])) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_ffn_scratch);
        if (e != cudaSuccess || !p) {
            const int code = e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction
                                 ? BQ_ERR_UNSUPPORTED
                                 : BQ_ERR_DEVICE;
            return fail(code, "%s: cudaGetSymbolAddress of the scratch array failed: %s", who, cudaGetErrorString(e));
        }
        addr[dev] = static_cast<uint16_t*>(p);
        ctx_id[dev] = current_context_id();  // the context cudaGetSymbolAddress made current
    }
    *out = addr[dev];
    return BQ_OK;
}

}  // namespace bq8

using namespace bq8;

extern "C" int ffn_q2_km_noalloc(const uint16_t* x, const bq_q2_weight* gate, const bq_q2_weight* up,
                                 const bq_q2_weight* down, uint16_t* out, uint32_t m, bq_stream_t stream) {
    const char* who = "ffn_q2_km_noalloc";
    if (m == 0) return ok();
    if (!gate || !up || !down) return fail(BQ_ERR_INVALID, "%s: NULL weight descriptor", who);
    if ((uint64_t)m * gate->n > (uint64_t)BQ_FFN_NOALLOC_MAX_ELEMS)
        return fail(BQ_ERR_INVALID, "%s: m * inter = %u * %u exceeds the built-in scratch of %u values per buffer",
                    who, m, gate->n, (unsigned)BQ_FFN_NOALLOC_MAX_ELEMS);
    uint16_t* scratch = nullptr;
    int st = scratch_address(&scratch, who);
    if (st) return st;
    // the same chain as ffn_q2_km (which checks every other argument), with its two
    // intermediates in the built-in array
    return ffn_q2_km(x, gate, up, down, scratch, scratch + BQ_FFN_NOALLOC_MAX_ELEMS, out, m, stream);
}
