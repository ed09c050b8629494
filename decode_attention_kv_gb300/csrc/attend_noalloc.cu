// attend_noalloc.cu -- kvd_attend_masked_noalloc: masked decode attention for
// callers that cannot allocate device memory.
//
// kvd_attend_masked needs a caller workspace for its per-split partial rows
// once the sequence axis is split across CTAs.  Some callers have no way to
// provide one: a host runtime whose allocator already owns all device memory
// and hands a plug-in only its inputs and outputs, an enqueue step that is
// forbidden to allocate, or a latency-critical loop that cannot afford
// cudaMalloc's implicit device synchronisation.  This entry point runs the
// very same split kernel and combine kernel with a workspace that lives in a
// fixed-size array compiled into the library (kNoAllocScratchBytes per
// device, held by every GPU that loads the library until the process exits).
//
// The array is shared by every call on a device and keeps whatever the last
// call left in it.  The attention kernel keeps its work counters in the
// array's leading bytes (kvd_plan.counter_bytes); they must be zero when a
// launch starts.  A completed launch
// leaves them at zero, but one whose bounded waits ran out (KVD_DEV_TIMEOUT)
// may not, so every call clears that block on the caller's stream
// (cudaMemsetAsync: stream-ordered, allocates nothing) before its launch.
// The partial rows need no clearing: each call writes the log-sum-exp of
// every split it reads and reads only partial rows it wrote.  Calls that may
// run at the same time on the GPU (different streams, or different host
// threads without ordering) race on the array and must be serialised by the
// caller.
#include <cstdio>
#include <mutex>

#include "kvd_device.cuh"
#include "kvd_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = KVD_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The workspace.  In host code this name is only a stand-in for the symbol,
// never a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char kvd_noalloc_scratch[kNoAllocScratchBytes];

// Driver entry point used to tell one context of a device from the next
// (after cudaDeviceReset the library's module is loaded again, possibly at
// another address).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
std::once_flag g_ctx_once;

std::mutex g_scratch_mutex;
struct ScratchEntry {
    CUcontext ctx;
    void* ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// Device address of the scratch array in the current device's current
// context, looked up with that device current the first time a context is
// seen, then cached.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(g_ctx_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    });
    // No context may be current yet on this thread (cudaGetDevice creates
    // none); the symbol lookup makes the primary context current, so the
    // context is asked for again after it.
    CUcontext ctx = nullptr;
    if (g_ctx_get_current) g_ctx_get_current(&ctx);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchEntry& ent = g_scratch[dev];
    if (!ent.ptr || !ctx || ent.ctx != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, kvd_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (g_ctx_get_current) g_ctx_get_current(&ctx);
        ent.ctx = ctx;
        ent.ptr = p;
    }
    *out = ent.ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" {

kvd_status kvd_attend_masked_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                     const uint8_t* mask, void* out, float* lse_out, int B,
                                     int Hq, int Hkv, int C, int D, float scale, kvd_dtype dtype,
                                     int num_splits, int32_t* dev_status, kvd_stream_t stream) {
    if (B < 1 || C < 1) {
        // Same argument rules as kvd_attend_masked (an empty batch is a no-op).
        return kvd_attend_masked(q, k_cache, v_cache, mask, out, lse_out, B, Hq, Hkv, C, D, scale,
                                 dtype, num_splits, nullptr, 0, dev_status, stream);
    }
    const size_t need =
        kvd_attend_masked_workspace_bytes(B, Hq, Hkv, C, D, dtype, num_splits);
    if (need > kNoAllocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "kvd_attend_masked_noalloc: these sizes need %zu bytes of split scratch, the "
                 "built-in scratch holds %zu; use kvd_attend_masked with a workspace or fewer "
                 "splits",
                 need, kNoAllocScratchBytes);
        kvd::set_last_error(msg);
        return KVD_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "kvd_attend_masked_noalloc: cudaGetSymbolAddress failed: %s",
                 cudaGetErrorString(e));
        kvd::set_last_error(msg);
        return KVD_ERR_CUDA;
    }
    // Work counters to zero first (a previous call's timed-out launch may have
    // left them set); stream-ordered before the launch.
    kvd_plan plan;
    const kvd_status sp = kvd_attend_masked_plan(B, Hq, Hkv, C, D, dtype, num_splits, &plan);
    if (sp != KVD_OK) return sp;
    const size_t counters = plan.counter_bytes > 256 ? plan.counter_bytes : 256;
    const cudaError_t ez = cudaMemsetAsync(scratch, 0, counters, (cudaStream_t)stream);
    if (ez != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "kvd_attend_masked_noalloc: clearing the counters failed: %s",
                 cudaGetErrorString(ez));
        kvd::set_last_error(msg);
        return KVD_ERR_CUDA;
    }
    return kvd_attend_masked(q, k_cache, v_cache, mask, out, lse_out, B, Hq, Hkv, C, D, scale,
                             dtype, num_splits, scratch, kNoAllocScratchBytes, dev_status, stream);
}

}  // extern "C"
