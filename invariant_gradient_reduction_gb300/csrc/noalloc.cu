// noalloc.cu -- det_scatter_reduce_noalloc: the scatter-reduce for callers
// that cannot allocate device memory when they call in.
//
// Some callers have no way to hand the library a workspace: code running
// inside a larger runtime whose allocator owns all device memory, a path
// that must not allocate once it has started (a latency-critical serving
// loop, for instance), or a fixed interface with no argument through which a
// scratch buffer could travel.  For them this entry point takes its scratch
// -- the fp32 partial slots of hot destinations -- from a fixed array that
// lives in the library's own device image.  The module loader reserves it on
// every GPU the library is loaded on, and it stays reserved until the process
// exits.  Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "common.cuh"
#include "plan_internal.cuh"

namespace detr {

// Maximum scratch: 16 MiB of fp32 partial slots (for example 32768 slots of a
// 128-wide row, or 1024 slots of a 4096-wide row).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on each device, looked up with that
// device current (the host-side symbol is only a stand-in and must never be
// handed to a kernel), together with the id of the context it was looked up
// in: after a device reset the module is loaded again in a new context and
// the array may have moved, so a changed context id means a new lookup.
struct ScratchEntry {
    void* addr;
    unsigned long long ctx_id;
};
static ScratchEntry g_scratch[kNoAllocMaxDevices] = {};
static std::mutex g_scratch_mu;

// Id of the current context (0 if there is none yet or the driver cannot say),
// through the driver's entry points, so that the library needs no link-time
// dependency on the driver library.
static unsigned long long current_context_id()
{
    using GetCurrent = int (*)(void**);
    using GetId = int (*)(void*, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static bool resolved = false;
    if (!resolved) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
        resolved = true;
    }
    void* ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == 0 && ctx && get_id(ctx, &id) == 0) return id;
    return 0;
}

static det_status scratch_address(void** out)
{
    int dev = 0;
    DETR_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kNoAllocMaxDevices) return DET_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry& e = g_scratch[dev];
    if (!e.addr || e.ctx_id == 0 || current_context_id() != e.ctx_id) {
        void* p = nullptr;
        DETR_CUDA(cudaGetSymbolAddress(&p, g_noalloc_scratch));  // also makes the context current
        if (!p) return DET_ERR_CUDA;
        e.addr = p;
        e.ctx_id = current_context_id();
    }
    *out = e.addr;
    return DET_OK;
}

}  // namespace detr

using namespace detr;

extern "C" det_status det_scatter_reduce_noalloc(det_plan plan, const void* const* x_shards,
                                                 const int64_t* shard_rows, int32_t P, det_dtype x_dtype,
                                                 int64_t ldx, int64_t H, const float* w, void* out, int64_t ldo,
                                                 det_dtype out_dtype, const det_opts* opts, void* stream)
{
    if (!plan) return DET_ERR_ARG;
    size_t need = 0;
    det_status s = det_scatter_workspace_size(plan, H, &need);
    if (s) return s;
    if (need > kNoAllocScratchBytes) return DET_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    s = scratch_address(&scratch);
    if (s) return s;
    // The partial slots need no clearing: every slot is written by the first
    // pass before the second pass reads it.  The whole array is passed as the
    // workspace, so the aliasing checks of det_scatter_reduce cover all of it.
    return det_scatter_reduce(plan, x_shards, shard_rows, P, x_dtype, ldx, H, w, out, ldo, out_dtype, scratch,
                              kNoAllocScratchBytes, opts, stream);
}
