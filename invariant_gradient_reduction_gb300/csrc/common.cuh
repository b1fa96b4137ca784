// common.cuh -- internal helpers shared by the translation units of
// libdetreduce.so (never installed, never seen by callers).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "det_reduce.h"

namespace detr {

// Limits: sizes and offsets of the destination lists are int32 on the device.
constexpr int64_t kMaxRows = 2147483646;  // N, M <= 2^31 - 2
constexpr int kMaxDevices = 64;            // per-device caches

// Canonical fold: consecutive chunks of this many terms are folded left to right.
constexpr int kChunk = 32;
constexpr int kDefaultSegLog2 = 3;
constexpr int kMinSegLog2 = 3;
constexpr int kMaxSegLog2 = 6;

// ---- status plumbing (host) ----
void set_last_cuda_error(cudaError_t e);
inline det_status cuda_fail(cudaError_t e)
{
    set_last_cuda_error(e);
    return DET_ERR_CUDA;
}
#define DETR_CUDA(call)                                   \
    do {                                                  \
        cudaError_t detr_e_ = (call);                     \
        if (detr_e_ != cudaSuccess) return detr::cuda_fail(detr_e_); \
    } while (0)
void count_launch();
#define DETR_LAUNCHED()                                   \
    do {                                                  \
        cudaError_t detr_e_ = cudaGetLastError();         \
        if (detr_e_ != cudaSuccess) return detr::cuda_fail(detr_e_); \
        detr::count_launch();                             \
    } while (0)

// Programmatic dependent launch.  A kernel launched by launch_after_previous()
// may begin while the kernel before it on the stream is still running (its
// launch and start-up overlap that kernel's tail); it calls pdl_wait() before
// it reads anything earlier work wrote, and that wait returns once the
// earlier kernel has finished and its writes are visible.  A kernel that
// calls pdl_launch_dependents() lets the kernel after it start early.  Both
// instructions do nothing for kernels launched the ordinary way.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_after_previous(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                         cudaStream_t st, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t a, size_t b) { return (a + b - 1) / b * b; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// SM count of the current device (cached per device).
det_status current_sm_count(int* sms);

// Allow `bytes` of dynamic shared memory for `func` on the current device
// (cudaFuncSetAttribute, called once per kernel, device and larger size).
det_status allow_dynamic_smem(const void* func, size_t bytes);

// Half-open byte ranges [a, a+na) and [b, b+nb) overlap?
inline bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

inline int dtype_size(det_dtype t) { return t == DET_F32 ? 4 : 2; }
inline bool dtype_ok(det_dtype t) { return t == DET_F32 || t == DET_BF16; }

// Where the physical rows live: shard q holds rows [row_begin[q], row_begin[q+1]).
struct ShardTable {
    const unsigned char* base[DET_MAX_SHARDS];
    long long row_begin[DET_MAX_SHARDS + 1];
    int P;
};

// Checks the shard arguments and fills the table.  x_bytes_of_shard[q]
// receives the byte extent of shard q (for alias checks).
det_status make_shard_table(const void* const* x_shards, const int64_t* shard_rows, int32_t P,
                            int64_t N, int64_t ldx, int64_t H, det_dtype x_dtype, ShardTable* t,
                            size_t* x_bytes_of_shard);

// ---- device helpers ----

// Address of physical row r (the staging lane calls this once per term).
__device__ __forceinline__ const unsigned char* shard_row(const ShardTable& t, long long r, long long ldx_bytes)
{
    int q = 0;
    while (q + 1 < t.P && r >= t.row_begin[q + 1]) ++q;
    return t.base[q] + (r - t.row_begin[q]) * ldx_bytes;
}

// 16-byte streaming load: each source row is read once, so do not keep it in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// bf16 pair (low half = first element) -> two exact binary32 values.
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

}  // namespace detr
