// api.cu -- status codes, version, argument helpers shared by the entry points.
#include <atomic>
#include <mutex>
#include <unordered_map>

#include "common.cuh"

namespace detr {

static thread_local int g_last_cuda_error = 0;
static std::atomic<long long> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void set_last_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }

static std::atomic<int> g_sm_count[kMaxDevices];

det_status current_sm_count(int* sms)
{
    int dev = 0;
    DETR_CUDA(cudaGetDevice(&dev));
    if (dev >= 0 && dev < kMaxDevices) {
        const int c = g_sm_count[dev].load(std::memory_order_relaxed);
        if (c > 0) { *sms = c; return DET_OK; }
    }
    DETR_CUDA(cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev));
    if (*sms <= 0) *sms = 1;
    if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(*sms, std::memory_order_relaxed);
    return DET_OK;
}

// Largest dynamic shared memory already allowed per (kernel, device).
static std::mutex g_attr_mu;
static std::unordered_map<const void*, size_t> g_attr_set[kMaxDevices];

det_status allow_dynamic_smem(const void* func, size_t bytes)
{
    if (bytes <= 48 * 1024) return DET_OK;
    int dev = 0;
    DETR_CUDA(cudaGetDevice(&dev));
    const bool cacheable = dev >= 0 && dev < kMaxDevices;
    if (cacheable) {
        std::lock_guard<std::mutex> lock(g_attr_mu);
        auto it = g_attr_set[dev].find(func);
        if (it != g_attr_set[dev].end() && it->second >= bytes) return DET_OK;
    }
    DETR_CUDA(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)));
    if (cacheable) {
        std::lock_guard<std::mutex> lock(g_attr_mu);
        size_t& v = g_attr_set[dev][func];
        v = std::max(v, bytes);
    }
    return DET_OK;
}

det_status make_shard_table(const void* const* x_shards, const int64_t* shard_rows, int32_t P,
                            int64_t N, int64_t ldx, int64_t H, det_dtype x_dtype, ShardTable* t,
                            size_t* x_bytes_of_shard)
{
    if (P < 1) return DET_ERR_ARG;
    if (P > DET_MAX_SHARDS) return DET_ERR_UNSUPPORTED;
    if (!x_shards || !shard_rows) return DET_ERR_ARG;
    if (!dtype_ok(x_dtype)) return DET_ERR_DTYPE;
    if (H < 0 || ldx < H || ldx > (int64_t(1) << 40)) return DET_ERR_ARG;
    int64_t begin = 0;
    const int es = dtype_size(x_dtype);
    for (int q = 0; q < P; ++q) {
        if (shard_rows[q] < 0) return DET_ERR_ARG;
        if (shard_rows[q] > 0 && H > 0 && !x_shards[q]) return DET_ERR_ARG;
        if (!aligned(x_shards[q], static_cast<size_t>(es))) return DET_ERR_ARG;
        t->base[q] = static_cast<const unsigned char*>(x_shards[q]);
        t->row_begin[q] = begin;
        x_bytes_of_shard[q] = shard_rows[q] > 0
            ? static_cast<size_t>((shard_rows[q] - 1) * ldx + H) * static_cast<size_t>(es) : 0;
        begin += shard_rows[q];
        if (begin > kMaxRows) return DET_ERR_UNSUPPORTED;
    }
    if (begin != N) return DET_ERR_ARG;
    for (int q = P; q < DET_MAX_SHARDS; ++q) { t->base[q] = nullptr; t->row_begin[q] = begin; }
    t->row_begin[P] = begin;
    t->row_begin[DET_MAX_SHARDS] = begin;
    t->P = P;
    return DET_OK;
}

}  // namespace detr

extern "C" {

const char* det_status_str(det_status s)
{
    switch (s) {
    case DET_OK: return "ok";
    case DET_ERR_ARG: return "invalid argument (null, negative, stride, alignment or aliasing)";
    case DET_ERR_DTYPE: return "unsupported dtype";
    case DET_ERR_INDEX_RANGE: return "destination index outside [0, M)";
    case DET_ERR_ORDER_KEY: return "two sources of one destination share an order key";
    case DET_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DET_ERR_CUDA: return "CUDA error (see det_last_cuda_error)";
    case DET_ERR_TIMEOUT: return "bounded device wait expired";
    case DET_ERR_UNSUPPORTED: return "size beyond a documented limit";
    default: return "unknown status";
    }
}

int32_t det_last_cuda_error(void) { return detr::g_last_cuda_error; }

int32_t det_version(void) { return (1 << 16) | 0; }

int64_t det_kernel_launches(void) { return detr::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
