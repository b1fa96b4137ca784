// atomic.cu -- the NON-deterministic baseline: scatter_add_ with atomics.
//
// Only for measuring what determinism costs.  Concurrent atomic adds to one
// address lose no update, but the scheduler decides who adds first, so the
// result's last bits change from run to run ("DeepSeek-V4 book, Ch 09", the
// glossary entry on atomicAdd; "Megatron-LM determinism developer reference",
// section 3.1, the scatter_add_ default branch).  One warp per source row;
// 16-byte loads; 16-byte vector atomics where the accumulator allows.
#include <algorithm>

#include "common.cuh"

namespace detr {

constexpr int kAtomicThreads = 256;
constexpr int kAtomicWarps = kAtomicThreads / 32;

struct AtomicArgs {
    const int* idx;
    long long N, M;
    long long ldx_bytes;
    int H;
    int V;         // vectors per row
    const float* w;
    float* acc;    // fp32 accumulator [M][lda]
    long long lda;
    int* flags;    // flags[0]: sources with idx outside [0, M)
};

template <typename XT, bool VECTOR, bool VATOM>
__global__ void __launch_bounds__(kAtomicThreads)
atomic_scatter_kernel(const __grid_constant__ AtomicArgs a, const __grid_constant__ ShardTable tbl)
{
    constexpr int VEC = VECTOR ? 16 / static_cast<int>(sizeof(XT)) : 1;
    const int lane = threadIdx.x & 31;
    const long long nwarps = static_cast<long long>(gridDim.x) * kAtomicWarps;
    for (long long i = static_cast<long long>(blockIdx.x) * kAtomicWarps + (threadIdx.x >> 5); i < a.N; i += nwarps) {
        const int m = a.idx[i];
        if (m < 0 || m >= a.M) {
            if (lane == 0) atomicAdd(a.flags, 1);
            continue;
        }
        const unsigned char* row = shard_row(tbl, i, a.ldx_bytes);
        const float wv = a.w ? a.w[i] : 1.0f;
        float* dst = a.acc + static_cast<long long>(m) * a.lda;
        for (int v = lane; v < a.V; v += 32) {
            float xf[VEC];
            if (VECTOR) {
                const uint4 r = ld_stream_v4(row + static_cast<long long>(v) * 16);
                if (sizeof(XT) == 2) {
                    const uint32_t u[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        xf[(2 * k) % VEC] = bf16lo(u[k]);
                        xf[(2 * k + 1) % VEC] = bf16hi(u[k]);
                    }
                } else {
                    xf[0] = __uint_as_float(r.x);
                    xf[1 % VEC] = __uint_as_float(r.y);
                    xf[2 % VEC] = __uint_as_float(r.z);
                    xf[3 % VEC] = __uint_as_float(r.w);
                }
            } else {
                if (sizeof(XT) == 2)
                    xf[0] = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row) + v)) << 16);
                else
                    xf[0] = __ldg(reinterpret_cast<const float*>(row) + v);
            }
            if (a.w) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) xf[e] = __fmul_rn(wv, xf[e]);
            }
            float* d = dst + static_cast<long long>(v) * VEC;
            if (VATOM) {
#pragma unroll
                for (int e = 0; e < VEC; e += 4)
                    atomicAdd(reinterpret_cast<float4*>(d + e), make_float4(xf[e], xf[(e + 1) % VEC], xf[(e + 2) % VEC], xf[(e + 3) % VEC]));
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) atomicAdd(d + e, xf[e]);
            }
        }
    }
}

// fp32 accumulator [M][H] -> bf16 out [M][ldo], nearest even.  Rows over the
// y dimension of the grid (and a loop), columns over x: no division per
// element.  VEC8: 8 columns per thread, two 16-byte loads and one 16-byte
// store (H a multiple of 8, out 16-byte aligned, ldo a multiple of 8).
template <bool VEC8>
__global__ void __launch_bounds__(256)
cast_bf16_kernel(const float* __restrict__ acc, long long M, int H, __nv_bfloat16* __restrict__ out, long long ldo)
{
    const int per_row = VEC8 ? H / 8 : H;
    for (long long m = blockIdx.y; m < M; m += gridDim.y) {
        const float* a = acc + m * H;
        __nv_bfloat16* o = out + m * ldo;
        for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < per_row; c += gridDim.x * blockDim.x) {
            if (VEC8) {
                const float4 lo = __ldcs(reinterpret_cast<const float4*>(a) + 2 * c);
                const float4 hi = __ldcs(reinterpret_cast<const float4*>(a) + 2 * c + 1);
                __nv_bfloat162 p0 = __floats2bfloat162_rn(lo.x, lo.y), p1 = __floats2bfloat162_rn(lo.z, lo.w);
                __nv_bfloat162 p2 = __floats2bfloat162_rn(hi.x, hi.y), p3 = __floats2bfloat162_rn(hi.z, hi.w);
                uint4 pk;
                pk.x = *reinterpret_cast<uint32_t*>(&p0);
                pk.y = *reinterpret_cast<uint32_t*>(&p1);
                pk.z = *reinterpret_cast<uint32_t*>(&p2);
                pk.w = *reinterpret_cast<uint32_t*>(&p3);
                reinterpret_cast<uint4*>(o)[c] = pk;
            } else {
                o[c] = __float2bfloat16_rn(a[c]);
            }
        }
    }
}

template <typename XT>
static void launch_atomic(bool vec, bool vatom, const AtomicArgs& a, const ShardTable& t, int grid, cudaStream_t st)
{
    if (vec && vatom) atomic_scatter_kernel<XT, true, true><<<grid, kAtomicThreads, 0, st>>>(a, t);
    else if (vec) atomic_scatter_kernel<XT, true, false><<<grid, kAtomicThreads, 0, st>>>(a, t);
    else atomic_scatter_kernel<XT, false, false><<<grid, kAtomicThreads, 0, st>>>(a, t);
}

}  // namespace detr

using namespace detr;

extern "C" {

det_status det_atomic_workspace_size(int64_t M, int64_t H, det_dtype out_dtype, size_t* bytes)
{
    if (!bytes || M < 0 || H < 0) return DET_ERR_ARG;
    if (!dtype_ok(out_dtype)) return DET_ERR_DTYPE;
    if (M > kMaxRows || H > kMaxRows) return DET_ERR_UNSUPPORTED;
    *bytes = 256 + (out_dtype == DET_BF16 ? static_cast<size_t>(M) * static_cast<size_t>(H) * 4 : 0);
    return DET_OK;
}

}  // extern "C"

// det_atomic_scatter_reduce (accumulate = false: out zeroed first) and
// det_atomic_index_add (true: fp32 out only, added to in place).
static det_status atomic_impl(const int32_t* idx, int64_t N, int64_t M, const void* const* x_shards,
                              const int64_t* shard_rows, int32_t P, det_dtype x_dtype, int64_t ldx, int64_t H,
                              const float* w, void* out, int64_t ldo, det_dtype out_dtype, void* workspace,
                              size_t ws_bytes, const det_opts* opts, void* stream, bool accumulate)
{
    if (accumulate && out_dtype != DET_F32) return DET_ERR_UNSUPPORTED;
    if (N < 0 || M < 0) return DET_ERR_ARG;
    if (N > kMaxRows || M > kMaxRows) return DET_ERR_UNSUPPORTED;
    if (!dtype_ok(x_dtype) || !dtype_ok(out_dtype)) return DET_ERR_DTYPE;
    if (H < 0 || ldo < H) return DET_ERR_ARG;
    if (H > kMaxRows) return DET_ERR_UNSUPPORTED;
    if ((N > 0 && !idx) || !aligned(idx, 4) || !aligned(w, 4)) return DET_ERR_ARG;
    ShardTable tbl;
    size_t xbytes[DET_MAX_SHARDS] = {};
    det_status s = make_shard_table(x_shards, shard_rows, P, N, ldx, H, x_dtype, &tbl, xbytes);
    if (s) return s;
    const int osz = dtype_size(out_dtype);
    if (M > 0 && H > 0 && !out) return DET_ERR_ARG;
    if (!aligned(out, static_cast<size_t>(osz))) return DET_ERR_ARG;
    size_t need = 0;
    s = det_atomic_workspace_size(M, H, out_dtype, &need);
    if (s) return s;
    if (!workspace || !aligned(workspace, 256) || ws_bytes < need) return DET_ERR_WORKSPACE;
    const size_t out_bytes = M > 0 && H > 0 ? static_cast<size_t>((M - 1) * ldo + H) * osz : 0;
    for (int q = 0; q < P; ++q)
        if (overlaps(out, out_bytes, x_shards[q], xbytes[q])) return DET_ERR_ARG;
    if (overlaps(out, out_bytes, workspace, ws_bytes) || overlaps(out, out_bytes, w, w ? static_cast<size_t>(N) * 4 : 0) ||
        overlaps(out, out_bytes, idx, static_cast<size_t>(N) * 4))
        return DET_ERR_ARG;

    cudaStream_t st = as_stream(stream);
    int* flags = static_cast<int*>(workspace);
    DETR_CUDA(cudaMemsetAsync(flags, 0, 256, st));
    if (M == 0 || H == 0) return DET_OK;
    AtomicArgs a{};
    a.idx = idx;
    a.N = N;
    a.M = M;
    a.H = static_cast<int>(H);
    a.w = w;
    a.flags = flags;
    if (out_dtype == DET_F32) {
        a.acc = static_cast<float*>(out);
        a.lda = ldo;
        if (!accumulate)
            DETR_CUDA(cudaMemset2DAsync(out, static_cast<size_t>(ldo) * 4, 0, static_cast<size_t>(H) * 4,
                                        static_cast<size_t>(M), st));
    } else {
        a.acc = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + 256);
        a.lda = H;
        DETR_CUDA(cudaMemsetAsync(a.acc, 0, static_cast<size_t>(M) * H * 4, st));
    }
    const int xsz = dtype_size(x_dtype);
    const int VEC = 16 / xsz;
    bool vec = (H % VEC == 0) && ((ldx * xsz) % 16 == 0);
    for (int q = 0; q < P; ++q)
        if (shard_rows[q] > 0 && !aligned(x_shards[q], 16)) vec = false;
    const bool vatom = vec && aligned(a.acc, 16) && a.lda % 4 == 0;
    a.V = static_cast<int>(vec ? H / VEC : H);
    a.ldx_bytes = ldx * xsz;
    int64_t grid64 = opts && opts->grid_ctas > 0 ? opts->grid_ctas : cdiv(N, kAtomicWarps);
    grid64 = std::max<int64_t>(1, std::min<int64_t>(grid64, 2147483647));
    const int grid = static_cast<int>(grid64);
    if (N > 0) {
        if (x_dtype == DET_BF16) launch_atomic<uint16_t>(vec, vatom, a, tbl, grid, st);
        else launch_atomic<float>(vec, vatom, a, tbl, grid, st);
        DETR_LAUNCHED();
    }
    if (out_dtype == DET_BF16) {
        const bool v8 = H % 8 == 0 && aligned(out, 16) && ldo % 8 == 0 && aligned(a.acc, 16);
        const int64_t per_row = v8 ? H / 8 : H;
        const unsigned int gx = static_cast<unsigned int>(std::max<int64_t>(1, std::min<int64_t>(cdiv(per_row, 256), 64)));
        const unsigned int gy = static_cast<unsigned int>(std::max<int64_t>(1, std::min<int64_t>(M, 65535)));
        if (M > 0 && H > 0) {
            if (v8)
                cast_bf16_kernel<true><<<dim3(gx, gy), 256, 0, st>>>(a.acc, M, a.H, static_cast<__nv_bfloat16*>(out), ldo);
            else
                cast_bf16_kernel<false><<<dim3(gx, gy), 256, 0, st>>>(a.acc, M, a.H, static_cast<__nv_bfloat16*>(out), ldo);
            DETR_LAUNCHED();
        }
    }
    if (opts && opts->debug_checks) {
        int bad = 0;
        DETR_CUDA(cudaMemcpyAsync(&bad, flags, sizeof(int), cudaMemcpyDeviceToHost, st));
        DETR_CUDA(cudaStreamSynchronize(st));
        if (bad) return DET_ERR_INDEX_RANGE;
    }
    return DET_OK;
}

extern "C" {

det_status det_atomic_scatter_reduce(const int32_t* idx, int64_t N, int64_t M, const void* const* x_shards,
                                     const int64_t* shard_rows, int32_t P, det_dtype x_dtype, int64_t ldx, int64_t H,
                                     const float* w, void* out, int64_t ldo, det_dtype out_dtype, void* workspace,
                                     size_t ws_bytes, const det_opts* opts, void* stream)
{
    return atomic_impl(idx, N, M, x_shards, shard_rows, P, x_dtype, ldx, H, w, out, ldo, out_dtype, workspace,
                       ws_bytes, opts, stream, false);
}

det_status det_atomic_index_add(const int32_t* idx, int64_t N, int64_t M, const void* const* x_shards,
                                const int64_t* shard_rows, int32_t P, det_dtype x_dtype, int64_t ldx, int64_t H,
                                const float* w, void* out, int64_t ldo, det_dtype out_dtype, void* workspace,
                                size_t ws_bytes, const det_opts* opts, void* stream)
{
    return atomic_impl(idx, N, M, x_shards, shard_rows, P, x_dtype, ldx, H, w, out, ldo, out_dtype, workspace,
                       ws_bytes, opts, stream, true);
}

}  // extern "C"
