// splitk.cu -- split-id-ordered split-K reduce.
//
// The mHC backward cannot avoid split-K (output width 24, K = 7168): every
// K-split writes its own buffer and a deterministic reduce kernel sums them
// in split-id order ("DeepSeek-V4 book, Ch 09: Batch invariance and
// determinism", section 3.3).  Here the sum over s is the same canonical fold
// as the scatter-reduce: chunks of 32 splits folded left to right, then the
// level-wise pairwise tree with the odd chunk carried up.  A thread owns four
// consecutive outputs (16-byte loads) and one chunk slot; neighbouring lanes
// fold neighbouring chunks and meet through xor shuffles.  With exactly two
// chunks (33..64 splits) and 16-byte rows, one thread folds both, one after
// the other, with eight loads in flight instead of four: fewer, deeper load
// rounds per thread (measured 19.2 us against 20.7 us for the two-slot split
// on the 56-split mHC reduce, where a plain read of the same 88 MB takes
// 18.3 us on the same clock).
#include <algorithm>

#include "common.cuh"

namespace detr {

constexpr int kSplitThreads = 256;
constexpr int kSplitBatch = 4;
// Six CTAs per SM (at most 40 registers a thread) when one round of chunk
// slots covers all splits: the 56-split, 393216-output reduce then runs as one
// wave of resident CTAs, where 64 registers left a quarter of the CTAs for a
// second wave.  Deeper counters (more rounds) keep four.
constexpr int kSplitMinBlocks = 6;
constexpr int kMaxSplitSlotsLog2 = 3;
constexpr int kMaxSplitRounds = 127;

struct SplitArgs {
    const float* P;
    long long ldp;
    long long nvec;     // output vectors (VEC outputs each)
    long long items;    // nvec << slots_log2
    void* out;
    int S;
    int slots_log2;
    int out_vec;
};

template <int DR, int VEC>
__device__ __forceinline__ void sk_push(float (&stk)[DR][VEC], unsigned int cnt, float* node)
{
    unsigned int c = cnt;
    bool placed = false;
#pragma unroll
    for (int L = 0; L < DR; ++L) {
        if (!placed) {
            if (c & 1u) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) node[e] = __fadd_rn(stk[L][e], node[e]);
                c >>= 1;
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) stk[L][e] = node[e];
                placed = true;
            }
        }
    }
}

template <typename OT, bool VECTOR, int DR>
__global__ void __launch_bounds__(kSplitThreads, DR == 1 ? kSplitMinBlocks : 4) splitk_kernel(const __grid_constant__ SplitArgs a)
{
    constexpr int VEC = VECTOR ? 4 : 1;
    const int lane = threadIdx.x & 31;
    const int slots = 1 << a.slots_log2;
    const int nch = (a.S + kChunk - 1) / kChunk;
    const int nrounds = (nch + slots - 1) >> a.slots_log2;
    const long long gwarp = (static_cast<long long>(blockIdx.x) * kSplitThreads + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * kSplitThreads) >> 5;
    for (long long base = gwarp * 32; base < a.items; base += nwarps * 32) {
        const long long item = base + lane;
        const bool valid = item < a.items;
        const long long v = item >> a.slots_log2;
        const int slot = static_cast<int>(item & (slots - 1));
        const long long e0 = v * VEC;
        float stk[DR][VEC];
        unsigned int cnt = 0;
        for (int r = 0; r < nrounds; ++r) {
            const int c = r * slots + slot;
            float acc[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
            if (valid && c < nch) {
                const int s_lo = c * kChunk;
                const int cnt_c = min(kChunk, a.S - s_lo);
                const float* col = a.P + static_cast<long long>(s_lo) * a.ldp + e0;
                for (int jb = 0; jb < cnt_c; jb += kSplitBatch) {
                    float vals[kSplitBatch][VEC];
#pragma unroll
                    for (int q = 0; q < kSplitBatch; ++q) {
                        if (jb + q < cnt_c) {
                            const float* src = col + static_cast<long long>(jb + q) * a.ldp;
                            if (VECTOR) {
                                const uint4 u = ld_stream_v4(src);
                                vals[q][0] = __uint_as_float(u.x);
                                if (VEC > 1) {
                                    vals[q][VEC > 1 ? 1 : 0] = __uint_as_float(u.y);
                                    vals[q][VEC > 2 ? 2 : 0] = __uint_as_float(u.z);
                                    vals[q][VEC > 3 ? 3 : 0] = __uint_as_float(u.w);
                                }
                            } else {
                                vals[q][0] = __ldcs(src);
                            }
                        }
                    }
#pragma unroll
                    for (int q = 0; q < kSplitBatch; ++q) {
                        if (jb + q < cnt_c) {
                            if (jb + q == 0) {
#pragma unroll
                                for (int e = 0; e < VEC; ++e) acc[e] = vals[q][e];
                            } else {
#pragma unroll
                                for (int e = 0; e < VEC; ++e) acc[e] = __fadd_rn(acc[e], vals[q][e]);
                            }
                        }
                    }
                }
            }
            for (int lvl = 0; lvl < a.slots_log2; ++lvl) {
                float pv[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) pv[e] = __shfl_xor_sync(0xffffffffu, acc[e], 1 << lvl);
                const int mine = r * slots + ((slot >> lvl) << lvl);
                const int theirs = r * slots + (((slot ^ (1 << lvl)) >> lvl) << lvl);
                if (mine < nch && theirs < nch) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) acc[e] = __fadd_rn(acc[e], pv[e]);
                } else if (mine >= nch) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) acc[e] = pv[e];
                }
            }
            sk_push<DR, VEC>(stk, cnt, acc);
            ++cnt;
        }
        float res[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) res[e] = 0.0f;
        bool have = false;
#pragma unroll
        for (int L = 0; L < DR; ++L) {
            if ((cnt >> L) & 1u) {
                if (!have) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) res[e] = stk[L][e];
                    have = true;
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) res[e] = __fadd_rn(stk[L][e], res[e]);
                }
            }
        }
        if (valid && slot == 0) {
            if (sizeof(OT) == 4) {
                float* o = static_cast<float*>(a.out) + e0;
                if (VECTOR && a.out_vec) *reinterpret_cast<float4*>(o) = make_float4(res[0], res[VEC > 1 ? 1 : 0], res[VEC > 2 ? 2 : 0], res[VEC > 3 ? 3 : 0]);
                else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) o[e] = res[e];
                }
            } else {
                __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + e0;
                if (VECTOR && a.out_vec) {
                    __nv_bfloat162 t0 = __floats2bfloat162_rn(res[0], res[VEC > 1 ? 1 : 0]);
                    __nv_bfloat162 t1 = __floats2bfloat162_rn(res[VEC > 2 ? 2 : 0], res[VEC > 3 ? 3 : 0]);
                    uint2 pk;
                    pk.x = *reinterpret_cast<uint32_t*>(&t0);
                    pk.y = *reinterpret_cast<uint32_t*>(&t1);
                    *reinterpret_cast<uint2*>(o) = pk;
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) o[e] = __float2bfloat16_rn(res[e]);
                }
            }
        }
    }
}

// Two chunks, 16-byte rows: thread v folds rows [0, 32) and [32, S) of its
// four columns left to right, eight loads in flight, then adds the two chunk
// nodes (the whole pairwise tree of two leaves).
constexpr int kTwoChunkBatch = 8;

// Rows [j0, j1) of one 16-byte column folded left to right from the first.
__device__ __forceinline__ float4 fold_column(const float* col, long long ldp, int j0, int j1)
{
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int jb = j0; jb < j1; jb += kTwoChunkBatch) {
        uint4 u[kTwoChunkBatch];
#pragma unroll
        for (int q = 0; q < kTwoChunkBatch; ++q)
            if (jb + q < j1) u[q] = ld_stream_v4(col + static_cast<long long>(jb + q) * ldp);
#pragma unroll
        for (int q = 0; q < kTwoChunkBatch; ++q) {
            if (jb + q < j1) {
                const float4 x = make_float4(__uint_as_float(u[q].x), __uint_as_float(u[q].y),
                                             __uint_as_float(u[q].z), __uint_as_float(u[q].w));
                if (jb + q == j0) {
                    acc = x;
                } else {
                    acc.x = __fadd_rn(acc.x, x.x);
                    acc.y = __fadd_rn(acc.y, x.y);
                    acc.z = __fadd_rn(acc.z, x.z);
                    acc.w = __fadd_rn(acc.w, x.w);
                }
            }
        }
    }
    return acc;
}

template <typename OT>
__global__ void __launch_bounds__(kSplitThreads, 3) splitk_two_chunk_kernel(const __grid_constant__ SplitArgs a)
{
    for (long long v = static_cast<long long>(blockIdx.x) * kSplitThreads + threadIdx.x; v < a.nvec;
         v += static_cast<long long>(gridDim.x) * kSplitThreads) {
    const float* col = a.P + v * 4;
    const float4 n0 = fold_column(col, a.ldp, 0, kChunk);
    const float4 n1 = fold_column(col, a.ldp, kChunk, a.S);
    const float res[4] = {__fadd_rn(n0.x, n1.x), __fadd_rn(n0.y, n1.y), __fadd_rn(n0.z, n1.z), __fadd_rn(n0.w, n1.w)};
    const long long e0 = v * 4;
    if (sizeof(OT) == 4) {
        float* o = static_cast<float*>(a.out) + e0;
        if (a.out_vec) *reinterpret_cast<float4*>(o) = make_float4(res[0], res[1], res[2], res[3]);
        else {
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = res[e];
        }
    } else {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + e0;
        if (a.out_vec) {
            __nv_bfloat162 t0 = __floats2bfloat162_rn(res[0], res[1]);
            __nv_bfloat162 t1 = __floats2bfloat162_rn(res[2], res[3]);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&t0);
            pk.y = *reinterpret_cast<uint32_t*>(&t1);
            *reinterpret_cast<uint2*>(o) = pk;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = __float2bfloat16_rn(res[e]);
        }
    }
    }
}

template <typename OT, bool VECTOR>
static void launch_splitk(int DR, const SplitArgs& a, int grid, cudaStream_t st)
{
    if (DR <= 1) splitk_kernel<OT, VECTOR, 1><<<grid, kSplitThreads, 0, st>>>(a);
    else if (DR <= 4) splitk_kernel<OT, VECTOR, 4><<<grid, kSplitThreads, 0, st>>>(a);
    else splitk_kernel<OT, VECTOR, 7><<<grid, kSplitThreads, 0, st>>>(a);
}

}  // namespace detr

using namespace detr;

extern "C" det_status det_splitk_reduce(const float* partials, int32_t S, int64_t count, int64_t ldp, void* out,
                                        det_dtype out_dtype, const det_opts* opts, void* stream)
{
    if (!dtype_ok(out_dtype)) return DET_ERR_DTYPE;
    if (S < 0 || count < 0 || ldp < count) return DET_ERR_ARG;
    if (count == 0) return DET_OK;
    if (!out || (S > 0 && !partials)) return DET_ERR_ARG;
    if (!aligned(partials, 4) || !aligned(out, static_cast<size_t>(dtype_size(out_dtype)))) return DET_ERR_ARG;
    if (ldp > (int64_t(1) << 40) || count > (int64_t(1) << 40)) return DET_ERR_UNSUPPORTED;
    const size_t pbytes = S > 0 ? static_cast<size_t>((S - 1) * ldp + count) * 4 : 0;
    if (overlaps(out, static_cast<size_t>(count) * dtype_size(out_dtype), partials, pbytes)) return DET_ERR_ARG;
    const int nch = (S + kChunk - 1) / kChunk;
    int slots_log2 = 0;
    while ((1 << slots_log2) < nch && slots_log2 < kMaxSplitSlotsLog2) ++slots_log2;
    const int rounds = (nch + (1 << slots_log2) - 1) >> slots_log2;
    if (rounds > kMaxSplitRounds) return DET_ERR_UNSUPPORTED;
    const int DR = rounds <= 1 ? 1 : (rounds <= 15 ? 4 : 7);
    const bool vec = aligned(partials, 16) && ldp % 4 == 0 && count % 4 == 0;
    SplitArgs a{};
    a.P = partials;
    a.ldp = ldp;
    a.nvec = vec ? count / 4 : count;
    a.slots_log2 = slots_log2;
    a.items = a.nvec << slots_log2;
    a.out = out;
    a.S = S;
    a.out_vec = aligned(out, 16);
    int64_t grid64 = opts && opts->grid_ctas > 0 ? opts->grid_ctas : cdiv(a.items, kSplitThreads);
    grid64 = std::max<int64_t>(1, std::min<int64_t>(grid64, 2147483647));
    cudaStream_t st = as_stream(stream);
    if (S == 0) {
        // no terms: every output is +0.0
        DETR_CUDA(cudaMemsetAsync(out, 0, static_cast<size_t>(count) * dtype_size(out_dtype), st));
        return DET_OK;
    }
    if (vec && nch == 2) {
        SplitArgs b = a;  // one thread per 16-byte column, both chunks
        b.slots_log2 = 0;
        b.items = a.nvec;
        int64_t g2 = opts && opts->grid_ctas > 0 ? opts->grid_ctas : cdiv(a.nvec, kSplitThreads);
        g2 = std::max<int64_t>(1, std::min<int64_t>(g2, 2147483647));
        if (out_dtype == DET_BF16) splitk_two_chunk_kernel<__nv_bfloat16><<<static_cast<int>(g2), kSplitThreads, 0, st>>>(b);
        else splitk_two_chunk_kernel<float><<<static_cast<int>(g2), kSplitThreads, 0, st>>>(b);
        DETR_LAUNCHED();
        if (opts && opts->debug_checks) DETR_CUDA(cudaStreamSynchronize(st));
        return DET_OK;
    }
    const int grid = static_cast<int>(grid64);
    if (out_dtype == DET_BF16) {
        if (vec) launch_splitk<__nv_bfloat16, true>(DR, a, grid, st);
        else launch_splitk<__nv_bfloat16, false>(DR, a, grid, st);
    } else {
        if (vec) launch_splitk<float, true>(DR, a, grid, st);
        else launch_splitk<float, false>(DR, a, grid, st);
    }
    DETR_LAUNCHED();
    if (opts && opts->debug_checks) DETR_CUDA(cudaStreamSynchronize(st));
    return DET_OK;
}
