// gather_async.cu -- vector-path gather-reduce with asynchronous copies.
//
// Same work decomposition and the same arithmetic as the register-staged
// kernel in gather.cu (warp task = plan unit x H-tiles; lanes = chunk slot x
// 16-byte column; left-to-right fold per chunk, xor-shuffle tree per round,
// binary counter over rounds), but every lane moves its 16-byte pieces of the
// source rows with cp.async into its own column of a per-warp shared-memory
// ring.  The warp issues batch b + 3 before it folds batch b, so up to 12 KB
// per warp stay in flight without holding registers, and the next round's
// source list is read while the current round streams.  A lane only ever
// reads the bytes it copied itself, so cp.async.wait_group is the only
// synchronisation the data needs.  The hot-destination segments, the sparse
// key scatter (256-byte rows) and any wide-row problem with long lists go
// through here.
#include "common.cuh"
#include "gather_internal.cuh"
#include "plan_internal.cuh"
#include "reduce_common.cuh"

namespace detr {

constexpr int kAsyncThreads = kAsyncWarps * 32;
constexpr int kAsyncBatch = 8;                            // terms per batch
constexpr int kAsyncBatchesPerRound = kChunk / kAsyncBatch;
constexpr int kAsyncDepth = 4;                            // ring slots per lane
constexpr int kAsyncLook = kAsyncDepth - 1;               // batches in flight ahead of the fold
constexpr int kAsyncMaxSlots = 8;
constexpr int kSlotPad = 34;  // staging stride per slot: slots land in different banks

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// bytes of shared memory per warp: two staging buffers (row pointer + weight
// per term of a round), the ring, and the binary-counter stack
__host__ __device__ constexpr size_t async_warp_bytes(int S, int levels, int vec)
{
    return static_cast<size_t>(2) * S * kSlotPad * (sizeof(void*) + sizeof(float)) +
           static_cast<size_t>(kAsyncDepth) * kAsyncBatch * 32 * 16 +
           static_cast<size_t>(levels) * vec * 32 * sizeof(float);
}

template <typename XT, typename OT>
__global__ void __launch_bounds__(kAsyncThreads)
gather_async_kernel(const __grid_constant__ GatherArgs a, const __grid_constant__ ShardTable tbl)
{
    using LD = Loader<XT, true>;
    constexpr int VEC = LD::VEC;
    extern __shared__ __align__(16) unsigned char smem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int S = 1 << a.S_log2;
    const int T = 1 << a.T_log2;
    const int lane_t = lane & (T - 1);
    const int slot = lane >> a.T_log2;
    const int SR = S * kSlotPad;  // staging entries per round (padded)
    unsigned char* wbase = smem + static_cast<size_t>(warp) * async_warp_bytes(S, a.levels, VEC);
    const unsigned char** sptr = reinterpret_cast<const unsigned char**>(wbase);  // [2][SR]
    float* swt = reinterpret_cast<float*>(wbase + static_cast<size_t>(2) * SR * sizeof(void*));  // [2][SR]
    unsigned char* ring = wbase + static_cast<size_t>(2) * SR * (sizeof(void*) + sizeof(float));
    const uint32_t ring_lane = smem_addr(ring) + lane * 16;
    float* stk = reinterpret_cast<float*>(ring + static_cast<size_t>(kAsyncDepth) * kAsyncBatch * 32 * 16);
    const bool has_w = a.w != nullptr;
    const long long seg_terms = static_cast<long long>(kChunk) << a.g;

    const long long nwarps = static_cast<long long>(gridDim.x) * kAsyncWarps;
    long long n_tasks, n_seg;
    if (!task_counts(a, &n_tasks, &n_seg)) return;
    for (long long task = static_cast<long long>(blockIdx.x) * kAsyncWarps + warp; task < n_tasks;
         task += nwarps) {
        int t0, t1;
        const long long u = task_unit(a, task, n_seg, &t0, &t1);
        const int4 ud = unit_at(a, u, n_seg);
        const int m = ud.x, seg = ud.y;
        const int lo = a.row_ptr[m], hi = a.row_ptr[m + 1];
        int beg = lo, end = hi;
        if (seg >= 0) {
            beg = lo + static_cast<int>(seg * seg_terms);
            end = static_cast<int>(min(static_cast<long long>(beg) + seg_terms, static_cast<long long>(hi)));
        }
        const int n = end - beg;
        const int nch = (n + kChunk - 1) / kChunk;
        const int nrounds = (nch + S - 1) >> a.S_log2;
        const int nb = nrounds * kAsyncBatchesPerRound;


        // stage round r of the list into buffer r & 1: row pointers and weights
        auto stage_round = [&](int r) {
            const int bufo = (r & 1) * SR;
#pragma unroll
            for (int s2 = 0; s2 < kAsyncMaxSlots; ++s2) {
                if (s2 < S) {
                    const int c2 = r * S + s2;
                    const int j = beg + c2 * kChunk + lane;
                    const unsigned char* p = nullptr;
                    float wv = 1.0f;
                    if (c2 < nch && j < end) {
                        const int i = a.perm[j];
                        p = shard_row(tbl, i, a.ldx_bytes);
                        if (has_w) wv = a.w[i];
                    }
                    sptr[bufo + s2 * kSlotPad + lane] = p;
                    swt[bufo + s2 * kSlotPad + lane] = wv;
                }
            }
        };

        for (int tile = t0; tile < t1; ++tile) {
            const int v = tile * T + lane_t;
            const int e0 = v * VEC;
            const bool active = e0 < a.H;
            const long long eoff = static_cast<long long>(e0) * sizeof(XT);
            unsigned int cnt = 0;
            float acc[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
            // next round's list, read ahead: perm values, then row pointers and weights
            int pre_i[kAsyncMaxSlots];
            const unsigned char* pre_p[kAsyncMaxSlots];
            float pre_w[kAsyncMaxSlots];

            __syncwarp();
            if (nrounds > 0) stage_round(0);
            __syncwarp();

            for (int b = 0; b < nb + kAsyncLook; ++b) {
                if (b < nb) {
                    const int r = b >> 2, q = b & 3;
                    if (q == 0 && r > 0) {
                        const int bufo = (r & 1) * SR;
#pragma unroll
                        for (int s2 = 0; s2 < kAsyncMaxSlots; ++s2) {
                            if (s2 < S) {
                                sptr[bufo + s2 * kSlotPad + lane] = pre_p[s2];
                                swt[bufo + s2 * kSlotPad + lane] = pre_w[s2];
                            }
                        }
                        __syncwarp();
                    }
                    if (q == 0 && r + 1 < nrounds) {
#pragma unroll
                        for (int s2 = 0; s2 < kAsyncMaxSlots; ++s2) {
                            pre_i[s2] = -1;
                            if (s2 < S) {
                                const int c2 = (r + 1) * S + s2;
                                const int j = beg + c2 * kChunk + lane;
                                if (c2 < nch && j < end) pre_i[s2] = a.perm[j];
                            }
                        }
                    }
                    if (q == 2 && r + 1 < nrounds) {
#pragma unroll
                        for (int s2 = 0; s2 < kAsyncMaxSlots; ++s2) {
                            pre_p[s2] = nullptr;
                            pre_w[s2] = 1.0f;
                            if (s2 < S && pre_i[s2] >= 0) {
                                pre_p[s2] = shard_row(tbl, pre_i[s2], a.ldx_bytes);
                                if (has_w) pre_w[s2] = a.w[pre_i[s2]];
                            }
                        }
                    }
                    // issue batch b: terms 8q .. 8q+7 of this lane's chunk of round r
                    const int c = r * S + slot;
                    if (c < nch && active) {
                        const int cnt_c = min(kChunk, n - c * kChunk);
                        const unsigned char* const* myp = sptr + (r & 1) * SR + slot * kSlotPad;
                        const uint32_t dst = ring_lane + (b % kAsyncDepth) * (kAsyncBatch * 32 * 16);
#pragma unroll
                        for (int qq = 0; qq < kAsyncBatch; ++qq) {
                            const int j = q * kAsyncBatch + qq;
                            if (j < cnt_c) cp_async16(dst + qq * 512, myp[j] + eoff);
                        }
                    }
                }
                cp_async_commit();
                if (b >= kAsyncLook) {
                    cp_async_wait<kAsyncLook>();
                    // fold batch bb
                    const int bb = b - kAsyncLook;
                    const int r = bb >> 2, q = bb & 3;
                    const int c = r * S + slot;
                    if (c < nch) {
                        const int cnt_c = min(kChunk, n - c * kChunk);
                        const float* myw = swt + (r & 1) * SR + slot * kSlotPad;
                        const unsigned char* src = ring + (bb % kAsyncDepth) * (kAsyncBatch * 32 * 16) + lane * 16;
#pragma unroll
                        for (int qq = 0; qq < kAsyncBatch; ++qq) {
                            const int j = q * kAsyncBatch + qq;
                            if (j < cnt_c) {
                                float xf[VEC];
                                if (active) {
                                    const uint4 raw = *reinterpret_cast<const uint4*>(src + qq * 512);
                                    LD::expand(raw, xf);
                                } else {
#pragma unroll
                                    for (int e = 0; e < VEC; ++e) xf[e] = 0.0f;
                                }
                                fold_term<VEC>(acc, xf, has_w, has_w ? myw[j] : 1.0f, j == 0);
                            }
                        }
                    }
                    if (q == kAsyncBatchesPerRound - 1) {
                        // end of round r: level-wise tree over the slots, then the counter
                        for (int lvl = 0; lvl < a.S_log2; ++lvl) {
                            const int off = 1 << (a.T_log2 + lvl);
                            float pv[VEC];
#pragma unroll
                            for (int e = 0; e < VEC; ++e) pv[e] = __shfl_xor_sync(0xffffffffu, acc[e], off);
                            const int mine = r * S + ((slot >> lvl) << lvl);
                            const int theirs = r * S + (((slot ^ (1 << lvl)) >> lvl) << lvl);
                            if (mine < nch && theirs < nch) {
#pragma unroll
                                for (int e = 0; e < VEC; ++e) acc[e] = __fadd_rn(acc[e], pv[e]);
                            } else if (mine >= nch) {
#pragma unroll
                                for (int e = 0; e < VEC; ++e) acc[e] = pv[e];
                            }
                        }
                        scounter_push<VEC>(stk, 32, lane, cnt, acc);
                        ++cnt;
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
                    }
                }
            }
            float res[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) res[e] = 0.0f;  // empty destination: +0.0
            scounter_collapse<VEC>(stk, 32, lane, cnt, res);
            if (slot == 0 && active) {
                if (seg < 0) {
                    store_out<OT, VEC>(a.out, static_cast<long long>(m) * a.ldo + e0, res, a.out_vec != 0);
                } else {
                    float* o = a.part + static_cast<long long>(ud.z) * a.ldpart + e0;
#pragma unroll
                    for (int e = 0; e < VEC; e += 4)
                        *reinterpret_cast<float4*>(o + e) = make_float4(res[e], res[e + 1], res[e + 2], res[e + 3]);
                }
            }
        }
    }
}

size_t async_smem_bytes(int S_log2, int levels, int vec)
{
    return async_warp_bytes(1 << S_log2, levels, vec) * kAsyncWarps;
}

template <typename XT, typename OT>
static det_status launch_async_t(const GatherArgs& a, const ShardTable& t, int grid, cudaStream_t st)
{
    const size_t smem = async_smem_bytes(a.S_log2, a.levels, Loader<XT, true>::VEC);
    {
        const det_status a_ = allow_dynamic_smem(reinterpret_cast<const void*>(gather_async_kernel<XT, OT>), smem);
        if (a_) return a_;
    }
    if (grid <= 0) {
        int per_sm = 1, sms = 1;
        DETR_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_async_kernel<XT, OT>, kAsyncThreads,
                                                                smem));
        det_status s = current_sm_count(&sms);
        if (s) return s;
        grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cdiv(a.n_tasks, kAsyncWarps),
                                                                        int64_t(std::max(per_sm, 1)) * sms)));
    }
    gather_async_kernel<XT, OT><<<grid, kAsyncThreads, smem, st>>>(a, t);
    DETR_LAUNCHED();
    return DET_OK;
}

det_status launch_gather_async(det_dtype x_dtype, det_dtype out_dtype, const GatherArgs& a, const ShardTable& t,
                               int grid, cudaStream_t st)
{
    if (x_dtype == DET_BF16 && out_dtype == DET_BF16) return launch_async_t<uint16_t, __nv_bfloat16>(a, t, grid, st);
    if (x_dtype == DET_BF16) return launch_async_t<uint16_t, float>(a, t, grid, st);
    if (out_dtype == DET_BF16) return launch_async_t<float, __nv_bfloat16>(a, t, grid, st);
    return launch_async_t<float, float>(a, t, grid, st);
}

}  // namespace detr
