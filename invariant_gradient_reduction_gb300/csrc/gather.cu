// gather.cu -- the deterministic gather-reduce (destination-major) and the
// second pass for hot destinations.
//
// One warp task = one unit of the plan (a whole destination, or one hot
// segment of 2^g chunks) x a group of H-tiles.  Inside a warp, lanes are
// (slot, vector): T lanes cover one H-tile of a source row with 16-byte
// loads, and 32/T slots fold different chunks of 32 terms at the same time.
// Each lane folds its chunk left to right in registers; the slots of one
// round are combined by a level-wise tree over xor shuffles, in which an
// absent right neighbour leaves its left neighbour unchanged (the odd carry);
// the round nodes, which are aligned tree nodes, go into a binary counter
// whose merge order is exactly the level-wise pairwise tree.  None of these
// choices changes a bit: each output element is the canonical sum of its
// terms.
//
// The problem and its constraints: the MoE token combine index_add_ versus
// scatter_add_ ("Megatron-LM determinism developer reference", section 3.1);
// the sparse-attention backward scatter onto hot keys ("DeepSeek-V4 book, Ch
// 09", section 3.1); private slots merged in a fixed order instead of writers
// racing on one address ("Bit-exact training interview notes", table "where
// nondeterminism comes from").
#include <algorithm>

#include "common.cuh"
#include "gather_internal.cuh"
#include "plan_internal.cuh"
#include "reduce_common.cuh"

namespace detr {

constexpr int kGatherThreads = 256;
constexpr int kGatherWarps = kGatherThreads / 32;
constexpr int kBatch = 8;
constexpr int kStagePad = 33;
constexpr int kFinishThreads = 256;
#ifndef DETR_FINISH_FV
#define DETR_FINISH_FV 4
#endif


#ifndef DETR_GATHER_MIN_BLOCKS
#define DETR_GATHER_MIN_BLOCKS 3
#endif

// ACC: compiled for index_add_ (a.accumulate set: the canonical sum is added
// to out, destinations without terms are left untouched), with the
// destination tile requested early; the scatter-reduce instantiations keep
// the code (and register allocation) without that request.  BESIDE (with
// ACC): the instantiation that runs beside the ring kernel (a.beside_ring),
// with its wait for the previous grid at the end; a separate instantiation,
// since the wait at the end cost the others 12 bytes more of spills.
template <typename XT, typename OT, bool VECTOR, bool ACC, bool BESIDE>
__global__ void __launch_bounds__(kGatherThreads, DETR_GATHER_MIN_BLOCKS)
gather_reduce_kernel(const __grid_constant__ GatherArgs a, const __grid_constant__ ShardTable tbl)
{
    using LD = Loader<XT, VECTOR>;
    constexpr int VEC = LD::VEC;
    extern __shared__ __align__(16) unsigned char smem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int S = 1 << a.S_log2;
    const int T = 1 << a.T_log2;
    const int lane_t = lane & (T - 1);
    const int slot = lane >> a.T_log2;
    const unsigned char** sptr =
        reinterpret_cast<const unsigned char**>(smem) + static_cast<size_t>(warp) * S * kStagePad;
    float* swt = reinterpret_cast<float*>(reinterpret_cast<const unsigned char**>(smem) +
                                          static_cast<size_t>(kGatherWarps) * S * kStagePad) +
                 static_cast<size_t>(warp) * S * kStagePad;
    float* stk = reinterpret_cast<float*>(reinterpret_cast<const unsigned char**>(smem) +
                                          static_cast<size_t>(kGatherWarps) * S * kStagePad) +
                 static_cast<size_t>(kGatherWarps) * S * kStagePad +
                 static_cast<size_t>(warp) * a.levels * VEC * 32;
    const bool has_w = a.w != nullptr;
    const long long seg_terms = static_cast<long long>(kChunk) << a.g;

    const long long nwarps = static_cast<long long>(gridDim.x) * kGatherWarps;
    // Behind the fixed-stage kernel (only_long) the counts are the plan's,
    // which had finished before that kernel started: they are read before
    // the wait for it, so that a launch with nothing to do ends as soon as
    // that kernel does.  Every launch waits for the grid before it, at the
    // latest before it ends.
    if (!BESIDE && !a.only_long) pdl_wait();  // the plan (or whatever wrote x and w) has finished
    pdl_launch_dependents();                  // the hot-destination pass may be launched now
    long long n_tasks, n_seg;
    const bool counted = task_counts(a, &n_tasks, &n_seg);
    if (!BESIDE && a.only_long) pdl_wait();
    if (!counted) {
        if (BESIDE) pdl_wait();
        return;
    }
    for (long long task = static_cast<long long>(blockIdx.x) * kGatherWarps + warp; task < n_tasks;
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
        if (a.accumulate && n == 0) continue;  // index_add_ leaves it untouched
        const int nch = (n + kChunk - 1) / kChunk;
        const int nrounds = (nch + S - 1) >> a.S_log2;

        bool staged = false;

        for (int tile = t0; tile < t1; ++tile) {
            const int v = tile * T + lane_t;
            const int e0 = v * VEC;
            const bool active = e0 < a.H;
            // index_add_ reads the destination tile only after the fold: ask
            // for it into L1 now, so that the read overlaps the source loads
            if (ACC && slot == 0 && active && seg < 0)
                asm volatile("prefetch.global.L1 [%0];" ::"l"(static_cast<const char*>(a.out) +
                                                            (static_cast<long long>(m) * a.ldo + e0) * sizeof(OT)));
            unsigned int cnt = 0;
            for (int r = 0; r < nrounds; ++r) {
                if (nrounds > 1 || !staged) {
                    __syncwarp();
                    for (int s2 = 0; s2 < S; ++s2) {
                        const int c2 = r * S + s2;
                        const int j = beg + c2 * kChunk + lane;
                        const unsigned char* p = nullptr;
                        float wv = 1.0f;
                        if (c2 < nch && j < end) {
                            const int i = a.perm[j];
                            p = shard_row(tbl, i, a.ldx_bytes);
                            if (has_w) wv = a.w[i];
                        }
                        sptr[s2 * kStagePad + lane] = p;
                        swt[s2 * kStagePad + lane] = wv;
                    }
                    __syncwarp();
                    staged = true;
                }
                // fold this lane's chunk, left to right from its first term
                const int c = r * S + slot;
                float acc[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
                if (c < nch) {
                    const int cnt_c = min(kChunk, n - c * kChunk);
                    const unsigned char** myp = sptr + slot * kStagePad;
                    const float* myw = swt + slot * kStagePad;
                    const long long eoff = static_cast<long long>(e0) * sizeof(XT);
                    for (int jb = 0; jb < cnt_c; jb += kBatch) {
                        typename LD::Raw raw[kBatch];
#pragma unroll
                        for (int q = 0; q < kBatch; ++q)
                            if (jb + q < cnt_c && active) raw[q] = LD::load(myp[jb + q] + eoff);
#pragma unroll
                        for (int q = 0; q < kBatch; ++q) {
                            if (jb + q < cnt_c) {
                                float xf[VEC];
                                if (active) LD::expand(raw[q], xf);
                                else {
#pragma unroll
                                    for (int e = 0; e < VEC; ++e) xf[e] = 0.0f;
                                }
                                fold_term<VEC>(acc, xf, has_w, has_w ? myw[jb + q] : 1.0f, jb + q == 0);
                            }
                        }
                    }
                }
                // level-wise tree over the slots of this round (xor partners)
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
            }
            float res[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) res[e] = 0.0f;  // empty destination: +0.0
            scounter_collapse<VEC>(stk, 32, lane, cnt, res);
            if (slot == 0 && active) {
                if (seg < 0) {
                    const long long off = static_cast<long long>(m) * a.ldo + e0;
                    if (!a.accumulate) store_out<OT, VEC>(a.out, off, res, a.out_vec != 0);
                    else if (n > 0) add_store_out<OT, VEC>(a.out, off, res, a.out_vec != 0);
                } else {
                    float* o = a.part + static_cast<long long>(ud.z) * a.ldpart + e0;
                    if (VEC % 4 == 0) {
#pragma unroll
                        for (int e = 0; e < VEC; e += 4)
                            *reinterpret_cast<float4*>(o + e) = make_float4(res[e], res[e + 1], res[e + 2], res[e + 3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) o[e] = res[e];
                    }
                }
            }
        }
    }
    if (BESIDE) pdl_wait();  // this grid ends after the ring kernel beside it
}

// Second pass for hot destinations: the level-wise tree over the row's
// segment nodes (aligned nodes of 2^g chunks), in segment order, through the
// binary counter (stack in shared memory, FV columns per thread).  An item
// is FV adjacent columns of one hot row (FV = 4: 16-byte loads of the
// partials, when H and the partial rows allow them).
template <typename OT, int FV>
__global__ void __launch_bounds__(kFinishThreads)
finish_kernel(const int4* finish, long long n_items, int H, const float* part, long long ldpart, void* out,
              long long ldo, const int* dev_counters, int accumulate)
{
    extern __shared__ float fstk[];  // [levels][FV][kFinishThreads]
    const int HV = H / FV;           // H % FV == 0
    // The plan's counts (it had finished before the gather pass started) are
    // read before the wait, so that a launch without hot destinations ends as
    // soon as the gather pass does
    if (dev_counters)
        n_items = dev_counters[kCtrErrIndex] | dev_counters[kCtrErrDup]
                      ? 0
                      : static_cast<long long>(dev_counters[kCtrHot]) * HV;
    pdl_wait();  // the gather pass has written every partial slot
    if (dev_counters && n_items > 0 && dev_counters[kCtrErrTimeout]) return;  // a gather kernel gave up
    for (long long t = static_cast<long long>(blockIdx.x) * kFinishThreads + threadIdx.x; t < n_items;
         t += static_cast<long long>(gridDim.x) * kFinishThreads) {
        const long long row_task = t / HV;
        const int h = static_cast<int>(t - row_task * HV) * FV;
        const int4 ft = finish[row_task];
        const int m = ft.x, s0 = ft.y, ns = ft.z;
        unsigned int cnt = 0;
        for (int s = 0; s < ns; s += kBatch) {
            float v[kBatch][FV];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                if (s + q < ns) {
                    const float* src = part + static_cast<long long>(s0 + s + q) * ldpart + h;
                    if constexpr (FV == 4) {
                        const float4 f = __ldcs(reinterpret_cast<const float4*>(src));
                        v[q][0] = f.x;
                        v[q][1] = f.y;
                        v[q][2] = f.z;
                        v[q][3] = f.w;
                    } else if constexpr (FV == 2) {
                        const float2 f = __ldcs(reinterpret_cast<const float2*>(src));
                        v[q][0] = f.x;
                        v[q][1] = f.y;
                    } else {
#pragma unroll
                        for (int e = 0; e < FV; ++e) v[q][e] = __ldcs(src + e);
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                if (s + q < ns) {
                    scounter_push<FV>(fstk, kFinishThreads, threadIdx.x, cnt, v[q]);
                    ++cnt;
                }
            }
        }
        float res[FV];
#pragma unroll
        for (int e = 0; e < FV; ++e) res[e] = 0.0f;
        scounter_collapse<FV>(fstk, kFinishThreads, threadIdx.x, cnt, res);
        if (accumulate) add_store_out<OT, FV>(out, static_cast<long long>(m) * ldo + h, res, false);
        else store_out<OT, FV>(out, static_cast<long long>(m) * ldo + h, res, false);
    }
}

template <typename XT, typename OT, bool VECTOR, bool ACC, bool BESIDE>
static det_status launch_gather_t(const GatherArgs& a, const ShardTable& t, int grid, cudaStream_t st)
{
    constexpr int VEC = Loader<XT, VECTOR>::VEC;
    const size_t smem = static_cast<size_t>(kGatherWarps) *
                        ((1 << a.S_log2) * kStagePad * (sizeof(void*) + sizeof(float)) +
                         static_cast<size_t>(a.levels) * VEC * 32 * sizeof(float));
    {
        const det_status a_ = allow_dynamic_smem(reinterpret_cast<const void*>(gather_reduce_kernel<XT, OT, VECTOR, ACC, BESIDE>), smem);
        if (a_) return a_;
        // An explicit shared-memory / L1 split: without one, the CTAs that a
        // dependent launch places on SMs just left by a kernel with a large
        // shared-memory footprint (the cluster plan: 222 KB per CTA) keep its
        // split and run ~33% slower with a small L1 (measured: the 16 SMs of
        // that plan's cluster held the reduce 74 us, 440 against 366 us per
        // EP-invariance step).  Half the SM's shared memory, or what the
        // resident CTAs need if that is more; preferring the largest L1
        // instead halved the occupancy.
        // Beside the index_add_ ring kernel: all of it, for that kernel's ring.
        static int carve_set = -1;
        int dev = 0, smem_sm = 0;
        DETR_CUDA(cudaGetDevice(&dev));
        DETR_CUDA(cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev));
        const size_t need = static_cast<size_t>(DETR_GATHER_MIN_BLOCKS) * (smem + 1024);
        int pct = smem_sm > 0 ? std::min<int>(100, std::max<int>(50, static_cast<int>(cdiv(
                                                                        static_cast<int64_t>(need) * 100, smem_sm))))
                              : 50;
        if (BESIDE) pct = 100;
        if (pct != carve_set) {
            DETR_CUDA(cudaFuncSetAttribute(reinterpret_cast<const void*>(gather_reduce_kernel<XT, OT, VECTOR, ACC, BESIDE>),
                                           cudaFuncAttributePreferredSharedMemoryCarveout, pct));
            carve_set = pct;
        }
    }
    if (grid <= 0) {
        // persistent: as many CTAs as fit at once; warps take tasks round-robin
        int per_sm = 1, sms = 1;
        DETR_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_reduce_kernel<XT, OT, VECTOR, ACC, BESIDE>,
                                                                kGatherThreads, smem));
        det_status s = current_sm_count(&sms);
        if (s) return s;
        // beside the ring kernel (544 threads of 64 registers and most of the
        // shared memory on every SM) one CTA of this kernel fits per SM
        if (BESIDE) per_sm = 1;
        grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cdiv(a.n_tasks, kGatherWarps),
                                                                        int64_t(std::max(per_sm, 1)) * sms)));
    }
    DETR_CUDA(launch_after_previous(gather_reduce_kernel<XT, OT, VECTOR, ACC, BESIDE>, dim3(grid), dim3(kGatherThreads), smem, st,
                                    a, t));
    DETR_LAUNCHED();
    return DET_OK;
}

template <typename XT, typename OT, bool VECTOR>
static det_status launch_gather(const GatherArgs& a, const ShardTable& t, int grid, cudaStream_t st)
{
    // beside the ring kernel: 16-byte rows only
    if (!a.accumulate)
        return VECTOR && a.beside_ring ? launch_gather_t<XT, OT, VECTOR, false, VECTOR>(a, t, grid, st)
                                       : launch_gather_t<XT, OT, VECTOR, false, false>(a, t, grid, st);
    return VECTOR && a.beside_ring ? launch_gather_t<XT, OT, VECTOR, true, VECTOR>(a, t, grid, st)
                                   : launch_gather_t<XT, OT, VECTOR, true, false>(a, t, grid, st);
}

template <typename XT, typename OT>
static det_status launch_gather_vec(bool vec, const GatherArgs& a, const ShardTable& t, int grid, cudaStream_t st)
{
    return vec ? launch_gather<XT, OT, true>(a, t, grid, st) : launch_gather<XT, OT, false>(a, t, grid, st);
}

// Wait for the stream and report a CUDA error or an expired device wait.
static det_status debug_sync_status(det_plan plan, cudaStream_t st)
{
    DETR_CUDA(cudaStreamSynchronize(st));
    int h = 0;
    DETR_CUDA(cudaMemcpy(&h, plan->counters + kCtrErrTimeout, sizeof(int), cudaMemcpyDeviceToHost));
    return h ? DET_ERR_TIMEOUT : DET_OK;
}

static int log2_floor(int64_t v)
{
    int r = 0;
    while ((int64_t(1) << (r + 1)) <= v) ++r;
    return r;
}

}  // namespace detr

using namespace detr;

extern "C" {

det_status det_scatter_workspace_size(det_plan plan, int64_t H, size_t* bytes)
{
    if (!plan || !bytes || H < 0) return DET_ERR_ARG;
    if (H > kMaxRows) return DET_ERR_UNSUPPORTED;
    const int64_t ldpart = (H + 7) / 8 * 8;
    const int64_t segs = plan->counts_on_host ? plan->n_segments
                                              : 2 * cdiv(plan->N, static_cast<int64_t>(kChunk) << plan->g) + 1;
    *bytes = static_cast<size_t>(segs) * static_cast<size_t>(ldpart) * sizeof(float);
    return DET_OK;
}

}  // extern "C"

// det_scatter_reduce (accumulate = false) and det_index_add (true).
static det_status scatter_reduce_impl(det_plan plan, const void* const* x_shards, const int64_t* shard_rows,
                                      int32_t P, det_dtype x_dtype, int64_t ldx, int64_t H, const float* w, void* out,
                                      int64_t ldo, det_dtype out_dtype, void* workspace, size_t ws_bytes,
                                      const det_opts* opts, void* stream, bool accumulate)
{
    if (!plan) return DET_ERR_ARG;
    if (!dtype_ok(x_dtype) || !dtype_ok(out_dtype)) return DET_ERR_DTYPE;
    if (H < 0 || ldo < H) return DET_ERR_ARG;
    if (H > kMaxRows) return DET_ERR_UNSUPPORTED;
    ShardTable tbl;
    size_t xbytes[DET_MAX_SHARDS] = {};
    det_status s = make_shard_table(x_shards, shard_rows, P, plan->N, ldx, H, x_dtype, &tbl, xbytes);
    if (s) return s;
    const int64_t M = plan->M;
    const int osz = dtype_size(out_dtype);
    if (M > 0 && H > 0 && !out) return DET_ERR_ARG;
    if (!aligned(out, static_cast<size_t>(osz)) || !aligned(w, 4)) return DET_ERR_ARG;
    if (ldo > (int64_t(1) << 40)) return DET_ERR_ARG;
    const size_t out_bytes = M > 0 && H > 0 ? static_cast<size_t>((M - 1) * ldo + H) * osz : 0;
    size_t need = 0;
    det_scatter_workspace_size(plan, H, &need);
    if (need > 0 && (!workspace || !aligned(workspace, 256) || ws_bytes < need)) return DET_ERR_WORKSPACE;
    for (int q = 0; q < P; ++q)
        if (overlaps(out, out_bytes, x_shards[q], xbytes[q])) return DET_ERR_ARG;
    if (overlaps(out, out_bytes, w, w ? static_cast<size_t>(plan->N) * 4 : 0) ||
        overlaps(out, out_bytes, plan->ws, plan->ws_bytes) || overlaps(out, out_bytes, workspace, ws_bytes))
        return DET_ERR_ARG;
    if (need > 0 && overlaps(workspace, need, plan->ws, plan->ws_bytes)) return DET_ERR_ARG;
    if (M == 0 || H == 0) return DET_OK;

    const int xsz = dtype_size(x_dtype);
    const int VEC = 16 / xsz;
    bool vec = (H % VEC == 0) && ((ldx * xsz) % 16 == 0);
    for (int q = 0; q < P; ++q)
        if (shard_rows[q] > 0 && !aligned(x_shards[q], 16)) vec = false;
    const int64_t V = vec ? H / VEC : H;

    GatherArgs a{};
    int T_log2 = V >= 32 ? 5 : std::max(2, log2_floor(V) + ((V & (V - 1)) ? 1 : 0));
    a.T_log2 = T_log2;
    a.S_log2 = 5 - T_log2;
    a.ntiles = static_cast<int>(cdiv(V, int64_t(1) << T_log2));
    a.H = static_cast<int>(H);
    a.g = plan->g;
    const bool dev_counts = !plan->counts_on_host;  // async plan: counts stay on the device
    a.accumulate = accumulate ? 1 : 0;
    a.seg_units = plan->seg_units;
    a.row_units = plan->row_units;
    a.n_seg = dev_counts ? 0 : plan->n_segments + plan->n_long;
    a.dev_counters = dev_counts ? plan->counters : nullptr;
    const int64_t n_units = dev_counts ? std::max<int64_t>(1, M) : plan->n_units;  // estimate when unknown
    a.row_ptr = plan->row_ptr;
    a.perm = plan->perm;
    a.w = w;
    a.ldx_bytes = ldx * xsz;
    a.out = out;
    a.ldo = ldo;
    a.out_vec = aligned(out, 16) && (ldo * osz) % 16 == 0;
    a.part = static_cast<float*>(workspace);
    a.ldpart = (H + 7) / 8 * 8;

    int sms = 0;
    s = current_sm_count(&sms);
    if (s) return s;
    // Tiles per warp task: about 16 KB of source data per task amortises the
    // task's list lookups, while keeping at least two tasks per resident warp
    // (measured best on the MoE combine and EP-invariance shapes; the split
    // changes no bit).
    const int64_t avg_terms = std::max<int64_t>(1, plan->N / std::max<int64_t>(1, n_units));
    const int64_t tile_bytes = (int64_t(1) << T_log2) * (vec ? 16 : xsz);
    int tpg = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(a.ntiles, 16384 / (avg_terms * tile_bytes))));
    const int64_t min_tasks = static_cast<int64_t>(sms) * 24 * 2;
    while (tpg > 1 && n_units * cdiv(a.ntiles, tpg) < min_tasks) tpg = static_cast<int>(cdiv(tpg, 2));
    if (opts && opts->tiles_per_task > 0) tpg = std::min(opts->tiles_per_task, a.ntiles);
    a.tiles_per_group = tpg;
    a.tile_groups = static_cast<int>(cdiv(a.ntiles, tpg));
    // A hot segment has 32 * 2^g terms, whatever the average: its tasks, and
    // those of the long rows (2..2^g chunks) listed after the segments, get
    // their own, narrower tile groups (about 16 KB of sources each too).
    const int64_t seg_terms = int64_t(kChunk) << plan->g;
    int tpgs = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(a.ntiles, 16384 / (seg_terms * tile_bytes))));
    if (opts && opts->tiles_per_task > 0) tpgs = std::min(opts->tiles_per_task, a.ntiles);
    a.seg_tiles_per_group = tpgs;
    a.seg_tile_groups = static_cast<int>(cdiv(a.ntiles, tpgs));
    const int64_t max_segs_all = 2 * cdiv(plan->N, seg_terms) + 1;
    const int64_t max_tg = std::max(a.tile_groups, a.seg_tile_groups);
    a.n_tasks = dev_counts ? plan->M * max_tg + max_segs_all * a.seg_tile_groups  // an upper bound
                           : a.n_seg * a.seg_tile_groups +
                                 (plan->n_units - a.n_seg - (accumulate ? plan->n_empty : 0)) * a.tile_groups;

    // Binary-counter depth: enough levels for the longest unit's rounds.
    const int64_t G = int64_t(1) << plan->g;
    const int64_t max_chunks = dev_counts ? G : std::min(cdiv(plan->max_row_len, kChunk), G);
    const int64_t max_rounds = std::max<int64_t>(1, cdiv(max_chunks, int64_t(1) << a.S_log2));
    a.levels = log2_floor(max_rounds) + 1;

    // 0 = persistent grid sized by occupancy in the launcher
    const int grid = opts && opts->grid_ctas > 0 ? opts->grid_ctas : 0;
    cudaStream_t st = as_stream(stream);

    const int path = opts ? opts->gather_path : 0;
    if (path < 0 || path > 3 || (opts && (opts->tiles_per_task < 0 || opts->reserved[0])))
        return DET_ERR_ARG;
    // Wide rows with at most 32 terms per destination (the MoE combine): TMA-staged kernel.
    int tile_elems = 0, tile_stride = 0, bulk_tiles = 0;
    const bool bulk_ok = vec && !dev_counts && !accumulate && plan->max_row_len <= 32 && H * xsz >= 1024 &&
                         plan->n_units > 0 &&
                         bulk_plan_tiles(H, xsz, plan->max_row_len, &tile_elems, &tile_stride, &bulk_tiles);
    // with sources in several shards a producer warp also looks up each
    // term's shard: one alone fell behind (EP-invariance, 8 shards: 347
    // against 335 us for the register-staged kernel), two keep up (309
    // against 335 us), so auto takes it for shards where the kernel runs two
    const bool bulk_auto =
        bulk_ok && (P == 1 || plan->n_units * bulk_tiles >= static_cast<int64_t>(kBulkTwoProducerItems) * sms);
    // The ring kernel: the destinations of at most one chunk (for index_add_
    // the ones with terms: 1..32; for the scatter-reduce also the empty ones,
    // which it writes as +0.0) are TMA-staged into a byte ring of shared
    // memory, the longer ones stay on the register-staged kernel (and the
    // finish pass).  Its copies need 16-byte x tiles (and, for index_add_,
    // out tiles): out rows 16-byte aligned and H a multiple of the quantum.
    // With an unwaited plan it reads its unit count from the plan's counter
    // block.
    const int64_t n_ring = dev_counts ? -1
                                      : plan->n_units - plan->n_segments - plan->n_long -
                                            (accumulate ? plan->n_empty : 0);
    const int ring_quantum = accumulate ? std::max(16 / xsz, 16 / osz) : 16 / xsz;
    const bool ring_ok = vec && a.out_vec && H % ring_quantum == 0 && n_ring != 0;
    // Auto: the fixed-stage bulk kernel where it applies (a waited plan whose
    // destinations all have at most 32 terms), else the ring for one shard
    // (its producer's shard lookup is on its critical path) of rows of 1 KB
    // or more: always for index_add_ (embedding backward: 128 against 181 us
    // for the register-staged kernel alone), for the scatter-reduce when the
    // sources are 1 GiB or more, where the ring's start (a claim, the list,
    // the bounds and the perm entries before the first copy) is amortised
    // (EP-invariance step with an unwaited plan: 332 against 354 us; the MoE
    // combine's 268 MB: 70.5 against 68.7 us).
    const bool ring_auto = ring_ok && P == 1 && H * xsz >= 1024 &&
                           (accumulate || static_cast<double>(plan->N) * static_cast<double>(H * xsz) >= 1073741824.0);
    // Behind an unwaited plan whose row lengths may all be <= 32 (unknown on
    // the host): the fixed-stage kernel reads the longest from the counter
    // block and tiles on the device, and does nothing if it is longer; the
    // register-staged kernel after it works only in that case.  MoE step:
    // 66.6 us, against 68.6 us on the register-staged kernel and 71 us on the
    // ring; EP-invariance step: 329 against 353 and 333 us.
    int te32 = 0, st32 = 0, nt32 = 0;
    const bool bulk_dev_auto = !accumulate && dev_counts && vec && H * xsz >= 1024 && M > 0 &&
                               (P == 1 || M >= static_cast<int64_t>(kBulkTwoProducerItems) * sms) &&
                               bulk_plan_tiles(H, xsz, kChunk, &te32, &st32, &nt32);
    bool use_bulk = false, use_ring = false, use_bulk_dev = false;
    if (path == 3) {
        if (bulk_ok) use_bulk = true;
        else if (ring_ok) use_ring = true;
        else return DET_ERR_UNSUPPORTED;
    } else if (path == 0) {
        if (bulk_auto) use_bulk = true;
        else if (bulk_dev_auto) use_bulk_dev = true;
        else if (ring_auto) use_ring = true;
    }
    if (path == 2 && !vec) return DET_ERR_UNSUPPORTED;
    if (accumulate && path == 2) return DET_ERR_UNSUPPORTED;
    if (use_ring) {
        RingArgs b{};
        b.units = plan->row_units;  // the one-chunk units come first in row_units, then the empty ones
        b.n_units = n_ring;
        b.H = a.H;
        b.quantum = ring_quantum;
        // index_add_: 128 KB, which leaves room on the SM for the CTA of the
        // register-staged kernel beside it (the embedding backward's long
        // rows); the scatter-reduce: 192 KB, three of the MoE and EP shapes'
        // 64 KB items in flight (EP-invariance step: 332 against 353 us with
        // 128 KB)
        b.ring_bytes = (accumulate ? 128 : 192) * 1024;
        b.row_ptr = plan->row_ptr;
        b.perm = plan->perm;
        b.w = w;
        b.ldx_bytes = a.ldx_bytes;
        b.out = out;
        b.ldo = ldo;
        b.status = plan->counters;
        b.dev_counters = dev_counts ? plan->counters : nullptr;
        int64_t bgrid = opts && opts->grid_ctas > 0 ? opts->grid_ctas
                                                    : (dev_counts ? sms : std::min<int64_t>(n_ring, sms));
        bgrid = std::max<int64_t>(1, std::min<int64_t>(bgrid, 2147483647));
        // as for the fixed-stage kernel below: embedding backward step 161.7
        // against 166.4 us launched the ordinary way
        b.dependent = dev_counts && plan->late_release;
        s = launch_gather_ring(x_dtype, out_dtype, accumulate, b, tbl, static_cast<int>(bgrid), st);
        if (s) return s;
        // The register-staged kernel takes the units of more than one chunk,
        // beside the ring kernel: launched as its programmatic dependent, it
        // starts at once on the shared memory the ring leaves free (one CTA
        // per SM) and waits for the ring kernel only before it ends.  On the
        // embedding backward: 128 us, against 150 us with the two kernels one
        // after the other and 181 us with the register-staged kernel alone.
        a.beside_ring = 1;
        // With only the long units, at one CTA per SM, a warp folding a hot
        // segment of 256 terms over 512-byte tiles waits for 32 dependent
        // rounds of loads, and the warps that drew two such tasks ended last.
        // Narrower tiles with two chunk slots per warp (2 chunks folded at
        // once over 256-byte tiles) halve each chain and double the tasks
        // (the split changes no bit).  Embedding backward: 126 us, against
        // 131 us with 512-byte tiles, 130 us with 128-byte and 161 us with
        // 64-byte ones.
        constexpr int kBesideTlog2 = 4;
        if (a.T_log2 > kBesideTlog2) {
            a.T_log2 = kBesideTlog2;
            a.S_log2 = 5 - a.T_log2;
            a.ntiles = static_cast<int>(cdiv(V, int64_t(1) << a.T_log2));
            const int64_t tb = (int64_t(1) << a.T_log2) * (vec ? 16 : xsz);
            int tps = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(a.ntiles, 16384 / (seg_terms * tb))));
            if (opts && opts->tiles_per_task > 0) tps = std::min(opts->tiles_per_task, a.ntiles);
            a.seg_tiles_per_group = tps;
            a.seg_tile_groups = static_cast<int>(cdiv(a.ntiles, tps));
            a.tiles_per_group = std::min(a.tiles_per_group, a.ntiles);
            a.tile_groups = static_cast<int>(cdiv(a.ntiles, a.tiles_per_group));
            a.levels = log2_floor(std::max<int64_t>(1, cdiv(max_chunks, int64_t(1) << a.S_log2))) + 1;
            if (dev_counts) a.n_tasks = plan->M * a.tile_groups + max_segs_all * a.seg_tile_groups;
        }
        if (!dev_counts) a.n_tasks = a.n_seg * a.seg_tile_groups;
    }
    // Where it applies (the row counts are on the host, every destination has
    // at most 32 terms, rows of 1 KB or more, one shard) the bulk kernel is the default:
    // with its producer reading source rows four items ahead it measured
    // 52.9 against 53.9 us (MoE combine) and 324 against 327 us
    // (EP-invariance).  Everything else takes the register-staged kernel.
    if (use_bulk || use_bulk_dev) {
        BulkArgs b{};
        b.units = plan->row_units;
        b.n_items = plan->n_units * bulk_tiles;
        b.ntiles = bulk_tiles;
        b.tile_elems = tile_elems;
        b.tile_stride = tile_stride;
        b.H = a.H;
        b.out_vec = a.out_vec;
        b.row_ptr = plan->row_ptr;
        b.perm = plan->perm;
        b.w = w;
        b.ldx_bytes = a.ldx_bytes;
        b.out = out;
        b.ldo = ldo;
        b.status = plan->counters;
        b.dev_counters = use_bulk_dev ? plan->counters : nullptr;
        int64_t bgrid = opts && opts->grid_ctas > 0 ? opts->grid_ctas
                                                    : (use_bulk_dev ? sms : std::min<int64_t>(b.n_items, sms));
        bgrid = std::max<int64_t>(1, std::min<int64_t>(bgrid, 2147483647));
        // Behind an unwaited plan whose kernel releases the kernel after it
        // only for its last phase (the owner plan, the two-pass cluster plan,
        // the route cluster kernel), as that kernel's programmatic
        // dependent: MoE step 62.6 against 64.5 us launched the ordinary
        // way, route plan + combine 62.4 against 64.5 us.
        s = launch_gather_bulk(x_dtype, out_dtype, b, tbl, static_cast<int>(bgrid), use_bulk_dev && plan->late_release,
                               st);
        if (s) return s;
        if (use_bulk_dev) {
            a.only_long = 1;  // the register-staged kernel below: only if some destination is longer
        } else {
            if (opts && opts->debug_checks) return debug_sync_status(plan, st);
            return DET_OK;
        }
    }
    if (a.n_tasks > 0 && vec && path == 2) {
        // 16-byte rows: asynchronous copies into a shared-memory ring
        s = launch_gather_async(x_dtype, out_dtype, a, tbl, grid, st);
        if (s) return s;
    } else if (a.n_tasks > 0) {
        if (x_dtype == DET_BF16 && out_dtype == DET_BF16) s = launch_gather_vec<uint16_t, __nv_bfloat16>(vec, a, tbl, grid, st);
        else if (x_dtype == DET_BF16) s = launch_gather_vec<uint16_t, float>(vec, a, tbl, grid, st);
        else if (out_dtype == DET_BF16) s = launch_gather_vec<float, __nv_bfloat16>(vec, a, tbl, grid, st);
        else s = launch_gather_vec<float, float>(vec, a, tbl, grid, st);
        if (s) return s;
    }
    // Hot destinations: a second pass.  With device-side counts it runs
    // whenever a hot destination is possible, on a grid-stride launch.
    const bool maybe_hot = dev_counts ? plan->N > (int64_t(kChunk) << plan->g) : plan->n_hot_rows > 0;
    if (maybe_hot) {
        const int64_t max_row = dev_counts ? plan->N : plan->max_row_len;
        // four adjacent columns per thread where the partial rows allow
        // 16-byte loads (a quarter of the threads, each with four times the
        // bytes in flight): sparse key scatter reduce 404.3 -> 401.4 us (two
        // columns: 401.5 us)
        int fv = DETR_FINISH_FV;
        while (fv > 1 && !(H % fv == 0 && a.ldpart % fv == 0 && aligned(a.part, 4 * fv))) fv /= 2;
        const long long items = (dev_counts ? (cdiv(plan->N, (int64_t(kChunk) << plan->g) + 1) + 1) * H
                                            : plan->n_hot_rows * H) / fv;
        // behind the fixed-stage kernel it has work only when some row is
        // longer than 32 terms (then it loops over its grid): a small grid
        // ends sooner when it has none
        const int64_t fcap = int64_t(sms) * (use_bulk_dev ? 2 : 16);
        const int64_t fgrid64 = dev_counts ? std::min<int64_t>(cdiv(items, kFinishThreads), fcap)
                                           : cdiv(items, kFinishThreads);
        const unsigned int fgrid = static_cast<unsigned int>(std::max<int64_t>(1, fgrid64));
        const int64_t max_segs = cdiv(cdiv(max_row, kChunk), G);
        const size_t fsmem = static_cast<size_t>(log2_floor(std::max<int64_t>(1, max_segs)) + 1) * kFinishThreads *
                             fv * sizeof(float);
        const int* dc = dev_counts ? plan->counters : nullptr;
        const int4* fin = plan->finish;
        const float* part = a.part;
        auto kern = out_dtype == DET_BF16
                        ? (fv == 4 ? finish_kernel<__nv_bfloat16, 4>
                                   : fv == 2 ? finish_kernel<__nv_bfloat16, 2> : finish_kernel<__nv_bfloat16, 1>)
                        : (fv == 4 ? finish_kernel<float, 4> : fv == 2 ? finish_kernel<float, 2> : finish_kernel<float, 1>);
        {
            const det_status a_ = allow_dynamic_smem(reinterpret_cast<const void*>(kern), fsmem);
            if (a_) return a_;
        }
        DETR_CUDA(launch_after_previous(kern, dim3(fgrid), dim3(kFinishThreads), fsmem, st, fin, items, a.H, part,
                                        a.ldpart, out, ldo, dc, a.accumulate));
        DETR_LAUNCHED();
    }
    if (opts && opts->debug_checks) return debug_sync_status(plan, st);
    return DET_OK;
}

extern "C" {

det_status det_scatter_reduce(det_plan plan, const void* const* x_shards, const int64_t* shard_rows, int32_t P,
                              det_dtype x_dtype, int64_t ldx, int64_t H, const float* w, void* out, int64_t ldo,
                              det_dtype out_dtype, void* workspace, size_t ws_bytes, const det_opts* opts,
                              void* stream)
{
    return scatter_reduce_impl(plan, x_shards, shard_rows, P, x_dtype, ldx, H, w, out, ldo, out_dtype, workspace,
                               ws_bytes, opts, stream, false);
}

det_status det_index_add(det_plan plan, const void* const* x_shards, const int64_t* shard_rows, int32_t P,
                         det_dtype x_dtype, int64_t ldx, int64_t H, const float* w, void* out, int64_t ldo,
                         det_dtype out_dtype, void* workspace, size_t ws_bytes, const det_opts* opts, void* stream)
{
    return scatter_reduce_impl(plan, x_shards, shard_rows, P, x_dtype, ldx, H, w, out, ldo, out_dtype, workspace,
                               ws_bytes, opts, stream, true);
}

}  // extern "C"
