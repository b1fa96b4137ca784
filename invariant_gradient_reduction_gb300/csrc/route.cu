// route.cu -- the sorted router top-k, and the MoE route plan: the dispatch
// layout and the combine plan made straight from top-k expert ids.
//
// The sorted router top-k is one of the named hot spots of the deterministic
// path ("Megatron-LM determinism developer reference", section 3.3).  The
// dispatch rows follow the stable (expert id, original token id) order of
// the MoE backward ("DeepSeek-V4 book, Ch 09: Batch invariance and
// determinism", section 3.2), and the combine adds every dispatch row back
// into its token (the index_add_ of the op catalog, Megatron-LM reference,
// section 3.1).  Everything here is selection and integer work, exact on any
// grid.
//
// Top-k: one warp per token.  Lane l holds the keys of experts l, l+32, ...:
// the score's IEEE totalOrder key as the high word and the complement of the
// expert id as the low word, so that the greatest pair is the greatest score
// with the lowest id.  Round r takes the warp maximum of the lanes' heads
// (two 32-bit redux.sync votes: the high word, then the low word among the
// lanes that hold that high word); the one lane that holds it drops it.
//
// Route plan.  Slot i = t*k + j is token t's j-th choice.  The dispatch rows
// are the slots sorted stably by expert, so the combine's terms of token t
// (its k dispatch rows in ascending order) are its slots in (expert, j)
// order, and every token has exactly k terms: row_ptr[t] = t*k and the work
// units follow in closed form.  The only cross-token quantity is the rank of
// a slot among the earlier slots of its expert.
//   One cluster kernel (E <= 256 experts, up to 16 CTAs x 8192 slots): each
//   CTA ranks its slice of whole tokens per expert (ballots per expert-id bit,
//   warps in order), publishes its expert counts in shared memory, reads
//   those of the other CTAs across the cluster (the earlier ones give its
//   offsets, all of them the expert offsets), stages its rows in expert order
//   and writes them out in runs; then each slot's rank inside its token gives
//   the combine list.
//   Otherwise: the destination-list plan over the expert ids (which is this
//   same stable sort by expert) followed by two kernels that turn it into the
//   dispatch arrays and the combine plan.
#include <cooperative_groups.h>

#include <algorithm>
#include <new>

#include "block_scan.cuh"
#include "common.cuh"
#include "plan_internal.cuh"

namespace cg = cooperative_groups;

namespace detr {

// ------------------------------------------------------------------------
// sorted router top-k
// ------------------------------------------------------------------------

constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkMaxE = 1024;
constexpr int kTopkMaxK = 32;

// IEEE 754 totalOrder of binary32 as an unsigned order of the bit pattern u:
// a clear sign bit is set, a set sign bit inverts the whole pattern.  The
// scores are read and ranked as integers throughout, never as floats, so no
// NaN pattern goes through a floating-point comparison.
__device__ __forceinline__ unsigned int total_order_key(unsigned int u)
{
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned int total_order_bits(unsigned int key)
{
    return (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
}

// Lane state of the top-k selection: the keys of its experts as (hi, lo) =
// (totalOrder key of the score, 2^32 - 1 - expert id); a larger pair is a
// greater score, or an equal score with a lower id.  Padding (no expert) is
// (0, 0), below every real pair, whose lo is at least 2^32 - 1024.
// Up to 8 keys a lane sorts them once (descending) and the round's winner
// shifts its list; with more it keeps them unsorted and the winner rescans.
template <int ITEMS>
struct TopkLane {
    unsigned int hi[ITEMS], lo[ITEMS];
    static constexpr bool kSorted = ITEMS <= 8;

    __device__ __forceinline__ static bool greater(unsigned int ah, unsigned int al, unsigned int bh, unsigned int bl)
    {
        return ah > bh || (ah == bh && al > bl);
    }

    __device__ __forceinline__ void prepare()
    {
        if constexpr (kSorted) {
#pragma unroll
            for (int pass = 0; pass < ITEMS; ++pass) {  // odd-even transposition sort
#pragma unroll
                for (int i = pass & 1; i + 1 < ITEMS; i += 2) {
                    if (greater(hi[i + 1], lo[i + 1], hi[i], lo[i])) {
                        const unsigned int th = hi[i], tl = lo[i];
                        hi[i] = hi[i + 1];
                        lo[i] = lo[i + 1];
                        hi[i + 1] = th;
                        lo[i + 1] = tl;
                    }
                }
            }
        } else {
            best_to_front();
        }
    }

    // Unsorted lists keep their greatest pair at index 0.
    __device__ __forceinline__ void best_to_front()
    {
#pragma unroll
        for (int i = 1; i < ITEMS; ++i) {
            if (greater(hi[i], lo[i], hi[0], lo[0])) {
                const unsigned int th = hi[i], tl = lo[i];
                hi[i] = hi[0];
                lo[i] = lo[0];
                hi[0] = th;
                lo[0] = tl;
            }
        }
    }

    // Drops the head (this lane won the round).
    __device__ __forceinline__ void pop()
    {
        if constexpr (kSorted) {
#pragma unroll
            for (int i = 0; i + 1 < ITEMS; ++i) {
                hi[i] = hi[i + 1];
                lo[i] = lo[i + 1];
            }
            hi[ITEMS - 1] = 0u;
            lo[ITEMS - 1] = 0u;
        } else {
            hi[0] = 0u;
            lo[0] = 0u;
            best_to_front();
        }
    }
};

template <int ITEMS>
__global__ void __launch_bounds__(kTopkThreads)
router_topk_kernel(const unsigned int* __restrict__ scores, long long T, int E, long long lds, int k,
                   int renormalize, int* __restrict__ ids, unsigned int* __restrict__ w)
{
    const int lane = threadIdx.x & 31;
    const long long nwarps = static_cast<long long>(gridDim.x) * kTopkWarps;
    for (long long t = static_cast<long long>(blockIdx.x) * kTopkWarps + (threadIdx.x >> 5); t < T; t += nwarps) {
        const unsigned int* s = scores + t * lds;
        TopkLane<ITEMS> L;
#pragma unroll
        for (int it = 0; it < ITEMS; ++it) {  // all loads first
            const int e = it * 32 + lane;
            L.hi[it] = e < E ? total_order_key(__ldg(s + e)) : 0u;
            L.lo[it] = e < E ? 0xFFFFFFFFu - static_cast<unsigned int>(e) : 0u;
        }
        L.prepare();
        int my_e = 0;
        unsigned int my_s = 0u;
        for (int r = 0; r < k; ++r) {
            const unsigned int h = __reduce_max_sync(0xffffffffu, L.hi[0]);
            const unsigned int l = __reduce_max_sync(0xffffffffu, L.hi[0] == h ? L.lo[0] : 0u);
            if (L.hi[0] == h && L.lo[0] == l) L.pop();  // one lane: the expert ids differ
            if (lane == r) {
                my_e = static_cast<int>(0xFFFFFFFFu - l);
                my_s = total_order_bits(h);
            }
        }
        if (renormalize) {  // sum left to right from the greatest, then one division each
            const float v = __uint_as_float(my_s);
            float sum = __shfl_sync(0xffffffffu, v, 0);
            for (int r = 1; r < k; ++r) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, v, r));
            my_s = __float_as_uint(__fdiv_rn(v, sum));
        }
        if (lane < k) {
            ids[t * k + lane] = my_e;
            if (w) w[t * k + lane] = my_s;
        }
    }
}

// ------------------------------------------------------------------------
// route plan: pieces shared by both methods
// ------------------------------------------------------------------------

// Work units of token t, whose list has k terms: the closed form of the
// destination-list plan's classes (a hot row's segments and finish task, a
// long row, or a short / empty row).
__device__ __forceinline__ void write_token_units(long long t, int k, int g, int4* seg_units, int4* row_units,
                                                  int4* finish)
{
    const int nch = (k + kChunk - 1) / kChunk;
    const int tt = static_cast<int>(t);
    if (nch > (1 << g)) {
        const int nseg = (nch + (1 << g) - 1) >> g;
        const int b = tt * nseg;
        finish[t] = make_int4(tt, b, nseg, 0);
        for (int s = 0; s < nseg; ++s) seg_units[b + s] = make_int4(tt, s, b + s, 0);
    } else if (nch > 1) {
        seg_units[t] = make_int4(tt, -1, 0, 0);
    } else {
        row_units[t] = make_int4(tt, -1, 0, 0);
    }
}

// The counter block of the combine plan: T rows of k terms each.
__device__ __forceinline__ void write_route_counters(long long T, int k, int g, int err, int* counters)
{
    const int nch = (k + kChunk - 1) / kChunk;
    const int t = static_cast<int>(T);
    int segs = 0, hot = 0, lng = 0, shrt = 0, empty = 0;
    if (nch > (1 << g)) {
        hot = t;
        segs = t * ((nch + (1 << g) - 1) >> g);
    } else if (nch > 1) {
        lng = t;
    } else if (nch == 1) {
        shrt = t;
    } else {
        empty = t;
    }
    for (int i = 0; i < kCtrCount; ++i) counters[i] = 0;
    counters[kCtrErrIndex] = err ? 1 : 0;
    counters[kCtrSegs] = segs;
    counters[kCtrNormal] = lng + shrt + empty;
    counters[kCtrHot] = hot;
    counters[kCtrMaxLen] = T > 0 ? k : 0;
    counters[kCtrLong] = lng;
    counters[kCtrBig] = segs + lng;
    counters[kCtrShort] = shrt;
    counters[kCtrEmpty] = empty;
}

// ------------------------------------------------------------------------
// route plan: one cluster kernel
// ------------------------------------------------------------------------

constexpr int kRouteWarps = kCluThreads / 32;
constexpr int kRouteMaxE = 256;         // an expert id fits one byte and one ranking digit
constexpr int kRouteMaxSlice = 8192;    // slots of one CTA
constexpr int kRouteTargetSlice = 2048;

struct RouteShared {
    int pos[kRouteMaxSlice];                  // dispatch row of each slot of the slice
    int stage_tok[kRouteMaxSlice];            // token of each staged row (expert-major)
    float stage_w[kRouteMaxSlice];            // its weight
    int whist[kRouteWarps * kRouteMaxE];      // per-warp expert counts, then warp offsets
    int tot[kRouteMaxE];                      // this CTA's slots per expert (read by the cluster)
    int cstart[kRouteMaxE];                   // first staged position of each expert
    int delta[kRouteMaxE];                    // staged position q of expert e is dispatch row q + delta[e]
    int ws[kRouteWarps + 1];                  // scan scratch
    int bad;                                  // an id outside [0, E) (read by the cluster)
    unsigned char ex[kRouteMaxSlice];         // expert of each slot
    unsigned char stage_e[kRouteMaxSlice];    // expert of each staged row
};

// CTA c owns tokens [c*Tc, (c+1)*Tc) and their slots; item it of lane l of
// warp w is slot w*32*ITEMS + it*32 + l of the slice.  kmagic = ceil(2^32 / k)
// turns the division of a slice position s < 2^13 by k into a multiply:
// (s * kmagic) >> 32 exceeds s / k by less than s / 2^32 < 1/k, so its floor
// is exact.
__device__ __forceinline__ int div_k(int s, unsigned long long kmagic)
{
    return static_cast<int>((static_cast<unsigned long long>(s) * kmagic) >> 32);
}

template <int ITEMS>
__global__ void __launch_bounds__(kCluThreads, 1)
route_cluster_kernel(const int* __restrict__ ids, const float* __restrict__ tw, long long T, int k,
                     unsigned long long kmagic, int E, int Tc, int g, int* __restrict__ expert_offsets,
                     int* __restrict__ row_token, float* __restrict__ row_w,
                     int* __restrict__ slot_row, int* __restrict__ row_ptr, int* __restrict__ perm,
                     int4* __restrict__ seg_units, int4* __restrict__ row_units, int4* __restrict__ finish,
                     int* __restrict__ counters)
{
    cg::cluster_group cl = cg::this_cluster();
    extern __shared__ __align__(16) unsigned char route_smem[];
    RouteShared& S = *reinterpret_cast<RouteShared*>(route_smem);
    const int C = static_cast<int>(cl.num_blocks());
    const int c = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long N = T * k;
    const long long t0 = min(T, static_cast<long long>(c) * Tc);
    const long long t1 = min(T, t0 + Tc);
    const long long s0 = t0 * k;
    const int cnt = static_cast<int>((t1 - t0) * k);  // <= ITEMS * kCluThreads
    const int wbase = warp * 32 * ITEMS;
    unsigned int lt;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));

    // 1. the slice, and each slot's rank among the earlier slots of its
    //    expert in its warp
    int d[ITEMS], rank[ITEMS];
    float wv[ITEMS];
    bool bad = false;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {  // all loads first
        const int s = wbase + it * 32 + lane;
        d[it] = 0;
        rank[it] = 0;
        wv[it] = 0.0f;
        if (s < cnt) {
            const int e = __ldg(ids + s0 + s);
            if (e < 0 || e >= E) bad = true;
            else d[it] = e;
            if (tw) wv[it] = __ldg(tw + s0 + s);
        }
    }
    for (int i = tid; i < kRouteWarps * kRouteMaxE; i += kCluThreads) S.whist[i] = 0;
    __syncthreads();
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int nl = cnt - (wbase + it * 32);
        const unsigned int live = nl >= 32 ? 0xffffffffu : (nl <= 0 ? 0u : (1u << nl) - 1u);
        if (live == 0u) continue;  // uniform over the warp
        const bool valid = (live >> lane) & 1u;
        const unsigned int peers = digit_peers(d[it], live);
        int* h = &S.whist[warp * kRouteMaxE + d[it]];
        const int old = *h;
        rank[it] = old + __popc(peers & lt);
        __syncwarp();
        if (valid && (peers & lt) == 0u) *h = old + __popc(peers);
        __syncwarp();
        if (valid) S.ex[wbase + it * 32 + lane] = static_cast<unsigned char>(d[it]);
    }
    const int cta_bad = __syncthreads_or(bad);

    // 2. per expert: warp offsets in warp order, this CTA's count, and the
    //    first staged position
    int tot = 0;
    if (tid < kRouteMaxE) {
        for (int w = 0; w < kRouteWarps; ++w) {
            const int v = S.whist[w * kRouteMaxE + tid];
            S.whist[w * kRouteMaxE + tid] = tot;
            tot += v;
        }
    }
    int unused;
    const int cst = block_excl_scan<kCluThreads>(tot, S.ws, &unused);
    if (tid < kRouteMaxE) {
        S.tot[tid] = tot;
        S.cstart[tid] = cst;
    }
    if (tid == 0) S.bad = cta_bad;
    cl.sync();  // every CTA's counts are published

    // 3. the cluster's counts: this expert's slots in earlier CTAs, and in all
    int before = 0, grand = 0, peer_bad = 0;
    if (tid < E) {
        int v[kCluMaxCtas];
#pragma unroll
        for (int r = 0; r < kCluMaxCtas; ++r)  // all remote loads in flight at once
            v[r] = r < C ? *cl.map_shared_rank(&S.tot[tid], r) : 0;
#pragma unroll
        for (int r = 0; r < kCluMaxCtas; ++r) {
            grand += v[r];
            before += r < c ? v[r] : 0;
        }
    }
    if (tid < C) peer_bad = *cl.map_shared_rank(&S.bad, tid);
    const int any_bad = __syncthreads_or(peer_bad);  // consumes every remote value
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");  // done reading the others
    if (any_bad) {
        if (c == 0 && tid == 0) write_route_counters(T, k, g, 1, counters);
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        return;  // nothing else is written
    }
    int total;
    const int off = block_excl_scan<kCluThreads>(tid < E ? grand : 0, S.ws, &total);
    if (tid < kRouteMaxE) S.delta[tid] = off + before - S.cstart[tid];
    if (c == 0 && tid <= E) expert_offsets[tid] = off;  // off at tid = E is the total, N
    __syncthreads();

    // 4. each slot's staged position and dispatch row
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int s = wbase + it * 32 + lane;
        if (s < cnt) {
            const int e = d[it];
            const int q = S.cstart[e] + S.whist[warp * kRouteMaxE + e] + rank[it];
            const int p = q + S.delta[e];
            S.pos[s] = p;
            S.stage_tok[q] = static_cast<int>(t0) + div_k(s, kmagic);
            S.stage_w[q] = wv[it];
            S.stage_e[q] = static_cast<unsigned char>(e);
            if (slot_row) slot_row[s0 + s] = p;
        }
    }
    __syncthreads();

    // The reduce may be launched now, for the last two phases (it waits for
    // this grid to finish): released at the kernel's start, the fixed-stage
    // gather behind an unwaited route plan would hold the other SMs through
    // the whole plan; launched the ordinary way it started later (route plan
    // + combine 64.5 us, against 62.4 us released here).
    pdl_launch_dependents();
    // 5. the dispatch rows go out in runs of consecutive rows per expert
    for (int q = tid; q < cnt; q += kCluThreads) {
        const int p = q + S.delta[S.stage_e[q]];
        row_token[p] = S.stage_tok[q];
        if (row_w) row_w[p] = S.stage_w[q];
    }

    // 6. the combine plan: token t's terms are its dispatch rows in ascending
    //    order, i.e. its slots in (expert, j) order
    for (int s = tid; s < cnt; s += kCluThreads) {
        const int first = div_k(s, kmagic) * k;
        const int j = s - first;
        const int e = S.ex[s];
        int r = 0;
        for (int j2 = 0; j2 < k; ++j2) {
            const int e2 = S.ex[first + j2];
            r += (e2 < e) || (e2 == e && j2 < j);
        }
        perm[s0 + first + r] = S.pos[s];
    }
    for (long long t = t0 + tid; t < t1; t += kCluThreads) {
        row_ptr[t] = static_cast<int>(t * k);
        write_token_units(t, k, g, seg_units, row_units, finish);
    }
    if (c == C - 1 && tid == 0) row_ptr[T] = static_cast<int>(N);
    if (c == 0 && tid == 0) write_route_counters(T, k, g, 0, counters);
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Route-kernel geometry for (T, k, E): CTAs, tokens per CTA, slots per thread
// (1, 2, 4 or 8); false where the cluster kernel does not apply.
static bool route_cluster_shape(int64_t T, int k, int E, int* C, int* Tc, int* items)
{
    const int64_t N = T * k;
    if (T <= 0 || k <= 0 || E > kRouteMaxE || N > int64_t(kCluMaxCtas) * kRouteMaxSlice) return false;
    const int64_t c = std::min<int64_t>(kCluMaxCtas, std::max<int64_t>(1, cdiv(N, kRouteTargetSlice)));
    const int64_t tc = cdiv(T, c);
    const int64_t slice = tc * k;
    if (slice > kRouteMaxSlice) return false;
    *C = static_cast<int>(cdiv(T, tc));
    *Tc = static_cast<int>(tc);
    *items = slice <= kCluThreads ? 1 : slice <= 2 * kCluThreads ? 2 : slice <= 4 * kCluThreads ? 4 : 8;
    return true;
}

// ------------------------------------------------------------------------
// route plan: from the destination-list plan over the expert ids
// ------------------------------------------------------------------------

constexpr int kRouteThreads = 256;

// Dispatch row p holds slot eperm[p] (the expert plan's list order); the
// expert plan's row_ptr is the expert offsets.  Without slots (N = 0) the
// expert plan is absent and only the offsets (all 0) are written.
__global__ void __launch_bounds__(kRouteThreads)
route_rows_kernel(const int* __restrict__ eperm, const int* __restrict__ erow_ptr, const int* __restrict__ ecounters,
                  long long N, int k, int E, const float* __restrict__ tw, int* __restrict__ expert_offsets,
                  int* __restrict__ row_token, float* __restrict__ row_w, int* __restrict__ slot_row)
{
    if (ecounters && ecounters[kCtrErrIndex]) return;
    const long long x = static_cast<long long>(blockIdx.x) * kRouteThreads + threadIdx.x;
    if (x < N) {
        const int slot = eperm[x];
        row_token[x] = slot / k;
        if (row_w) row_w[x] = tw[slot];
        slot_row[slot] = static_cast<int>(x);
    }
    if (x <= E) expert_offsets[x] = erow_ptr ? erow_ptr[x] : 0;  // no slots: every expert starts at 0
}

// The combine plan: slot x of token t lands at rank r of t's list, r its
// place in (expert, j) order; row_ptr, the units and the counter block.
__global__ void __launch_bounds__(kRouteThreads)
route_combine_kernel(const int* __restrict__ ids, long long T, int k, int g, const int* __restrict__ slot_row,
                     const int* __restrict__ ecounters, int* __restrict__ row_ptr, int* __restrict__ perm,
                     int4* __restrict__ seg_units, int4* __restrict__ row_units, int4* __restrict__ finish,
                     int* __restrict__ counters)
{
    pdl_launch_dependents();  // the reduce may be launched now; it waits for this grid to finish
    const int err = ecounters ? ecounters[kCtrErrIndex] : 0;
    const long long x = static_cast<long long>(blockIdx.x) * kRouteThreads + threadIdx.x;
    if (x == 0) write_route_counters(T, k, g, err, counters);
    if (err) return;
    const long long N = T * k;
    if (x < N) {
        const long long first = x - x % k;
        const int j = static_cast<int>(x - first);
        const int e = ids[x];
        int r = 0;
        for (int j2 = 0; j2 < k; ++j2) {
            const int e2 = ids[first + j2];
            r += (e2 < e) || (e2 == e && j2 < j);
        }
        perm[first + r] = slot_row[x];
    }
    if (x < T) {
        row_ptr[x] = static_cast<int>(x * k);
        write_token_units(x, k, g, seg_units, row_units, finish);
    }
    if (x == T) row_ptr[T] = static_cast<int>(N);
}

// ------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------

struct RouteLayout {
    size_t counters, row_ptr, perm, seg_units, row_units, finish, slot_row, eplan, total;
    size_t eplan_bytes;
};

static int64_t route_seg_units(int64_t T, int k, int g)
{
    const int64_t nch = cdiv(k, kChunk);
    if (nch > (int64_t(1) << g)) return T * ((nch + (int64_t(1) << g) - 1) >> g);
    return nch > 1 ? T : 0;
}

static det_status route_layout(int64_t T, int k, int E, int g, const det_opts* opts, RouteLayout* L)
{
    *L = RouteLayout{};
    const int64_t N = T * k;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + (bytes ? bytes : 1), 256);
        return at;
    };
    L->counters = take(kCtrCount * sizeof(int));
    L->row_ptr = take(static_cast<size_t>(T + 1) * sizeof(int));
    L->perm = take(static_cast<size_t>(N) * sizeof(int));
    L->seg_units = take(static_cast<size_t>(route_seg_units(T, k, g)) * sizeof(int4));
    L->row_units = take(static_cast<size_t>(T + 1) * sizeof(int4));
    L->finish = take(static_cast<size_t>(T) * sizeof(int4));
    L->slot_row = take(static_cast<size_t>(N) * sizeof(int));
    det_opts eo = opts ? *opts : det_opts{0, -1, 0, 0, 0, 0, 0, {0}};
    eo.plan_path = 1;
    eo.async_plan = 1;
    const det_status s = det_plan_workspace_size(N, E, 0, &eo, &L->eplan_bytes);
    if (s) return s;
    L->eplan = take(L->eplan_bytes);
    L->total = off;
    return DET_OK;
}

static det_status route_seg_log2(const det_opts* o, int* g)
{
    *g = kDefaultSegLog2;
    if (o && o->seg_chunks_log2 >= 0) {
        if (o->seg_chunks_log2 < kMinSegLog2 || o->seg_chunks_log2 > kMaxSegLog2) return DET_ERR_ARG;
        *g = o->seg_chunks_log2;
    }
    return DET_OK;
}

static det_status route_args(int64_t T, int32_t k, int32_t E)
{
    if (T < 0 || k < 0 || E < 1) return DET_ERR_ARG;
    if (T > kMaxRows || E > kMaxRows || (k > 0 && T > kMaxRows / k)) return DET_ERR_UNSUPPORTED;
    return DET_OK;
}

}  // namespace detr

using namespace detr;

extern "C" {

det_status det_router_topk(const float* scores, int64_t T, int32_t E, int64_t lds, int32_t k, int32_t renormalize,
                           int32_t* topk_ids, float* topk_w, void* stream)
{
    if (T < 0 || E < 1 || k < 1 || k > E || lds < E) return DET_ERR_ARG;
    if (E > kTopkMaxE || k > kTopkMaxK || T > kMaxRows || T * k > kMaxRows || lds > (int64_t(1) << 40))
        return DET_ERR_UNSUPPORTED;
    if (T == 0) return DET_OK;
    if (!scores || !topk_ids || (renormalize && !topk_w)) return DET_ERR_ARG;
    if (!aligned(scores, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4)) return DET_ERR_ARG;
    const size_t sbytes = static_cast<size_t>((T - 1) * lds + E) * 4;
    const size_t obytes = static_cast<size_t>(T * k) * 4;
    if (overlaps(scores, sbytes, topk_ids, obytes) || overlaps(scores, sbytes, topk_w, topk_w ? obytes : 0) ||
        overlaps(topk_ids, obytes, topk_w, topk_w ? obytes : 0))
        return DET_ERR_ARG;
    int sms = 0;
    det_status s = current_sm_count(&sms);
    if (s) return s;
    const int64_t want = cdiv(T, kTopkWarps);
    const unsigned int grid = static_cast<unsigned int>(std::min<int64_t>(want, int64_t(sms) * 8));
    cudaStream_t st = as_stream(stream);
    const long long t = T, ld = lds;
    const unsigned int* sb = reinterpret_cast<const unsigned int*>(scores);
    unsigned int* wb = reinterpret_cast<unsigned int*>(topk_w);
    const int items = E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : E <= 256 ? 8 : E <= 512 ? 16 : 32;
    switch (items) {
        case 1: router_topk_kernel<1><<<grid, kTopkThreads, 0, st>>>(sb, t, E, ld, k, renormalize, topk_ids, wb); break;
        case 2: router_topk_kernel<2><<<grid, kTopkThreads, 0, st>>>(sb, t, E, ld, k, renormalize, topk_ids, wb); break;
        case 4: router_topk_kernel<4><<<grid, kTopkThreads, 0, st>>>(sb, t, E, ld, k, renormalize, topk_ids, wb); break;
        case 8: router_topk_kernel<8><<<grid, kTopkThreads, 0, st>>>(sb, t, E, ld, k, renormalize, topk_ids, wb); break;
        case 16: router_topk_kernel<16><<<grid, kTopkThreads, 0, st>>>(sb, t, E, ld, k, renormalize, topk_ids, wb); break;
        default: router_topk_kernel<32><<<grid, kTopkThreads, 0, st>>>(sb, t, E, ld, k, renormalize, topk_ids, wb); break;
    }
    DETR_LAUNCHED();
    return DET_OK;
}

det_status det_moe_route_workspace_size(int64_t T, int32_t k, int32_t E, const det_opts* opts, size_t* bytes)
{
    if (!bytes) return DET_ERR_ARG;
    det_status s = route_args(T, k, E);
    if (s) return s;
    int g;
    s = route_seg_log2(opts, &g);
    if (s) return s;
    RouteLayout L;
    s = route_layout(T, k, E, g, opts, &L);
    if (s) return s;
    *bytes = L.total;
    return DET_OK;
}

det_status det_moe_route_plan(const int32_t* topk_ids, const float* topk_w, int64_t T, int32_t k, int32_t E,
                              int32_t* expert_offsets, int32_t* row_token, float* row_w, int32_t* slot_row,
                              void* workspace, size_t ws_bytes, const det_opts* opts, void* stream,
                              det_plan* out_plan)
{
    if (!out_plan) return DET_ERR_ARG;
    *out_plan = nullptr;
    det_status s = route_args(T, k, E);
    if (s) return s;
    int g;
    s = route_seg_log2(opts, &g);
    if (s) return s;
    if (opts && (opts->plan_path < 0 || opts->plan_path > 2 || opts->reserved[0])) return DET_ERR_ARG;
    const int64_t N = T * k;
    if (!expert_offsets || (N > 0 && (!topk_ids || !row_token)) || (row_w && !topk_w)) return DET_ERR_ARG;
    if (!aligned(topk_ids, 4) || !aligned(topk_w, 4) || !aligned(expert_offsets, 4) || !aligned(row_token, 4) ||
        !aligned(row_w, 4) || !aligned(slot_row, 4))
        return DET_ERR_ARG;
    RouteLayout L;
    s = route_layout(T, k, E, g, opts, &L);
    if (s) return s;
    if (!workspace || !aligned(workspace, 256) || ws_bytes < L.total) return DET_ERR_WORKSPACE;
    {  // no output may overlap an input, another output or the workspace
        const size_t nb = static_cast<size_t>(N) * 4;
        const void* p[7] = {topk_ids, topk_w, expert_offsets, row_token, row_w, slot_row, workspace};
        const size_t b[7] = {topk_ids ? nb : 0, topk_w ? nb : 0, static_cast<size_t>(E + 1) * 4,
                             row_token ? nb : 0, row_w ? nb : 0, slot_row ? nb : 0, ws_bytes};
        for (int i = 2; i < 7; ++i)
            for (int j = 0; j < i; ++j)
                if (overlaps(p[i], b[i], p[j], b[j])) return DET_ERR_ARG;
    }

    cudaStream_t st = as_stream(stream);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    int* counters = reinterpret_cast<int*>(ws + L.counters);
    int* row_ptr = reinterpret_cast<int*>(ws + L.row_ptr);
    int* perm = reinterpret_cast<int*>(ws + L.perm);
    int4* seg_units = reinterpret_cast<int4*>(ws + L.seg_units);
    int4* row_units = reinterpret_cast<int4*>(ws + L.row_units);
    int4* finish = reinterpret_cast<int4*>(ws + L.finish);
    const int plan_path = opts ? opts->plan_path : 0;

    bool done = false;
    int C = 0, Tc = 0, items = 0;
    if (plan_path != 1 && route_cluster_shape(T, k, E, &C, &Tc, &items)) {
        long long t = T;
        unsigned long long kmagic = ((1ull << 32) + static_cast<unsigned long long>(k) - 1) / static_cast<unsigned long long>(k);
        const int* ids_a = topk_ids;
        const float* tw_a = topk_w;
        int k_a = k, E_a = E;
        void* args[] = {&ids_a, &tw_a, &t, &k_a, &kmagic, &E_a, &Tc, &g, &expert_offsets, &row_token, &row_w, &slot_row,
                        &row_ptr, &perm, &seg_units, &row_units, &finish, &counters};
        const void* kern = items == 1   ? reinterpret_cast<const void*>(route_cluster_kernel<1>)
                           : items == 2 ? reinterpret_cast<const void*>(route_cluster_kernel<2>)
                           : items == 4 ? reinterpret_cast<const void*>(route_cluster_kernel<4>)
                                        : reinterpret_cast<const void*>(route_cluster_kernel<8>);
        const int variant = kCluVariantRoute + (items == 1 ? 0 : items == 2 ? 1 : items == 4 ? 2 : 3);
        s = launch_on_cluster(variant, kern, C, sizeof(RouteShared), st, args, &done);
        if (s) return s;
    }
    if (plan_path == 2 && !done) return DET_ERR_UNSUPPORTED;
    if (!done) {
        int* srow = slot_row ? slot_row : reinterpret_cast<int*>(ws + L.slot_row);
        const int* ecounters = nullptr;
        const int* eperm = nullptr;
        const int* erow_ptr = nullptr;
        if (N > 0) {
            // the stable sort of the slots by expert is the destination-list
            // plan over the expert ids
            det_opts eo = opts ? *opts : det_opts{0, -1, 0, 0, 0, 0, 0, {0}};
            eo.plan_path = plan_path == 1 ? 1 : 0;
            eo.async_plan = 1;
            det_plan ep = nullptr;
            s = det_reduce_plan(topk_ids, nullptr, N, E, ws + L.eplan, L.eplan_bytes, &eo, stream, &ep);
            if (s) return s;
            eperm = ep->perm;
            erow_ptr = ep->row_ptr;
            ecounters = ep->counters;
            det_plan_destroy(ep);
        }
        const unsigned int rgrid = static_cast<unsigned int>(cdiv(std::max<int64_t>(N, int64_t(E) + 1), kRouteThreads));
        route_rows_kernel<<<rgrid, kRouteThreads, 0, st>>>(eperm, erow_ptr, ecounters, N, k, E, topk_w,
                                                           expert_offsets, row_token, row_w, srow);
        DETR_LAUNCHED();
        const unsigned int cgrid = static_cast<unsigned int>(cdiv(std::max<int64_t>(N, T + 1), kRouteThreads));
        route_combine_kernel<<<cgrid, kRouteThreads, 0, st>>>(topk_ids, T, k, g, srow, ecounters, row_ptr, perm,
                                                              seg_units, row_units, finish, counters);
        DETR_LAUNCHED();
    }

    const bool async = opts && opts->async_plan;
    int h[kCtrCount] = {};
    if (!async) {
        DETR_CUDA(cudaMemcpyAsync(h, counters, sizeof(h), cudaMemcpyDeviceToHost, st));
        DETR_CUDA(cudaStreamSynchronize(st));
        if (h[kCtrErrIndex]) return DET_ERR_INDEX_RANGE;
    }
    det_plan_s* p = new (std::nothrow) det_plan_s();
    if (!p) return DET_ERR_ARG;
    p->N = N;
    p->M = T;
    p->g = g;
    p->ws = ws;
    p->ws_bytes = ws_bytes;
    p->counters = counters;
    p->row_ptr = row_ptr;
    p->perm = perm;
    p->seg_units = seg_units;
    p->row_units = row_units;
    p->finish = finish;
    p->late_release = done;  // the cluster kernel releases the reduce only for its last phases
    if (async) {
        p->counts_on_host = false;
        p->n_segments = p->n_units = p->n_hot_rows = p->max_row_len = p->n_long = p->n_empty = -1;
    } else {
        p->n_segments = h[kCtrSegs];
        p->n_units = static_cast<int64_t>(h[kCtrSegs]) + h[kCtrNormal];
        p->n_hot_rows = h[kCtrHot];
        p->max_row_len = h[kCtrMaxLen];
        p->n_long = h[kCtrLong];
        p->n_empty = h[kCtrEmpty];
    }
    *out_plan = p;
    return DET_OK;
}

}  // extern "C"
