// plan_cluster.cu -- the whole plan in one kernel on one thread-block cluster,
// for small problems ordered by source position (no src_id).
//
// The lists are the same as the multi-kernel plan's: the terms of destination
// m are the sources with idx[i] = m in ascending i ("DeepSeek-V4 book, Ch 09:
// Batch invariance and determinism", section 3.2), and the work list splits
// destinations with more than 2^g chunks into aligned segments.  All of it is
// integer work, so both methods give the same arrays.
//
// A small plan built from separate kernels is latency-bound: every kernel pays
// its launch and a few dependent round trips to L2.  Here one cluster of C CTAs
// (one per SM, C <= 16) keeps the sources in distributed shared memory, each
// CTA a slice of E consecutive positions, and runs every step between cluster
// barriers:
//   1. each CTA loads its slice of idx and checks the range;
//   2. per 8-bit digit of the destination, a stable LSD radix pass: the CTA
//      ranks its slice (peers of a digit from ballots, in element order, warps
//      in order), publishes its 256 digit counts and reads those of every CTA
//      of the cluster (the earlier CTAs give its offsets, all of them the digit
//      starts), stages its pairs in (digit, position) order in its own shared
//      memory and copies them out in runs, so that a warp's stores go to
//      consecutive words of one owner;
//   3. row_ptr: the first position of every key present is stored into the
//      shared memory of the CTA that owns the key's row range; each CTA then
//      takes suffix minima over its rows (an empty row starts where the next
//      present one does), bounded by the first position past its range, which
//      is the sum over the slices of their keys below the range end;
//   4. the work list: rows classified as whole-row units or hot rows, offsets
//      by scans inside the CTA and across the cluster; then perm, row_ptr, the
//      unit arrays and (CTA 0) the counter block go out to global memory.
// Cluster barriers are hardware barriers: no thread waits on a flag.
#include <cooperative_groups.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "block_scan.cuh"
#include "common.cuh"
#include "plan_internal.cuh"

namespace cg = cooperative_groups;

namespace detr {

constexpr int kCluWarps = kCluThreads / 32;
constexpr int kCluItems = 8;
constexpr int kCluRadix = 256;
constexpr int kCluMaxRowsPerCta = kCluRowsPerThread * kCluThreads;
static_assert(kCluThreads * kCluItems == kCluMaxSlice, "a slice is at most kCluItems per thread");
static_assert(kCluMaxCtas < 32, "the cluster-level scan runs on one warp");
static_assert(kCluThreads == 4 * kCluRadix && kCluMaxCtas % 4 == 0, "four readers per digit");

__device__ __forceinline__ long long min_ll(long long a, long long b) { return a < b ? a : b; }

struct CluShared {
    uint2 kv[kCluMaxSlice];          // this CTA's slice of the current order: {key, source position}
    uint2 stage[kCluMaxSlice];       // the same pairs in (digit, position) order, before they go out
    int rstart[kCluMaxRowsPerCta];   // first sorted position of each destination of this CTA, or INT_MAX
    int whist[kCluWarps * kCluRadix];  // per warp digit counts, then warp offsets
    int chist[kCluRadix];            // this CTA's digit counts (read by the cluster)
    int tstart[kCluRadix];           // first staged position of each digit
    int gbase[kCluRadix];            // first global position of this CTA's keys of each digit
    int cnt_lt[kCluMaxCtas];         // keys of this slice below the end of CTA r's rows (read by the cluster)
    int ws[5 * (kCluWarps + 1)];     // scan scratch
    int tot[6];                      // seg units, long, short rows, finish tasks, empty rows, longest row (read by the cluster)
    int base[5];                     // this CTA's offsets into the unit arrays
    int grand[6];                    // cluster totals
    int bad;                         // this CTA saw an index outside [0, M) (read by the cluster)
    int any_bad;
    int next_start;                  // first sorted position past this CTA's rows
};

// Minimum of v over the threads with a larger index (INT_MAX for the last
// thread), over 1024 threads.  Ends synchronised.
__device__ __forceinline__ int block_suffix_min_excl(int v, int* ws)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;  // min over lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl = min(incl, t);
    }
    if (lane == 0) ws[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int si = ws[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_down_sync(0xffffffffu, si, o);
            if (lane + o < 32) si = min(si, t);
        }
        ws[lane] = si;  // min over warps >= lane
    }
    __syncthreads();
    int next = __shfl_down_sync(0xffffffffu, incl, 1);
    if (lane == 31) next = INT_MAX;
    const int after = warp + 1 < kCluWarps ? ws[warp + 1] : INT_MAX;
    __syncthreads();
    return min(next, after);
}

// Cluster barrier whose arrival does not wait for this thread's earlier
// memory operations: for a CTA that only has to stay resident while other
// CTAs read its shared memory.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ int slice_len(long long N, int E, int r)
{
    const long long rem = N - static_cast<long long>(r) * E;
    return rem <= 0 ? 0 : (rem < E ? static_cast<int>(rem) : E);
}

__global__ void __launch_bounds__(kCluThreads, 1)
plan_cluster_kernel(const int* __restrict__ idx, long long N, long long M, int E, int np32, int g,
                    int* __restrict__ row_ptr, int* __restrict__ perm, int4* __restrict__ seg_units,
                    int4* __restrict__ row_units, int4* __restrict__ finish, int* __restrict__ counters)
{
    cg::cluster_group cl = cg::this_cluster();
    extern __shared__ __align__(16) unsigned char clu_smem[];
    CluShared& S = *reinterpret_cast<CluShared*>(clu_smem);
    const int C = static_cast<int>(cl.num_blocks());
    const int c = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cnt = slice_len(N, E, c);
    const long long c0 = static_cast<long long>(c) * E;
    // warp w owns the elements [w*ipw, (w+1)*ipw) of the slice, nk per lane
    const int ipw = (((cnt + kCluWarps - 1) / kCluWarps) + 31) & ~31;
    const int nk = ipw >> 5;  // <= kCluItems
    // rows [r_lo, r_hi) belong to this CTA
    const long long R = (M + C - 1) / C;
    const long long r_lo = min_ll(M, static_cast<long long>(c) * R);
    const long long r_hi = min_ll(M, r_lo + R);
    unsigned int lt;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
    if (tid == 0) S.tot[5] = 0;
    for (int i = tid; i < r_hi - r_lo; i += kCluThreads) S.rstart[i] = INT_MAX;

    // 1. the slice, in position order, into kv; in the passes item k of lane
    //    l of warp w is element w*ipw + k*32 + l
    bool bad = false;
    for (int i = tid; i < cnt; i += kCluThreads) {
        const unsigned int k = static_cast<unsigned int>(__ldg(idx + c0 + i));
        bad |= static_cast<long long>(k) >= M;
        S.kv[i] = make_uint2(k, static_cast<unsigned int>(c0 + i));
    }
    const int cta_bad = __syncthreads_or(bad);
    if (tid == 0) S.bad = cta_bad;

    // 2. stable radix passes over the destination digits.  The slice stays
    //    intact in kv until this CTA arrives at the pass's first cluster
    //    barrier (other CTAs write into it only after that barrier).
    unsigned int key[kCluItems];
    int rank[kCluItems];
    for (int pass = 0; pass < np32; ++pass) {
        const int shift = 8 * pass;
#pragma unroll
        for (int k = 0; k < kCluItems; ++k) {
            const int p = warp * ipw + k * 32 + lane;
            key[k] = k < nk && p < cnt ? S.kv[p].x : 0u;
        }
        for (int i = tid; i < kCluWarps * kCluRadix; i += kCluThreads) S.whist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kCluItems; ++k) {
            if (k >= nk) break;  // uniform over the block
            const int nlive = cnt - (warp * ipw + k * 32);  // lanes below this hold elements
            const unsigned int live = nlive >= 32 ? 0xffffffffu : (nlive <= 0 ? 0u : (1u << nlive) - 1u);
            const bool valid = (live >> lane) & 1u;
            const int d = static_cast<int>((key[k] >> shift) & 255u);
            const unsigned int peers = digit_peers(d, live);
            // every lane reads its digit's running count (no branch, no
            // shuffle); the lowest lane of each digit group writes it back
            const int old = S.whist[warp * kCluRadix + d];
            rank[k] = old + __popc(peers & lt);
            __syncwarp();
            if (valid && (peers & lt) == 0u) S.whist[warp * kCluRadix + d] = old + __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        int mine = 0;
        if (tid < kCluRadix) {
            for (int w = 0; w < kCluWarps; ++w) {
                const int x = S.whist[w * kCluRadix + tid];
                S.whist[w * kCluRadix + tid] = mine;
                mine += x;
            }
            S.chist[tid] = mine;
        }
        int sum_unused;
        const int lstart = block_excl_scan<kCluThreads>(tid < kCluRadix ? mine : 0, S.ws, &sum_unused);
        if (tid < kCluRadix) S.tstart[tid] = lstart;
        __syncthreads();
        // stage the slice in (digit, position) order; needs only this CTA's counts
#pragma unroll
        for (int k = 0; k < kCluItems; ++k) {
            const int p = warp * ipw + k * 32 + lane;
            if (k < nk && p < cnt) {
                const int d = static_cast<int>((key[k] >> shift) & 255u);
                const int lpos = S.tstart[d] + S.whist[warp * kCluRadix + d] + rank[k];  // in [0, cnt)
                S.stage[lpos] = S.kv[p];
            }
        }
        cl.sync();  // every CTA's digit counts are visible; the stage is complete
        if (pass == 0 && warp == kCluWarps - 1) {
            const int b = lane < C ? *cl.map_shared_rank(&S.bad, lane) : 0;
            const int any = __any_sync(0xffffffffu, b != 0);
            if (lane == 0) S.any_bad = any;
        }
        // digit d's counts in every CTA: thread (j, d) reads CTAs j, j+4, ...,
        // the four partial sums meet in the (now free) warp histogram
        int* part = S.whist;
        {
            const int d = tid & (kCluRadix - 1), j = tid >> 8;
            int pe = 0, pt = 0;
#pragma unroll
            for (int r4 = 0; r4 < kCluMaxCtas / 4; ++r4) {
                const int r = j + 4 * r4;
                if (r < C) {
                    const int x = *cl.map_shared_rank(&S.chist[d], r);
                    pt += x;
                    pe += r < c ? x : 0;
                }
            }
            part[tid] = pe;
            part[kCluThreads + tid] = pt;
        }
        __syncthreads();
        int excl = 0, tot = 0;
        if (tid < kCluRadix) {
#pragma unroll
            for (int j = 0; j < kCluThreads / kCluRadix; ++j) {
                excl += part[j * kCluRadix + tid];
                tot += part[kCluThreads + j * kCluRadix + tid];
            }
        }
        const int gstart = block_excl_scan<kCluThreads>(tid < kCluRadix ? tot : 0, S.ws, &sum_unused);
        if (tid < kCluRadix) S.gbase[tid] = gstart + excl;
        __syncthreads();
        for (int i = tid; i < cnt; i += kCluThreads) {
            const uint2 e = S.stage[i];
            const int d = static_cast<int>((e.x >> shift) & 255u);
            const int gpos = S.gbase[d] + (i - S.tstart[d]);  // in [0, N)
            const int owner = gpos / E;
            *cl.map_shared_rank(&S.kv[gpos - owner * E], owner) = e;
        }
        cl.sync();  // the pass's output is in place
    }

    // 3. the first position of every key present, stored with the key's row
    //    owner; this slice's keys below the end of every CTA's rows
    const bool any_bad = S.any_bad != 0;
    if (!any_bad) {
        for (int i = tid; i < cnt; i += kCluThreads) {
            const unsigned int k = S.kv[i].x;
            bool first;
            if (i > 0) first = S.kv[i - 1].x != k;
            else first = c == 0 || cl.map_shared_rank(S.kv, c - 1)[E - 1].x != k;
            if (first) {
                const unsigned int owner = k / static_cast<unsigned int>(R);  // k < M, R < 2^31
                *cl.map_shared_rank(&S.rstart[k - owner * static_cast<unsigned int>(R)], owner) =
                    static_cast<int>(c0 + i);
            }
        }
        if (tid < C) {
            const unsigned long long X = static_cast<unsigned long long>(min_ll(M, (tid + 1) * R));
            int lo = 0, hi = cnt;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (S.kv[mid].x < X) lo = mid + 1;
                else hi = mid;
            }
            S.cnt_lt[tid] = lo;
        }
    }
    cl.sync();  // row starts and counts are visible
    if (warp == 0) {
        int v = !any_bad && lane < C ? *cl.map_shared_rank(&S.cnt_lt[c], lane) : 0;
        v = __reduce_add_sync(0xffffffffu, v);
        if (lane == 0) S.next_start = v;
    }
    __syncthreads();

    // row_ptr over this CTA's rows: q consecutive rows per thread
    const int q = static_cast<int>((R + kCluThreads - 1) / kCluThreads);  // <= kCluRowsPerThread
    const long long t_lo = min_ll(r_hi, r_lo + static_cast<long long>(tid) * q);
    const long long t_hi = min_ll(r_hi, t_lo + q);
    const int nrows = any_bad ? 0 : static_cast<int>(t_hi - t_lo);
    int rp[kCluRowsPerThread];
    int run = INT_MAX;
#pragma unroll
    for (int j = kCluRowsPerThread - 1; j >= 0; --j) {
        rp[j] = INT_MAX;
        if (j < nrows) {
            run = min(run, S.rstart[t_lo - r_lo + j]);
            rp[j] = run;
        }
    }
    const int after = min(block_suffix_min_excl(run, S.ws), S.next_start);
#pragma unroll
    for (int j = 0; j < kCluRowsPerThread; ++j) rp[j] = min(rp[j], after);

    // 4. the work list: hot rows (more than 2^g chunks) give segment units and
    //    a finish task, rows of 2..2^g chunks a long whole-row unit, the
    //    others a short one (long ones listed first)
    const int G = 1 << g;
    int v4[5] = {0, 0, 0, 0, 0};  // segments, long rows, short rows, finish tasks, empty rows
    int mx = 0;
#pragma unroll
    for (int j = 0; j < kCluRowsPerThread; ++j) {
        if (j < nrows) {
            const int len = (j + 1 < nrows ? rp[j + 1] : after) - rp[j];
            const int nch = (len + 31) >> 5;
            if (nch > G) {
                v4[0] += (nch + G - 1) >> g;
                v4[3] += 1;
            } else if (nch > 1) {
                v4[1] += 1;
            } else if (nch == 1) {
                v4[2] += 1;
            } else {
                v4[4] += 1;
            }
            mx = max(mx, len);
        }
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0 && mx > 0) atomicMax(&S.tot[5], mx);
    int t4[5];
    block_excl_scan_n<kCluThreads, 5>(v4, S.ws, t4);
    if (tid == 0) {
        S.tot[0] = t4[0];
        S.tot[1] = t4[1];
        S.tot[2] = t4[2];
        S.tot[3] = t4[3];
        S.tot[4] = t4[4];
    }
    cl.sync();  // every CTA's totals are visible (no global store is pending here)
    if (warp == 0) {
        int v[5] = {0, 0, 0, 0, 0}, m = 0;
        if (lane < C) {
            const int* rt = cl.map_shared_rank(S.tot, lane);
#pragma unroll
            for (int j = 0; j < 5; ++j) v[j] = rt[j];
            m = rt[5];
        }
        int in[5] = {v[0], v[1], v[2], v[3], v[4]};
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
            for (int j = 0; j < 5; ++j) {
                const int t = __shfl_up_sync(0xffffffffu, in[j], o);
                if (lane >= o) in[j] += t;
            }
        }
        const int gm = __reduce_max_sync(0xffffffffu, m);
        if (lane == c) {
#pragma unroll
            for (int j = 0; j < 5; ++j) S.base[j] = in[j] - v[j];
        }
        if (lane == 31) {
#pragma unroll
            for (int j = 0; j < 5; ++j) S.grand[j] = in[j];
            S.grand[5] = gm;
        }
    }
    __syncthreads();
    // the last reads of other CTAs' shared memory are done: arrive now, write
    // the results, wait before leaving
    cluster_arrive_relaxed();
    // The reduce may be launched now, for this last phase (it waits for
    // this grid to finish).  Released at the kernel's start, the reduce's
    // ring kernel, one CTA per SM, would hold the SMs through the plan;
    // launched the ordinary way it started later: embedding backward step
    // 166.4 us, against 161.7 us with the release here and the ring kernel
    // as this kernel's programmatic dependent.
    pdl_launch_dependents();
    for (int i = tid; i < cnt; i += kCluThreads) perm[c0 + i] = static_cast<int>(S.kv[i].y);
    if (!any_bad) {
        int eA = v4[0] + S.base[0], eL = S.grand[0] + v4[1] + S.base[1], eS = v4[2] + S.base[2];
        int eC = v4[3] + S.base[3], eE = S.grand[2] + v4[4] + S.base[4];
#pragma unroll
        for (int j = 0; j < kCluRowsPerThread; ++j) {
            if (j < nrows) {
                const int m = static_cast<int>(t_lo + j);
                const int len = (j + 1 < nrows ? rp[j + 1] : after) - rp[j];
                const int nch = (len + 31) >> 5;
                row_ptr[m] = rp[j];
                if (nch > G) {
                    const int a = (nch + G - 1) >> g;
                    finish[eC++] = make_int4(m, eA, a, 0);
                    for (int s = 0; s < a; ++s) seg_units[eA + s] = make_int4(m, s, eA + s, 0);
                    eA += a;
                } else if (nch > 1) {
                    seg_units[eL++] = make_int4(m, -1, 0, 0);
                } else if (nch == 1) {
                    row_units[eS++] = make_int4(m, -1, 0, 0);
                } else {
                    row_units[eE++] = make_int4(m, -1, 0, 0);
                }
            }
        }
        if (c == 0 && tid == 0) row_ptr[M] = static_cast<int>(N);
    }
    if (c == 0 && tid < kCtrCount) {
        int v = 0;
        if (tid == kCtrErrIndex) v = any_bad ? 1 : 0;
        else if (!any_bad && tid == kCtrSegs) v = S.grand[0];
        else if (!any_bad && tid == kCtrLong) v = S.grand[1];
        else if (!any_bad && tid == kCtrNormal) v = S.grand[1] + S.grand[2] + S.grand[4];
        else if (!any_bad && tid == kCtrHot) v = S.grand[3];
        else if (!any_bad && tid == kCtrMaxLen) v = S.grand[5];
        else if (!any_bad && tid == kCtrBig) v = S.grand[0] + S.grand[1];
        else if (!any_bad && tid == kCtrShort) v = S.grand[2];
        else if (!any_bad && tid == kCtrEmpty) v = S.grand[4];
        counters[tid] = v;
    }
    cluster_wait();  // no CTA leaves while another may still read its shared memory
}

// ------------------------------------------------------------------------
// single-pass variant: at most 4096 destinations
// ------------------------------------------------------------------------
// With M <= 4096 the destination itself is the digit, so one counting pass
// sorts, and the destination counts it yields give row_ptr directly:
//   1. each CTA loads its slice; its warps rank it (peers of the whole
//      destination from one ballot per bit, in element order, warps in order)
//      against 8-bit per-warp counts of every destination;
//   2. each CTA owns R consecutive destinations: it reads their counts in
//      every CTA, writes each CTA's exclusive prefix back into that CTA's
//      shared memory, and takes the totals as row lengths, with their
//      work-list classification;
//   3. a scan over the CTAs' totals gives each range its first position, so
//      row_ptr of every owned destination;
//   4. every CTA copies all ranges' row_ptr (coalesced remote reads), and
//      source i goes to perm[row_ptr[key] + earlier CTAs + earlier warps +
//      rank].
constexpr int kOneMaxBins = 4096;
constexpr int kOneMaxSlice = 4096;
constexpr int kOneRowsPerThread = kOneMaxBins / kCluThreads;
static_assert(kOneMaxSlice / kCluWarps <= 255, "a warp's count of one destination fits a byte");
static_assert(kOneMaxBins / 4 <= kCluThreads, "one word of four counts per thread");

struct OneShared {
    uint2 kv[kOneMaxSlice];                               // {key, source position}
    unsigned short rank[kOneMaxSlice];                    // rank among equal keys inside the warp
    unsigned char whist[kCluWarps * kOneMaxBins];         // per warp count of every destination (< 256)
    int chist[kOneMaxBins];    // this CTA's count of each destination (read by the owners)
    int pref[kOneMaxBins];     // earlier CTAs' count of each destination (written by the owners)
    int rp[kOneMaxBins];       // row_ptr of the destinations this CTA owns (read by every CTA)
    int ws[6 * (kCluWarps + 1)];
    int tot[7];                // rows, seg units, long, short rows, finish tasks, empty rows, longest row
    int all_tot[kCluMaxCtas][7];  // every CTA's tot (written by that CTA)
    int bad;                   // this CTA saw an index outside [0, M) (read by every CTA)
    int any_bad;
};

// Lanes among `live` holding the same nbits-bit key as this lane.
__device__ __forceinline__ unsigned int key_peers(int d, unsigned int live, int nbits)
{
    unsigned int peers = live;
#pragma unroll
    for (int b = 0; b < 12; ++b) {
        if (b < nbits) {  // uniform
            const unsigned int set = __ballot_sync(0xffffffffu, (d >> b) & 1);
            peers &= ((d >> b) & 1) ? set : ~set;
        }
    }
    return peers;
}

__global__ void __launch_bounds__(kCluThreads, 1)
plan_cluster_one_kernel(const int* __restrict__ idx, long long N, long long M, int E, int nbits, int g,
                        int* __restrict__ row_ptr, int* __restrict__ perm, int4* __restrict__ seg_units,
                        int4* __restrict__ row_units, int4* __restrict__ finish, int* __restrict__ counters)
{
    cg::cluster_group cl = cg::this_cluster();
    extern __shared__ __align__(16) unsigned char clu_smem[];
    OneShared& S = *reinterpret_cast<OneShared*>(clu_smem);
    const int C = static_cast<int>(cl.num_blocks());
    const int c = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cnt = slice_len(N, E, c);
    const long long c0 = static_cast<long long>(c) * E;
    const int B = 1 << nbits;  // >= M
    const int R = static_cast<int>((M + C - 1) / C);  // destinations per owner, <= kOneMaxBins
    const int r_lo = static_cast<int>(min_ll(M, static_cast<long long>(c) * R));
    const int r_hi = static_cast<int>(min_ll(M, static_cast<long long>(r_lo) + R));
    unsigned int lt;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
    pdl_launch_dependents();  // the reduce may be launched now; it waits for this grid to finish
    unsigned int* wz = reinterpret_cast<unsigned int*>(S.whist);  // B is a multiple of 4
    for (int i = tid; i < kCluWarps * B / 4; i += kCluThreads) wz[i] = 0u;
    if (tid == 0) S.tot[6] = 0;

    // 1. the slice, then the ranking: warp w < 16 owns [w*ipw, (w+1)*ipw)
    bool bad = false;
    for (int i = tid; i < cnt; i += kCluThreads) {
        const unsigned int k = static_cast<unsigned int>(__ldg(idx + c0 + i));
        bad |= static_cast<long long>(k) >= M;
        S.kv[i] = make_uint2(k, static_cast<unsigned int>(c0 + i));
    }
    const int cta_bad = __syncthreads_or(bad);
    if (tid == 0) S.bad = cta_bad;
    const int ipw = (((cnt + kCluWarps - 1) / kCluWarps) + 31) & ~31;  // warp w owns [w*ipw, (w+1)*ipw)
    const int nk = ipw >> 5;  // <= 4
    {
        unsigned char* wh = S.whist + warp * B;
        for (int k = 0; k < nk; ++k) {
            const int p0 = warp * ipw + k * 32;
            const int nl = cnt - p0;
            const unsigned int live = nl >= 32 ? 0xffffffffu : (nl <= 0 ? 0u : (1u << nl) - 1u);
            if (live == 0u) break;  // uniform over the warp
            const int p = p0 + lane;
            const bool valid = (live >> lane) & 1u;
            const int d = valid ? static_cast<int>(S.kv[p].x & static_cast<unsigned int>(B - 1)) : 0;
            const unsigned int peers = key_peers(d, live, nbits);
            const int old = wh[d];
            if (valid) S.rank[p] = static_cast<unsigned short>(old + __popc(peers & lt));
            __syncwarp();
            if (valid && (peers & lt) == 0u) wh[d] = static_cast<unsigned char>(old + __popc(peers));
            __syncwarp();
        }
    }
    __syncthreads();
    // this CTA's count of every destination: thread t sums four destinations
    // (one word) over the 32 warps, bytes split into two 16-bit lanes
    if (tid < B / 4) {
        const unsigned int* wr = reinterpret_cast<const unsigned int*>(S.whist);
        unsigned int even = 0u, odd = 0u;
#pragma unroll 8
        for (int w = 0; w < kCluWarps; ++w) {
            const unsigned int x = wr[w * (B / 4) + tid];
            even += x & 0x00ff00ffu;
            odd += (x >> 8) & 0x00ff00ffu;
        }
        S.chist[4 * tid + 0] = static_cast<int>(even & 0xffffu);
        S.chist[4 * tid + 1] = static_cast<int>(odd & 0xffffu);
        S.chist[4 * tid + 2] = static_cast<int>(even >> 16);
        S.chist[4 * tid + 3] = static_cast<int>(odd >> 16);
    }
    cl.sync();  // every CTA's counts are visible
    if (warp == kCluWarps - 1) {
        const int b = lane < C ? *cl.map_shared_rank(&S.bad, lane) : 0;
        const int any = __any_sync(0xffffffffu, b != 0);
        if (lane == 0) S.any_bad = any;
    }
    __syncthreads();
    const bool any_bad = S.any_bad != 0;

    // 2. owned destinations [r_lo, r_hi), q consecutive per thread: counts in
    //    every CTA, each CTA's prefix written back, totals = row lengths
    const int q = (R + kCluThreads - 1) / kCluThreads;  // <= kOneRowsPerThread
    const int t_lo = min(r_hi, r_lo + tid * q);
    const int nrows = any_bad ? 0 : min(r_hi, t_lo + q) - t_lo;
    int len[kOneRowsPerThread];
#pragma unroll
    for (int j = 0; j < kOneRowsPerThread; ++j) {
        len[j] = 0;
        if (j < nrows) {
            const int m = t_lo + j;
            int x[kCluMaxCtas];
#pragma unroll
            for (int r = 0; r < kCluMaxCtas; ++r) x[r] = r < C ? *cl.map_shared_rank(&S.chist[m], r) : 0;
            int run = 0;
#pragma unroll
            for (int r = 0; r < kCluMaxCtas; ++r) {
                if (r < C) *cl.map_shared_rank(&S.pref[m], r) = run;
                run += x[r];
            }
            len[j] = run;
        }
    }
    const int G = 1 << g;
    // rows' sources, segment units, long rows (2..2^g chunks), short rows,
    // finish tasks, empty rows
    constexpr int NV = 6;
    int v5[NV] = {0, 0, 0, 0, 0, 0};
    int mx = 0;
#pragma unroll
    for (int j = 0; j < kOneRowsPerThread; ++j) {
        if (j < nrows) {
            const int nch = (len[j] + 31) >> 5;
            v5[0] += len[j];
            if (nch > G) {
                v5[1] += (nch + G - 1) >> g;
                v5[4] += 1;
            } else if (nch > 1) {
                v5[2] += 1;
            } else if (nch == 1) {
                v5[3] += 1;
            } else {
                v5[5] += 1;
            }
            mx = max(mx, len[j]);
        }
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0 && mx > 0) atomicMax(&S.tot[NV], mx);
    int t5[NV];
    block_excl_scan_n<kCluThreads, NV>(v5, S.ws, t5);  // ends synchronised: S.tot[NV] is final
    if (tid < (NV + 1) * C) {  // push this CTA's totals into every CTA
        const int r = tid / (NV + 1), f = tid - (NV + 1) * (tid / (NV + 1));
        int v = S.tot[NV];
#pragma unroll
        for (int j = 0; j < NV; ++j)
            if (f == j) v = t5[j];
        *cl.map_shared_rank(&S.all_tot[c][f], r) = v;
    }
    cl.sync();  // prefixes and every CTA's totals are visible

    // 3. bases from the CTAs' totals (every warp computes them itself); row_ptr
    //    of the owned destinations
    int base[NV], grand[NV + 1];
    {
        int v[NV] = {0, 0, 0, 0, 0, 0}, m = 0;
        if (lane < C) {
#pragma unroll
            for (int j = 0; j < NV; ++j) v[j] = S.all_tot[lane][j];
            m = S.all_tot[lane][NV];
        }
        int in[NV];
#pragma unroll
        for (int j = 0; j < NV; ++j) in[j] = v[j];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const int t = __shfl_up_sync(0xffffffffu, in[j], o);
                if (lane >= o) in[j] += t;
            }
        }
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            base[j] = __shfl_sync(0xffffffffu, in[j] - v[j], c);
            grand[j] = __shfl_sync(0xffffffffu, in[j], 31);
        }
        grand[NV] = __reduce_max_sync(0xffffffffu, m);
    }
    int rstart = v5[0] + base[0];
#pragma unroll
    for (int j = 0; j < kOneRowsPerThread; ++j) {
        if (j < nrows) {
            S.rp[t_lo + j - r_lo] = rstart;
            rstart += len[j];
        }
    }
    cl.sync();  // row_ptr of every range is visible

    // 4. perm.  First every range's row_ptr into this CTA, in place of the
    //    counts (no longer read): a warp reads 32 consecutive rows of one
    //    owner, where one remote read per source would cost a network request
    //    each.
    int* rp_all = S.chist;
    if (!any_bad) {
        for (int m = tid; m < M; m += kCluThreads) {
            const int o = m / R;
            rp_all[m] = cl.map_shared_rank(S.rp, o)[m - o * R];
        }
    }
    __syncthreads();
    if (!any_bad) {
        for (int i = tid; i < cnt; i += kCluThreads) {
            const uint2 e = S.kv[i];  // e.x < M
            const int w = i / ipw;
            int before = 0;  // equal keys in earlier warps of this CTA
            for (int v = 0; v < w; ++v) before += S.whist[v * B + e.x];
            const int pos = rp_all[e.x] + S.pref[e.x] + before + S.rank[i];
            perm[pos] = static_cast<int>(e.y);  // pos in [0, N)
        }
    }
    // the last reads of other CTAs' shared memory are done: arrive now, write
    // the lists, wait before leaving
    cluster_arrive_relaxed();
    if (!any_bad) {
        int eA = v5[1] + base[1], eL = grand[1] + v5[2] + base[2], eS = v5[3] + base[3], eC = v5[4] + base[4];
        int eE = grand[3] + v5[5] + base[5];
#pragma unroll
        for (int j = 0; j < kOneRowsPerThread; ++j) {
            if (j < nrows) {
                const int m = t_lo + j;
                const int nch = (len[j] + 31) >> 5;
                row_ptr[m] = S.rp[m - r_lo];
                if (nch > G) {
                    const int a = (nch + G - 1) >> g;
                    finish[eC++] = make_int4(m, eA, a, 0);
                    for (int s = 0; s < a; ++s) seg_units[eA + s] = make_int4(m, s, eA + s, 0);
                    eA += a;
                } else if (nch > 1) {
                    seg_units[eL++] = make_int4(m, -1, 0, 0);
                } else if (nch == 1) {
                    row_units[eS++] = make_int4(m, -1, 0, 0);
                } else {
                    row_units[eE++] = make_int4(m, -1, 0, 0);
                }
            }
        }
        if (c == 0 && tid == 0) row_ptr[M] = static_cast<int>(N);
    }
    if (c == 0 && tid < kCtrCount) {
        int v = 0;
        if (tid == kCtrErrIndex) v = any_bad ? 1 : 0;
        else if (!any_bad && tid == kCtrSegs) v = grand[1];
        else if (!any_bad && tid == kCtrLong) v = grand[2];
        else if (!any_bad && tid == kCtrNormal) v = grand[2] + grand[3] + grand[5];
        else if (!any_bad && tid == kCtrHot) v = grand[4];
        else if (!any_bad && tid == kCtrMaxLen) v = grand[NV];
        else if (!any_bad && tid == kCtrBig) v = grand[1] + grand[2];
        else if (!any_bad && tid == kCtrShort) v = grand[3];
        else if (!any_bad && tid == kCtrEmpty) v = grand[5];
        counters[tid] = v;
    }
    cluster_wait();  // no CTA leaves while another may still read its shared memory
}

// ------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------

namespace {
std::mutex g_clu_mu;
signed char g_clu_ok[kCluVariants][kMaxDevices][kCluMaxCtas + 1];  // [variant][device][C]: 0 unknown, 1 schedulable, -1 not
bool g_clu_attr[kCluVariants][kMaxDevices];

int bits_of(int64_t v)
{
    int b = 0;
    while (v > 0) { ++b; v >>= 1; }
    return b;
}
}  // namespace

det_status launch_on_cluster(int variant, const void* kern, int C, size_t smem, cudaStream_t st, void** args,
                             bool* launched)
{
    if (variant < 0 || variant >= kCluVariants || C < 1 || C > kCluMaxCtas) return DET_ERR_ARG;
    int dev = 0;
    DETR_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return DET_OK;
    {
        std::lock_guard<std::mutex> lock(g_clu_mu);
        if (!g_clu_attr[variant][dev]) {
            DETR_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
            DETR_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
            g_clu_attr[variant][dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned int>(C), 1, 1);
    cfg.blockDim = dim3(kCluThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned int>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    signed char ok;
    {
        std::lock_guard<std::mutex> lock(g_clu_mu);
        ok = g_clu_ok[variant][dev][C];
    }
    if (ok == 0) {
        int n = 0;
        const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) (void)cudaGetLastError();
        ok = (e == cudaSuccess && n >= 1) ? 1 : -1;
        std::lock_guard<std::mutex> lock(g_clu_mu);
        g_clu_ok[variant][dev][C] = ok;
    }
    if (ok < 0) return DET_OK;
    DETR_CUDA(cudaLaunchKernelExC(&cfg, kern, args));
    DETR_LAUNCHED();
    *launched = true;
    return DET_OK;
}

int plan_cluster_ctas(int64_t N, int64_t M)
{
    if (N <= 0 || N > static_cast<int64_t>(kCluMaxCtas) * kCluMaxSlice) return 0;
    const int C = static_cast<int>(std::min<int64_t>(kCluMaxCtas, std::max<int64_t>(1, cdiv(N, kCluTargetSlice))));
    if (cdiv(N, C) > kCluMaxSlice) return 0;
    if (cdiv(cdiv(M, C), kCluThreads) > kCluRowsPerThread) return 0;
    return C;
}

det_status launch_plan_cluster(const int32_t* idx, int64_t N, int64_t M, int g, int np32, int* row_ptr, int* perm,
                               int4* seg_units, int4* row_units, int4* finish, int* counters, bool two_pass,
                               cudaStream_t st, bool* launched)
{
    *launched = false;
    const int C = plan_cluster_ctas(N, M);
    if (C == 0) return DET_OK;
    int E = static_cast<int>(cdiv(N, C));
    if (M <= kOneMaxBins && E <= kOneMaxSlice) {
        long long n = N, m = M;
        int nbits = std::max(2, bits_of(M - 1));
        void* args[] = {&idx, &n, &m, &E, &nbits, &g, &row_ptr, &perm, &seg_units, &row_units, &finish, &counters};
        const det_status s = launch_on_cluster(kCluVariantOnePass, reinterpret_cast<const void*>(plan_cluster_one_kernel),
                                               C, sizeof(OneShared), st, args, launched);
        if (s || *launched) return s;
    }
    if (!two_pass) return DET_OK;
    long long n = N, m = M;
    void* args[] = {&idx, &n, &m, &E, &np32, &g, &row_ptr, &perm, &seg_units, &row_units, &finish, &counters};
    return launch_on_cluster(kCluVariantTwoPass, reinterpret_cast<const void*>(plan_cluster_kernel), C,
                             sizeof(CluShared), st, args, launched);
}

}  // namespace detr
