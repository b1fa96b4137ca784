// plan_owner.cu -- the plan for small and medium problems without order keys
// in one kernel spread over every SM: clusters of CTAs each own a range of
// destinations, and no cluster waits for another.
//
// The lists are the same as the other plan methods build: the terms of
// destination m are the sources with idx[i] = m in ascending i (the stable
// (expert id, original token id) order of "DeepSeek-V4 book, Ch 09: Batch
// invariance and determinism", section 3.2), and the work list splits
// destinations with more than 2^g chunks into aligned segments.  It is all
// integer work, so every method gives the same arrays.
//
// A plan over tens of thousands of sources is latency-bound: on a single
// cluster it is issue-bound on those few SMs, and as separate kernels it pays
// a launch and a round trip to L2 for every step.  Here K clusters of CS CTAs
// (CS = 8, one CTA per SM) each read all of idx between them (CTA s of a
// cluster reads slice s), which is small and stays in L2, so what crosses
// clusters is computed redundantly in every cluster instead of exchanged:
//   1. each CTA sweeps its slice: the range check, a count of every
//      destination (a full histogram in shared memory), and per-warp counts
//      of the destinations its cluster owns (warp w covers a contiguous
//      sub-range of the slice);
//   2. [cluster barrier] CTA s sums the cluster's histograms over its 1/CS of
//      the destinations (distributed shared memory), giving their lengths, and
//      classifies them for the work list: totals over all destinations and
//      over those before the cluster's range; it also turns its per-warp
//      counts of the owned rows into warp prefixes and a per-CTA count;
//   3. [cluster barrier] every CTA reads the CS partial totals: the sources
//      before the owned range are its first row_ptr, the units before it are
//      its offsets in the work list; the owned rows' lengths give their
//      offsets; each CTA writes row_ptr and the units of 1/CS of the owned
//      rows; the first CTA writes the counter block (an id outside [0, M),
//      flagged in step 1 and summed with the totals, stops every cluster
//      here with only the error flag written);
//   4. each warp reads its sub-range again in source order and places the
//      owned matches (peers of a row in a round of 32 from one ballot per
//      row-number bit): row start + earlier CTAs' and earlier warps' matches
//      of the row + rank.
// Cluster barriers are hardware barriers; nothing needs global memory zeroed
// first and no thread spins.
#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>

#include "block_scan.cuh"
#include "common.cuh"
#include "plan_internal.cuh"

namespace cg = cooperative_groups;

namespace detr {

constexpr int kCoThreads = 1024;
constexpr int kCoWarps = kCoThreads / 32;
constexpr int kCoClusters[3] = {8, 4, 2};  // cluster sizes tried, largest first (8 = the portable maximum)
constexpr int kCoBatch = 8;          // 16-byte loads in flight per lane in the counting sweep
constexpr int kCoScalarBatch = 8;    // 4-byte loads in flight per lane in the placing sweep
constexpr int kCoAgg = 15;           // published totals: 7 before the owned range, 7 over all destinations, bad ids
constexpr int kAggMax = 13;          // the longest row (a maximum, not a sum)
constexpr int kAggBad = 14;          // CTAs that saw an id outside [0, M)
constexpr size_t kCoMaxSmem = 200 * 1024;
static_assert(kOwnMaxRows <= kCoThreads, "one owned row per thread");
static_assert(kOwnMaxN / 32 < 65536, "a warp's count of one row fits 16 bits");

// Work-list class of a destination of len terms: v[0] sources, v[1] segment
// units and v[4] one finish task for a row of more than 2^g chunks, v[2] a
// long whole-row unit (2..2^g chunks), v[3] a short one (one chunk), v[5] an
// empty one.
__device__ __forceinline__ void row_classes(int len, int g, int v[6])
{
#pragma unroll
    for (int j = 0; j < 6; ++j) v[j] = 0;
    const int nch = (len + kChunk - 1) / kChunk;
    v[0] = len;
    if (nch > (1 << g)) {
        v[1] = (nch + (1 << g) - 1) >> g;
        v[4] = 1;
    } else if (nch > 1) {
        v[2] = 1;
    } else if (nch == 1) {
        v[3] = 1;
    } else {
        v[5] = 1;
    }
}

struct CoArgs {
    const int* idx;
    int N, M;
    int Rk;     // destinations per cluster
    int nb;     // bits of an owned row number (Rk - 1)
    int g;
    int sub;    // sources per warp sub-range (multiple of 128); a CTA slice is 32 * sub
    int B;      // destinations per CTA in the histogram sum (multiple of 4)
    int Mpad;   // histogram length (CS * B >= M)
    int Rw;     // 32-bit words per warp of packed 16-bit owned-row counts
    int* row_ptr;
    int* perm;
    int4* seg_units;
    int4* row_units;
    int4* finish;
    int* counters;
};

// Cluster barrier arrival that orders this thread's earlier memory accesses
// (its reads of other CTAs' shared memory) before it, without waiting.
__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Stable placement of up to 32 matches of one warp, in lane order: the lanes
// in `live` holding the same owned row rr are found from one ballot per bit of
// rr; each goes to its row's start for this CTA (rstart: row_ptr + earlier
// CTAs' matches) + the warp's running count of the row (earlier warps and
// earlier rounds) + its rank among its peers.
__device__ __forceinline__ void co_place(int rr, int pos, bool valid, unsigned int live, int nb,
                                         unsigned short* myc, const int* rstart, unsigned int lt_mask,
                                         int* perm)
{
    unsigned int peers = live;
    for (int b = 0; b < nb; ++b) {  // nb is uniform
        const unsigned int set = __ballot_sync(0xffffffffu, (rr >> b) & 1);
        peers &= ((rr >> b) & 1) ? set : ~set;
    }
    const int old = valid ? myc[rr] : 0;
    if (valid) perm[rstart[rr] + old + __popc(peers & lt_mask)] = pos;  // < N
    __syncwarp();
    if (valid && (peers & lt_mask) == 0u) myc[rr] = static_cast<unsigned short>(old + __popc(peers));
    __syncwarp();
}

// VEC: idx is 16-byte aligned (every sub-range starts at a multiple of 128
// sources, so every full group of four is one 16-byte load).  SHORT: a warp's
// sub-range is shorter than one round of either sweep (fewer than 1024
// sources), so both sweeps skip their batches past its end; with full rounds
// the unguarded loops measured faster.
template <bool VEC, int CS, bool SHORT>
__global__ void __launch_bounds__(kCoThreads, 1)
plan_owner_kernel(const __grid_constant__ CoArgs a)
{
    cg::cluster_group cl = cg::this_cluster();
    extern __shared__ __align__(16) int co_smem[];
    int* hist = co_smem;                                                   // [Mpad]: counts, then lengths (own bins)
    unsigned int* whist = reinterpret_cast<unsigned int*>(hist + a.Mpad);  // [warp][Rw]: 16-bit owned-row counts
    int* crow = reinterpret_cast<int*>(whist + kCoWarps * a.Rw);          // [Rk]: this CTA's count of each owned row
    int* rstart = crow + a.Rk;                                             // [Rk]: first position of this CTA's matches
    __shared__ int agg[kCoAgg];   // this CTA's partial totals (read by the cluster)
    __shared__ int sagg[kCoAgg];  // the cluster's totals
    __shared__ int ws[6 * (kCoWarps + 1)];

    const int s = static_cast<int>(cl.block_rank());
    const int k = static_cast<int>(blockIdx.x) / CS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = a.N, M = a.M, Rk = a.Rk;
    const int r_lo = k * Rk;
    const int nr = min(M - r_lo, Rk);  // >= 1: there are cdiv(M, Rk) clusters
    unsigned int lt_mask;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt_mask));

    for (int i = tid; i < a.Mpad; i += kCoThreads) hist[i] = 0;
    for (int i = tid; i < kCoWarps * a.Rw; i += kCoThreads) whist[i] = 0u;
    if (tid < kCoAgg) agg[tid] = 0;
    __syncthreads();

    // 1. count the warp's sub-range [wb, we) in groups of four per lane
    const int wb = (s * kCoWarps + warp) * a.sub;  // CS * 32 * sub < N + CS * 32 * 128 < 2^31
    const int we = min(N, wb + a.sub);
    unsigned int* mywh = whist + warp * a.Rw;
    const unsigned int ulo = static_cast<unsigned int>(r_lo), unr = static_cast<unsigned int>(nr);
    const unsigned int uM = static_cast<unsigned int>(M);
    // out-of-range ids are counted, and so are the padding slots past the end
    // (0xffffffff: out of range, never a match)
    unsigned int nbad = 0u, npad = 0u;
    for (int p0 = wb + 4 * lane; p0 < we; p0 += 128 * kCoBatch) {
        // batches that start past the sub-range hold no source of any lane
        // (warp-uniform): skipped, so a short sub-range costs only its own work
        const int nb = SHORT ? min(kCoBatch, (we - (p0 - 4 * lane) + 127) >> 7) : kCoBatch;
        int4 v[kCoBatch];
#pragma unroll
        for (int b = 0; b < kCoBatch; ++b) {  // all loads in flight first
            if (b >= nb) break;
            const int p = p0 + 128 * b;
            if (VEC && p + 3 < we) {
                v[b] = __ldg(reinterpret_cast<const int4*>(a.idx + p));
            } else {
                v[b].x = p < we ? __ldg(a.idx + p) : -1;
                v[b].y = p + 1 < we ? __ldg(a.idx + p + 1) : -1;
                v[b].z = p + 2 < we ? __ldg(a.idx + p + 2) : -1;
                v[b].w = p + 3 < we ? __ldg(a.idx + p + 3) : -1;
                npad += static_cast<unsigned int>(4 - min(4, max(0, we - p)));
            }
        }
#pragma unroll
        for (int b = 0; b < kCoBatch; ++b) {
            if (b >= nb) break;
            const unsigned int e[4] = {static_cast<unsigned int>(v[b].x), static_cast<unsigned int>(v[b].y),
                                       static_cast<unsigned int>(v[b].z), static_cast<unsigned int>(v[b].w)};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (e[j] < uM) atomicAdd(&hist[e[j]], 1);
                else ++nbad;  // a negative id is huge as unsigned
                const unsigned int rr = e[j] - ulo;
                if (rr < unr) atomicAdd(&mywh[rr >> 1], 1u << ((rr & 1u) * 16u));  // < 2^16 per warp
            }
        }
    }
    // an id outside [0, M) is counted nowhere; the flag goes out with the
    // totals and is acted on once they are read
    if (__any_sync(0xffffffffu, nbad != npad) && lane == 0) atomicOr(&agg[kAggBad], 1);
    cl.sync();  // every CTA's counts are visible

    // 2. lengths of this CTA's 1/CS of the destinations, and their classes:
    //    totals over those before the owned range (vb) and over all (va)
    int vb[7] = {0, 0, 0, 0, 0, 0, 0}, va[7] = {0, 0, 0, 0, 0, 0, 0};
    {
        const int m_lo = s * a.B, m_hi = min(M, m_lo + a.B);
        for (int m = m_lo + tid; m < m_hi; m += kCoThreads) {
            int len = 0;
#pragma unroll
            for (int r = 0; r < CS; ++r) len += cl.map_shared_rank(hist, r)[m];
            int v[6];
            row_classes(len, a.g, v);
#pragma unroll
            for (int j = 0; j < 6; ++j) {
                va[j] += v[j];
                if (m < r_lo) vb[j] += v[j];
            }
            va[6] = max(va[6], len);
            // the length replaces this CTA's own count of bin m, which no other
            // CTA reads (each reads only the bins it sums)
            hist[m] = len;
        }
    }
    // this CTA's count of each owned row; the per-warp counts become warp
    // prefixes (the two rows of a word belong to two threads of one warp:
    // each changes its half with an atomic add that leaves the other's half)
    if (tid < nr) {
        int run = 0;
        const int sh = (tid & 1) * 16;
        unsigned int* col = whist + (tid >> 1);
        // eight warps' counts read at once, then their eight independent updates
        for (int w0 = 0; w0 < kCoWarps; w0 += 8) {
            int x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = static_cast<int>((col[(w0 + j) * a.Rw] >> sh) & 0xffffu);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                atomicAdd(col + (w0 + j) * a.Rw, static_cast<unsigned int>(run - x[j]) << sh);  // the half becomes run
                run += x[j];
            }
        }
        crow[tid] = run;
    }
#pragma unroll
    for (int j = 0; j < 7; ++j) {
        const int tb = __reduce_add_sync(0xffffffffu, vb[j]);
        const int ta = j == 6 ? __reduce_max_sync(0xffffffffu, va[j]) : __reduce_add_sync(0xffffffffu, va[j]);
        if (lane == 0) {
            if (tb) atomicAdd(&agg[j], tb);
            if (ta) {
                if (j == 6) atomicMax(&agg[kAggMax], ta);
                else atomicAdd(&agg[7 + j], ta);
            }
        }
    }
    cl.sync();  // every CTA's partial totals, lengths and owned-row counts are visible

    // 3. the cluster's totals; the owned rows' lengths and this CTA's offsets
    if (tid < kCoAgg) {
        int t = 0;
#pragma unroll
        for (int r = 0; r < CS; ++r) {
            const int x = cl.map_shared_rank(agg, r)[tid];
            t = tid == kAggMax ? max(t, x) : t + x;
        }
        sagg[tid] = t;
    }
    int rlen = 0, before = 0;
    if (tid < nr) {
        const int m = r_lo + tid;
        rlen = cl.map_shared_rank(hist, m / a.B)[m];
#pragma unroll
        for (int r = 0; r < CS; ++r)
            if (r < s) before += cl.map_shared_rank(crow, r)[tid];
    }
    // the last reads of other CTAs' shared memory are done
    cluster_arrive_release();
    int roff_tot;
    const int roff = block_excl_scan<kCoThreads>(rlen, ws, &roff_tot);  // synchronises: sagg is visible
    if (sagg[kAggBad]) {
        // every cluster read all of idx, so every CTA takes this branch: only
        // the error flag is written
        if (k == 0 && s == 0 && tid < kCtrCount) a.counters[tid] = tid == kCtrErrIndex ? 1 : 0;
        cluster_wait_acquire();  // no CTA leaves while another may still read its shared memory
        return;
    }
    const int base = sagg[0];  // sources with idx < r_lo = row_ptr[r_lo]
    if (tid < nr) rstart[tid] = base + roff + before;
    // units of the owned rows, at offsets from the classes before each row
    int v6[6] = {0, 0, 0, 0, 0, 0};
    if (tid < nr) row_classes(rlen, a.g, v6);
    int t6[6];
    block_excl_scan_n<kCoThreads, 6>(v6, ws, t6);  // synchronises: rstart is visible
    const int q = (nr + CS - 1) / CS;
    if (tid < nr && tid >= s * q && tid < (s + 1) * q) {
        const int m = r_lo + tid;
        const int G = 1 << a.g;
        a.row_ptr[m] = base + roff;
        const int nch = (rlen + kChunk - 1) / kChunk;
        if (nch > G) {
            const int eA = sagg[1] + v6[1];
            const int na = (nch + G - 1) >> a.g;
            a.finish[sagg[4] + v6[4]] = make_int4(m, eA, na, 0);
            for (int j = 0; j < na; ++j) a.seg_units[eA + j] = make_int4(m, j, eA + j, 0);
        } else if (nch > 1) {
            a.seg_units[sagg[7 + 1] + sagg[2] + v6[2]] = make_int4(m, -1, 0, 0);
        } else if (nch == 1) {
            a.row_units[sagg[3] + v6[3]] = make_int4(m, -1, 0, 0);
        } else {
            a.row_units[sagg[7 + 3] + sagg[5] + v6[5]] = make_int4(m, -1, 0, 0);
        }
    }
    if (k == static_cast<int>(gridDim.x) / CS - 1 && s == 0 && tid == 0) a.row_ptr[M] = N;
    if (k == 0 && s == 0 && tid < kCtrCount) {
        const int* G7 = sagg + 7;  // sources, segs, long, short, finish, empty, longest (all destinations)
        int x = 0;
        if (tid == kCtrSegs) x = G7[1];
        else if (tid == kCtrLong) x = G7[2];
        else if (tid == kCtrNormal) x = G7[2] + G7[3] + G7[5];
        else if (tid == kCtrHot) x = G7[4];
        else if (tid == kCtrMaxLen) x = G7[6];
        else if (tid == kCtrBig) x = G7[1] + G7[2];
        else if (tid == kCtrShort) x = G7[3];
        else if (tid == kCtrEmpty) x = G7[5];
        a.counters[tid] = x;  // the error flags are 0
    }

    // The reduce may be launched now, for this kernel's last phase: it waits
    // for this grid to finish.  (Released at the kernel's start, the CTAs of
    // the fixed-stage gather, launched as a programmatic dependent, sat on
    // the SMs for the whole plan, and the MoE step took 65.2 us; released
    // here, 62.6 us, against 64.5 us with that gather launched the ordinary
    // way.)
    pdl_launch_dependents();
    // 4. place the matches: the sub-range again in source order, 32 per round
    unsigned short* myc = reinterpret_cast<unsigned short*>(mywh);
    for (int p0 = wb; p0 < we; p0 += 32 * kCoScalarBatch) {
        const int nb = SHORT ? min(kCoScalarBatch, (we - p0 + 31) >> 5) : kCoScalarBatch;  // rounds with a source (warp-uniform)
        unsigned int kk[kCoScalarBatch];
#pragma unroll
        for (int b = 0; b < kCoScalarBatch; ++b) {
            if (b >= nb) break;
            const int p = p0 + b * 32 + lane;
            kk[b] = p < we ? static_cast<unsigned int>(__ldg(a.idx + p)) : uM;
        }
#pragma unroll
        for (int b = 0; b < kCoScalarBatch; ++b) {
            if (b >= nb) break;
            const unsigned int rr = kk[b] - ulo;
            const bool valid = rr < unr;  // the padding M never matches: r_lo + nr <= M
            const unsigned int live = __ballot_sync(0xffffffffu, valid);
            if (live == 0u) continue;  // uniform
            co_place(valid ? static_cast<int>(rr) : 0, p0 + b * 32 + lane, valid, live, a.nb, myc, rstart,
                     lt_mask, a.perm);
        }
    }
    cluster_wait_acquire();  // no CTA leaves while another may still read its shared memory
}

// ------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------

namespace {
std::mutex g_co_mu;
int g_co_clusters[2][3][kMaxDevices];  // [vec][size][device]: clusters run at once; 0 unknown, -1 none

int bit_count(int64_t v)
{
    int b = 0;
    while (v > 0) { ++b; v >>= 1; }
    return b;
}

struct CoShape {
    int CS, K, Rk, sub, B, Mpad, Rw;
    size_t smem;
};

const void* co_kernel(int vec, int ci, int shrt = 0)
{
    static const void* k[2][2][3] = {
        {{reinterpret_cast<const void*>(plan_owner_kernel<false, 8, false>), reinterpret_cast<const void*>(plan_owner_kernel<false, 4, false>),
          reinterpret_cast<const void*>(plan_owner_kernel<false, 2, false>)},
         {reinterpret_cast<const void*>(plan_owner_kernel<true, 8, false>), reinterpret_cast<const void*>(plan_owner_kernel<true, 4, false>),
          reinterpret_cast<const void*>(plan_owner_kernel<true, 2, false>)}},
        {{reinterpret_cast<const void*>(plan_owner_kernel<false, 8, true>), reinterpret_cast<const void*>(plan_owner_kernel<false, 4, true>),
          reinterpret_cast<const void*>(plan_owner_kernel<false, 2, true>)},
         {reinterpret_cast<const void*>(plan_owner_kernel<true, 8, true>), reinterpret_cast<const void*>(plan_owner_kernel<true, 4, true>),
          reinterpret_cast<const void*>(plan_owner_kernel<true, 2, true>)}}};
    return k[shrt][vec][ci];
}

// Shape for clusters of CS CTAs, at most max_clusters of them (the number the
// device runs at once, so that they all run in one wave).
bool co_shape(int64_t N, int64_t M, int CS, int max_clusters, CoShape* sh)
{
    if (N < 1 || N > kOwnMaxN || M < 1 || M > kOwnMaxM || max_clusters < 1) return false;
    const int64_t K0 = std::min<int64_t>(max_clusters, M);
    const int64_t Rk = cdiv(M, K0);
    if (Rk > kOwnMaxRows) return false;
    sh->CS = CS;
    sh->Rk = static_cast<int>(Rk);
    sh->K = static_cast<int>(cdiv(M, Rk));
    sh->sub = static_cast<int>(cdiv(cdiv(N, int64_t(CS) * kCoWarps), 128) * 128);
    // a CTA's running count of one row (16 bits) covers at most its slice
    if (int64_t(sh->sub) * kCoWarps > 65535) return false;
    sh->B = static_cast<int>(cdiv(cdiv(M, CS), 4) * 4);
    sh->Mpad = sh->B * CS;
    sh->Rw = static_cast<int>(cdiv(Rk, 2));
    sh->smem = (static_cast<size_t>(sh->Mpad) + static_cast<size_t>(kCoWarps) * sh->Rw + 2 * static_cast<size_t>(Rk)) *
               sizeof(int);
    return sh->smem <= kCoMaxSmem;
}

cudaLaunchConfig_t co_config(const CoShape& sh, cudaLaunchAttribute* attr, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sh.K * sh.CS));
    cfg.blockDim = dim3(kCoThreads);
    cfg.dynamicSmemBytes = sh.smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sh.CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// How many clusters of size kCoClusters[ci] the current device runs at once
// with the largest shared memory the plan may ask for (cached per device).
det_status co_max_clusters(int vec, int ci, int* out)
{
    int dev = 0;
    DETR_CUDA(cudaGetDevice(&dev));
    *out = 0;
    if (dev < 0 || dev >= kMaxDevices) return DET_OK;
    std::lock_guard<std::mutex> lk(g_co_mu);
    int& n = g_co_clusters[vec][ci][dev];
    if (n == 0) {
        // both sweep variants (full and short rounds) launch with the same
        // block size, register limit and shared memory: one query serves both
        for (int shrt = 0; shrt < 2; ++shrt) {
            const det_status s = allow_dynamic_smem(co_kernel(vec, ci, shrt), kCoMaxSmem);
            if (s) return s;
        }
        const void* kern = co_kernel(vec, ci);
        CoShape sh{};
        sh.CS = kCoClusters[ci];
        sh.K = 1;
        sh.smem = kCoMaxSmem;
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = co_config(sh, attr, nullptr);
        int nclu = 0;
        DETR_CUDA(cudaOccupancyMaxActiveClusters(&nclu, kern, &cfg));
        n = nclu >= 1 ? nclu : -1;
    }
    *out = std::max(n, 0);
    return DET_OK;
}

// The largest cluster size whose clusters, all running at once, own at most
// kOwnMaxRows destinations each.
det_status co_pick(int64_t N, int64_t M, int vec, CoShape* sh, int* ci_out, bool* ok)
{
    *ok = false;
    for (int ci = 0; ci < 3; ++ci) {
        int maxc = 0;
        det_status s = co_max_clusters(vec, ci, &maxc);
        if (s) return s;
        if (co_shape(N, M, kCoClusters[ci], maxc, sh)) {
            *ci_out = ci;
            *ok = true;
            return DET_OK;
        }
    }
    return DET_OK;
}
}  // namespace

det_status launch_plan_owner(const int32_t* idx, int64_t N, int64_t M, int g, int* row_ptr, int* perm,
                             int4* seg_units, int4* row_units, int4* finish, int* counters, cudaStream_t st,
                             bool* launched)
{
    *launched = false;
    const int vec = aligned(idx, 16) ? 1 : 0;
    CoShape sh{};
    int ci = 0;
    bool ok = false;
    det_status s = co_pick(N, M, vec, &sh, &ci, &ok);
    if (s || !ok) return s;
    const void* kern = co_kernel(vec, ci, sh.sub < 128 * kCoBatch ? 1 : 0);
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = co_config(sh, attr, st);
    CoArgs a{};
    a.idx = idx;
    a.N = static_cast<int>(N);
    a.M = static_cast<int>(M);
    a.Rk = sh.Rk;
    a.nb = bit_count(sh.Rk - 1);
    a.g = g;
    a.sub = sh.sub;
    a.B = sh.B;
    a.Mpad = sh.Mpad;
    a.Rw = sh.Rw;
    a.row_ptr = row_ptr;
    a.perm = perm;
    a.seg_units = seg_units;
    a.row_units = row_units;
    a.finish = finish;
    a.counters = counters;
    void* args[] = {&a};
    DETR_CUDA(cudaLaunchKernelExC(&cfg, kern, args));
    DETR_LAUNCHED();
    *launched = true;
    return DET_OK;
}

}  // namespace detr
