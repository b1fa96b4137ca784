// plan_radix.cu -- the plan for large problems without order keys: stable
// 8-bit LSD radix passes over packed words, row lengths counted by the last
// pass, and the work list from one kernel.
//
// The lists are the same as the other plan methods build: the terms of
// destination m are the sources with idx[i] = m in ascending i (the stable
// (expert id, original token id) order of "DeepSeek-V4 book, Ch 09: Batch
// invariance and determinism", section 3.2; for the sparse-attention backward
// of section 3.1, the queries that chose key m, in query order).  It is all
// integer work, so every method gives the same arrays.
//
// For N < 2^24 sources and M <= 65536 destinations (one or two 8-bit digits):
//   per digit pass, three kernels, none of which waits for another CTA:
//     rx_count_kernel    digit counts of every tile of 4096 words, by a
//                        persistent grid that prefetches its next tile (the
//                        first pass also checks idx against M and zeroes the
//                        row counters);
//     rx_offset_kernel   one CTA per digit: exclusive scan of the digit's
//                        counts over the tiles (the first pass also gathers
//                        the tiles' range errors into the counter block);
//     rx_scatter_kernel  each tile ranks its words (peers of a digit from
//                        one ballot per digit bit, in element order, warps in
//                        order), stages them in shared memory in (digit,
//                        position) order and writes them in runs.  The first
//                        of two passes writes packed words (high digit << 24 |
//                        source), so the second reads 4 bytes per source, and
//                        beside each word its low digit (one byte); the last
//                        pass writes perm, and since its staged words are in
//                        destination order it also adds each run of one
//                        destination to that destination's row counter;
//   rx_units_count_kernel, rx_units_write_kernel
//                        row_ptr and the work list from the row counters:
//                        class totals per block of 1024 destinations, then
//                        each block's offsets from the blocks before it.
// Every kernel is a programmatic dependent of the one before it: it is
// launched while that one runs and waits (griddepcontrol.wait) before reading
// what it wrote.
#include <algorithm>

#include "block_scan.cuh"
#include "common.cuh"
#include "plan_internal.cuh"

namespace detr {

constexpr int kRxThreads = 256;
constexpr int kRxWarps = kRxThreads / 32;
constexpr int kRxItems = 16;
constexpr int kRxTile = kRxThreads * kRxItems;  // 4096 words per tile
constexpr int kRxRadix = 256;
constexpr int kRxUnitThreads = 1024;            // destinations per CTA of the work-list kernels
constexpr int kRxMaxUnitBlocks = 64;            // blocks of 1024 destinations (M <= 65536)
static_assert(kRxMaxUnitBlocks * 8 <= kRxUnitThreads, "one block total per thread");

// ------------------------------------------------------------------------
// counts
// ------------------------------------------------------------------------

// MODE 0: the words are idx (digit = low byte; ids checked against M).
// MODE 1: packed words of the first pass (digit = top byte).
// Persistent: CTA c counts tiles c, c + grid, ...; the next tile's 16-byte
// loads are in flight while the current one is counted (VEC: the words are
// 16-byte aligned).
constexpr int kRxCountVec = kRxTile / (4 * kRxThreads);  // 16-byte loads per thread per tile

template <bool VEC>
__device__ __forceinline__ void rx_load_tile(const int* in, int N, int t, int tid, uint4 (&v)[kRxCountVec])
{
#pragma unroll
    for (int j = 0; j < kRxCountVec; ++j) {
        const int p = t * kRxTile + 4 * (j * kRxThreads + tid);
        if (VEC && p + 3 < N) {
            v[j] = __ldg(reinterpret_cast<const uint4*>(in + p));
        } else {
            v[j].x = p < N ? static_cast<unsigned int>(__ldg(in + p)) : 0u;
            v[j].y = p + 1 < N ? static_cast<unsigned int>(__ldg(in + p + 1)) : 0u;
            v[j].z = p + 2 < N ? static_cast<unsigned int>(__ldg(in + p + 2)) : 0u;
            v[j].w = p + 3 < N ? static_cast<unsigned int>(__ldg(in + p + 3)) : 0u;
        }
    }
}

template <int MODE, bool VEC>
__global__ void __launch_bounds__(kRxThreads)
rx_count_kernel(const int* __restrict__ in, int N, unsigned int M, int* __restrict__ counts, int ntiles,
                int* __restrict__ tbad, int* __restrict__ zero_a, int zero_na)
{
    __shared__ int wh[kRxWarps * kRxRadix];
    const int tid = threadIdx.x, warp = tid >> 5;
    pdl_launch_dependents();  // the next kernel may be launched now; it waits for this grid to finish
    for (int i = tid; i < kRxWarps * kRxRadix; i += kRxThreads) wh[i] = 0;
    pdl_wait();  // whatever wrote idx (or the previous pass) has finished
    if (MODE == 0) {  // read by a later kernel of this plan only
        const int stride = static_cast<int>(gridDim.x) * kRxThreads;
        for (int i = static_cast<int>(blockIdx.x) * kRxThreads + tid; i < zero_na; i += stride) zero_a[i] = 0;
    }
    __syncthreads();
    int t = blockIdx.x;
    uint4 cur[kRxCountVec], nxt[kRxCountVec];
    if (t < ntiles) rx_load_tile<VEC>(in, N, t, tid, cur);
    int* mh = wh + warp * kRxRadix;
    for (; t < ntiles; t += gridDim.x) {
        const int tn = t + static_cast<int>(gridDim.x);
        if (tn < ntiles) rx_load_tile<VEC>(in, N, tn, tid, nxt);
        bool bad = false;
#pragma unroll
        for (int j = 0; j < kRxCountVec; ++j) {
            const int p = t * kRxTile + 4 * (j * kRxThreads + tid);
            const unsigned int e[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (p + c < N) {
                    if (MODE == 0) bad |= e[c] >= M;  // a negative id is huge as unsigned
                    atomicAdd(&mh[MODE == 0 ? (e[c] & 255u) : (e[c] >> 24)], 1);
                }
            }
        }
        const int b = __syncthreads_or(bad);
        if (MODE == 0 && tid == 0) tbad[t] = b;
        int c = 0;
#pragma unroll
        for (int q = 0; q < kRxWarps; ++q) {
            c += wh[q * kRxRadix + tid];
            wh[q * kRxRadix + tid] = 0;
        }
        counts[static_cast<long long>(tid) * ntiles + t] = c;
        __syncthreads();  // the histogram is zero again before the next tile's adds
#pragma unroll
        for (int j = 0; j < kRxCountVec; ++j) cur[j] = nxt[j];
    }
}

// One CTA per digit: exclusive scan of the digit's tile counts, in place, and
// the digit's total.  With tbad: CTA 0 also writes the counter block (the
// range-error flag; the work counts are written by the units kernel).
constexpr int kRxOffItems = 4;

__global__ void __launch_bounds__(kRxThreads)
rx_offset_kernel(int* __restrict__ counts, int ntiles, int* __restrict__ totals, const int* __restrict__ tbad,
                 int* __restrict__ counters)
{
    __shared__ int ws[kRxThreads / 32 + 1];
    pdl_launch_dependents();
    pdl_wait();
    int* row = counts + static_cast<long long>(blockIdx.x) * ntiles;
    int carry = 0;
    for (int t0 = 0; t0 < ntiles; t0 += kRxThreads * kRxOffItems) {
        int v[kRxOffItems];
        int sum = 0;
#pragma unroll
        for (int j = 0; j < kRxOffItems; ++j) {
            const int t = t0 + threadIdx.x * kRxOffItems + j;
            v[j] = t < ntiles ? row[t] : 0;
            sum += v[j];
        }
        int tot;
        int run = carry + block_excl_scan<kRxThreads>(sum, ws, &tot);
#pragma unroll
        for (int j = 0; j < kRxOffItems; ++j) {
            const int t = t0 + threadIdx.x * kRxOffItems + j;
            if (t < ntiles) row[t] = run;
            run += v[j];
        }
        carry += tot;
    }
    if (threadIdx.x == 0) totals[blockIdx.x] = carry;
    if (tbad && blockIdx.x == 0) {
        bool b = false;
        for (int t = threadIdx.x; t < ntiles; t += kRxThreads) b |= tbad[t] != 0;
        const int any = __syncthreads_or(b);
        if (threadIdx.x < kCtrCount) counters[threadIdx.x] = threadIdx.x == kCtrErrIndex ? any : 0;
    }
}

// ------------------------------------------------------------------------
// scatter
// ------------------------------------------------------------------------

// MODE 0: words are idx; the digit is the low byte; the output (first of two
// passes) is (high byte << 24 | source) with the low byte in lowd at the same
// position, or (single pass, M <= 256) perm.
// MODE 1: words are packed; the digit is the top byte; lowd holds each word's
// low byte; the output is perm.
// LAST: the output is perm and the staged runs of equal destinations are
// added to rowcnt.  Warp w owns words [w*32*ITEMS, (w+1)*32*ITEMS) of the
// tile, item k of lane l being word w*32*ITEMS + k*32 + l.
struct RxScatterShared {
    unsigned int sval[kRxTile];      // staged output words, in (digit, position) order
    unsigned short skey[kRxTile];    // staged destinations (LAST), or staged digits (first of two passes)
    unsigned char lomap[kRxTile];    // MODE 1: the low digit of each input word of the tile (from lowd)
    int whist[kRxWarps * kRxRadix];  // per warp running digit counts, then warp offsets
    int tstart[kRxRadix];            // first staged position of each digit
    int gbase[kRxRadix];             // global position of staged position 0 of each digit
    int ws[kRxThreads / 32 + 1];
};

// One tile; FULL: all kTile words exist (no bounds checks).
template <int MODE, bool LAST, bool FULL>
__device__ __forceinline__ void rx_scatter_tile(RxScatterShared& S, const int* __restrict__ in, int N,
                                                unsigned int* __restrict__ out, const int* __restrict__ offsets,
                                                const int* __restrict__ totals, unsigned char* __restrict__ lowd,
                                                int ntiles, int* __restrict__ rowcnt)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tile = blockIdx.x;
    const int base = tile * kRxTile;
    unsigned int lt_mask;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt_mask));

    const int wbase = base + warp * 32 * kRxItems;
    unsigned int wv[kRxItems];
#pragma unroll
    for (int k = 0; k < kRxItems; ++k) {  // all loads first
        const int p = wbase + k * 32 + lane;
        wv[k] = FULL || p < N ? static_cast<unsigned int>(__ldg(in + p)) : 0u;
    }
    const int tot_d = totals[tid];
    const int off_d = offsets[static_cast<long long>(tid) * ntiles + tile];
    int total_unused;
    const int dstart = block_excl_scan<kRxThreads>(tot_d, S.ws, &total_unused);  // orders the whist zeroing
    S.gbase[tid] = dstart + off_d;
    if (MODE == 1) {
        // the low digit of each input word, written beside it by the first
        // pass (16-byte loads from the 16-byte aligned array; the tail of
        // the last tile byte by byte, none past N)
        const int b0 = base + 16 * tid;
        if (FULL || b0 + 15 < N) {
            reinterpret_cast<uint4*>(S.lomap)[tid] = *reinterpret_cast<const uint4*>(lowd + b0);
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) S.lomap[16 * tid + j] = b0 + j < N ? lowd[b0 + j] : 0;
        }
        __syncthreads();
    }

    // rank inside the warp, item by item: every lane reads the warp's running
    // count of its digit, and the lowest lane of each digit group writes it
    // back advanced
    unsigned short rank[kRxItems];
#pragma unroll
    for (int k = 0; k < kRxItems; ++k) {
        const int nl = N - (wbase + k * 32);
        const unsigned int live = FULL || nl >= 32 ? 0xffffffffu : (nl <= 0 ? 0u : (1u << nl) - 1u);
        rank[k] = 0;
        if (!FULL && live == 0u) continue;  // uniform over the warp
        const bool valid = FULL || ((live >> lane) & 1u);
        const int d = static_cast<int>(MODE == 0 ? (wv[k] & 255u) : (wv[k] >> 24));
        const unsigned int peers = digit_peers(d, live);
        const int old = valid ? S.whist[warp * kRxRadix + d] : 0;  // lanes of one digit read one word
        const unsigned int below = peers & lt_mask;
        rank[k] = static_cast<unsigned short>(old + __popc(below));
        __syncwarp();  // every lane has read before the group's lowest lane writes
        if (valid && below == 0u) S.whist[warp * kRxRadix + d] = old + __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // per digit: offsets of the warps (warp order), tile counts, staged starts
    int tot = 0;
    {
        const int d = tid;
#pragma unroll
        for (int q = 0; q < kRxWarps; ++q) {
            const int c = S.whist[q * kRxRadix + d];
            S.whist[q * kRxRadix + d] = tot;
            tot += c;
        }
    }
    const int excl = block_excl_scan<kRxThreads>(tot, S.ws, &total_unused);
    S.tstart[tid] = excl;
    S.gbase[tid] -= excl;  // staged position i of digit d goes to gbase[d] + i
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kRxItems; ++k) {
        const int p = wbase + k * 32 + lane;
        if (FULL || p < N) {
            const unsigned int w = wv[k];
            const int d = static_cast<int>(MODE == 0 ? (w & 255u) : (w >> 24));
            const int pos = S.tstart[d] + S.whist[warp * kRxRadix + d] + rank[k];
            if (MODE == 0 && !LAST) {
                S.sval[pos] = ((w >> 8) << 24) | static_cast<unsigned int>(p);  // w < M <= 65536, p < 2^24
                S.skey[pos] = static_cast<unsigned short>(d);  // the low digit, written beside the word
            } else if (MODE == 0) {
                S.sval[pos] = static_cast<unsigned int>(p);
                S.skey[pos] = static_cast<unsigned short>(d);  // the destination itself (M <= 256)
            } else {
                S.sval[pos] = w & 0xffffffu;
                S.skey[pos] = static_cast<unsigned short>((d << 8) | S.lomap[p - base]);
            }
        }
    }
    __syncthreads();

    const int rem = N - base;
    const int nvalid = FULL || rem >= kRxTile ? kRxTile : rem;
    for (int i0 = 0; i0 < kRxTile; i0 += kRxThreads) {
        const int i = i0 + tid;
        unsigned int key = 0xffffffffu;
        if (i < nvalid) {
            key = S.skey[i];
            const int d = LAST && MODE == 1 ? static_cast<int>(key >> 8) : static_cast<int>(key);
            out[S.gbase[d] + i] = S.sval[i];  // in [0, N)
            if (MODE == 0 && !LAST) lowd[S.gbase[d] + i] = static_cast<unsigned char>(d);
        }
        if (LAST) {
            // runs of one destination inside this warp's 32 staged words: one
            // add of the run length per run (a run cut by the warp boundary is
            // added in two parts)
            const unsigned int prevk = __shfl_up_sync(0xffffffffu, key, 1);
            const bool start = i < nvalid && (lane == 0 || prevk != key);
            const unsigned int starts = __ballot_sync(0xffffffffu, start);
            const unsigned int validm = __ballot_sync(0xffffffffu, i < nvalid);
            if (start) {
                const unsigned int later = lane == 31 ? 0u : (starts & (0xffffffffu << (lane + 1)));
                const int end = later ? __ffs(later) - 1 : 32 - __clz(validm);
                atomicAdd(&rowcnt[key], end - lane);
            }
        }
    }
}

template <int MODE, bool LAST>
__global__ void __launch_bounds__(kRxThreads, 4)
rx_scatter_kernel(const int* __restrict__ in, int N, unsigned int* __restrict__ out, const int* __restrict__ offsets,
                  const int* __restrict__ totals, unsigned char* __restrict__ lowd, int ntiles,
                  int* __restrict__ rowcnt, const int* __restrict__ counters)
{
    extern __shared__ __align__(16) unsigned char rx_smem[];
    RxScatterShared& S = *reinterpret_cast<RxScatterShared*>(rx_smem);
    const int tid = threadIdx.x;
    pdl_launch_dependents();
    for (int i = tid; i < kRxWarps * kRxRadix; i += kRxThreads) S.whist[i] = 0;
    pdl_wait();  // the previous kernels' counts, offsets and words are visible
    // with an id out of range the row counters would be indexed out of range:
    // the last pass writes nothing (the plan reports the error)
    if (LAST && counters[kCtrErrIndex]) return;
    if ((static_cast<long long>(blockIdx.x) + 1) * kRxTile <= N)  // uniform over the CTA
        rx_scatter_tile<MODE, LAST, true>(S, in, N, out, offsets, totals, lowd, ntiles, rowcnt);
    else
        rx_scatter_tile<MODE, LAST, false>(S, in, N, out, offsets, totals, lowd, ntiles, rowcnt);
}

// ------------------------------------------------------------------------
// row_ptr and the work list
// ------------------------------------------------------------------------

// Work-list class of a destination of len terms: v[0] sources, v[1] segment
// units and v[4] one finish task for a row of more than 2^g chunks, v[2] a
// long whole-row unit (2..2^g chunks), v[3] a short one (one chunk), v[5] an
// empty one.
__device__ __forceinline__ void rx_row_classes(int len, int g, int v[6])
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

// The work list in two kernels over blocks of 1024 destinations:
//   rx_units_count_kernel  each block's class totals (6) and longest row;
//   rx_units_write_kernel  each CTA sums the totals of the blocks before its
//                          own (its offsets) and of all blocks (the region
//                          starts), scans its rows and writes row_ptr, the
//                          units and the finish tasks.
__global__ void __launch_bounds__(kRxUnitThreads)
rx_units_count_kernel(const int* __restrict__ rowcnt, int M, int g, int* __restrict__ btot,
                      const int* __restrict__ counters)
{
    __shared__ int stot[7];
    const int tid = threadIdx.x, lane = tid & 31;
    pdl_launch_dependents();
    if (tid < 7) stot[tid] = 0;
    pdl_wait();
    if (counters[kCtrErrIndex]) return;  // the same for every CTA
    const int m = blockIdx.x * kRxUnitThreads + tid;
    const int len = m < M ? rowcnt[m] : 0;
    int v[6];
    rx_row_classes(len, g, v);
    if (m >= M) v[5] = 0;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 6; ++k) {
        const int t = __reduce_add_sync(0xffffffffu, v[k]);
        if (lane == 0 && t) atomicAdd(&stot[k], t);
    }
    const int mx = __reduce_max_sync(0xffffffffu, len);
    if (lane == 0 && mx) atomicMax(&stot[6], mx);
    __syncthreads();
    if (tid < 7) btot[blockIdx.x * 8 + tid] = stot[tid];
}

__global__ void __launch_bounds__(kRxUnitThreads)
rx_units_write_kernel(const int* __restrict__ rowcnt, int N, int M, int g, const int* __restrict__ btot,
                      int* __restrict__ row_ptr, int4* __restrict__ seg_units, int4* __restrict__ row_units,
                      int4* __restrict__ finish, int* __restrict__ counters)
{
    __shared__ int ws[6 * (kRxUnitThreads / 32 + 1)];
    __shared__ int sbase[6], sgrand[7];
    const int tid = threadIdx.x;
    const int b = blockIdx.x, nblk = static_cast<int>(gridDim.x);
    pdl_launch_dependents();  // the reduce may be launched now; it waits for this grid to finish
    pdl_wait();
    if (counters[kCtrErrIndex]) return;  // the same for every CTA
    const int m = b * kRxUnitThreads + tid;
    const int len = m < M ? rowcnt[m] : 0;
    // every block's totals into shared memory at once (one load per thread),
    // then seven threads sum them
    __shared__ int sb[kRxMaxUnitBlocks * 8];
    if (tid < nblk * 8) sb[tid] = btot[tid];
    __syncthreads();
    if (tid < 7) {
        int pre = 0, all = 0;
        for (int q = 0; q < nblk; ++q) {
            const int x = sb[q * 8 + tid];
            if (tid == 6) {
                all = max(all, x);
            } else {
                all += x;
                if (q < b) pre += x;
            }
        }
        if (tid < 6) sbase[tid] = pre;
        sgrand[tid] = all;
    }
    int v[6];
    rx_row_classes(len, g, v);
    if (m >= M) v[5] = 0;
    int t6[6];
    block_excl_scan_n<kRxUnitThreads, 6>(v, ws, t6);  // synchronises: sbase, sgrand are visible
    if (m < M) {
        const int G = 1 << g;
        row_ptr[m] = sbase[0] + v[0];
        const int nch = (len + kChunk - 1) / kChunk;
        if (nch > G) {
            const int eA = sbase[1] + v[1];
            const int na = (nch + G - 1) >> g;
            finish[sbase[4] + v[4]] = make_int4(m, eA, na, 0);
            for (int q = 0; q < na; ++q) seg_units[eA + q] = make_int4(m, q, eA + q, 0);
        } else if (nch > 1) {
            seg_units[sgrand[1] + sbase[2] + v[2]] = make_int4(m, -1, 0, 0);
        } else if (nch == 1) {
            row_units[sbase[3] + v[3]] = make_int4(m, -1, 0, 0);
        } else {
            row_units[sgrand[3] + sbase[5] + v[5]] = make_int4(m, -1, 0, 0);
        }
        if (m == M - 1) row_ptr[M] = N;
    }
    if (b == 0 && tid < kCtrCount && tid != kCtrErrIndex) {
        const int* G7 = sgrand;
        int x = 0;
        if (tid == kCtrSegs) x = G7[1];
        else if (tid == kCtrLong) x = G7[2];
        else if (tid == kCtrNormal) x = G7[2] + G7[3] + G7[5];
        else if (tid == kCtrHot) x = G7[4];
        else if (tid == kCtrMaxLen) x = G7[6];
        else if (tid == kCtrBig) x = G7[1] + G7[2];
        else if (tid == kCtrShort) x = G7[3];
        else if (tid == kCtrEmpty) x = G7[5];
        counters[tid] = x;
    }
}

// ------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------

bool plan_radix_applies(int64_t N, int64_t M)
{
    return N >= 1 && N < (int64_t(1) << 24) && M >= 1 && M <= 65536;
}

int64_t plan_radix_tiles(int64_t N) { return std::max<int64_t>(1, cdiv(N, kRxTile)); }

int64_t plan_radix_blocks(int64_t M) { return std::max<int64_t>(1, cdiv(M, kRxUnitThreads)); }

det_status launch_plan_radix(const int32_t* idx, int64_t N, int64_t M, int g, const RadixBuffers& b,
                             cudaStream_t st)
{
    if (!plan_radix_applies(N, M)) return DET_ERR_UNSUPPORTED;
    const int n = static_cast<int>(N), ntiles = static_cast<int>(plan_radix_tiles(N));
    const unsigned int um = static_cast<unsigned int>(M);
    const bool two = M > kRxRadix;
    const size_t smem = sizeof(RxScatterShared);
    int sms = 1;
    { const det_status a_ = current_sm_count(&sms); if (a_) return a_; }
    const int cgrid = static_cast<int>(std::min<int64_t>(ntiles, int64_t(sms) * 4));
    const int* no_bad = nullptr;
    int* no_i = nullptr;
    const bool vec_idx = aligned(idx, 16);
    // pass 0: the low byte of idx
    DETR_CUDA(launch_after_previous(vec_idx ? rx_count_kernel<0, true> : rx_count_kernel<0, false>, dim3(cgrid),
                                    dim3(kRxThreads), 0, st, static_cast<const int*>(idx), n, um, b.counts, ntiles,
                                    b.tbad, b.rowcnt, static_cast<int>(M)));
    DETR_LAUNCHED();
    DETR_CUDA(launch_after_previous(rx_offset_kernel, dim3(kRxRadix), dim3(kRxThreads), 0, st, b.counts, ntiles,
                                    b.totals0, static_cast<const int*>(b.tbad), b.counters));
    DETR_LAUNCHED();
    if (two) {
        auto k0 = rx_scatter_kernel<0, false>;
        { const det_status a_ = allow_dynamic_smem(reinterpret_cast<const void*>(k0), smem); if (a_) return a_; }
        DETR_CUDA(launch_after_previous(k0, dim3(ntiles), dim3(kRxThreads), smem, st, static_cast<const int*>(idx), n,
                                        reinterpret_cast<unsigned int*>(b.packed), static_cast<const int*>(b.counts),
                                        static_cast<const int*>(b.totals0), b.lowd, ntiles, no_i,
                                        static_cast<const int*>(b.counters)));
        DETR_LAUNCHED();
        // pass 1: the high byte, from the packed words (16-byte aligned in the workspace)
        DETR_CUDA(launch_after_previous(rx_count_kernel<1, true>, dim3(cgrid), dim3(kRxThreads), 0, st,
                                        static_cast<const int*>(b.packed), n, um, b.counts, ntiles, no_i, no_i, 0));
        DETR_LAUNCHED();
        DETR_CUDA(launch_after_previous(rx_offset_kernel, dim3(kRxRadix), dim3(kRxThreads), 0, st, b.counts, ntiles,
                                        b.totals1, no_bad, no_i));
        DETR_LAUNCHED();
        auto k1 = rx_scatter_kernel<1, true>;
        { const det_status a_ = allow_dynamic_smem(reinterpret_cast<const void*>(k1), smem); if (a_) return a_; }
        DETR_CUDA(launch_after_previous(k1, dim3(ntiles), dim3(kRxThreads), smem, st,
                                        static_cast<const int*>(b.packed), n, reinterpret_cast<unsigned int*>(b.perm),
                                        static_cast<const int*>(b.counts), static_cast<const int*>(b.totals1),
                                        b.lowd, ntiles, b.rowcnt, static_cast<const int*>(b.counters)));
        DETR_LAUNCHED();
    } else {
        auto k0 = rx_scatter_kernel<0, true>;
        { const det_status a_ = allow_dynamic_smem(reinterpret_cast<const void*>(k0), smem); if (a_) return a_; }
        DETR_CUDA(launch_after_previous(k0, dim3(ntiles), dim3(kRxThreads), smem, st, static_cast<const int*>(idx), n,
                                        reinterpret_cast<unsigned int*>(b.perm), static_cast<const int*>(b.counts),
                                        static_cast<const int*>(b.totals0), static_cast<unsigned char*>(nullptr),
                                        ntiles, b.rowcnt, static_cast<const int*>(b.counters)));
        DETR_LAUNCHED();
    }
    const unsigned int nblk = static_cast<unsigned int>(cdiv(M, kRxUnitThreads));
    DETR_CUDA(launch_after_previous(rx_units_count_kernel, dim3(nblk), dim3(kRxUnitThreads), 0, st,
                                    static_cast<const int*>(b.rowcnt), static_cast<int>(M), g, b.btot,
                                    static_cast<const int*>(b.counters)));
    DETR_LAUNCHED();
    DETR_CUDA(launch_after_previous(rx_units_write_kernel, dim3(nblk), dim3(kRxUnitThreads), 0, st,
                                    static_cast<const int*>(b.rowcnt), n, static_cast<int>(M), g,
                                    static_cast<const int*>(b.btot), b.row_ptr, b.seg_units, b.row_units, b.finish,
                                    b.counters));
    DETR_LAUNCHED();
    return DET_OK;
}

}  // namespace detr
