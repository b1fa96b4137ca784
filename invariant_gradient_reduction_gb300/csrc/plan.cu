// plan.cu -- destination lists (CSR) and the reduce work list, multi-kernel
// method (small problems without order keys use one cluster kernel instead,
// plan_cluster.cu).
//
// The terms of destination m are the sources with idx[i] = m in ascending
// order key (src_id[i], default i): the stable (expert id, original token id)
// order the MoE backward sorts by ("DeepSeek-V4 book, Ch 09: Batch invariance
// and determinism", section 3.2).  Everything here is integer work and exact,
// so any correct method gives the same bytes.  This one:
//
//   1-2. per 8-bit digit (the order key's first when given, then the
//        destination's), a stable LSD radix pass in three kernels: digit
//        counts of every tile, their scan over the tiles, and a scatter in
//        which each tile ranks its keys and writes them to their places.  The
//        first destination pass checks idx against M;
//   3.   row_bounds_kernel: the first and one-past-last sorted position of
//        every destination present, from the boundaries of the sorted
//        destinations;
//   4.   the work list, counted per tile of destinations, scanned over the
//        tiles and written: row lengths give row_ptr, and each destination one
//        whole-row unit or (more than 2^g chunks) its segment units and a
//        finish task.
//
// No kernel here waits for another CTA: every cross-tile quantity goes
// through a separate counting kernel and a scan.
#include <algorithm>
#include <new>

#include "block_scan.cuh"
#include "common.cuh"
#include "plan_internal.cuh"

namespace detr {

// Sort tiles: large problems use 4096-key tiles (256 threads x 16 keys, three
// CTAs per SM for 32-bit keys), small ones 1024-key tiles (256 x 4) so that
// more CTAs share the work.
constexpr int kBigThreads = 256, kBigItems = 16;
constexpr int kSmallThreads = 256, kSmallItems = 4;
constexpr int64_t kSmallSortMaxN = 1 << 20;
constexpr int kRadix = 256;
constexpr int kUnitThreads = 256;  // one row per thread
// Auto takes the owner plan up to this many sources (where it applies).
constexpr int64_t kOwnAutoMaxN = int64_t(1) << 17;

enum KeyMode { KM_DIRECT = 0, KM_CARRY = 1, KM_GATHER = 2 };

// ------------------------------------------------------------------------
// keys
// ------------------------------------------------------------------------

template <typename K>
__device__ __forceinline__ K direct_key(const void* kin, long long p);
template <>
__device__ __forceinline__ unsigned int direct_key<unsigned int>(const void* kin, long long p)
{
    return static_cast<unsigned int>(static_cast<const int*>(kin)[p]);
}
template <>
__device__ __forceinline__ unsigned long long direct_key<unsigned long long>(const void* kin, long long p)
{
    // flip the sign bit so that unsigned digit order is signed int64 order
    return static_cast<unsigned long long>(static_cast<const long long*>(kin)[p]) ^ 0x8000000000000000ull;
}

template <typename K, int MODE>
__device__ __forceinline__ void load_kv(const void* kin, const int* vin, const int* gather, long long p,
                                        K& key, int& val)
{
    if (MODE == KM_DIRECT) {
        val = static_cast<int>(p);
        key = direct_key<K>(kin, p);
    } else if (MODE == KM_CARRY) {
        val = vin[p];
        key = static_cast<const K*>(kin)[p];
    } else {
        val = vin[p];
        key = static_cast<K>(static_cast<unsigned int>(gather[val]));
    }
}

template <typename K>
__device__ __forceinline__ int digit_of(K key, int shift)
{
    return static_cast<int>((key >> shift) & static_cast<K>(kRadix - 1));
}

// ------------------------------------------------------------------------
// 1-2. stable radix passes: count, offsets, scatter
// ------------------------------------------------------------------------

// One pass sorts by one 8-bit digit in three kernels; no CTA ever waits for
// another:
//   tile_count_kernel     the digit counts of every tile of the pass's input
//                         order, digit-major (counts[d * ntiles + t]); the
//                         first destination pass also checks idx against M;
//   tile_offset_kernel    one CTA per digit: exclusive scan of the digit's
//                         counts over the tiles (in place) and its total;
//   radix_scatter_kernel  each tile ranks its keys (peers of a digit from
//                         ballots, in element order, warps in order), stages
//                         them in shared memory in (digit, position) order and
//                         writes them to their places: the digit's start, plus
//                         the digit's keys in earlier tiles, plus the rank.
template <typename K, int MODE, int NT, int ITEMS>
__global__ void __launch_bounds__(NT)
tile_count_kernel(const void* kin, const int* vin, const int* gather, long long N, int shift, long long M_check,
                  int* counts, int ntiles, int* counters)
{
    __shared__ int h[kRadix];
    for (int i = threadIdx.x; i < kRadix; i += NT) h[i] = 0;
    __syncthreads();
    const long long base = static_cast<long long>(blockIdx.x) * NT * ITEMS;
    bool bad = false;
    K key[ITEMS];
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {  // all loads in flight first
        const long long p = base + static_cast<long long>(k) * NT + threadIdx.x;
        key[k] = 0;
        if (p < N) {
            int val;
            load_kv<K, MODE>(kin, vin, gather, p, key[k], val);
        }
    }
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        if (base + static_cast<long long>(k) * NT + threadIdx.x < N) {
            if (M_check > 0 && static_cast<long long>(key[k]) >= M_check) bad = true;
            atomicAdd(&h[digit_of<K>(key[k], shift)], 1);
        }
    }
    if (M_check > 0 && __syncthreads_or(bad) && threadIdx.x == 0) atomicOr(&counters[kCtrErrIndex], 1);
    __syncthreads();
    for (int i = threadIdx.x; i < kRadix; i += NT) counts[static_cast<long long>(i) * ntiles + blockIdx.x] = h[i];
}

constexpr int kOffThreads = 256;
constexpr int kOffItems = 4;

__global__ void __launch_bounds__(kOffThreads)
tile_offset_kernel(int* counts, int ntiles, int* totals)
{
    __shared__ int ws[kOffThreads / 32 + 1];
    int* row = counts + static_cast<long long>(blockIdx.x) * ntiles;
    int carry = 0;
    for (int t0 = 0; t0 < ntiles; t0 += kOffThreads * kOffItems) {
        int v[kOffItems];
        int sum = 0;
#pragma unroll
        for (int j = 0; j < kOffItems; ++j) {
            const int t = t0 + threadIdx.x * kOffItems + j;
            v[j] = t < ntiles ? row[t] : 0;
            sum += v[j];
        }
        int tot;
        int run = carry + block_excl_scan<kOffThreads>(sum, ws, &tot);
#pragma unroll
        for (int j = 0; j < kOffItems; ++j) {
            const int t = t0 + threadIdx.x * kOffItems + j;
            if (t < ntiles) row[t] = run;
            run += v[j];
        }
        carry += tot;
    }
    if (threadIdx.x == 0) totals[blockIdx.x] = carry;
}

// Warp w owns elements [w*32*ITEMS, (w+1)*32*ITEMS) of the tile, item k of
// lane l being element w*32*ITEMS + k*32 + l.
template <typename K, int MODE, int NT, int ITEMS, bool WRITE_KEYS>
__global__ void __launch_bounds__(NT, sizeof(K) == 4 ? 3 : 2)  // three 32-bit-key tiles per SM
radix_scatter_kernel(const void* kin, const int* vin, const int* gather, K* kout, int* vout, const int* offsets,
                     const int* totals, int ntiles, long long N, int shift)
{
    constexpr int W = NT / 32;
    constexpr int TILE = NT * ITEMS;
    extern __shared__ __align__(16) unsigned char smem[];
    K* skeys = reinterpret_cast<K*>(smem);
    int* svals = reinterpret_cast<int*>(skeys + TILE);
    int* whist = svals + TILE;                // [W][kRadix]
    int* tstart = whist + W * kRadix;
    int* gbase = tstart + kRadix;
    int* ws = gbase + kRadix;                 // scan scratch (NT/32 + 1)

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tile = blockIdx.x;
    const long long base = static_cast<long long>(tile) * TILE;
    for (int i = threadIdx.x; i < W * kRadix; i += NT) whist[i] = 0;
    const int tot_d = threadIdx.x < kRadix ? totals[threadIdx.x] : 0;
    const int off_d = threadIdx.x < kRadix ? offsets[static_cast<long long>(threadIdx.x) * ntiles + tile] : 0;
    unsigned int lt;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));

    K key[ITEMS];
    int val[ITEMS];
    int rank[ITEMS];
    const long long wbase = base + static_cast<long long>(warp) * 32 * ITEMS;  // item k of lane l: wbase + k*32 + l
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {  // all loads first
        const long long p = wbase + k * 32 + lane;
        key[k] = 0;
        val[k] = 0;
        if (p < N) load_kv<K, MODE>(kin, vin, gather, p, key[k], val[k]);
    }
    int total_unused;
    const int dstart = block_excl_scan<NT>(tot_d, ws, &total_unused);  // also orders the whist zeroing
    if (threadIdx.x < kRadix) gbase[threadIdx.x] = dstart + off_d;

    // rank inside the warp: every lane reads its digit's running count, the
    // lowest lane of each digit group writes it back
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const long long nl = N - (wbase + k * 32);
        const unsigned int live = nl >= 32 ? 0xffffffffu : (nl <= 0 ? 0u : (1u << nl) - 1u);
        if (live == 0u) continue;  // uniform over the warp
        const bool valid = (live >> lane) & 1u;
        const int d = digit_of<K>(key[k], shift);
        const unsigned int peers = digit_peers(d, live);
        const int old = whist[warp * kRadix + d];
        rank[k] = old + __popc(peers & lt);
        __syncwarp();
        if (valid && (peers & lt) == 0u) whist[warp * kRadix + d] = old + __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // per digit: offsets of the warps (warp order), tile counts, staged starts
    int tot = 0;
    if (threadIdx.x < kRadix) {
        const int d = threadIdx.x;
        for (int w = 0; w < W; ++w) {
            const int c = whist[w * kRadix + d];
            whist[w * kRadix + d] = tot;
            tot += c;
        }
    }
    const int excl = block_excl_scan<NT>(tot, ws, &total_unused);
    if (threadIdx.x < kRadix) {
        tstart[threadIdx.x] = excl;
        gbase[threadIdx.x] -= excl;  // staged position i of digit d goes to gbase[d] + i
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        if (wbase + k * 32 + lane < N) {
            const int dk = digit_of<K>(key[k], shift);
            const int pos = tstart[dk] + whist[warp * kRadix + dk] + rank[k];
            skeys[pos] = key[k];
            svals[pos] = val[k];
        }
    }
    __syncthreads();

    const long long rem = N - base;
    const int nvalid = rem < TILE ? static_cast<int>(rem) : TILE;
    for (int i = threadIdx.x; i < nvalid; i += NT) {
        const K kk = skeys[i];
        const long long g = static_cast<long long>(gbase[digit_of<K>(kk, shift)]) + i;  // in [0, N)
        if (WRITE_KEYS) kout[g] = kk;
        vout[g] = svals[i];
    }
}

template <typename K, int NT, int ITEMS>
static size_t pass_smem_bytes()
{
    return static_cast<size_t>(NT * ITEMS) * (sizeof(K) + sizeof(int)) +
           static_cast<size_t>((NT / 32) * kRadix + 2 * kRadix + NT / 32 + 1) * sizeof(int);
}

// Sources of one destination must carry distinct order keys.
__global__ void dup_key_kernel(const int* skeys, const int* perm, const long long* src_id, long long N, int* counters)
{
    const long long p = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x + 1;
    if (p >= N) return;
    if (skeys[p] == skeys[p - 1] && src_id[perm[p]] == src_id[perm[p - 1]]) atomicOr(&counters[kCtrErrDup], 1);
}

// ------------------------------------------------------------------------
// 3. row_ptr and the work list
// ------------------------------------------------------------------------

// Marks the sorted run of every destination present: rstart[k] = its first
// position, rend[k] = one past its last (both stay 0 for an absent one).
// kBoundItems positions per thread, all loads in flight.
constexpr int kBoundItems = 4;

__global__ void __launch_bounds__(kUnitThreads)
row_bounds_kernel(const int* skeys, long long N, long long M, int* rstart, int* rend, const int* counters)
{
    if (counters[kCtrErrIndex]) return;  // keys may be out of range
    const long long base = static_cast<long long>(blockIdx.x) * kUnitThreads * kBoundItems + threadIdx.x;
    int k[kBoundItems], prev[kBoundItems], next[kBoundItems];
#pragma unroll
    for (int j = 0; j < kBoundItems; ++j) {
        const long long p = base + static_cast<long long>(j) * kUnitThreads;
        k[j] = p < N ? skeys[p] : -1;
        prev[j] = p > 0 && p < N ? skeys[p - 1] : -1;
        next[j] = p + 1 < N ? skeys[p + 1] : -1;
    }
#pragma unroll
    for (int j = 0; j < kBoundItems; ++j) {
        const long long p = base + static_cast<long long>(j) * kUnitThreads;
        if (p >= N || k[j] < 0 || k[j] >= M) continue;
        if (prev[j] != k[j]) rstart[k[j]] = static_cast<int>(p);
        if (next[j] != k[j]) rend[k[j]] = static_cast<int>(p + 1);
    }
}

// The work list in three kernels (no CTA waits for another), over tiles of
// kUnitThreads destinations, one per thread:
//   units_count_kernel  each tile's totals: sources (row lengths), hot
//                       segments, long, short and empty whole-row units,
//                       finish tasks; and the longest list;
//   units_scan_kernel   one CTA: exclusive scans of the six totals over the
//                       tiles, and the grand totals into the counter block;
//   units_write_kernel  row_ptr, and the units: hot rows (more than 2^g
//                       chunks) give `seg` segment units and one finish task,
//                       rows of 2..2^g chunks a long whole-row unit (listed
//                       after the segments), the others a short one (empty
//                       destinations after the ones with terms).
constexpr int kUnitVals = 6;  // sources, segments, long rows, short rows, finish tasks, empty rows

struct RowClass {
    int v[kUnitVals];
};

__device__ __forceinline__ RowClass classify_row(const int* rstart, const int* rend, long long m, long long M, int g)
{
    RowClass r{{0, 0, 0, 0, 0, 0}};
    if (m < M) {
        r.v[0] = rend[m] - rstart[m];
        const int nch = (r.v[0] + kChunk - 1) / kChunk;
        if (nch > (1 << g)) {
            r.v[1] = (nch + (1 << g) - 1) >> g;
            r.v[4] = 1;
        } else if (nch > 1) {
            r.v[2] = 1;
        } else if (nch == 1) {
            r.v[3] = 1;
        } else {
            r.v[5] = 1;
        }
    }
    return r;
}

__global__ void __launch_bounds__(kUnitThreads)
units_count_kernel(const int* rstart, const int* rend, long long M, int g, int* tile_tot, int* counters)
{
    __shared__ int ws[kUnitThreads / 32 + 1];
    if (counters[kCtrErrIndex]) return;
    const long long m = static_cast<long long>(blockIdx.x) * kUnitThreads + threadIdx.x;
    const RowClass r = classify_row(rstart, rend, m, M, g);
    const int mx = __reduce_max_sync(0xffffffffu, r.v[0]);
    if ((threadIdx.x & 31) == 0 && mx > 0) atomicMax(&counters[kCtrMaxLen], mx);
#pragma unroll
    for (int j = 0; j < kUnitVals; ++j) {
        int t;
        block_excl_scan<kUnitThreads>(r.v[j], ws, &t);
        if (threadIdx.x == 0) tile_tot[static_cast<long long>(blockIdx.x) * kUnitVals + j] = t;
    }
}

constexpr int kUnitScanThreads = 1024;

__global__ void __launch_bounds__(kUnitScanThreads)
units_scan_kernel(int* tile_tot, int nut, int* counters)
{
    __shared__ int ws[kUnitScanThreads / 32 + 1];
    if (counters[kCtrErrIndex]) return;
    int carry[kUnitVals] = {0, 0, 0, 0, 0, 0};
    for (int t0 = 0; t0 < nut; t0 += kUnitScanThreads) {
        const int t = t0 + threadIdx.x;
#pragma unroll
        for (int j = 0; j < kUnitVals; ++j) {
            int* slot = tile_tot + static_cast<long long>(t) * kUnitVals + j;
            const int v = t < nut ? *slot : 0;
            int tot;
            const int e = block_excl_scan<kUnitScanThreads>(v, ws, &tot);
            if (t < nut) *slot = carry[j] + e;
            carry[j] += tot;
        }
    }
    if (threadIdx.x == 0) {
        counters[kCtrSegs] = carry[1];
        counters[kCtrLong] = carry[2];
        counters[kCtrNormal] = carry[2] + carry[3] + carry[5];
        counters[kCtrHot] = carry[4];
        counters[kCtrBig] = carry[1] + carry[2];
        counters[kCtrShort] = carry[3];
        counters[kCtrEmpty] = carry[5];
    }
}

__global__ void __launch_bounds__(kUnitThreads)
units_write_kernel(const int* rstart, const int* rend, long long N, long long M, int g, const int* tile_off,
                   int* row_ptr, int4* seg_units, int4* row_units, int4* finish, const int* counters)
{
    __shared__ int ws[kUnitThreads / 32 + 1];
    pdl_launch_dependents();  // the reduce may be launched now; it waits for this grid to finish
    if (counters[kCtrErrIndex]) return;
    const long long m = static_cast<long long>(blockIdx.x) * kUnitThreads + threadIdx.x;
    const RowClass r = classify_row(rstart, rend, m, M, g);
    int e[kUnitVals];
#pragma unroll
    for (int j = 0; j < kUnitVals; ++j) {
        int unused;
        e[j] = tile_off[static_cast<long long>(blockIdx.x) * kUnitVals + j] +
               block_excl_scan<kUnitThreads>(r.v[j], ws, &unused);
    }
    if (m < M) {
        row_ptr[m] = e[0];
        if (r.v[4]) {
            finish[e[4]] = make_int4(static_cast<int>(m), e[1], r.v[1], 0);
            for (int s = 0; s < r.v[1]; ++s) seg_units[e[1] + s] = make_int4(static_cast<int>(m), s, e[1] + s, 0);
        } else if (r.v[2]) {
            seg_units[counters[kCtrSegs] + e[2]] = make_int4(static_cast<int>(m), -1, 0, 0);
        } else if (r.v[3]) {
            row_units[e[3]] = make_int4(static_cast<int>(m), -1, 0, 0);
        } else {
            row_units[counters[kCtrShort] + e[5]] = make_int4(static_cast<int>(m), -1, 0, 0);
        }
    }
    if (m == M - 1) row_ptr[M] = static_cast<int>(N);
}

// ------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------

struct PlanLayout {
    // zeroed at the start of every multi-kernel plan: counters, row_ptr and
    // the destinations' run bounds
    size_t counters, row_ptr, rstart, rend, zero_end;
    size_t utot;
    size_t counts, totals, perm, skeys, k32_tmp, v_tmp, k64_a, k64_b, va, vb, seg_units, row_units, finish, rx_tbad, rx_tot1, rx_btot, total;
    int ntiles, nut, npass;
    int64_t max_segs, max_rows, max_finish;
};

static int sort_tile(int64_t N)
{
    return N <= kSmallSortMaxN ? kSmallThreads * kSmallItems : kBigThreads * kBigItems;
}

static int bit_length(int64_t v)
{
    int b = 0;
    while (v > 0) { ++b; v >>= 1; }
    return b;
}

static int dest_passes(int64_t M) { return (std::max(1, bit_length(M - 1)) + 7) / 8; }

static PlanLayout plan_layout(int64_t N, int64_t M, bool with_src, int g)
{
    PlanLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + (bytes ? bytes : 1), 256);
        return at;
    };
    L.ntiles = static_cast<int>(std::max<int64_t>(1, cdiv(N, sort_tile(N))));
    L.nut = static_cast<int>(std::max<int64_t>(1, cdiv(M, kUnitThreads)));
    L.npass = dest_passes(M) + (with_src ? 8 : 0);
    const int64_t seg_terms = static_cast<int64_t>(kChunk) << g;
    L.max_finish = cdiv(N, seg_terms) + 1;
    L.max_segs = 2 * cdiv(N, seg_terms) + 1 + std::min<int64_t>(M, N / (kChunk + 1) + 1);  // + long rows
    L.max_rows = M + 1;
    L.counters = take(kCtrCount * sizeof(int));
    L.row_ptr = take(static_cast<size_t>(M + 1) * sizeof(int));
    L.rstart = take(static_cast<size_t>(M) * sizeof(int));
    L.rend = take(static_cast<size_t>(M) * sizeof(int));
    L.zero_end = off;
    L.utot = take(static_cast<size_t>(L.nut) * kUnitVals * sizeof(int));
    L.counts = take(static_cast<size_t>(kRadix) * L.ntiles * sizeof(int));
    L.totals = take(static_cast<size_t>(kRadix) * sizeof(int));
    L.perm = take(static_cast<size_t>(N) * sizeof(int));
    L.skeys = take(static_cast<size_t>(N) * sizeof(int));
    L.k32_tmp = take(static_cast<size_t>(N) * sizeof(int));
    L.v_tmp = take(static_cast<size_t>(N) * sizeof(int));
    if (with_src) {
        L.k64_a = take(static_cast<size_t>(N) * 8);
        L.k64_b = take(static_cast<size_t>(N) * 8);
        L.va = take(static_cast<size_t>(N) * sizeof(int));
        L.vb = take(static_cast<size_t>(N) * sizeof(int));
    }
    L.seg_units = take(static_cast<size_t>(L.max_segs) * sizeof(int4));
    L.row_units = take(static_cast<size_t>(L.max_rows) * sizeof(int4));
    L.finish = take(static_cast<size_t>(L.max_finish) * sizeof(int4));
    L.rx_tbad = take(static_cast<size_t>(plan_radix_tiles(N)) * sizeof(int));
    L.rx_tot1 = take(static_cast<size_t>(kRadix) * sizeof(int));
    L.rx_btot = take(static_cast<size_t>(plan_radix_blocks(M)) * 8 * sizeof(int));
    L.total = off;
    return L;
}

static det_status counter_status(const int* h)
{
    if (h[kCtrErrIndex]) return DET_ERR_INDEX_RANGE;
    if (h[kCtrErrTimeout]) return DET_ERR_TIMEOUT;
    if (h[kCtrErrDup]) return DET_ERR_ORDER_KEY;
    return DET_OK;
}

static void set_counts(det_plan_s* p, const int* h)
{
    p->n_segments = h[kCtrSegs];
    p->n_units = static_cast<int64_t>(h[kCtrSegs]) + h[kCtrNormal];
    p->n_hot_rows = h[kCtrHot];
    p->max_row_len = h[kCtrMaxLen];
    p->n_long = h[kCtrLong];
    p->n_empty = h[kCtrEmpty];
}

static det_status resolve_seg_log2(const det_opts* o, int* g)
{
    *g = kDefaultSegLog2;
    if (o && o->seg_chunks_log2 >= 0) {
        if (o->seg_chunks_log2 < kMinSegLog2 || o->seg_chunks_log2 > kMaxSegLog2) return DET_ERR_ARG;
        *g = o->seg_chunks_log2;
    }
    return DET_OK;
}

template <typename K, int MODE, int NT, int ITEMS, bool WRITE_KEYS>
static det_status radix_pass_t(const void* kin, const int* vin, const int* gather, K* kout, int* vout, int* counts,
                               int* totals, int64_t N, int ntiles, int shift, int64_t M_check, int* counters,
                               cudaStream_t st)
{
    tile_count_kernel<K, MODE, NT, ITEMS><<<ntiles, NT, 0, st>>>(kin, vin, gather, N, shift, M_check, counts, ntiles,
                                                                 counters);
    DETR_LAUNCHED();
    tile_offset_kernel<<<kRadix, kOffThreads, 0, st>>>(counts, ntiles, totals);
    DETR_LAUNCHED();
    const size_t smem = pass_smem_bytes<K, NT, ITEMS>();
    auto kern = radix_scatter_kernel<K, MODE, NT, ITEMS, WRITE_KEYS>;
    { const det_status a_ = allow_dynamic_smem(reinterpret_cast<const void*>(kern), smem); if (a_) return a_; }
    kern<<<ntiles, NT, smem, st>>>(kin, vin, gather, kout, vout, counts, totals, ntiles, N, shift);
    DETR_LAUNCHED();
    return DET_OK;
}

template <typename K, int MODE, bool WRITE_KEYS>
static det_status radix_pass(bool small, const void* kin, const int* vin, const int* gather, K* kout, int* vout,
                             int* counts, int* totals, int64_t N, int ntiles, int shift, int64_t M_check,
                             int* counters, cudaStream_t st)
{
    if (small)
        return radix_pass_t<K, MODE, kSmallThreads, kSmallItems, WRITE_KEYS>(kin, vin, gather, kout, vout, counts,
                                                                             totals, N, ntiles, shift, M_check,
                                                                             counters, st);
    return radix_pass_t<K, MODE, kBigThreads, kBigItems, WRITE_KEYS>(kin, vin, gather, kout, vout, counts, totals, N,
                                                                     ntiles, shift, M_check, counters, st);
}

}  // namespace detr

using namespace detr;

extern "C" {

det_status det_plan_workspace_size(int64_t N, int64_t M, int32_t with_src_id, const det_opts* opts,
                                   size_t* bytes)
{
    if (!bytes || N < 0 || M < 0) return DET_ERR_ARG;
    if (N > kMaxRows || M > kMaxRows) return DET_ERR_UNSUPPORTED;
    int g;
    det_status s = resolve_seg_log2(opts, &g);
    if (s) return s;
    *bytes = plan_layout(N, M, with_src_id != 0, g).total;
    return DET_OK;
}

det_status det_reduce_plan(const int32_t* idx, const int64_t* src_id, int64_t N, int64_t M, void* workspace,
                           size_t ws_bytes, const det_opts* opts, void* stream, det_plan* out_plan)
{
    if (!out_plan) return DET_ERR_ARG;
    *out_plan = nullptr;
    if (N < 0 || M < 0) return DET_ERR_ARG;
    if (N > kMaxRows || M > kMaxRows) return DET_ERR_UNSUPPORTED;
    if (N > 0 && !idx) return DET_ERR_ARG;
    if (!aligned(idx, 4) || !aligned(src_id, 8)) return DET_ERR_ARG;
    int g;
    det_status s = resolve_seg_log2(opts, &g);
    if (s) return s;
    if (opts && (opts->plan_path < 0 || opts->plan_path > 4 || opts->reserved[0])) return DET_ERR_ARG;
    const bool with_src = src_id != nullptr && N > 0;
    const PlanLayout L = plan_layout(N, M, with_src, g);
    if (!workspace || !aligned(workspace, 256) || ws_bytes < L.total) return DET_ERR_WORKSPACE;
    if (overlaps(workspace, ws_bytes, idx, static_cast<size_t>(N) * 4) ||
        overlaps(workspace, ws_bytes, src_id, src_id ? static_cast<size_t>(N) * 8 : 0))
        return DET_ERR_ARG;
    if (N > 0 && M == 0) return DET_ERR_INDEX_RANGE;

    cudaStream_t st = as_stream(stream);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    int* counters = reinterpret_cast<int*>(ws + L.counters);
    int* row_ptr = reinterpret_cast<int*>(ws + L.row_ptr);
    int* counts = reinterpret_cast<int*>(ws + L.counts);
    int* totals = reinterpret_cast<int*>(ws + L.totals);
    int* perm = reinterpret_cast<int*>(ws + L.perm);
    int* skeys = reinterpret_cast<int*>(ws + L.skeys);
    int* k32_tmp = reinterpret_cast<int*>(ws + L.k32_tmp);
    int* v_tmp = reinterpret_cast<int*>(ws + L.v_tmp);
    int4* seg_units = reinterpret_cast<int4*>(ws + L.seg_units);
    int4* row_units = reinterpret_cast<int4*>(ws + L.row_units);
    int4* finish = reinterpret_cast<int4*>(ws + L.finish);

    const int np32 = dest_passes(M);
    const int plan_path = opts ? opts->plan_path : 0;
    bool one_kernel_set = false;  // a single-cluster or owner plan was enqueued
    if ((plan_path == 0 || plan_path == 3) && !with_src && N > 0 && (plan_path == 3 || N <= kOwnAutoMaxN)) {
        s = launch_plan_owner(idx, N, M, g, row_ptr, perm, seg_units, row_units, finish, counters, st,
                              &one_kernel_set);
        if (s) return s;
        if (plan_path == 3 && !one_kernel_set) return DET_ERR_UNSUPPORTED;
    }
    const bool owner_plan = one_kernel_set;
    bool cluster_late = false;  // the two-pass cluster kernel, which releases the reduce for its last phase
    if (plan_path == 3 && (with_src || N == 0)) return DET_ERR_UNSUPPORTED;
    if (!one_kernel_set && (plan_path == 0 || plan_path == 2) && !with_src && N > 0) {
        // Auto takes the two-pass cluster kernel only up to 65536 sources: after
        // it, on a 131072-source, 16384-destination plan, the reduce ran ~70 us
        // longer than after the multi-kernel plan, more than the 15 us the plan
        // itself saves; on a 32768-source, 131072-destination plan it saved 35 us.
        const bool two_pass = plan_path == 2 || N <= (int64_t(1) << 16);
        s = launch_plan_cluster(idx, N, M, g, np32, row_ptr, perm, seg_units, row_units, finish, counters,
                                two_pass, st, &one_kernel_set);
        if (s) return s;
        cluster_late = two_pass && one_kernel_set;
        if (plan_path == 2 && !one_kernel_set) return DET_ERR_UNSUPPORTED;
    }
    if (plan_path == 2 && !one_kernel_set) return DET_ERR_UNSUPPORTED;
    if (!one_kernel_set && (plan_path == 0 || plan_path == 4) && !with_src && plan_radix_applies(N, M)) {
        RadixBuffers rb{};
        rb.counts = counts;
        rb.tbad = reinterpret_cast<int*>(ws + L.rx_tbad);
        rb.totals0 = totals;
        rb.totals1 = reinterpret_cast<int*>(ws + L.rx_tot1);
        rb.packed = reinterpret_cast<int*>(ws + L.k32_tmp);
        rb.lowd = ws + L.skeys;  // 4N bytes, unused by this method
        rb.perm = perm;
        rb.rowcnt = reinterpret_cast<int*>(ws + L.rstart);
        rb.btot = reinterpret_cast<int*>(ws + L.rx_btot);
        rb.row_ptr = row_ptr;
        rb.seg_units = seg_units;
        rb.row_units = row_units;
        rb.finish = finish;
        rb.counters = counters;
        s = launch_plan_radix(idx, N, M, g, rb, st);
        if (s) return s;
        one_kernel_set = true;
    }
    if (plan_path == 4 && !one_kernel_set) return DET_ERR_UNSUPPORTED;
    const bool one_cluster = one_kernel_set;
    if (!one_cluster) {
    DETR_CUDA(cudaMemsetAsync(ws, 0, L.zero_end, st));

    if (N > 0) {
        const int ntiles = L.ntiles;
        const bool small = N <= kSmallSortMaxN;
        const int64_t noM = 0;  // no range check in this pass
        const int* vals_in = nullptr;
        if (with_src) {
            unsigned long long* k64[2] = {reinterpret_cast<unsigned long long*>(ws + L.k64_a),
                                          reinterpret_cast<unsigned long long*>(ws + L.k64_b)};
            int* v64[2] = {reinterpret_cast<int*>(ws + L.va), reinterpret_cast<int*>(ws + L.vb)};
            for (int j = 0; j < 8; ++j) {
                const int o = j & 1;
                if (j == 0)
                    s = radix_pass<unsigned long long, KM_DIRECT, true>(small, src_id, nullptr, nullptr, k64[o], v64[o],
                                                                        counts, totals, N, ntiles, 0, noM, counters,
                                                                        st);
                else
                    s = radix_pass<unsigned long long, KM_CARRY, true>(small, k64[o ^ 1], v64[o ^ 1], nullptr, k64[o],
                                                                       v64[o], counts, totals, N, ntiles, 8 * j, noM,
                                                                       counters, st);
                if (s) return s;
            }
            vals_in = v64[1];
        }
        // destination passes; the first checks idx against M, the last writes
        // the sorted destinations, where the work list finds row_ptr
        for (int j = 0; j < np32; ++j) {
            const bool to_final = ((np32 - 1 - j) % 2) == 0;
            unsigned int* ko = reinterpret_cast<unsigned int*>(to_final ? skeys : k32_tmp);
            int* vo = to_final ? perm : v_tmp;
            const unsigned int* ki = reinterpret_cast<const unsigned int*>(to_final ? k32_tmp : skeys);
            const int* vi = to_final ? v_tmp : perm;
            if (j == 0 && with_src)
                s = radix_pass<unsigned int, KM_GATHER, true>(small, nullptr, vals_in, idx, ko, vo, counts, totals, N,
                                                              ntiles, 0, M, counters, st);
            else if (j == 0)
                s = radix_pass<unsigned int, KM_DIRECT, true>(small, idx, nullptr, nullptr, ko, vo, counts, totals, N,
                                                              ntiles, 0, M, counters, st);
            else
                s = radix_pass<unsigned int, KM_CARRY, true>(small, ki, vi, nullptr, ko, vo, counts, totals, N, ntiles,
                                                             8 * j, noM, counters, st);
            if (s) return s;
        }
        if (with_src && N > 1) {
            dup_key_kernel<<<static_cast<unsigned int>(cdiv(N - 1, 256)), 256, 0, st>>>(
                skeys, perm, reinterpret_cast<const long long*>(src_id), N, counters);
            DETR_LAUNCHED();
        }
    }
    if (M > 0) {
        int* rstart = reinterpret_cast<int*>(ws + L.rstart);
        int* rend = reinterpret_cast<int*>(ws + L.rend);
        if (N > 0) {
            const unsigned int bgrid = static_cast<unsigned int>(cdiv(N, int64_t(kUnitThreads) * kBoundItems));
            row_bounds_kernel<<<bgrid, kUnitThreads, 0, st>>>(skeys, N, M, rstart, rend, counters);
            DETR_LAUNCHED();
        }
        int* tile_tot = reinterpret_cast<int*>(ws + L.utot);
        units_count_kernel<<<L.nut, kUnitThreads, 0, st>>>(rstart, rend, M, g, tile_tot, counters);
        DETR_LAUNCHED();
        units_scan_kernel<<<1, kUnitScanThreads, 0, st>>>(tile_tot, L.nut, counters);
        DETR_LAUNCHED();
        units_write_kernel<<<L.nut, kUnitThreads, 0, st>>>(rstart, rend, N, M, g, tile_tot, row_ptr, seg_units,
                                                           row_units, finish, counters);
        DETR_LAUNCHED();
    }
    }  // multi-kernel plan
    const bool async = opts && opts->async_plan;
    int h[kCtrCount] = {};
    if (!async) {
        DETR_CUDA(cudaMemcpyAsync(h, counters, sizeof(h), cudaMemcpyDeviceToHost, st));
        DETR_CUDA(cudaStreamSynchronize(st));
        const det_status e = counter_status(h);
        if (e) return e;
    }

    det_plan_s* p = new (std::nothrow) det_plan_s();
    if (!p) return DET_ERR_ARG;
    p->N = N;
    p->M = M;
    p->g = g;
    p->ws = ws;
    p->ws_bytes = ws_bytes;
    p->counters = counters;
    p->row_ptr = row_ptr;
    p->perm = perm;
    p->seg_units = seg_units;
    p->row_units = row_units;
    p->finish = finish;
    p->late_release = owner_plan || cluster_late;
    if (async) {
        p->counts_on_host = false;
        p->n_segments = p->n_units = p->n_hot_rows = p->max_row_len = p->n_long = p->n_empty = -1;
    } else {
        set_counts(p, h);
    }
    *out_plan = p;
    return DET_OK;
}

det_status det_plan_status(det_plan plan, void* stream)
{
    if (!plan) return DET_ERR_ARG;
    if (plan->counts_on_host) return DET_OK;
    int h[kCtrCount];
    cudaStream_t st = as_stream(stream);
    DETR_CUDA(cudaMemcpyAsync(h, plan->counters, sizeof(h), cudaMemcpyDeviceToHost, st));
    DETR_CUDA(cudaStreamSynchronize(st));
    const det_status e = counter_status(h);
    if (e) return e;
    set_counts(plan, h);
    plan->counts_on_host = true;
    return DET_OK;
}

det_status det_plan_destroy(det_plan plan)
{
    delete plan;
    return DET_OK;
}

det_status det_plan_describe(det_plan plan, det_plan_desc* d)
{
    if (!plan || !d) return DET_ERR_ARG;
    d->N = plan->N;
    d->M = plan->M;
    d->seg_chunks_log2 = plan->g;
    d->reserved = 0;
    d->row_ptr = plan->row_ptr;
    d->perm = plan->perm;
    d->n_units = plan->n_units;
    d->n_segments = plan->n_segments;
    d->n_hot_rows = plan->n_hot_rows;
    d->max_row_len = plan->max_row_len;
    return DET_OK;
}

}  // extern "C"
