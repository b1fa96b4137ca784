// plan.cu -- destination lists (CSR) and the reduce work list.
//
// The terms of destination m are the sources with idx[i] = m in ascending
// order key (src_id[i], default i): the stable (expert id, original token id)
// order the MoE backward sorts by ("DeepSeek-V4 book, Ch 09: Batch invariance
// and determinism", section 3.2).  Everything here is integer work and exact,
// so any correct method gives the same bytes; this one is a stable LSD radix
// sort in 8-bit digits (order keys first when given, then the destination),
// followed by a boundary pass that writes row_ptr and a three-phase scan that
// writes the work list.  No kernel waits on another CTA.
#include <algorithm>
#include <new>

#include "common.cuh"
#include "plan_internal.cuh"

namespace detr {

constexpr int kSortThreads = 512;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kItems = 16;
constexpr int kTile = kSortThreads * kItems;  // keys per sort tile
constexpr int kRadix = 256;
constexpr int kUnitThreads = 256;
constexpr int kUnitRowsPerThread = 16;
constexpr int kUnitTile = kUnitThreads * kUnitRowsPerThread;

enum KeyMode { KM_DIRECT = 0, KM_CARRY = 1, KM_GATHER = 2 };

// ------------------------------------------------------------------------
// block scans
// ------------------------------------------------------------------------

// Exclusive scan of one int per thread over a block of NT threads; *total gets
// the block sum.  `ws` is shared scratch of NT/32 + 1 ints.  Ends synchronised.
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int* ws, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) ws[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int s = lane < NT / 32 ? ws[lane] : 0;
        int si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(0xffffffffu, si, o);
            if (lane >= o) si += t;
        }
        if (lane < NT / 32) ws[lane] = si - s;
        if (lane == 31) ws[NT / 32] = si;
    }
    __syncthreads();
    int r = incl - v + ws[warp];
    *total = ws[NT / 32];
    __syncthreads();
    return r;
}

// ------------------------------------------------------------------------
// radix sort passes
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

// Per-tile digit histogram; the first destination pass also range-checks idx.
template <typename K, int MODE, bool CHECK>
__global__ void __launch_bounds__(kSortThreads)
radix_count_kernel(const void* kin, const int* vin, const int* gather, int* counts, long long N, int ntiles,
                   int shift, unsigned int M, int* counters)
{
    __shared__ int hist[kRadix];
    for (int d = threadIdx.x; d < kRadix; d += kSortThreads) hist[d] = 0;
    __syncthreads();
    const long long base = static_cast<long long>(blockIdx.x) * kTile;
    bool bad = false;
    for (int i = threadIdx.x; i < kTile; i += kSortThreads) {
        const long long p = base + i;
        if (p >= N) break;
        K key;
        int val;
        load_kv<K, MODE>(kin, vin, gather, p, key, val);
        if (CHECK && static_cast<unsigned long long>(key) >= M) bad = true;
        atomicAdd(&hist[digit_of<K>(key, shift)], 1);
    }
    if (CHECK && __syncthreads_or(bad) && threadIdx.x == 0) atomicOr(&counters[kCtrErrIndex], 1);
    __syncthreads();
    for (int d = threadIdx.x; d < kRadix; d += kSortThreads)
        counts[static_cast<long long>(d) * ntiles + blockIdx.x] = hist[d];
}

// One CTA per digit: exclusive scan of that digit's per-tile counts, in place.
__global__ void __launch_bounds__(256) radix_colscan_kernel(int* counts, int* col_total, int ntiles)
{
    __shared__ int ws[256 / 32 + 1];
    int* row = counts + static_cast<long long>(blockIdx.x) * ntiles;
    int carry = 0;
    for (int base = 0; base < ntiles; base += 256 * 4) {
        const int i0 = base + threadIdx.x * 4;
        int v[4], s = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[k] = i0 + k < ntiles ? row[i0 + k] : 0;
            s += v[k];
        }
        int total;
        int run = carry + block_excl_scan<256>(s, ws, &total);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (i0 + k < ntiles) { row[i0 + k] = run; run += v[k]; }
        carry += total;
    }
    if (threadIdx.x == 0) col_total[blockIdx.x] = carry;
}

// Stable scatter of one tile: ranks inside a warp come from match_any in
// element order, warps are offset per digit in warp order, the tile is staged
// in shared memory in sorted order and written out coalesced.
template <typename K, int MODE>
__global__ void __launch_bounds__(kSortThreads)
radix_scatter_kernel(const void* kin, const int* vin, const int* gather, K* kout, int* vout,
                     const int* counts, const int* col_total, long long N, int ntiles, int shift)
{
    extern __shared__ __align__(16) unsigned char smem[];
    K* skeys = reinterpret_cast<K*>(smem);
    int* svals = reinterpret_cast<int*>(skeys + kTile);
    int* whist = svals + kTile;               // [kSortWarps][kRadix]
    int* tstart = whist + kSortWarps * kRadix;
    int* gbase = tstart + kRadix;
    int* ws = gbase + kRadix;                 // scan scratch

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kSortWarps * kRadix; i += kSortThreads) whist[i] = 0;
    __syncthreads();

    const long long base = static_cast<long long>(blockIdx.x) * kTile;
    unsigned int lt;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));

    K key[kItems];
    int val[kItems];
    int rank[kItems];
    int dig[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const long long p = base + static_cast<long long>(warp) * 32 * kItems + k * 32 + lane;
        const bool valid = p < N;
        int d = kRadix;  // sentinel: invalid lanes only match each other
        if (valid) {
            load_kv<K, MODE>(kin, vin, gather, p, key[k], val[k]);
            d = digit_of<K>(key[k], shift);
        }
        const unsigned int peers = __match_any_sync(0xffffffffu, d);
        const int leader = __ffs(peers) - 1;
        int old = 0;
        if (valid && lane == leader) {
            old = whist[warp * kRadix + d];
            whist[warp * kRadix + d] = old + __popc(peers);
        }
        old = __shfl_sync(0xffffffffu, old, leader);
        rank[k] = old + __popc(peers & lt);
        dig[k] = valid ? d : -1;
        __syncwarp();
    }
    __syncthreads();

    // per digit: offsets of the warps (warp order), tile totals
    int tot = 0;
    if (threadIdx.x < kRadix) {
        const int d = threadIdx.x;
        int run = 0;
        for (int w = 0; w < kSortWarps; ++w) {
            const int c = whist[w * kRadix + d];
            whist[w * kRadix + d] = run;
            run += c;
        }
        tot = run;
    }
    int total_unused;
    const int excl = block_excl_scan<kSortThreads>(tot, ws, &total_unused);
    const int ctot = threadIdx.x < kRadix ? col_total[threadIdx.x] : 0;
    const int dstart = block_excl_scan<kSortThreads>(ctot, ws, &total_unused);
    if (threadIdx.x < kRadix) {
        const int d = threadIdx.x;
        tstart[d] = excl;
        gbase[d] = dstart + counts[static_cast<long long>(d) * ntiles + blockIdx.x] - excl;
    }
    __syncthreads();

#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        if (dig[k] >= 0) {
            const int pos = tstart[dig[k]] + whist[warp * kRadix + dig[k]] + rank[k];
            skeys[pos] = key[k];
            svals[pos] = val[k];
        }
    }
    __syncthreads();

    const long long rem = N - base;
    const int nvalid = rem < kTile ? static_cast<int>(rem) : kTile;
    for (int i = threadIdx.x; i < nvalid; i += kSortThreads) {
        const K kk = skeys[i];
        const long long g = static_cast<long long>(gbase[digit_of<K>(kk, shift)]) + i;
        kout[g] = kk;
        vout[g] = svals[i];
    }
}

template <typename K>
static size_t scatter_smem_bytes()
{
    return static_cast<size_t>(kTile) * (sizeof(K) + sizeof(int)) +
           static_cast<size_t>(kSortWarps * kRadix + 2 * kRadix + kSortThreads / 32 + 1) * sizeof(int);
}

// ------------------------------------------------------------------------
// row_ptr from the sorted destinations; order-key uniqueness
// ------------------------------------------------------------------------

__global__ void row_ptr_kernel(const int* skeys, long long N, long long M, int* row_ptr,
                               const long long* src_id, const int* perm, int* counters)
{
    if (counters[kCtrErrIndex]) return;
    const long long p = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (p > N) return;
    if (p < N) {
        const long long k = skeys[p];
        const long long prev = p == 0 ? -1 : skeys[p - 1];
        for (long long m = prev + 1; m <= k; ++m) row_ptr[m] = static_cast<int>(p);
        if (src_id && p > 0 && prev == k && src_id[perm[p]] == src_id[perm[p - 1]])
            atomicOr(&counters[kCtrErrDup], 1);
    } else {
        const long long last = N == 0 ? -1 : skeys[N - 1];
        for (long long m = last + 1; m <= M; ++m) row_ptr[m] = static_cast<int>(N);
    }
}

// ------------------------------------------------------------------------
// work list: whole destinations, and hot destinations split into segments
// ------------------------------------------------------------------------

struct RowWork {
    int seg;     // hot segments of this row (0 if not hot)
    int normal;  // 1 if the row is one whole unit
    int hot;     // 1 if the row needs a finish task
};

__device__ __forceinline__ RowWork row_work(const int* row_ptr, long long m, int g, int* len)
{
    const int n = row_ptr[m + 1] - row_ptr[m];
    *len = n;
    const int nch = (n + kChunk - 1) / kChunk;
    const int G = 1 << g;
    RowWork r;
    if (nch > G) { r.seg = (nch + G - 1) >> g; r.normal = 0; r.hot = 1; }
    else { r.seg = 0; r.normal = 1; r.hot = 0; }
    return r;
}

__global__ void __launch_bounds__(kUnitThreads)
units_count_kernel(const int* row_ptr, long long M, int g, int* upart, int nut, int* counters)
{
    __shared__ int ws[kUnitThreads / 32 + 1];
    if (counters[kCtrErrIndex]) return;
    const long long m0 = static_cast<long long>(blockIdx.x) * kUnitTile + threadIdx.x * kUnitRowsPerThread;
    int a = 0, b = 0, c = 0, mx = 0;
    for (int k = 0; k < kUnitRowsPerThread; ++k) {
        const long long m = m0 + k;
        if (m >= M) break;
        int len;
        const RowWork r = row_work(row_ptr, m, g, &len);
        a += r.seg; b += r.normal; c += r.hot;
        mx = max(mx, len);
    }
    int ta, tb, tc;
    block_excl_scan<kUnitThreads>(a, ws, &ta);
    block_excl_scan<kUnitThreads>(b, ws, &tb);
    block_excl_scan<kUnitThreads>(c, ws, &tc);
    if (threadIdx.x == 0) {
        upart[blockIdx.x] = ta;
        upart[nut + blockIdx.x] = tb;
        upart[2 * nut + blockIdx.x] = tc;
    }
    if (mx > 0) atomicMax(&counters[kCtrMaxLen], mx);
}

__global__ void __launch_bounds__(1024) units_scan_kernel(int* upart, int nut, int* counters)
{
    __shared__ int ws[1024 / 32 + 1];
    if (counters[kCtrErrIndex]) return;
    for (int arr = 0; arr < 3; ++arr) {
        int* v = upart + arr * nut;
        int carry = 0;
        for (int base = 0; base < nut; base += 1024) {
            const int i = base + threadIdx.x;
            const int x = i < nut ? v[i] : 0;
            int total;
            const int e = block_excl_scan<1024>(x, ws, &total);
            if (i < nut) v[i] = carry + e;
            carry += total;
        }
        if (threadIdx.x == 0) counters[kCtrSegs + arr] = carry;
    }
}

__global__ void __launch_bounds__(kUnitThreads)
units_emit_kernel(const int* row_ptr, long long M, int g, const int* upart, int nut, const int* counters,
                  int4* units, int4* finish)
{
    __shared__ int ws[kUnitThreads / 32 + 1];
    if (counters[kCtrErrIndex]) return;
    const long long m0 = static_cast<long long>(blockIdx.x) * kUnitTile + threadIdx.x * kUnitRowsPerThread;
    int a = 0, b = 0, c = 0;
    for (int k = 0; k < kUnitRowsPerThread; ++k) {
        const long long m = m0 + k;
        if (m >= M) break;
        int len;
        const RowWork r = row_work(row_ptr, m, g, &len);
        a += r.seg; b += r.normal; c += r.hot;
    }
    int t;
    int ao = block_excl_scan<kUnitThreads>(a, ws, &t) + upart[blockIdx.x];
    int bo = block_excl_scan<kUnitThreads>(b, ws, &t) + upart[nut + blockIdx.x] + counters[kCtrSegs];
    int co = block_excl_scan<kUnitThreads>(c, ws, &t) + upart[2 * nut + blockIdx.x];
    for (int k = 0; k < kUnitRowsPerThread; ++k) {
        const long long m = m0 + k;
        if (m >= M) break;
        int len;
        const RowWork r = row_work(row_ptr, m, g, &len);
        if (r.hot) {
            finish[co++] = make_int4(static_cast<int>(m), ao, r.seg, 0);
            for (int s = 0; s < r.seg; ++s) units[ao + s] = make_int4(static_cast<int>(m), s, ao + s, 0);
            ao += r.seg;
        } else {
            units[bo++] = make_int4(static_cast<int>(m), -1, 0, 0);
        }
    }
}

// ------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------

struct PlanLayout {
    size_t row_ptr, perm, skeys, k32_tmp, v_tmp, k64_a, k64_b, va, vb, counts, col_total, units, finish,
        upart, counters, total;
    int ntiles, nut;
    int64_t max_units, max_finish;
};

static PlanLayout plan_layout(int64_t N, int64_t M, bool with_src, int g)
{
    PlanLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + (bytes ? bytes : 1), 256);
        return at;
    };
    L.ntiles = static_cast<int>(std::max<int64_t>(1, cdiv(N, kTile)));
    L.nut = static_cast<int>(std::max<int64_t>(1, cdiv(M, kUnitTile)));
    const int64_t seg_terms = static_cast<int64_t>(kChunk) << g;
    L.max_finish = cdiv(N, seg_terms) + 1;
    L.max_units = M + 2 * cdiv(N, seg_terms) + 1;
    L.counters = take(kCtrCount * sizeof(int));
    L.row_ptr = take(static_cast<size_t>(M + 1) * sizeof(int));
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
    L.counts = take(static_cast<size_t>(kRadix) * L.ntiles * sizeof(int));
    L.col_total = take(kRadix * sizeof(int));
    L.units = take(static_cast<size_t>(L.max_units) * sizeof(int4));
    L.finish = take(static_cast<size_t>(L.max_finish) * sizeof(int4));
    L.upart = take(static_cast<size_t>(3) * L.nut * sizeof(int));
    L.total = off;
    return L;
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

static int bit_length(int64_t v)
{
    int b = 0;
    while (v > 0) { ++b; v >>= 1; }
    return b;
}

template <typename K, int MODE, bool CHECK>
static det_status radix_pass(const void* kin, const int* vin, const int* gather, K* kout, int* vout,
                             int* counts, int* col_total, int64_t N, int ntiles, int shift, int64_t M,
                             int* counters, cudaStream_t st)
{
    radix_count_kernel<K, MODE, CHECK><<<ntiles, kSortThreads, 0, st>>>(
        kin, vin, gather, counts, N, ntiles, shift, static_cast<unsigned int>(M), counters);
    DETR_LAUNCHED();
    radix_colscan_kernel<<<kRadix, 256, 0, st>>>(counts, col_total, ntiles);
    DETR_LAUNCHED();
    const size_t smem = scatter_smem_bytes<K>();
    DETR_CUDA(cudaFuncSetAttribute(radix_scatter_kernel<K, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem)));
    radix_scatter_kernel<K, MODE><<<ntiles, kSortThreads, smem, st>>>(kin, vin, gather, kout, vout, counts,
                                                                    col_total, N, ntiles, shift);
    DETR_LAUNCHED();
    return DET_OK;
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
    int* perm = reinterpret_cast<int*>(ws + L.perm);
    int* skeys = reinterpret_cast<int*>(ws + L.skeys);
    int* k32_tmp = reinterpret_cast<int*>(ws + L.k32_tmp);
    int* v_tmp = reinterpret_cast<int*>(ws + L.v_tmp);
    int* counts = reinterpret_cast<int*>(ws + L.counts);
    int* col_total = reinterpret_cast<int*>(ws + L.col_total);
    int4* units = reinterpret_cast<int4*>(ws + L.units);
    int4* finish = reinterpret_cast<int4*>(ws + L.finish);
    int* upart = reinterpret_cast<int*>(ws + L.upart);

    DETR_CUDA(cudaMemsetAsync(counters, 0, kCtrCount * sizeof(int), st));

    if (N > 0) {
        const int ntiles = L.ntiles;
        const int* vals_in = nullptr;
        if (with_src) {
            unsigned long long* k64[2] = {reinterpret_cast<unsigned long long*>(ws + L.k64_a),
                                          reinterpret_cast<unsigned long long*>(ws + L.k64_b)};
            int* v64[2] = {reinterpret_cast<int*>(ws + L.va), reinterpret_cast<int*>(ws + L.vb)};
            for (int j = 0; j < 8; ++j) {
                const int o = j & 1;
                if (j == 0)
                    s = radix_pass<unsigned long long, KM_DIRECT, false>(src_id, nullptr, nullptr, k64[o], v64[o],
                                                                         counts, col_total, N, ntiles, 0, M,
                                                                         counters, st);
                else
                    s = radix_pass<unsigned long long, KM_CARRY, false>(k64[o ^ 1], v64[o ^ 1], nullptr, k64[o],
                                                                        v64[o], counts, col_total, N, ntiles,
                                                                        8 * j, M, counters, st);
                if (s) return s;
            }
            vals_in = v64[1];
        }
        const int np32 = (std::max(1, bit_length(M - 1)) + 7) / 8;
        for (int j = 0; j < np32; ++j) {
            const bool to_final = ((np32 - 1 - j) % 2) == 0;
            unsigned int* ko = reinterpret_cast<unsigned int*>(to_final ? skeys : k32_tmp);
            int* vo = to_final ? perm : v_tmp;
            const unsigned int* ki = reinterpret_cast<const unsigned int*>(to_final ? k32_tmp : skeys);
            const int* vi = to_final ? v_tmp : perm;
            if (j == 0 && with_src)
                s = radix_pass<unsigned int, KM_GATHER, true>(nullptr, vals_in, idx, ko, vo, counts, col_total, N,
                                                              ntiles, 0, M, counters, st);
            else if (j == 0)
                s = radix_pass<unsigned int, KM_DIRECT, true>(idx, nullptr, nullptr, ko, vo, counts, col_total, N,
                                                              ntiles, 0, M, counters, st);
            else
                s = radix_pass<unsigned int, KM_CARRY, false>(ki, vi, nullptr, ko, vo, counts, col_total, N, ntiles,
                                                              8 * j, M, counters, st);
            if (s) return s;
        }
    }
    row_ptr_kernel<<<static_cast<unsigned int>(cdiv(N + 1, 256)), 256, 0, st>>>(
        skeys, N, M, row_ptr, with_src ? reinterpret_cast<const long long*>(src_id) : nullptr, perm, counters);
    DETR_LAUNCHED();
    if (M > 0) {
        units_count_kernel<<<L.nut, kUnitThreads, 0, st>>>(row_ptr, M, g, upart, L.nut, counters);
        DETR_LAUNCHED();
        units_scan_kernel<<<1, 1024, 0, st>>>(upart, L.nut, counters);
        DETR_LAUNCHED();
        units_emit_kernel<<<L.nut, kUnitThreads, 0, st>>>(row_ptr, M, g, upart, L.nut, counters, units, finish);
        DETR_LAUNCHED();
    }
    int h[kCtrCount];
    DETR_CUDA(cudaMemcpyAsync(h, counters, sizeof(h), cudaMemcpyDeviceToHost, st));
    DETR_CUDA(cudaStreamSynchronize(st));
    if (h[kCtrErrIndex]) return DET_ERR_INDEX_RANGE;
    if (h[kCtrErrDup]) return DET_ERR_ORDER_KEY;

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
    p->units = units;
    p->finish = finish;
    p->n_segments = h[kCtrSegs];
    p->n_units = static_cast<int64_t>(h[kCtrSegs]) + h[kCtrNormal];
    p->n_hot_rows = h[kCtrHot];
    p->max_row_len = h[kCtrMaxLen];
    *out_plan = p;
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
