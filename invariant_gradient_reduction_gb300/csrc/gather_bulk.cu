// gather_bulk.cu -- gather-reduce for wide rows with few terms (the MoE
// combine: top-k <= 32 rows of several KB per destination), staged by TMA.
//
// A persistent CTA = one producer warp + sixteen consumer warps.  The producer
// walks the CTA's work items (destination, H-tile) in order; for each it
// reads the destination's source list, writes the weights to shared memory
// and issues one cp.async.bulk per source row tile into a ring of shared
// memory stages, completing on the stage's mbarrier.  Consumers wait for the
// stage, fold the (at most 32) terms of every 16-byte column left to right --
// the whole canonical fold when a destination has a single chunk -- round to
// the output type and store, then release the stage.  The bulk copies keep
// ~100 KB per SM in flight without registers, which is what the
// register-staged gather could not reach.
//
// Every mbarrier wait is bounded; on expiry the CTA records kCtrErrTimeout in
// the plan's counter block, drains the copies it issued (also bounded) and
// returns.
#include "bulk_copy.cuh"
#include "common.cuh"
#include "gather_internal.cuh"
#include "plan_internal.cuh"

namespace detr {

constexpr int kBulkConsumerWarps = 16;
constexpr int kBulkConsumers = kBulkConsumerWarps * 32;
constexpr int kBulkThreads = kBulkConsumers + 32;
#ifndef DETR_BULK_STAGES
#define DETR_BULK_STAGES 3
#endif
#ifndef DETR_BULK_STAGE_KB
#define DETR_BULK_STAGE_KB 64
#endif
constexpr int kBulkStages = DETR_BULK_STAGES;
constexpr int kBulkStageBytes = DETR_BULK_STAGE_KB * 1024;
constexpr int kBulkMaxTerms = 32;
// Producer warps of the fixed-stage kernel: items alternate between them
// when a CTA has at least kBulkTwoProducerItems items (EP-invariance, ~215
// items per CTA: 303 against 306.5 us); with fewer one producer works alone
// (MoE combine, 27 items per CTA: 52.2 us with two, 51.4 with one).
constexpr int kBulkProducers = 2;
constexpr int kBulkStageThreads = kBulkConsumers + 32 * kBulkProducers;
// The producers' unit pipeline: perm entries copied into shared memory
// kPipePermAhead units (items) ahead, weights kPipeWAhead ahead, in
// kPipeSlots slots.
constexpr int kPipePermAhead = 12;
constexpr int kPipeWAhead = 6;
constexpr int kPipeSlots = 16;
static_assert(kPipePermAhead == 2 * kPipeWAhead && kPipeSlots > kPipePermAhead, "unit pipeline distances");
constexpr int kBulkVecPerThread = 1;  // tile <= 8 KB = 512 16-byte vectors

struct BulkStageMeta {
    int m;      // destination
    int n;      // terms
    int col0;   // first element of the tile
    int bytes;  // bytes per term in this tile
};

template <typename XT>
struct BulkVec;
template <>
struct BulkVec<uint16_t> {
    static constexpr int VEC = 8;
    static __device__ __forceinline__ void expand(const uint4& r, float* f)
    {
        f[0] = bf16lo(r.x); f[1] = bf16hi(r.x); f[2] = bf16lo(r.y); f[3] = bf16hi(r.y);
        f[4] = bf16lo(r.z); f[5] = bf16hi(r.z); f[6] = bf16lo(r.w); f[7] = bf16hi(r.w);
    }
};
template <>
struct BulkVec<float> {
    static constexpr int VEC = 4;
    static __device__ __forceinline__ void expand(const uint4& r, float* f)
    {
        f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
    }
};

template <typename OT, int VEC>
__device__ __forceinline__ void bulk_store(void* base, long long off, const float* v, bool vec)
{
    if (sizeof(OT) == 4) {
        float* o = static_cast<float*>(base) + off;
        if (vec) {
#pragma unroll
            for (int e = 0; e < VEC; e += 4)
                *reinterpret_cast<float4*>(o + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[e] = v[e];
        }
    } else {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(base) + off;
        if (vec) {
            uint32_t pk[VEC / 2];
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                __nv_bfloat162 t = __floats2bfloat162_rn(v[e], v[e + 1]);
                pk[e / 2] = *reinterpret_cast<uint32_t*>(&t);
            }
            if (VEC == 8) *reinterpret_cast<uint4*>(o) = make_uint4(pk[0], pk[1 % (VEC / 2)], pk[2 % (VEC / 2)], pk[3 % (VEC / 2)]);
            else *reinterpret_cast<uint2*>(o) = make_uint2(pk[0], pk[1 % (VEC / 2)]);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[e] = __float2bfloat16_rn(v[e]);
        }
    }
}

// Tiling of rows of H elements for destinations of at most `terms` terms:
// the fewest H-tiles of at most 8 KB whose staged rows fit one stage (the
// host's bulk_plan_tiles, for a plan whose counts are on the device).
__device__ __forceinline__ bool bulk_tiles_dev(int H, int xsz, int terms, int* te, int* stride, int* nt)
{
    const long long row_bytes = static_cast<long long>(H) * xsz;
    for (int k = 1; k <= 64; ++k) {
        const long long tb = ((row_bytes + k - 1) / k + 15) / 16 * 16;
        if (tb > 16LL * kBulkConsumers * kBulkVecPerThread) continue;
        const long long st = (tb + 127) / 128 * 128;
        if (st * terms > kBulkStageBytes) continue;
        *te = static_cast<int>(tb / xsz);
        *stride = static_cast<int>(st);
        *nt = static_cast<int>((H + *te - 1) / *te);
        return true;
    }
    return false;
}

template <typename XT, typename OT>
__global__ void __launch_bounds__(kBulkStageThreads, 1)
gather_bulk_kernel(const __grid_constant__ BulkArgs a, const __grid_constant__ ShardTable tbl)
{
    using BV = BulkVec<XT>;
    constexpr int VEC = BV::VEC;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* stage_buf = smem;  // kBulkStages x kBulkStageBytes
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBulkStages * kBulkStageBytes);
    uint64_t* empty = full + kBulkStages;
    float* swt = reinterpret_cast<float*>(empty + kBulkStages);            // [kBulkStages][32]
    BulkStageMeta* meta = reinterpret_cast<BulkStageMeta*>(swt + kBulkStages * kBulkMaxTerms);
    // each producer's item pipeline: perm [kPipeSlots][32], weights [kPipeSlots][32], (destination, terms, tile) [kPipeSlots][3]
    int* pu_base = reinterpret_cast<int*>(meta + kBulkStages);
    constexpr int kPuInts = kPipeSlots * (32 + 32 + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(pu_base + kBulkProducers * kPuInts);

    pdl_wait();  // as a programmatic dependent (behind an unwaited plan): the plan has finished
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ long long s_items;
    __shared__ int s_tile[4];  // elements, staged stride, tiles per row, producers
    if (threadIdx.x == 0) {
        for (int s = 0; s < kBulkStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBulkConsumerWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        long long ni = a.n_items;
        int te = a.tile_elems, st = a.tile_stride, nt = a.ntiles;
        if (a.dev_counters) {  // written by the plan's kernels, which finished before this grid started
            const int* c = a.dev_counters;
            ni = 0;
            if (!(c[kCtrErrIndex] | c[kCtrErrDup] | c[kCtrErrTimeout]) && c[kCtrMaxLen] <= kBulkMaxTerms &&
                bulk_tiles_dev(a.H, static_cast<int>(sizeof(XT)), max(1, c[kCtrMaxLen]), &te, &st, &nt))
                ni = static_cast<long long>(c[kCtrShort] + c[kCtrEmpty]) * nt;  // every unit: none is longer
        }
        s_items = ni;
        s_tile[0] = te;
        s_tile[1] = st;
        s_tile[2] = nt;
        s_tile[3] = ni >= static_cast<long long>(kBulkTwoProducerItems) * gridDim.x ? kBulkProducers : 1;
    }
    __syncthreads();

    const long long n_items = s_items;
    const int tile_elems = s_tile[0], tile_stride = s_tile[1], ntiles = s_tile[2], nprod = s_tile[3];
    // the next kernel may be launched now: behind an unwaited plan the
    // register-staged kernel, which reads only the plan's counts before it
    // waits for this grid (its launch then overlaps this kernel, not its end)
    pdl_launch_dependents();
    if (warp >= kBulkConsumerWarps) {
        // ---------------- producer warps ----------------
        // Item k of this CTA is blockIdx.x + k * gridDim.x; producer pw of
        // nprod issues the items k = pw, pw + nprod, ... (its item j is k =
        // j * nprod + pw) into stage k % kBulkStages, so that the
        // stages fill in item order, as the consumers take them.  One
        // producer warp had spent ~1 us of its own instructions per 64 KB
        // item (27 items per CTA on the MoE combine), waiting for a free
        // stage only a third of its time.  Nothing a producer waits for per
        // item is a load issued for that item: the
        // list entries are read in batches of 32 items (lane l = item 32b +
        // l), a batch's entries two batches ahead and their row_ptr bounds
        // one batch ahead; each item's perm entries are copied into a
        // shared-memory slot kPipePermAhead items ahead and its weights
        // kPipeWAhead items ahead (cp.async, one commit group per item).  A
        // ring of registers shifted one slot per item had made every item
        // wait for the loads issued one item before: the producer issued an
        // item every ~1.7 us and waited for a free stage 4% of the time.
        const int pw = warp - kBulkConsumerWarps;
        if (pw >= nprod) return;
        int* pu_perm = pu_base + pw * kPuInts;
        float* pu_w = reinterpret_cast<float*>(pu_perm + kPipeSlots * 32);
        int* pu_mnt = pu_perm + kPipeSlots * 64;
        const long long g = gridDim.x;
        auto item_of = [&](long long j) { return blockIdx.x + (j * nprod + pw) * g; };
        auto list_m = [&](long long b) -> int {  // lane l: the list entry of this producer's item 32 b + l, or -1
            const long long it = item_of(32 * b + lane);
            return it < n_items ? a.units[it / ntiles].x : -1;
        };
        // A: the batch being entered; X: the next (bounds issued one batch
        // ago); Y: the one after (list entries)
        int A_m = -1, A_lo = 0, A_hi = 0;
        int X_m = list_m(0), X_lo = 0, X_hi = 0;
        int Y_m = list_m(1);
        if (X_m >= 0) { X_lo = a.row_ptr[X_m]; X_hi = a.row_ptr[X_m + 1]; }
        long long batch = -1;  // the batch held in A
        auto enter = [&](long long q) {  // item q into slot q % kPipeSlots, its perm copies issued
            if ((q >> 5) != batch) {     // q grows by one per call: the next batch
                A_m = X_m; A_lo = X_lo; A_hi = X_hi;
                X_m = Y_m;
                X_lo = X_hi = 0;
                if (X_m >= 0) { X_lo = a.row_ptr[X_m]; X_hi = a.row_ptr[X_m + 1]; }
                ++batch;
                Y_m = list_m(batch + 2);
            }
            const int l = static_cast<int>(q & 31);
            const int m = __shfl_sync(0xffffffffu, A_m, l);
            const int lo = __shfl_sync(0xffffffffu, A_lo, l);
            const int n = m < 0 ? 0 : __shfl_sync(0xffffffffu, A_hi, l) - lo;
            const int sl = static_cast<int>(q % kPipeSlots);
            if (lane == 0) {
                pu_mnt[3 * sl] = m;
                pu_mnt[3 * sl + 1] = n;
                pu_mnt[3 * sl + 2] = ntiles == 1 ? 0 : static_cast<int>(item_of(q) % ntiles);
            }
            if (lane < n) cp_async4(&pu_perm[sl * 32 + lane], a.perm + lo + lane);
        };
        auto fetch_w = [&](long long q) {  // item q's weights (its perm entries have landed)
            const int sl = static_cast<int>(q % kPipeSlots);
            if (a.w && lane < pu_mnt[3 * sl + 1]) cp_async4(&pu_w[sl * 32 + lane], a.w + pu_perm[sl * 32 + lane]);
        };
        // commit group G_j holds perm(j + kPipePermAhead) and w(j + kPipeWAhead);
        // item k needs G_{k - kPipeWAhead} and older
        for (int j = -kPipePermAhead; j < 0; ++j) {
            if (j >= -kPipeWAhead) {
                cp_async_wait_pending<kPipeWAhead - 1>();
                __syncwarp();
                fetch_w(j + kPipeWAhead);
            }
            enter(j + kPipePermAhead);
            cp_async_commit_group();
        }
        for (long long j = 0; item_of(j) < n_items; ++j) {
            cp_async_wait_pending<kPipeWAhead - 1>();
            __syncwarp();
            const int sl = static_cast<int>(j % kPipeSlots);
            const long long k = j * nprod + pw;  // the CTA's item index: its stage and phase
            const int cm = pu_mnt[3 * sl], cn = pu_mnt[3 * sl + 1], ct = pu_mnt[3 * sl + 2];
            const int ri = lane < cn ? pu_perm[sl * 32 + lane] : 0;
            const float rw = a.w && lane < cn ? pu_w[sl * 32 + lane] : 1.0f;
            const int s = static_cast<int>(k % kBulkStages);
            const uint32_t ph = static_cast<uint32_t>((k / kBulkStages) & 1);
            bool ok = true;
            if (k >= kBulkStages) ok = mbar_wait_bounded(&empty[s], ph ^ 1u);
            if (!__all_sync(0xffffffffu, ok) || *abort_flag) {
                if (lane == 0) { *abort_flag = 1; atomicOr(a.status + kCtrErrTimeout, 1); }
                break;
            }
            const int col0 = ct * tile_elems;
            const int bytes = min(tile_elems, a.H - col0) * static_cast<int>(sizeof(XT));
            if (lane < cn) swt[s * kBulkMaxTerms + lane] = rw;
            if (lane == 0) meta[s] = BulkStageMeta{cm, cn, col0, bytes};
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(cn * bytes));
            __syncwarp();
            if (lane < cn)
                bulk_g2s(stage_buf + static_cast<size_t>(s) * kBulkStageBytes + static_cast<size_t>(lane) * tile_stride,
                         shard_row(tbl, ri, a.ldx_bytes) + static_cast<long long>(col0) * sizeof(XT),
                         static_cast<uint32_t>(bytes), &full[s]);
            fetch_w(j + kPipeWAhead);
            enter(j + kPipePermAhead);
            cp_async_commit_group();
        }
        cp_async_wait_pending<0>();  // no copy into shared memory outlives the kernel
        return;
    }

    // ---------------- consumer warps ----------------
    const int ctid = threadIdx.x;  // 0 .. kBulkConsumers-1
    long long k = 0;
    long long item = blockIdx.x;
    for (; item < n_items; item += gridDim.x, ++k) {
        const int s = static_cast<int>(k % kBulkStages);
        const uint32_t ph = static_cast<uint32_t>((k / kBulkStages) & 1);
        const bool ok = mbar_wait_bounded(&full[s], ph);
        if (!ok || *abort_flag) {
            *abort_flag = 1;
            atomicOr(a.status + kCtrErrTimeout, 1);
            break;
        }
        const BulkStageMeta md = meta[s];
        const unsigned char* buf = stage_buf + static_cast<size_t>(s) * kBulkStageBytes;
        const float* wts = swt + s * kBulkMaxTerms;
        const int nvec = md.bytes / 16;
#pragma unroll
        for (int r = 0; r < kBulkVecPerThread; ++r) {
            const int v = ctid + r * kBulkConsumers;
            if (v < nvec) {
                float acc[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;  // empty destination: +0.0
                for (int j = 0; j < md.n; ++j) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(buf + static_cast<size_t>(j) * tile_stride + v * 16);
                    float xf[VEC];
                    BV::expand(raw, xf);
                    if (a.w) {
                        const float wv = wts[j];
#pragma unroll
                        for (int e = 0; e < VEC; ++e) xf[e] = __fmul_rn(wv, xf[e]);
                    }
                    if (j == 0) {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[e] = xf[e];
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[e] = __fadd_rn(acc[e], xf[e]);
                    }
                }
                bulk_store<OT, VEC>(a.out, static_cast<long long>(md.m) * a.ldo + md.col0 + v * VEC, acc,
                                    a.out_vec != 0);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (item < n_items) {
        // aborted: drain the copies this CTA may still have in flight (bounded)
        for (int s = 0; s < kBulkStages; ++s) {
            const long long kk = k + s;
            const uint32_t ph = static_cast<uint32_t>((kk / kBulkStages) & 1);
            mbar_wait_bounded(&full[kk % kBulkStages], ph);
        }
    }
}

template <typename XT, typename OT>
static det_status launch_bulk_t(const BulkArgs& a, const ShardTable& t, int grid, bool dependent, cudaStream_t st)
{
    const size_t smem = bulk_smem_bytes();
    {
        const det_status a_ = allow_dynamic_smem(reinterpret_cast<const void*>(gather_bulk_kernel<XT, OT>), smem);
        if (a_) return a_;
    }
    if (dependent) {
        DETR_CUDA(launch_after_previous(gather_bulk_kernel<XT, OT>, dim3(grid), dim3(kBulkStageThreads), smem, st, a, t));
    } else {
        gather_bulk_kernel<XT, OT><<<grid, kBulkStageThreads, smem, st>>>(a, t);
    }
    DETR_LAUNCHED();
    return DET_OK;
}

size_t bulk_smem_bytes()
{
    return static_cast<size_t>(kBulkStages) * kBulkStageBytes + 2 * kBulkStages * sizeof(uint64_t) +
           kBulkStages * kBulkMaxTerms * sizeof(float) + kBulkStages * sizeof(BulkStageMeta) +
           static_cast<size_t>(kBulkProducers) * kPipeSlots * (32 + 32 + 3) * sizeof(int) + 16;
}

bool bulk_plan_tiles(int64_t H, int xsz, int64_t max_terms, int* tile_elems, int* tile_stride, int* ntiles)
{
    if (max_terms > kBulkMaxTerms) return false;
    const int64_t row_bytes = H * xsz;
    const int64_t terms = std::max<int64_t>(1, max_terms);
    for (int64_t k = 1; k <= 64; ++k) {
        const int64_t tb = (cdiv(row_bytes, k) + 15) / 16 * 16;  // 16-byte multiple
        if (tb > 16 * kBulkConsumers * kBulkVecPerThread) continue;
        const int64_t stride = (tb + 127) / 128 * 128;
        if (stride * terms > kBulkStageBytes) continue;
        *tile_elems = static_cast<int>(tb / xsz);
        *tile_stride = static_cast<int>(stride);
        *ntiles = static_cast<int>(cdiv(H, tb / xsz));
        return true;
    }
    return false;
}

det_status launch_gather_bulk(det_dtype x_dtype, det_dtype out_dtype, const BulkArgs& a, const ShardTable& t, int grid,
                              bool dependent, cudaStream_t st)
{
    if (x_dtype == DET_BF16 && out_dtype == DET_BF16)
        return launch_bulk_t<uint16_t, __nv_bfloat16>(a, t, grid, dependent, st);
    if (x_dtype == DET_BF16) return launch_bulk_t<uint16_t, float>(a, t, grid, dependent, st);
    if (out_dtype == DET_BF16) return launch_bulk_t<float, __nv_bfloat16>(a, t, grid, dependent, st);
    return launch_bulk_t<float, float>(a, t, grid, dependent, st);
}

// ------------------------------------------------------------------------
// destinations of at most one chunk: a byte ring of whole items
// ------------------------------------------------------------------------
//
// The embedding backward's rows have mostly one to three terms, and each
// touched gradient row is read and written once: with a fixed stage per item
// the stages would hold a few KB each.  Here an item is one H-tile of one
// destination -- its n term tiles and, for index_add_ (ACC), the
// destination's old tile -- sized per n (as wide as fits 64 KB, at most 8 KB
// of sources for the 512 consumer threads), and the producer packs
// consecutive items into a byte ring of shared memory (its size a launch
// argument), up to kRingSlots items in flight.  A consumer thread folds its
// 16-byte column of the n terms left to right (the canonical fold of a
// single chunk; +0.0 for a destination without terms), adds the result to
// the old value once (__fadd_rn) for index_add_, rounds to the output type
// and stores.  The producer reuses ring bytes only after the items that held
// them are consumed (their empty barriers, oldest first), and ends with an
// item marked last that tells the consumers to stop.
constexpr int kRingSlots = 8;
static_assert((kRingSlots & (kRingSlots - 1)) == 0, "a power of two");
constexpr int kRingChunk = 8;       // units per claim
constexpr int kRingItemMax = 64 * 1024;
constexpr int kRingSpinCheck = 1024;  // consumer try_waits between looks at the abort flag

struct RingMeta {
    int m;       // destination (n < 0: no more items)
    int n;       // terms
    int col0;    // first element of the tile
    int elems;   // elements in the tile
    int off;     // ring offset of the first term tile; the old tile (ACC) follows the n term tiles
    int stride;  // bytes between term tiles (128-byte multiple)
};

struct RingTile {
    int te;      // tile width in elements
    int stride;  // staged bytes per term tile
    int obytes;  // staged bytes of the old destination tile (0 without ACC)
    int nt;      // tiles per row
};

__device__ __forceinline__ long long ring_cdiv(long long a, long long b) { return (a + b - 1) / b; }

// Tiling of a destination with n terms: the fewest tiles for which a tile of
// x is at most 8 KB (one 16-byte column per consumer thread) and the item
// (n term tiles + the old tile, each rounded to 128 bytes) fits kRingItemMax.
__device__ __forceinline__ RingTile ring_tile(int n, int H, int q, int xsz, int osz)
{
    RingTile t{};
    const long long per_elem = static_cast<long long>(n) * xsz + osz;
    int nt = static_cast<int>(max(ring_cdiv(static_cast<long long>(H) * xsz, 16LL * kBulkConsumers),
                                  ring_cdiv(static_cast<long long>(H) * per_elem, static_cast<long long>(kRingItemMax))));
    nt = max(nt, 1);
    for (;; ++nt) {
        const int te = static_cast<int>((ring_cdiv(H, nt) + q - 1) / q * q);
        const int stride = (te * xsz + 127) / 128 * 128;
        const int ob = (te * osz + 127) / 128 * 128;
        if (te * xsz <= 16 * kBulkConsumers && static_cast<long long>(n) * stride + ob <= kRingItemMax) {
            t.te = te;
            t.stride = stride;
            t.obytes = ob;
            t.nt = static_cast<int>(ring_cdiv(H, te));
            return t;
        }
    }
}

// The old destination values of one 16-byte column of x (VEC elements).
template <typename OT, int VEC>
__device__ __forceinline__ void ring_load_old(const unsigned char* p, float* old)
{
    if (sizeof(OT) == 4) {
#pragma unroll
        for (int e = 0; e < VEC; e += 4) {
            const float4 t = *reinterpret_cast<const float4*>(p + e * 4);
            old[e] = t.x; old[e + 1] = t.y; old[e + 2] = t.z; old[e + 3] = t.w;
        }
    } else {
        const unsigned short* o = reinterpret_cast<const unsigned short*>(p);
#pragma unroll
        for (int e = 0; e < VEC; ++e) old[e] = __uint_as_float(static_cast<uint32_t>(o[e]) << 16);
    }
}

// At most 64 registers: with one CTA of the register-staged kernel (8 warps
// of 80 registers) beside it, the SM sub-partition that holds 5 of this
// kernel's 17 warps needs 5 x 2048 + 2 x 2560 <= 16384 registers; at 70
// registers the second CTA did not fit and the two kernels ran one after
// the other (201 against 128 us on the embedding backward).
template <typename XT, typename OT, bool ACC>
__global__ void __maxnreg__(64)
gather_ring_kernel(const __grid_constant__ RingArgs a, const __grid_constant__ ShardTable tbl)
{
    using BV = BulkVec<XT>;
    constexpr int VEC = BV::VEC;
    constexpr int XSZ = static_cast<int>(sizeof(XT));
    constexpr int OSZ = static_cast<int>(sizeof(OT));
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t R = static_cast<uint32_t>(a.ring_bytes);  // a multiple of 128, at least 2 * kRingItemMax
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + R);
    uint64_t* empty = full + kRingSlots;
    uint32_t* charge = reinterpret_cast<uint32_t*>(empty + kRingSlots);      // producer's: ring bytes each slot's item holds
    float* swt = reinterpret_cast<float*>(charge + kRingSlots);              // [kRingSlots][32]
    RingMeta* meta = reinterpret_cast<RingMeta*>(swt + kRingSlots * kBulkMaxTerms);
    RingTile* tiles = reinterpret_cast<RingTile*>(meta + kRingSlots);       // [kBulkMaxTerms + 1], by n
    int* pu_perm = reinterpret_cast<int*>(tiles + kBulkMaxTerms + 1);       // producer's unit pipeline [kPipeSlots][32]
    float* pu_w = reinterpret_cast<float*>(pu_perm + kPipeSlots * 32);      // [kPipeSlots][32]
    int* pu_mn = reinterpret_cast<int*>(pu_w + kPipeSlots * 32);            // [kPipeSlots][2]: destination, terms
    volatile int* abort_flag = reinterpret_cast<volatile int*>(pu_mn + kPipeSlots * 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRingSlots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBulkConsumerWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (threadIdx.x <= kBulkMaxTerms) tiles[threadIdx.x] = ring_tile(threadIdx.x, a.H, a.quantum, XSZ, ACC ? OSZ : 0);
    // Launched the ordinary way, or as the plan's programmatic dependent and
    // past this wait, so everything before this grid has finished: the
    // kernel for the other destinations may start now and run beside this
    // one (it reads the plan without waiting, writes other rows, and waits
    // for this grid before it ends).  (Behind a plan that released it at
    // the plan's start, this kernel made the MoE step 3 us and the
    // EP-invariance step 4 us slower: its CTAs sat on the SMs through the
    // whole plan.)
    pdl_wait();
    pdl_launch_dependents();
    __syncthreads();

    long long n_units = a.n_units;
    if (a.dev_counters) {  // written by the plan's kernels, which finished before this grid started
        const int* c = a.dev_counters;
        n_units = (c[kCtrErrIndex] | c[kCtrErrDup] | c[kCtrErrTimeout]) ? 0
                                                                         : c[kCtrShort] + (ACC ? 0 : c[kCtrEmpty]);
    }
    if (warp == kBulkConsumerWarps) {
        // ---------------- producer warp ----------------
        // Units come in chunks of kRingChunk list entries: this CTA's first
        // two chunks are fixed (chunk c = list entries (c * grid + CTA) *
        // kRingChunk ...), later ones are claimed from a counter in the plan's
        // counter block, so that CTAs whose units were cheaper take more (the
        // units differ in cost up to tenfold; with a fixed round-robin the
        // last CTA ended ~30% after the first).  Nothing the producer waits
        // for per unit is a load issued for that unit: a chunk's claim, its
        // list entries and their row_ptr bounds are issued one chunk apart,
        // its perm entries are copied into a shared-memory slot
        // kPipePermAhead units ahead and its weights kPipeWAhead units ahead
        // (cp.async, one commit group per unit).  (A ring of registers
        // shifted one slot per unit had made every unit wait for the load
        // issued one unit before.)
        const long long G = gridDim.x;
        int* ring_next = a.status + kCtrRingNext;
        auto chunk_m = [&](long long base) -> int {  // lane l < kRingChunk: list entry base + l, or -1
            return lane < kRingChunk && base + lane < n_units ? a.units[base + lane].x : -1;
        };
        const long long dyn0 = 2 * G * kRingChunk;  // claimed chunks start after the fixed ones
        // A: the chunk being entered (lane l = its unit l); X: the next (bounds
        // issued one chunk ago); Y: the one after (list entries); zclaim (lane
        // 0): the claim of the one after that
        int A_m = -1, A_lo = 0, A_hi = 0;
        int X_m = chunk_m(static_cast<long long>(blockIdx.x) * kRingChunk), X_lo = 0, X_hi = 0;
        int Y_m = chunk_m((G + blockIdx.x) * kRingChunk);
        int zclaim = 0;  // lane 0: raw counter value of the claim (read one chunk later)
        if (lane == 0) zclaim = atomicAdd(ring_next, kRingChunk);
        if (X_m >= 0) { X_lo = a.row_ptr[X_m]; X_hi = a.row_ptr[X_m + 1]; }
        long long chunk = -1;  // the chunk held in A
        auto advance = [&]() {
            A_m = X_m; A_lo = X_lo; A_hi = X_hi;
            X_m = Y_m;
            X_lo = X_hi = 0;
            if (X_m >= 0) { X_lo = a.row_ptr[X_m]; X_hi = a.row_ptr[X_m + 1]; }
            const long long zb = dyn0 + __shfl_sync(0xffffffffu, zclaim, 0);
            Y_m = chunk_m(zb);
            if (lane == 0 && zb < n_units) zclaim = atomicAdd(ring_next, kRingChunk);
            ++chunk;
        };
        // unit q of this CTA enters the pipeline: its list entry into slot
        // q % kPipeSlots (destination -1: no more units), its perm copies issued
        auto enter = [&](long long q) {
            if (q / kRingChunk != chunk) advance();  // q grows by one per call
            const int l = static_cast<int>(q % kRingChunk);
            const int m = __shfl_sync(0xffffffffu, A_m, l);
            const int lo = __shfl_sync(0xffffffffu, A_lo, l);
            const int n = m < 0 ? 0 : __shfl_sync(0xffffffffu, A_hi, l) - lo;
            const int sl = static_cast<int>(q % kPipeSlots);
            if (lane == 0) { pu_mn[2 * sl] = m; pu_mn[2 * sl + 1] = n; }
            if (lane < n) cp_async4(&pu_perm[sl * 32 + lane], a.perm + lo + lane);
        };
        // weights of unit q (its perm entries have landed)
        auto fetch_w = [&](long long q) {
            const int sl = static_cast<int>(q % kPipeSlots);
            if (a.w && lane < pu_mn[2 * sl + 1]) cp_async4(&pu_w[sl * 32 + lane], a.w + pu_perm[sl * 32 + lane]);
        };
        // Commit group G_j (j >= -kPipePermAhead) holds perm(j + kPipePermAhead)
        // and w(j + kPipeWAhead): unit j needs G_{j - kPipeWAhead} and older,
        // which leaves kPipeWAhead - 1 groups pending.  The prologue issues
        // G_{-kPipePermAhead} .. G_{-1}.
        for (int j = -kPipePermAhead; j < 0; ++j) {
            if (j >= -kPipeWAhead) {
                cp_async_wait_pending<kPipeWAhead - 1>();
                __syncwarp();
                fetch_w(j + kPipeWAhead);
            }
            enter(j + kPipePermAhead);
            cp_async_commit_group();
        }
        // The ring: head is the offset where the next item may start, free
        // the bytes not held by items in flight.  An item never wraps: when
        // it does not fit before the end, it starts at 0 and also holds the
        // bytes it skipped (its charge), which come free with it.
        uint32_t k = 0;     // items issued (modulo 2^32)
        uint32_t tail = 0;  // items known to be consumed (all items below it)
        uint32_t head = 0, free_bytes = R;
        bool ok = true;
        // Ring bytes [start, start + bytes) for item k, after the consumers
        // have freed them; false if a wait expired.
        auto reserve = [&](uint32_t bytes, uint32_t* start, uint32_t* held) -> bool {
            const uint32_t skip = head + bytes > R ? R - head : 0u;
            const uint32_t need = skip + bytes;
            while (static_cast<int>(k - tail) >= kRingSlots || free_bytes < need) {
                const uint32_t ts = tail & (kRingSlots - 1);
                const bool w_ok = mbar_wait_bounded(&empty[ts], (tail / kRingSlots) & 1u);
                if (!__all_sync(0xffffffffu, w_ok) || *abort_flag) return false;
                free_bytes += charge[ts];
                ++tail;
            }
            *start = skip ? 0u : head;
            head = *start + bytes;
            if (head == R) head = 0;
            free_bytes -= need;
            *held = need;
            return true;
        };
        for (long long ku = 0; ok; ++ku) {
            // perm(ku), w(ku) and perm(ku + kPipeWAhead) have landed: G_{ku - kPipeWAhead} and older
            cp_async_wait_pending<kPipeWAhead - 1>();
            __syncwarp();
            const int sl = static_cast<int>(ku % kPipeSlots);
            const int cm = pu_mn[2 * sl], cn = pu_mn[2 * sl + 1];
            if (cm < 0) break;  // no more units (the claims come in order)
            const RingTile tl = tiles[cn];
            const int ri = lane < cn ? pu_perm[sl * 32 + lane] : 0;
            const float rw = a.w && lane < cn ? pu_w[sl * 32 + lane] : 1.0f;
            const unsigned char* xrow = lane < cn ? shard_row(tbl, ri, a.ldx_bytes) : nullptr;
            const unsigned char* orow = static_cast<const unsigned char*>(a.out) + static_cast<long long>(cm) * a.ldo * OSZ;
            const uint32_t bytes = static_cast<uint32_t>(cn * tl.stride + tl.obytes);
            for (int t = 0; t < tl.nt; ++t) {
                const int col0 = t * tl.te;
                const int elems = min(tl.te, a.H - col0);
                uint32_t start = 0, held = 0;
                if (!reserve(bytes, &start, &held)) { ok = false; break; }
                const uint32_t s = k & (kRingSlots - 1);
                if (a.w && lane < cn) swt[s * kBulkMaxTerms + lane] = rw;
                if (lane == 0) {
                    meta[s] = RingMeta{cm, cn, col0, elems, static_cast<int>(start), tl.stride};
                    charge[s] = held;
                }
                __syncwarp();
                // the copies may complete before the expected byte count is
                // set: the count goes below zero until then, and the phase
                // cannot complete before this one arrival
                const uint32_t xb = static_cast<uint32_t>(elems * XSZ), ob = static_cast<uint32_t>(elems * OSZ);
                if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(cn) * xb + (ACC ? ob : 0u));
                if (lane < cn)
                    bulk_g2s(ring + start + lane * tl.stride, xrow + static_cast<long long>(col0) * XSZ, xb, &full[s]);
                if (ACC && lane == 31)
                    bulk_g2s(ring + start + cn * tl.stride, orow + static_cast<long long>(col0) * OSZ, ob, &full[s]);
                ++k;
            }
            if (!ok) break;
            // G_ku: w(ku + kPipeWAhead) (its perm entries are in G_{ku - kPipeWAhead}), perm(ku + kPipePermAhead)
            fetch_w(ku + kPipeWAhead);
            enter(ku + kPipePermAhead);
            cp_async_commit_group();
        }
        cp_async_wait_pending<0>();  // no copy into shared memory outlives the kernel
        if (ok) {
            // the end marker: an item of no bytes, marked last, in the next slot
            uint32_t start = 0, held = 0;
            ok = reserve(0, &start, &held);
            if (ok) {
                const uint32_t s = k & (kRingSlots - 1);
                if (lane == 0) {
                    meta[s] = RingMeta{0, -1, 0, 0, 0, 0};
                    charge[s] = 0;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[s]);
                ++k;
            }
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(a.status + kCtrErrTimeout, 1);
        }
        // every copy this CTA issued lands before it exits: the items not
        // known to be consumed are the last of their slots (bounded waits)
        for (uint32_t j = static_cast<int>(k - tail) > kRingSlots ? k - kRingSlots : tail; j != k; ++j)
            mbar_wait_bounded(&full[j & (kRingSlots - 1)], (j / kRingSlots) & 1u);
        // the last CTA to get here (after every claim of every CTA) sets the
        // claim counter back to 0 for the next call with this plan
        if (lane == 0) {
            __threadfence();
            if (atomicAdd(a.status + kCtrRingDone, 1) == static_cast<int>(gridDim.x) - 1) {
                a.status[kCtrRingNext] = 0;
                a.status[kCtrRingDone] = 0;
                __threadfence();
            }
        }
        return;
    }

    // ---------------- consumer warps ----------------
    const int ctid = threadIdx.x;  // 0 .. kBulkConsumers-1
    for (uint32_t k = 0;; ++k) {
        const uint32_t s = k & (kRingSlots - 1);
        const uint32_t ph = (k / kRingSlots) & 1u;
        bool ok = false;
        for (unsigned long long it = 0; it < kBulkWaitLimit; ++it) {
            if (mbar_try_wait(&full[s], ph)) { ok = true; break; }
            if ((it & (kRingSpinCheck - 1)) == kRingSpinCheck - 1 && *abort_flag) break;
        }
        if (!ok || *abort_flag) {
            *abort_flag = 1;
            atomicOr(a.status + kCtrErrTimeout, 1);
            break;
        }
        const RingMeta md = meta[s];
        if (md.n < 0) break;  // no more items
        const unsigned char* buf = ring + md.off;
        const float* wts = swt + s * kBulkMaxTerms;
        const int nvec = md.elems * XSZ / 16;
        if (ctid < nvec) {
            float acc[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;  // a destination without terms: +0.0
            for (int j = 0; j < md.n; ++j) {
                const uint4 raw = *reinterpret_cast<const uint4*>(buf + j * md.stride + ctid * 16);
                float xf[VEC];
                BV::expand(raw, xf);
                if (a.w) {
                    const float wv = wts[j];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) xf[e] = __fmul_rn(wv, xf[e]);
                }
                if (j == 0) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) acc[e] = xf[e];
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) acc[e] = __fadd_rn(acc[e], xf[e]);
                }
            }
            if (ACC) {
                float old[VEC];
                ring_load_old<OT, VEC>(buf + md.n * md.stride + ctid * VEC * OSZ, old);
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] = __fadd_rn(old[e], acc[e]);
            }
            bulk_store<OT, VEC>(a.out, static_cast<long long>(md.m) * a.ldo + md.col0 + ctid * VEC, acc, true);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

size_t ring_smem_bytes(int ring_bytes)
{
    return static_cast<size_t>(ring_bytes) + 2 * kRingSlots * sizeof(uint64_t) + kRingSlots * sizeof(uint32_t) +
           kRingSlots * kBulkMaxTerms * sizeof(float) + kRingSlots * sizeof(RingMeta) +
           (kBulkMaxTerms + 1) * sizeof(RingTile) + kPipeSlots * 32 * (sizeof(int) + sizeof(float)) +
           kPipeSlots * 2 * sizeof(int) + 16;
}

template <typename XT, typename OT, bool ACC>
static det_status launch_ring_t(const RingArgs& a, const ShardTable& t, int grid, cudaStream_t st)
{
    if (a.ring_bytes % 128 || a.ring_bytes < 2 * kRingItemMax) return DET_ERR_ARG;
    const size_t smem = ring_smem_bytes(a.ring_bytes);
    {
        const det_status a_ =
            allow_dynamic_smem(reinterpret_cast<const void*>(gather_ring_kernel<XT, OT, ACC>), smem);
        if (a_) return a_;
        // all of the SM's shared memory: the register-staged kernel that runs
        // beside it needs the rest of it on the same SM
        static bool carve_set = false;
        if (!carve_set) {
            DETR_CUDA(cudaFuncSetAttribute(reinterpret_cast<const void*>(gather_ring_kernel<XT, OT, ACC>),
                                           cudaFuncAttributePreferredSharedMemoryCarveout, 100));
            carve_set = true;
        }
    }
    if (a.dependent) {
        DETR_CUDA(launch_after_previous(gather_ring_kernel<XT, OT, ACC>, dim3(grid), dim3(kBulkThreads), smem, st, a, t));
    } else {
        gather_ring_kernel<XT, OT, ACC><<<grid, kBulkThreads, smem, st>>>(a, t);
    }
    DETR_LAUNCHED();
    return DET_OK;
}

template <bool ACC>
static det_status launch_ring_acc(det_dtype x_dtype, det_dtype out_dtype, const RingArgs& a, const ShardTable& t,
                                  int grid, cudaStream_t st)
{
    if (x_dtype == DET_BF16 && out_dtype == DET_BF16) return launch_ring_t<uint16_t, __nv_bfloat16, ACC>(a, t, grid, st);
    if (x_dtype == DET_BF16) return launch_ring_t<uint16_t, float, ACC>(a, t, grid, st);
    if (out_dtype == DET_BF16) return launch_ring_t<float, __nv_bfloat16, ACC>(a, t, grid, st);
    return launch_ring_t<float, float, ACC>(a, t, grid, st);
}

det_status launch_gather_ring(det_dtype x_dtype, det_dtype out_dtype, bool accumulate, const RingArgs& a,
                              const ShardTable& t, int grid, cudaStream_t st)
{
    return accumulate ? launch_ring_acc<true>(x_dtype, out_dtype, a, t, grid, st)
                      : launch_ring_acc<false>(x_dtype, out_dtype, a, t, grid, st);
}

}  // namespace detr
