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
constexpr int kBulkStages = 3;
constexpr int kBulkStageBytes = 64 * 1024;
constexpr int kBulkMaxTerms = 32;
constexpr int kBulkLook = 4;  // items whose source rows the producer reads ahead
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

template <typename XT, typename OT>
__global__ void __launch_bounds__(kBulkThreads, 1)
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
    volatile int* abort_flag = reinterpret_cast<volatile int*>(meta + kBulkStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kBulkStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBulkConsumerWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const long long n_items = a.n_items;
    if (warp == kBulkConsumerWarps) {
        // ---------------- producer warp ----------------
        // Item k of this CTA is blockIdx.x + k * gridDim.x.  The list lookups
        // run 32 items ahead (lane l holds item kb + l of the current and of
        // the next batch).  The source rows of the next kBulkLook items are
        // read ahead too (lane = term; an item's perm entries kBulkLook items
        // before its copies, its weights two items before), so that after an
        // L2 flush no item waits on its perm -> weight chain: the one
        // producer warp issues every copy, and that chain was its critical
        // path.
        const long long g = gridDim.x;
        int bm = 0, blo = 0, bn = -1, nm = 0, nlo = 0, nn = -1;
        auto fetch_meta = [&](long long kb, int& fm, int& flo, int& fn) {
            const long long it = blockIdx.x + (kb + lane) * g;
            fn = -1;
            if (it < n_items) {
                fm = a.units[it / a.ntiles].x;
                flo = a.row_ptr[fm];
                fn = a.row_ptr[fm + 1] - flo;
            }
        };
        fetch_meta(0, bm, blo, bn);
        fetch_meta(32, nm, nlo, nn);
        long long batch = 0;  // bm/blo/bn hold items [32 batch, 32 batch + 32), nm/nlo/nn the next 32
        // the ring: slot d holds item k + d
        int rm[kBulkLook], rn[kBulkLook], rt[kBulkLook], ri[kBulkLook];
        float rw[kBulkLook];
        auto enter = [&](long long q, int d) {  // item q into slot d: its list entry and its perm loads
            const int jq = static_cast<int>(q & 31);
            const bool here = (q >> 5) == batch;
            const int m = __shfl_sync(0xffffffffu, here ? bm : nm, jq);
            const int lo = __shfl_sync(0xffffffffu, here ? blo : nlo, jq);
            const int n = __shfl_sync(0xffffffffu, here ? bn : nn, jq);
            rm[d] = m;
            rn[d] = n;
            rt[d] = static_cast<int>((blockIdx.x + q * g) % a.ntiles);
            ri[d] = lane < n ? a.perm[lo + lane] : 0;
            rw[d] = 1.0f;
        };
#pragma unroll
        for (int d = 0; d < kBulkLook; ++d) enter(d, d);
        if (a.w) {
            if (lane < rn[0]) rw[0] = a.w[ri[0]];
            if (lane < rn[1]) rw[1] = a.w[ri[1]];
        }
        for (long long k = 0; blockIdx.x + k * g < n_items; ++k) {
            const int s = static_cast<int>(k % kBulkStages);
            const uint32_t ph = static_cast<uint32_t>((k / kBulkStages) & 1);
            bool ok = true;
            if (k >= kBulkStages) ok = mbar_wait_bounded(&empty[s], ph ^ 1u);
            if (!__all_sync(0xffffffffu, ok) || *abort_flag) {
                if (lane == 0) { *abort_flag = 1; atomicOr(a.status + kCtrErrTimeout, 1); }
                break;
            }
            const int cm = rm[0], cn = rn[0];
            const int col0 = rt[0] * a.tile_elems;
            const int bytes = min(a.tile_elems, a.H - col0) * static_cast<int>(sizeof(XT));
            if (lane < cn) swt[s * kBulkMaxTerms + lane] = rw[0];
            if (lane == 0) meta[s] = BulkStageMeta{cm, cn, col0, bytes};
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(cn * bytes));
            __syncwarp();
            if (lane < cn)
                bulk_g2s(stage_buf + static_cast<size_t>(s) * kBulkStageBytes + static_cast<size_t>(lane) * a.tile_stride,
                         shard_row(tbl, ri[0], a.ldx_bytes) + static_cast<long long>(col0) * sizeof(XT),
                         static_cast<uint32_t>(bytes), &full[s]);
            // advance: the list batch, the ring, the weights two items ahead
            const long long q = k + kBulkLook;
            if ((q >> 5) > batch + 1) {
                batch += 1;
                bm = nm; blo = nlo; bn = nn;
                fetch_meta(32 * (batch + 1), nm, nlo, nn);
            }
#pragma unroll
            for (int d = 0; d + 1 < kBulkLook; ++d) {
                rm[d] = rm[d + 1]; rn[d] = rn[d + 1]; rt[d] = rt[d + 1]; ri[d] = ri[d + 1]; rw[d] = rw[d + 1];
            }
            enter(q, kBulkLook - 1);
            if (a.w && lane < rn[1]) rw[1] = a.w[ri[1]];
        }
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
                    const uint4 raw = *reinterpret_cast<const uint4*>(buf + static_cast<size_t>(j) * a.tile_stride + v * 16);
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
static det_status launch_bulk_t(const BulkArgs& a, const ShardTable& t, int grid, cudaStream_t st)
{
    const size_t smem = bulk_smem_bytes();
    {
        const det_status a_ = allow_dynamic_smem(reinterpret_cast<const void*>(gather_bulk_kernel<XT, OT>), smem);
        if (a_) return a_;
    }
    gather_bulk_kernel<XT, OT><<<grid, kBulkThreads, smem, st>>>(a, t);
    DETR_LAUNCHED();
    return DET_OK;
}

size_t bulk_smem_bytes()
{
    return static_cast<size_t>(kBulkStages) * kBulkStageBytes + 2 * kBulkStages * sizeof(uint64_t) +
           kBulkStages * kBulkMaxTerms * sizeof(float) + kBulkStages * sizeof(BulkStageMeta) + 16;
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
                              cudaStream_t st)
{
    if (x_dtype == DET_BF16 && out_dtype == DET_BF16) return launch_bulk_t<uint16_t, __nv_bfloat16>(a, t, grid, st);
    if (x_dtype == DET_BF16) return launch_bulk_t<uint16_t, float>(a, t, grid, st);
    if (out_dtype == DET_BF16) return launch_bulk_t<float, __nv_bfloat16>(a, t, grid, st);
    return launch_bulk_t<float, float>(a, t, grid, st);
}

// ------------------------------------------------------------------------
// index_add_ on one-chunk destinations: a byte ring of whole items
// ------------------------------------------------------------------------
//
// The embedding backward's rows have mostly one to three terms, and each
// touched gradient row is read and written once: with a fixed stage per item
// the stages would hold a few KB each.  Here an item is one H-tile of one
// destination -- its n term tiles and the destination's old tile -- sized per
// n (as wide as fits 64 KB, at most 8 KB of sources for the 512 consumer
// threads), and the producer packs consecutive items into a 160 KB ring of
// shared memory, up to kAccSlots items in flight.  A consumer thread folds
// its 16-byte column of the n terms left to right (the canonical fold of a
// single chunk), adds the result to the old value once (__fadd_rn), rounds to
// the output type and stores.  The producer reuses ring bytes only after the
// items that held them are consumed (their empty barriers, oldest first), and
// ends with an item of no terms that tells the consumers to stop.

// The ring leaves room on the SM for one CTA of the register-staged kernel,
// which runs the longer destinations beside this kernel (128, 160 and 176 KB
// rings measured the same on the embedding backward).
constexpr int kAccSlots = 8;
constexpr int kAccRingBytes = 160 * 1024;
static_assert(kAccRingBytes >= 2 * (64 * 1024), "an item that does not fit the ring's tail must fit its head");
constexpr int kAccItemMax = 64 * 1024;
constexpr int kAccSpinCheck = 1024;  // consumer try_waits between looks at the abort flag

struct AccMeta {
    int m;       // destination (n < 0: no more items)
    int n;       // terms
    int col0;    // first element of the tile
    int elems;   // elements in the tile
    int off;     // ring offset of the first term tile; the old tile follows the n term tiles
    int stride;  // bytes between term tiles (128-byte multiple)
};

struct AccTile {
    int te;      // tile width in elements
    int stride;  // staged bytes per term tile
    int obytes;  // staged bytes of the old destination tile
    int nt;      // tiles per row
};

// Tiling of a destination with n terms: the fewest tiles for which a tile of
// x is at most 8 KB (one 16-byte column per consumer thread) and the item
// (n term tiles + the old tile, each rounded to 128 bytes) fits kAccItemMax.
__device__ __forceinline__ long long acc_cdiv(long long a, long long b) { return (a + b - 1) / b; }

__device__ __forceinline__ AccTile acc_tile(int n, int H, int q, int xsz, int osz)
{
    AccTile t{};
    const long long per_elem = static_cast<long long>(n) * xsz + osz;
    int nt = static_cast<int>(max(acc_cdiv(static_cast<long long>(H) * xsz, 16LL * kBulkConsumers),
                                  acc_cdiv(static_cast<long long>(H) * per_elem, static_cast<long long>(kAccItemMax))));
    nt = max(nt, 1);
    for (;; ++nt) {
        const int te = static_cast<int>((acc_cdiv(H, nt) + q - 1) / q * q);
        const int stride = (te * xsz + 127) / 128 * 128;
        const int ob = (te * osz + 127) / 128 * 128;
        if (te * xsz <= 16 * kBulkConsumers && static_cast<long long>(n) * stride + ob <= kAccItemMax) {
            t.te = te;
            t.stride = stride;
            t.obytes = ob;
            t.nt = static_cast<int>(acc_cdiv(H, te));
            return t;
        }
    }
}

// The old destination values of one 16-byte column of x (VEC elements).
template <typename OT, int VEC>
__device__ __forceinline__ void acc_load_old(const unsigned char* p, float* old)
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
template <typename XT, typename OT>
__global__ void __maxnreg__(64)
gather_bulk_acc_kernel(const __grid_constant__ BulkAccArgs a, const __grid_constant__ ShardTable tbl)
{
    using BV = BulkVec<XT>;
    constexpr int VEC = BV::VEC;
    constexpr int XSZ = static_cast<int>(sizeof(XT));
    constexpr int OSZ = static_cast<int>(sizeof(OT));
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;  // kAccRingBytes
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kAccRingBytes);
    uint64_t* empty = full + kAccSlots;
    long long* slot_end = reinterpret_cast<long long*>(empty + kAccSlots);  // producer's: ring end of each slot's item
    float* swt = reinterpret_cast<float*>(slot_end + kAccSlots);           // [kAccSlots][32]
    AccMeta* meta = reinterpret_cast<AccMeta*>(swt + kAccSlots * kBulkMaxTerms);
    AccTile* tiles = reinterpret_cast<AccTile*>(meta + kAccSlots);         // [kBulkMaxTerms + 1], by n
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tiles + kBulkMaxTerms + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kAccSlots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBulkConsumerWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (threadIdx.x <= kBulkMaxTerms) tiles[threadIdx.x] = acc_tile(threadIdx.x, a.H, a.quantum, XSZ, OSZ);
    // the kernel for the other destinations may start now and run beside
    // this one (it writes other rows; it waits for this grid before it ends)
    pdl_launch_dependents();
    __syncthreads();

    long long n_units = a.n_units;
    if (a.dev_counters) {  // written by the plan's kernels, which finished before this grid started
        const int* c = a.dev_counters;
        n_units = (c[kCtrErrIndex] | c[kCtrErrDup] | c[kCtrErrTimeout]) ? 0 : c[kCtrShort];
    }
    if (warp == kBulkConsumerWarps) {
        // ---------------- producer warp ----------------
        // Unit k of this CTA is blockIdx.x + k * gridDim.x; lane l holds the
        // list entry of unit kb + l of the current and of the next batch of
        // 32, and the source rows of the next kBulkLook units are read ahead
        // (lane = term), as in the fixed-stage kernel above.
        const long long g = gridDim.x;
        int bm = 0, blo = 0, bn = -1, nm = 0, nlo = 0, nn = -1;
        auto fetch_meta = [&](long long kb, int& fm, int& flo, int& fn) {
            const long long u = blockIdx.x + (kb + lane) * g;
            fn = -1;
            if (u < n_units) {
                fm = a.units[u].x;
                flo = a.row_ptr[fm];
                fn = a.row_ptr[fm + 1] - flo;
            }
        };
        fetch_meta(0, bm, blo, bn);
        fetch_meta(32, nm, nlo, nn);
        long long batch = 0;
        int rm[kBulkLook], rn[kBulkLook], ri[kBulkLook];
        float rw[kBulkLook];
        auto enter = [&](long long q, int d) {
            const int jq = static_cast<int>(q & 31);
            const bool here = (q >> 5) == batch;
            const int m = __shfl_sync(0xffffffffu, here ? bm : nm, jq);
            const int lo = __shfl_sync(0xffffffffu, here ? blo : nlo, jq);
            const int n = __shfl_sync(0xffffffffu, here ? bn : nn, jq);
            rm[d] = m;
            rn[d] = n;
            ri[d] = lane < n ? a.perm[lo + lane] : 0;
            rw[d] = 1.0f;
        };
#pragma unroll
        for (int d = 0; d < kBulkLook; ++d) enter(d, d);
        if (a.w) {
            if (lane < rn[0]) rw[0] = a.w[ri[0]];
            if (lane < rn[1]) rw[1] = a.w[ri[1]];
        }
        long long k = 0;      // items issued
        long long tail = 0;   // items known to be consumed (all items below it)
        long long pos = 0;    // unwrapped ring position of the next item
        long long cend = 0;   // unwrapped ring end of item tail - 1 (0 before any)
        bool ok = true;
        // Ring bytes [start, start + bytes) for item k, after the consumers
        // have freed them; false if a wait expired.
        auto reserve = [&](long long bytes, long long* start) -> bool {
            long long s0 = pos;
            const long long r = s0 % kAccRingBytes;
            if (r + bytes > kAccRingBytes) s0 += kAccRingBytes - r;  // items never wrap
            const long long e = s0 + bytes;
            while (tail + kAccSlots <= k || e > cend + kAccRingBytes) {
                const int ts = static_cast<int>(tail % kAccSlots);
                const uint32_t tph = static_cast<uint32_t>((tail / kAccSlots) & 1);
                const bool w_ok = mbar_wait_bounded(&empty[ts], tph);
                if (!__all_sync(0xffffffffu, w_ok) || *abort_flag) return false;
                cend = slot_end[ts];
                ++tail;
            }
            pos = e;
            *start = s0;
            return true;
        };
        for (long long ku = 0; ok && blockIdx.x + ku * g < n_units; ++ku) {
            const int cm = rm[0], cn = rn[0];
            const AccTile tl = tiles[cn];
            const unsigned char* xrow = lane < cn ? shard_row(tbl, ri[0], a.ldx_bytes) : nullptr;
            const unsigned char* orow = static_cast<const unsigned char*>(a.out) + static_cast<long long>(cm) * a.ldo * OSZ;
            for (int t = 0; t < tl.nt; ++t) {
                const int col0 = t * tl.te;
                const int elems = min(tl.te, a.H - col0);
                const long long bytes = static_cast<long long>(cn) * tl.stride + tl.obytes;
                long long start = 0;
                if (!reserve(bytes, &start)) { ok = false; break; }
                const int s = static_cast<int>(k % kAccSlots);
                const int off = static_cast<int>(start % kAccRingBytes);
                if (lane < cn) swt[s * kBulkMaxTerms + lane] = rw[0];
                if (lane == 0) {
                    meta[s] = AccMeta{cm, cn, col0, elems, off, tl.stride};
                    slot_end[s] = start + bytes;
                }
                __syncwarp();
                const uint32_t xb = static_cast<uint32_t>(elems * XSZ), ob = static_cast<uint32_t>(elems * OSZ);
                if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(cn) * xb + ob);
                __syncwarp();
                if (lane < cn)
                    bulk_g2s(ring + off + lane * tl.stride, xrow + static_cast<long long>(col0) * XSZ, xb, &full[s]);
                if (lane == 31)
                    bulk_g2s(ring + off + cn * tl.stride, orow + static_cast<long long>(col0) * OSZ, ob, &full[s]);
                ++k;
            }
            if (!ok) break;
            // advance: the list batch, the ring of units, the weights two units ahead
            const long long q = ku + kBulkLook;
            if ((q >> 5) > batch + 1) {
                batch += 1;
                bm = nm; blo = nlo; bn = nn;
                fetch_meta(32 * (batch + 1), nm, nlo, nn);
            }
#pragma unroll
            for (int d = 0; d + 1 < kBulkLook; ++d) {
                rm[d] = rm[d + 1]; rn[d] = rn[d + 1]; ri[d] = ri[d + 1]; rw[d] = rw[d + 1];
            }
            enter(q, kBulkLook - 1);
            if (a.w && lane < rn[1]) rw[1] = a.w[ri[1]];
        }
        if (ok) {
            // the end marker: an item of no terms in the next slot
            long long start = 0;
            ok = reserve(0, &start);
            if (ok) {
                const int s = static_cast<int>(k % kAccSlots);
                if (lane == 0) meta[s] = AccMeta{0, -1, 0, 0, 0, 0};
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
        for (long long j = max(tail, k - kAccSlots); j < k; ++j)
            mbar_wait_bounded(&full[j % kAccSlots], static_cast<uint32_t>((j / kAccSlots) & 1));
        return;
    }

    // ---------------- consumer warps ----------------
    const int ctid = threadIdx.x;  // 0 .. kBulkConsumers-1
    for (long long k = 0;; ++k) {
        const int s = static_cast<int>(k % kAccSlots);
        const uint32_t ph = static_cast<uint32_t>((k / kAccSlots) & 1);
        bool ok = false;
        for (unsigned long long it = 0; it < kBulkWaitLimit; ++it) {
            if (mbar_try_wait(&full[s], ph)) { ok = true; break; }
            if ((it & (kAccSpinCheck - 1)) == kAccSpinCheck - 1 && *abort_flag) break;
        }
        if (!ok || *abort_flag) {
            *abort_flag = 1;
            atomicOr(a.status + kCtrErrTimeout, 1);
            break;
        }
        const AccMeta md = meta[s];
        if (md.n < 0) break;  // no more items
        const unsigned char* buf = ring + md.off;
        const float* wts = swt + s * kBulkMaxTerms;
        const int nvec = md.elems * XSZ / 16;
        if (ctid < nvec) {
            float acc[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
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
            float old[VEC];
            acc_load_old<OT, VEC>(buf + md.n * md.stride + ctid * VEC * OSZ, old);
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[e] = __fadd_rn(old[e], acc[e]);
            bulk_store<OT, VEC>(a.out, static_cast<long long>(md.m) * a.ldo + md.col0 + ctid * VEC, acc, true);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

size_t bulk_acc_smem_bytes()
{
    return static_cast<size_t>(kAccRingBytes) + 2 * kAccSlots * sizeof(uint64_t) + kAccSlots * sizeof(long long) +
           kAccSlots * kBulkMaxTerms * sizeof(float) + kAccSlots * sizeof(AccMeta) +
           (kBulkMaxTerms + 1) * sizeof(AccTile) + 16;
}

template <typename XT, typename OT>
static det_status launch_bulk_acc_t(const BulkAccArgs& a, const ShardTable& t, int grid, cudaStream_t st)
{
    const size_t smem = bulk_acc_smem_bytes();
    {
        const det_status a_ =
            allow_dynamic_smem(reinterpret_cast<const void*>(gather_bulk_acc_kernel<XT, OT>), smem);
        if (a_) return a_;
        // all of the SM's shared memory: the register-staged kernel that runs
        // beside it needs the rest of it on the same SM
        static bool carve_set = false;
        if (!carve_set) {
            DETR_CUDA(cudaFuncSetAttribute(reinterpret_cast<const void*>(gather_bulk_acc_kernel<XT, OT>),
                                           cudaFuncAttributePreferredSharedMemoryCarveout, 100));
            carve_set = true;
        }
    }
    gather_bulk_acc_kernel<XT, OT><<<grid, kBulkThreads, smem, st>>>(a, t);
    DETR_LAUNCHED();
    return DET_OK;
}

det_status launch_gather_bulk_acc(det_dtype x_dtype, det_dtype out_dtype, const BulkAccArgs& a, const ShardTable& t,
                                  int grid, cudaStream_t st)
{
    if (x_dtype == DET_BF16 && out_dtype == DET_BF16) return launch_bulk_acc_t<uint16_t, __nv_bfloat16>(a, t, grid, st);
    if (x_dtype == DET_BF16) return launch_bulk_acc_t<uint16_t, float>(a, t, grid, st);
    if (out_dtype == DET_BF16) return launch_bulk_acc_t<float, __nv_bfloat16>(a, t, grid, st);
    return launch_bulk_acc_t<float, float>(a, t, grid, st);
}

}  // namespace detr
