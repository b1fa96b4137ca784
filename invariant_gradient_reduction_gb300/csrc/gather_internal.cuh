// gather_internal.cuh -- entry of the TMA-staged gather-reduce (gather_bulk.cu)
// used by the dispatcher in gather.cu.
#pragma once

#include <algorithm>

#include "common.cuh"
#include "plan_internal.cuh"

namespace detr {

// Arguments of the warp-task gather-reduce kernels (gather.cu, gather_async.cu).
struct GatherArgs {
    const int4* seg_units;
    const int4* row_units;
    long long n_seg;      // units below n_seg have more than one chunk (hot segments, then long rows)
    long long n_tasks;
    int tile_groups;      // task groups per whole-row unit
    int tiles_per_group;
    int seg_tile_groups;  // task groups per hot-segment unit (segments are the longest units)
    int seg_tiles_per_group;
    int ntiles;           // H-tiles per row
    int H;
    int T_log2;           // lanes per H-tile (row vector count)
    int S_log2;           // chunk slots per warp = 32 >> T_log2
    int g;                // a segment covers 2^g chunks
    int out_vec;          // vector stores to out allowed
    int levels;           // binary-counter levels a unit can need (floor(log2(rounds)) + 1)
    const int* row_ptr;
    const int* perm;
    const float* w;
    long long ldx_bytes;
    void* out;
    long long ldo;
    float* part;
    long long ldpart;
    const int* dev_counters;  // non-null: read the work counts (and plan errors) from the device
    int accumulate;           // add to out (index_add_); destinations without terms stay untouched
    int only_long;            // behind the fixed-stage bulk kernel of an unwaited plan: no work unless some
                              // destination has more than 32 terms (the bulk kernel did nothing then)
    int beside_ring;          // beside the ring kernel, which takes the one-chunk units: only the units of
                              // more than one chunk, and the wait for the previous grid (the ring kernel;
                              // everything before it had finished when it started) at the end
};

// Work counts of a launch: from the host, or from the plan's counter block
// when the plan did not wait.  Returns false if the plan recorded an error
// (the kernel then writes nothing).
__device__ __forceinline__ bool task_counts(const GatherArgs& a, long long* n_tasks, long long* n_seg)
{
    *n_tasks = a.n_tasks;
    *n_seg = a.n_seg;
    if (a.dev_counters) {
        const int* c = a.dev_counters;
        if (c[kCtrErrIndex] | c[kCtrErrDup] | c[kCtrErrTimeout]) return false;
        *n_seg = c[kCtrBig];
        // index_add_ has nothing to do for the empty destinations (listed last)
        if (a.only_long && c[kCtrMaxLen] <= kChunk) {
            *n_tasks = 0;
            return true;
        }
        *n_tasks = static_cast<long long>(c[kCtrBig]) * a.seg_tile_groups +
                   (a.beside_ring ? 0LL
                                  : static_cast<long long>(c[kCtrShort] + (a.accumulate ? 0 : c[kCtrEmpty])) *
                                        a.tile_groups);
    }
    return true;
}

// Vector-path gather with per-lane asynchronous copies into a shared-memory ring.
size_t async_smem_bytes(int S_log2, int levels, int vec);
det_status launch_gather_async(det_dtype x_dtype, det_dtype out_dtype, const GatherArgs& a,
                               const ShardTable& t, int grid, cudaStream_t st);
constexpr int kAsyncWarps = 4;

struct BulkArgs {
    const int4* units;     // whole-destination units (every list has <= 32 terms, so no segments)
    long long n_items;     // units x tiles
    int ntiles;            // H-tiles per row
    int tile_elems;        // elements per H-tile (the last tile may be shorter)
    int tile_stride;       // bytes between staged rows in shared memory (128-byte multiple)
    int H;
    int out_vec;
    const int* row_ptr;
    const int* perm;
    const float* w;
    long long ldx_bytes;
    void* out;
    long long ldo;
    int* status;           // counter block; kCtrErrTimeout is set if a bounded wait expires
    const int* dev_counters;  // non-null (plan that did not wait): the items and the tiling follow from the
                              // counter block; none when some destination has more than 32 terms
};

// Task -> (unit, first and one-past-last H-tile): the units of more than one
// chunk first (hot segments, then long rows), each in seg_tile_groups tasks,
// then the short whole-row units in tile_groups tasks.
__device__ __forceinline__ long long task_unit(const GatherArgs& a, long long task, long long n_seg, int* t0, int* t1)
{
    const long long seg_tasks = n_seg * a.seg_tile_groups;
    long long u;
    int tg, tpg;
    if (task < seg_tasks) {
        u = task / a.seg_tile_groups;
        tg = static_cast<int>(task - u * a.seg_tile_groups);
        tpg = a.seg_tiles_per_group;
    } else {
        const long long r = task - seg_tasks;
        const long long ur = r / a.tile_groups;
        tg = static_cast<int>(r - ur * a.tile_groups);
        tpg = a.tiles_per_group;
        u = n_seg + ur;
    }
    *t0 = tg * tpg;
    *t1 = min(*t0 + tpg, a.ntiles);
    return u;
}

__device__ __forceinline__ int4 unit_at(const GatherArgs& a, long long u, long long n_seg)
{
    return u < n_seg ? a.seg_units[u] : a.row_units[u - n_seg];
}

// The fixed-stage kernel runs two producer warps from this many items per CTA
// (one below); with sources in several shards only two keep up with the
// per-term shard lookups, so auto takes it for shards from there.
constexpr int kBulkTwoProducerItems = 64;

size_t bulk_smem_bytes();
// Tile a row of H elements so that max_terms staged tiles fit one stage; false if not possible.
bool bulk_plan_tiles(int64_t H, int xsz, int64_t max_terms, int* tile_elems, int* tile_stride, int* ntiles);
// dependent: launched as a programmatic dependent of the kernel before it
// (the kernel waits for that one before it reads anything).
det_status launch_gather_bulk(det_dtype x_dtype, det_dtype out_dtype, const BulkArgs& a, const ShardTable& t,
                              int grid, bool dependent, cudaStream_t st);

// The destinations of at most one chunk (1..32 terms; for the scatter-reduce
// also those without terms), TMA-staged: each item is a destination's H-tile
// with its term tiles (and, for index_add_, the old destination tile), packed
// into a byte ring of shared memory.
struct RingArgs {
    const int4* units;     // the one-chunk whole-destination units (row_units[0 .. n_units))
    long long n_units;
    int H;
    int quantum;           // tile widths are multiples of this many elements (16-byte copies)
    int ring_bytes;        // shared-memory ring: a multiple of 128, at least 128 KB
    const int* row_ptr;
    const int* perm;
    const float* w;
    long long ldx_bytes;
    void* out;             // 16-byte aligned rows (ldo * sizeof(out) a multiple of 16)
    long long ldo;
    int* status;           // counter block; kCtrErrTimeout is set if a bounded wait expires
    const int* dev_counters;  // non-null (plan that did not wait): n_units is the block's count of
                              // such units, or 0 if the plan recorded an error
    int dependent;            // launched as a programmatic dependent of the kernel before it (the plan)
};

size_t ring_smem_bytes(int ring_bytes);
det_status launch_gather_ring(det_dtype x_dtype, det_dtype out_dtype, bool accumulate, const RingArgs& a,
                              const ShardTable& t, int grid, cudaStream_t st);

}  // namespace detr
