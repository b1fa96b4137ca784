// plan_internal.cuh -- the plan handle and the device counter block, shared by
// plan.cu (which builds a plan) and gather.cu (which runs it).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <vector_types.h>

#include "det_reduce.h"

namespace detr {

// int32 counter block at the start of the plan workspace.
enum {
    kCtrErrIndex = 0,  // some idx outside [0, M)
    kCtrErrDup = 1,    // two sources of one destination share an order key
    kCtrSegs = 2,      // hot segments (units that write partial slots)
    kCtrNormal = 3,    // whole-destination units
    kCtrHot = 4,       // destinations split into segments (finish tasks)
    kCtrMaxLen = 5,    // longest destination list
    kCtrErrTimeout = 6,  // a bounded wait inside a reduce kernel expired
    kCtrLong = 7,      // whole-destination units of 2..2^g chunks (in seg_units, after the segments)
    kCtrBig = 8,       // units of more than one chunk: hot segments + long whole rows
    kCtrShort = 9,     // whole-destination units of 1..32 terms (row_units)
    kCtrEmpty = 10,    // destinations without terms (row_units, after the short ones)
    kCtrRingNext = 11, // index_add ring kernel: next unclaimed chunk of units (0 between calls)
    kCtrRingDone = 12, // index_add ring kernel: CTAs finished (0 between calls)
    kCtrCount = 16
};

// Single-cluster plan (plan_cluster.cu): up to kCluMaxCtas CTAs of 1024
// threads, each holding a slice of at most kCluMaxSlice sources (about
// kCluTargetSlice when there are enough sources) and at most
// kCluRowsPerThread destinations per thread.
constexpr int kCluMaxCtas = 16;
constexpr int kCluMaxSlice = 8192;
constexpr int kCluTargetSlice = 2048;
constexpr int kCluRowsPerThread = 8;

constexpr int kCluThreads = 1024;  // threads of every CTA of a cluster kernel

// Cluster kernels of the library, each with its own cache of whether the
// device can schedule it.
enum {
    kCluVariantTwoPass = 0,    // plan_cluster_kernel
    kCluVariantOnePass = 1,    // plan_cluster_one_kernel
    kCluVariantRoute = 2,      // route_cluster_kernel, one variant per items-per-thread count (4 of them)
    kCluVariants = 6
};

// Launches a kernel of kCluThreads-thread CTAs on one cluster of C CTAs with
// `smem` bytes of dynamic shared memory (args as for cudaLaunchKernel).
// *launched stays false if the device cannot schedule such a cluster; the
// answer is cached per (variant, device, C).
det_status launch_on_cluster(int variant, const void* kern, int C, size_t smem, cudaStream_t st, void** args,
                             bool* launched);

// CTAs the single-cluster plan would use for (N, M); 0 where it does not apply.
int plan_cluster_ctas(int64_t N, int64_t M);

// Enqueues the single-cluster plan when it applies and the device can
// schedule the cluster (*launched = true); otherwise does nothing.  The
// single-pass kernel is taken where it applies; the two-pass kernel only when
// two_pass is set.  Writes row_ptr, perm, the three unit arrays and the whole
// counter block.
det_status launch_plan_cluster(const int32_t* idx, int64_t N, int64_t M, int g, int np32, int* row_ptr, int* perm,
                               int4* seg_units, int4* row_units, int4* finish, int* counters, bool two_pass,
                               cudaStream_t st, bool* launched);

// Owner plan (plan_owner.cu): clusters of 8, 4 or 2 CTAs (one per SM) each
// own at most kOwnMaxRows consecutive destinations and together read all
// N <= kOwnMaxN sources; M <= kOwnMaxM (a full histogram per CTA).
constexpr int64_t kOwnMaxN = int64_t(1) << 18;
constexpr int64_t kOwnMaxM = int64_t(1) << 15;
constexpr int kOwnMaxRows = 1024;

// Enqueues the owner plan (one kernel) when it applies and the device can
// schedule its clusters (*launched = true); otherwise does nothing.  Writes
// row_ptr, perm, the three unit arrays and the whole counter block.
det_status launch_plan_owner(const int32_t* idx, int64_t N, int64_t M, int g, int* row_ptr, int* perm,
                             int4* seg_units, int4* row_units, int4* finish, int* counters, cudaStream_t st,
                             bool* launched);

// Radix plan (plan_radix.cu): no order keys, 1 <= N < 2^24, M <= 65536.
struct RadixBuffers {
    int* counts;     // [256][tiles]
    int* tbad;       // [tiles]
    int* totals0;    // [256]
    int* totals1;    // [256]
    int* packed;     // [N]
    unsigned char* lowd;  // [N], 16-byte aligned: the low digit of each packed word
    int* perm;       // [N]
    int* rowcnt;     // [M]
    int* btot;       // [plan_radix_blocks(M) * 8]
    int* row_ptr;    // [M+1]
    int4* seg_units;
    int4* row_units;
    int4* finish;
    int* counters;
};
bool plan_radix_applies(int64_t N, int64_t M);
int64_t plan_radix_tiles(int64_t N);
int64_t plan_radix_blocks(int64_t M);
// Enqueues the radix plan (DET_ERR_UNSUPPORTED where it does not apply).
// Writes row_ptr, perm, the three unit arrays and the whole counter block.
det_status launch_plan_radix(const int32_t* idx, int64_t N, int64_t M, int g, const RadixBuffers& b,
                             cudaStream_t st);

}  // namespace detr

// Host handle.  Device arrays live in the caller's plan workspace.
//   seg_units[u] = {row m, segment s, partial slot, 0} for the hot segments,
//                  then {row m, -1, 0, 0} for the n_long whole-row units of
//                  2..2^g chunks: the units with more than one chunk;
//   row_units[u] = {row m, -1, 0, 0} for the other whole-row units: those
//                  with terms, then the empty ones (which index_add skips);
//   finish[k]    = {row m, first partial slot, number of segments, 0}.
// Work unit u of the reduce is seg_units[u] for u < n_segments + n_long,
// else row_units[u - n_segments - n_long] (the longest units first).
struct det_plan_s {
    int64_t N = 0, M = 0;
    int g = 3;                       // a hot segment covers 2^g chunks of 32 terms
    unsigned char* ws = nullptr;
    size_t ws_bytes = 0;
    int* counters = nullptr;         // [kCtrCount]
    int* row_ptr = nullptr;          // [M+1]
    int* perm = nullptr;             // [N]
    int4* seg_units = nullptr;
    int4* row_units = nullptr;
    int4* finish = nullptr;
    int64_t n_units = 0, n_segments = 0, n_hot_rows = 0, max_row_len = 0, n_long = 0, n_empty = 0;
    bool counts_on_host = true;      // false for an async plan until det_plan_status
    bool late_release = false;       // built by a kernel that lets the kernel after it start only for its
                                     // last phase (the owner plan, the two-pass cluster plan, the route
                                     // cluster kernel)
};
