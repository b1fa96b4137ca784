// gather_internal.cuh -- entry of the TMA-staged gather-reduce (gather_bulk.cu)
// used by the dispatcher in gather.cu.
#pragma once

#include <algorithm>

#include "common.cuh"

namespace detr {

struct BulkArgs {
    const int4* units;     // whole-destination units (every list has <= 32 terms)
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
};

size_t bulk_smem_bytes();
// Tile a row of H elements so that max_terms staged tiles fit one stage; false if not possible.
bool bulk_plan_tiles(int64_t H, int xsz, int64_t max_terms, int* tile_elems, int* tile_stride, int* ntiles);
det_status launch_gather_bulk(det_dtype x_dtype, det_dtype out_dtype, const BulkArgs& a, const ShardTable& t,
                              int grid, cudaStream_t st);

}  // namespace detr
