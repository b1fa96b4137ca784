// block_scan.cuh -- block scan and warp ranking primitives of the plan kernels.
#pragma once

namespace detr {

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

// Exclusive scans of NV ints per thread over a block of NT threads at once;
// tot gets the block sums.  `ws` is shared scratch of NV * (NT/32 + 1) ints.
// Ends synchronised.
template <int NT, int NV>
__device__ __forceinline__ void block_excl_scan_n(int v[NV], int* ws, int tot[NV])
{
    constexpr int W = NT / 32;
    static_assert(NV <= W && W <= 32, "one warp per value scans the warp sums");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        incl[j] = v[j];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl[j], o);
            if (lane >= o) incl[j] += t;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int j = 0; j < NV; ++j) ws[j * (W + 1) + warp] = incl[j];
    }
    __syncthreads();
    if (warp < NV) {
        const int s = lane < W ? ws[warp * (W + 1) + lane] : 0;
        int si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, si, o);
            if (lane >= o) si += t;
        }
        if (lane < W) ws[warp * (W + 1) + lane] = si - s;
        if (lane == 31) ws[warp * (W + 1) + W] = si;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        tot[j] = ws[j * (W + 1) + W];
        v[j] = incl[j] - v[j] + ws[j * (W + 1) + warp];
    }
    __syncthreads();
}

// Lanes among `live` holding the same 8-bit digit as this lane, from one
// ballot per digit bit.  Warp votes are the ranking's main cost (measured on
// GB300: a few cycles each per SM sub-partition, while one match.any costs
// about 250), so there is no separate vote for
// validity and callers skip items that no lane holds.
__device__ __forceinline__ unsigned int digit_peers(int d, unsigned int live)
{
    unsigned int peers = live;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const unsigned int set = __ballot_sync(0xffffffffu, (d >> b) & 1);
        peers &= ((d >> b) & 1) ? set : ~set;
    }
    return peers;
}

}  // namespace detr
