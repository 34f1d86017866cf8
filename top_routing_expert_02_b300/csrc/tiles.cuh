// Tile bookkeeping for grouped GEMMs over variable-length expert segments.
//
// Expert e owns rows [offsets[e], offsets[e] + kept[e]) of the permuted
// buffers.  Its rows are cut into ceil(kept[e] / BM) M-tiles; mstart[] is the
// running count of M-tiles (mstart[0] = 0, mstart[E] = all M-tiles).  The
// table is rebuilt on the device from kept[] by every block, so no host
// round trip is needed to learn the segment sizes.
#pragma once
#include "common.cuh"

// Warp-wide inclusive scan of ceil(kept / BM); writes mstart[0..E].
template <int BM>
__device__ __forceinline__ void build_mtile_prefix(const int32_t* __restrict__ kept, int E, int* mstart,
                                                   int lane)
{
    int carry = 0;
    for (int b = 0; b < E; b += 32) {
        const int e = b + lane;
        int v = (e < E) ? (__ldg(kept + e) + BM - 1) / BM : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int nb = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += nb;
        }
        if (e < E) mstart[e + 1] = carry + v;
        carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) mstart[0] = 0;
}

// Largest e with mstart[e] <= mt  (i.e. mstart[e] <= mt < mstart[e+1]).
__device__ __forceinline__ int find_expert(const int* mstart, int E, int mt)
{
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (mstart[mid] <= mt) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}
