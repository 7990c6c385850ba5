// Block-wide exclusive prefix sum for 1024-thread blocks, in thread order (deterministic).
#pragma once
#include <cstdint>

namespace ds {

// Returns the exclusive prefix of `v` over threads 0..threadIdx.x-1 and writes the block
// total to *total.  Needs 33 ints of shared scratch; all threads of the block must call it.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T *scratch, T *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        T w = lane < nwarps ? scratch[lane] : T(0);
        T s = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            T y = __shfl_up_sync(0xFFFFFFFFu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < nwarps) scratch[lane] = s - w;   // exclusive warp offsets
        if (lane == 31) scratch[32] = s;
    }
    __syncthreads();
    const T res = scratch[warp] + x - v;
    *total = scratch[32];
    __syncthreads();
    return res;
}

// Cumulative boundaries for an inverse-CDF search over per-thread masses v >= 0: buf[t] is the
// exclusive prefix of thread t (parallel scan, fixed order) and buf[blockDim.x] the total.
// Thread t's interval is [buf[t], buf[t+1]); read both ends from buf.  Consecutive intervals
// cover [0, total) even where rounding makes the sequence dip, so a target in range falls in at
// least one of them; take the lowest such thread.  buf holds blockDim.x + 1 floats; scratch 33.
__device__ __forceinline__ void block_cdf_bounds(float v, float *buf, float *scratch)
{
    float tot;
    const float ex = block_exclusive_scan(v, scratch, &tot);
    buf[threadIdx.x] = ex;
    if (threadIdx.x == 0) buf[blockDim.x] = tot;
    __syncthreads();
}

}  // namespace ds
