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

}  // namespace ds
