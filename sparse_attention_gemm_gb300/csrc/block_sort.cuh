// block_sort.cuh -- block-wide helpers on shared memory: bitonic sort of
// 32-bit keys and an inclusive block scan.
#pragma once

#include <stdint.h>

namespace dsa {

// Sorts s[0 .. n) ascending in place; n must be a power of two.  All threads
// of the block call it; it ends with __syncthreads().
template <typename Key>
__device__ void bitonic_sort_smem(Key* s, int n) {
  __syncthreads();
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int ixj = i ^ j;
        if (ixj > i) {
          Key a = s[i], b = s[ixj];
          bool up = (i & k) == 0;
          if ((a > b) == up) {
            s[i] = b;
            s[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Inclusive prefix sum of one value per thread over the block (blockDim.x a
// multiple of 32, at most 1024).  `scratch` holds 32 ints of shared memory.
// Returns the inclusive sum for this thread; *total receives the block sum.
__device__ __forceinline__ int block_inclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int res = v + (warp > 0 ? scratch[warp - 1] : 0);
  if (total) *total = scratch[nwarps - 1];
  __syncthreads();
  return res;
}

}  // namespace dsa
