// Block-wide exclusive prefix sum for blocks of up to 1024 threads (a
// multiple of 32).  Two barriers; `scratch` holds 33 ints of shared memory.
#pragma once

#include <stdint.h>

namespace isk {

template <typename I>
__device__ __forceinline__ I block_exclusive_scan(I x, I* scratch, I* total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  I inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const I y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    I w = lane < nwarps ? scratch[lane] : I(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const I y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;                 // inclusive warp totals
  }
  __syncthreads();
  const I before = warp > 0 ? scratch[warp - 1] : I(0);
  *total = scratch[nwarps - 1];
  __syncthreads();                     // scratch may be reused right after
  return before + inc - x;
}

// The same sum with one barrier: each warp scans with shuffles and publishes
// its total; after the barrier every thread adds up the totals of the warps
// before its own.  `scratch` holds NWARPS ints and is read after the barrier,
// so it may be written again only once every thread has passed a later
// barrier: back-to-back calls alternate between two buffers.
template <int NWARPS, typename I>
__device__ __forceinline__ I block_exclusive_scan_1bar(I x, I* scratch, I* total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  I inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const I y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  I before = I(0), tot = I(0);
#pragma unroll
  for (int w = 0; w < NWARPS; ++w) {
    const I t = scratch[w];
    if (w < warp) before += t;
    tot += t;
  }
  *total = tot;
  return before + inc - x;
}

}  // namespace isk
