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

}  // namespace isk
