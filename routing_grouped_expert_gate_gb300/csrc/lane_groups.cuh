// Reductions over a group of G consecutive lanes of a warp (G a power of two
// up to 32; G = 32 is the whole warp, in the same order as warp_max/warp_sum).
#pragma once

#include <cuda_runtime.h>

namespace moe {

template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o, G));
  return v;
}
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o, G);
  return v;
}

}  // namespace moe
