// Warp arg-max by reduction: an order-preserving unsigned key of a float lets redux.sync (a warp
// max / min over 32-bit integers) find the largest value and then the smallest index holding it.
#pragma once

#include <cstdint>

namespace dfl {

// Order-preserving unsigned key of a float, -0.0 counted as +0.0 so that equal values tie;
// key_float inverts it.
__device__ __forceinline__ uint32_t float_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Over the lanes with `active`: the largest key, then the smallest `index` among the lanes holding
// it (every lane gets both). Inactive lanes take part with key 0, below every float's key.
__device__ __forceinline__ void warp_max_min_index(uint32_t key, bool active, uint32_t index, uint32_t& kmax,
                                                   uint32_t& imin) {
  kmax = __reduce_max_sync(0xffffffffu, active ? key : 0u);
  imin = __reduce_min_sync(0xffffffffu, (active && key == kmax) ? index : 0xffffffffu);
}

}  // namespace dfl
