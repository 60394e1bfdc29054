// INT8 quantisation of one (token, KV head) row, shared by the INT8 append
// and the fused INT8 decode step so that both write identical bytes: amax =
// max |x|, scale = amax / 127 and code = round-half-even(x / scale) clamped to
// [-127, 127], both divisions IEEE fp32; amax == 0 gives scale 0 and zero
// codes.
#pragma once

#include <stdint.h>

namespace pkv {

// Codes of the two values x0 (dim lane) and x1 (dim lane + 32) of a row held
// across the warp, and the row's scale.
__device__ __forceinline__ float quantize_pair(float x0, float x1, int8_t& c0, int8_t& c1) {
  const uint32_t a = max(__float_as_uint(x0) & 0x7FFFFFFFu, __float_as_uint(x1) & 0x7FFFFFFFu);
  const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, a));  // |x| bits order as |x|
  const float scale = __fdiv_rn(amax, 127.f);
  if (amax == 0.f) {
    c0 = c1 = 0;
    return 0.f;
  }
  c0 = (int8_t)max(-127, min(127, __float2int_rn(__fdiv_rn(x0, scale))));
  c1 = (int8_t)max(-127, min(127, __float2int_rn(__fdiv_rn(x1, scale))));
  return scale;
}

}  // namespace pkv
