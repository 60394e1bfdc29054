// RoPE rotation of one bf16 pair, shared by the append and the fused
// decode-with-append kernels so that both write identical bytes.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace pkv {

// r0 = x0*c - x1*s, r1 = x0*s + x1*c, every operation rounded to nearest in
// fp32 (no contraction into FMA), then rounded to bf16 nearest-even.  Pairs
// are (i, i + 32) of a 64-wide head (half-split convention).
__device__ __forceinline__ void rope_pair(uint16_t x0b, uint16_t x1b, float c, float s,
                                          uint16_t& r0b, uint16_t& r1b) {
  const float x0 = __uint_as_float((uint32_t)x0b << 16);
  const float x1 = __uint_as_float((uint32_t)x1b << 16);
  const float r0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
  const float r1 = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
  r0b = __bfloat16_as_ushort(__float2bfloat16_rn(r0));
  r1b = __bfloat16_as_ushort(__float2bfloat16_rn(r1));
}

}  // namespace pkv
