// Byte format of one INT8 (page, KV head) block of the pool, PKV_I8_BLOCK_BYTES
// = 2176 bytes ("Lifecycle and Memory Model", section "Per-request /
// handle-owned memory", names INT8 K/V storage; the format is this library's).
// Written by kv_append_rope_int8 and the fused INT8 decode step, read by the
// INT8 decode.
//
//   * a code c in [-127, 127] is stored as the byte c + 128;
//   * K codes, bytes 0 .. 1023: slot t, dim d at 64 t + d;
//   * V codes, bytes 1024 .. 2047, by slot pairs: slot t is member t % 2 of
//     pair p = t / 2, and dim d of a pair is the byte pair at
//       1024 + 128 p + 16 ((d % 8) ^ (2 (p % 4))) + 2 (d / 8) + member;
//   * scales, bytes 2048 .. 2175, fp32, in groups of four: group j = 0..7
//     at 2048 + 16 j holds the K scales of slots j and j + 8, then their V
//     scales.
//
// Why: decode lane (g8, c) = (lane / 4, lane % 4) multiplies rows g8 and
// g8 + 8 of the page (S^T = K q'^T), whose K codes it reads as two 16-byte
// rows, and whose four scales are one 16-byte group; for O^T = V^T P'^T it
// needs dims g8 + 8 j (j = 0..7) of the slot pairs c and c + 4, which are one
// 16-byte chunk of each pair.  The XOR spreads the eight lanes of a
// quarter-warp over all 32 banks.
#pragma once

#include <stdint.h>

namespace pkv {

__host__ __device__ constexpr uint32_t i8_k_byte(int t, int d) { return 64u * (uint32_t)t + (uint32_t)d; }
__host__ __device__ constexpr uint32_t i8_v_byte(int t, int d) {
  return 1024u + 128u * (uint32_t)(t >> 1) + 16u * (uint32_t)((d & 7) ^ (2 * ((t >> 1) & 3))) +
         2u * (uint32_t)(d >> 3) + (uint32_t)(t & 1);
}
__host__ __device__ constexpr uint32_t i8_k_scale_byte(int t) {
  return 2048u + 16u * (uint32_t)(t & 7) + 4u * (uint32_t)(t >> 3);
}
__host__ __device__ constexpr uint32_t i8_v_scale_byte(int t) { return i8_k_scale_byte(t) + 8u; }

// the stored byte of a code
__host__ __device__ constexpr uint8_t i8_code_byte(int8_t code) { return (uint8_t)((uint8_t)code ^ 0x80u); }

}  // namespace pkv
