// Host-side helpers shared by the C-ABI entry points (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Make the device that owns `stream` current for this thread (the current
// device is kept for the legacy default stream).  Returns PKV_OK or
// PKV_ERR_CUDA.
int bind_stream_device(void* stream, int* device_out);

// Number of SMs of `device` (cached after the first query).
int sm_count(int device);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Remember a failure description for pkv_last_error() (per thread).
void set_last_error(const char* where, const char* what);

inline int cuda_status(cudaError_t e, const char* where = "cuda") {
  if (e == cudaSuccess) return PKV_OK;
  set_last_error(where, cudaGetErrorString(e));
  (void)cudaGetLastError();  // clear the non-sticky error state for the next call
  return PKV_ERR_CUDA;
}

// TMA tensor map of the pool [num_pages][2][8][16][64] bf16 viewed as
// (dim 64, slot 16, head 8, page * 2 + kv), box {64, 16, 1, 2} (the K then V
// tile of one (page, head)), 128-byte swizzle; cached per thread for the
// last (pool, num_pages).  Returns PKV_OK or PKV_ERR_CUDA.
int make_pool_map(CUtensorMap* map, const void* pool, int num_pages);
// The same view with a one-tile box {64, 16, 1, 1}.
int make_pool_tile_map(CUtensorMap* map, const void* pool, int num_pages);

// The host-side argument checks of paged_gqa_decode that need no workspace
// and no CUDA call (sizes, null pointers, alignment, the scale): PKV_OK or
// the status the decode call would return for these arguments.
int decode_check_args(const void* q, const void* kv_pool, int num_pages,
                      const int32_t* block_tables, int bt_row_stride, int max_blocks,
                      const int32_t* seq_lens, int num_seqs, const void* out, float scale);
}  // namespace pkv
