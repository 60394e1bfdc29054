// The pool's TMA tensor map, shared by the decode and prefill kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>
#include <stdio.h>

#include "internal.h"

namespace pkv {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    else
      (void)cudaGetLastError();
  });
  return fn;
}

// Pool viewed as a 4-D tensor: dim (64), token slot (16), head (8),
// page * 2 + kv.  One box {64, 16, 1, 2} = the K and V tiles of one (page,
// head), 2 x 2 KiB, stored in shared memory with the 128-byte swizzle (16
// rows of 128 bytes each, so the V tile starts a fresh swizzle period).
int make_pool_map(CUtensorMap* map, const void* pool, int num_pages) {
  struct Cached {
    const void* ptr = nullptr;
    int pages = 0;
    CUtensorMap map;
  };
  static thread_local Cached cache;
  if (cache.ptr == pool && cache.pages == num_pages) {
    *map = cache.map;
    return PKV_OK;
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) {
    set_last_error("cudaGetDriverEntryPointByVersion", "cuTensorMapEncodeTiled unavailable");
    return PKV_ERR_CUDA;
  }
  // (dim, token, head, 2 page + K/V): one box {64, 16, 1, 2} is the K tile and
  // then the V tile of one (page, head), 4 KiB, in a single copy
  const cuuint64_t dims[4] = {64, 16, PKV_NUM_KV_HEADS, (cuuint64_t)num_pages * 2};
  const cuuint64_t strides[3] = {128, 2048, 2048 * PKV_NUM_KV_HEADS};
  const cuuint32_t box[4] = {64, 16, 1, 2};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[64];
    snprintf(msg, sizeof(msg), "CUresult %d", (int)r);
    set_last_error("cuTensorMapEncodeTiled", msg);
    return PKV_ERR_CUDA;
  }
  cache.ptr = pool;
  cache.pages = num_pages;
  cache.map = *map;
  return PKV_OK;
}

// The same view with a one-tile box {64, 16, 1, 1}: the K tile (kv = 0) or
// the V tile (kv = 1) of one (page, head) alone, so that the tiles of
// consecutive pages can be placed back to back in shared memory.
int make_pool_tile_map(CUtensorMap* map, const void* pool, int num_pages) {
  struct Cached {
    const void* ptr = nullptr;
    int pages = 0;
    CUtensorMap map;
  };
  static thread_local Cached cache;
  if (cache.ptr == pool && cache.pages == num_pages) {
    *map = cache.map;
    return PKV_OK;
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) {
    set_last_error("cudaGetDriverEntryPointByVersion", "cuTensorMapEncodeTiled unavailable");
    return PKV_ERR_CUDA;
  }
  // (dim, token, head, 2 page + K/V): one box {64, 16, 1, 2} is the K tile and
  // then the V tile of one (page, head), 4 KiB, in a single copy
  const cuuint64_t dims[4] = {64, 16, PKV_NUM_KV_HEADS, (cuuint64_t)num_pages * 2};
  const cuuint64_t strides[3] = {128, 2048, 2048 * PKV_NUM_KV_HEADS};
  const cuuint32_t box[4] = {64, 16, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[64];
    snprintf(msg, sizeof(msg), "CUresult %d", (int)r);
    set_last_error("cuTensorMapEncodeTiled", msg);
    return PKV_ERR_CUDA;
  }
  cache.ptr = pool;
  cache.pages = num_pages;
  cache.map = *map;
  return PKV_OK;
}

}  // namespace pkv
