// The pool's TMA tensor maps, shared by the decode and prefill kernels.
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

// One encoded map per (base pointer, extent) and kind, cached per thread:
// the encode is a host-side driver call of a few microseconds.
struct MapCache {
  const void* ptr = nullptr;
  long long extent = -1;
  CUtensorMap map;
};

static int encode_4d(MapCache& cache, CUtensorMap* map, const void* base, long long extent,
                     const cuuint64_t (&dims)[4], const cuuint64_t (&strides)[3],
                     const cuuint32_t (&box)[4], CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  if (cache.ptr == base && cache.extent == extent) {
    *map = cache.map;
    return PKV_OK;
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) {
    set_last_error("cudaGetDriverEntryPointByVersion", "cuTensorMapEncodeTiled unavailable");
    return PKV_ERR_CUDA;
  }
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, dtype, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[64];
    snprintf(msg, sizeof(msg), "CUresult %d", (int)r);
    set_last_error("cuTensorMapEncodeTiled", msg);
    return PKV_ERR_CUDA;
  }
  cache.ptr = base;
  cache.extent = extent;
  cache.map = *map;
  return PKV_OK;
}

// Pool viewed as a 4-D tensor: dim (64), token slot (16), head (8),
// page * 2 + kv.  One box {64, 16, 1, 2} = the K and V tiles of one (page,
// head), 2 x 2 KiB, stored in shared memory with the 128-byte swizzle (16
// rows of 128 bytes each, so the V tile starts a fresh swizzle period).
int make_pool_map(CUtensorMap* map, const void* pool, int num_pages) {
  static thread_local MapCache cache;
  const cuuint64_t dims[4] = {64, 16, PKV_NUM_KV_HEADS, (cuuint64_t)num_pages * 2};
  const cuuint64_t strides[3] = {128, 2048, 2048 * PKV_NUM_KV_HEADS};
  const cuuint32_t box[4] = {64, 16, 1, 2};
  return encode_4d(cache, map, pool, num_pages, dims, strides, box);
}

// The same view with a one-tile box {64, 16, 1, 1}: the K tile (kv = 0) or
// the V tile (kv = 1) of one (page, head) alone, so that the tiles of
// consecutive pages can be placed back to back in shared memory.
int make_pool_tile_map(CUtensorMap* map, const void* pool, int num_pages) {
  static thread_local MapCache cache;
  const cuuint64_t dims[4] = {64, 16, PKV_NUM_KV_HEADS, (cuuint64_t)num_pages * 2};
  const cuuint64_t strides[3] = {128, 2048, 2048 * PKV_NUM_KV_HEADS};
  const cuuint32_t box[4] = {64, 16, 1, 1};
  return encode_4d(cache, map, pool, num_pages, dims, strides, box);
}

}  // namespace pkv
