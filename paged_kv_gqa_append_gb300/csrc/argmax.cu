// Next-token argmax over FP32 logits ("Architecture et flux d'inference" of
// the samir-vllm article: the final logits are FP32 and a GPU argmax selects
// the next token).  Result per row: the first index of the largest non-NaN
// value; 0 when every value is NaN.
//
// One CTA per row.  Each thread keeps the best (value, index) of a strided
// share of the row (16-byte streaming loads when the row is 16-byte aligned);
// warp shuffles, then one shared-memory round, reduce the pairs under the
// same total order (larger value first, then lower index, NaN last), which
// is associative and commutative, so the result does not depend on the
// reduction order.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "pkv.h"

namespace pkv {
namespace {

constexpr int kArgThreads = 256;

// (v, i) before (bv, bi)?  bi < 0 marks "nothing yet"; a NaN never wins.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  if (i < 0 || isnan(v)) return false;
  if (bi < 0) return true;
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void take(float v, int i, float& bv, int& bi) {
  if (better(v, i, bv, bi)) {
    bv = v;
    bi = i;
  }
}

__global__ void __launch_bounds__(kArgThreads) argmax_kernel(const float* __restrict__ x, int vocab,
                                                             long long stride,
                                                             int32_t* __restrict__ out) {
  const float* row = x + (size_t)blockIdx.x * (size_t)stride;
  float bv = 0.f;
  int bi = -1;
  if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
    const int n4 = vocab / 4;
    const float4* r4 = reinterpret_cast<const float4*>(row);
    for (int k = threadIdx.x; k < n4; k += kArgThreads) {
      const float4 v = __ldcs(r4 + k);
      take(v.x, 4 * k, bv, bi);
      take(v.y, 4 * k + 1, bv, bi);
      take(v.z, 4 * k + 2, bv, bi);
      take(v.w, 4 * k + 3, bv, bi);
    }
    for (int i = 4 * n4 + threadIdx.x; i < vocab; i += kArgThreads) take(__ldcs(row + i), i, bv, bi);
  } else {
    for (int i = threadIdx.x; i < vocab; i += kArgThreads) take(__ldcs(row + i), i, bv, bi);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_down_sync(0xffffffffu, bv, o);
    const int oi = __shfl_down_sync(0xffffffffu, bi, o);
    take(ov, oi, bv, bi);
  }
  __shared__ float sv[kArgThreads / 32];
  __shared__ int si[kArgThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    bv = lane < kArgThreads / 32 ? sv[lane] : 0.f;
    bi = lane < kArgThreads / 32 ? si[lane] : -1;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      const float ov = __shfl_down_sync(0xffffffffu, bv, o);
      const int oi = __shfl_down_sync(0xffffffffu, bi, o);
      take(ov, oi, bv, bi);
    }
    if (lane == 0) out[blockIdx.x] = bi < 0 ? 0 : bi;
  }
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_argmax_f32(const float* logits, int rows, int vocab, long long row_stride,
                              int32_t* out_ids, void* stream) {
  if (rows < 0 || vocab < 1 || row_stride < vocab) return PKV_ERR_INVALID_ARGUMENT;
  if (rows == 0) return PKV_OK;
  if (!logits || !out_ids) return PKV_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) || (reinterpret_cast<uintptr_t>(out_ids) & 3u))
    return PKV_ERR_MISALIGNED;
  int dev = 0;
  const int rc = pkv::bind_stream_device(stream, &dev);
  if (rc != PKV_OK) return rc;
  pkv::argmax_kernel<<<rows, pkv::kArgThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      logits, vocab, row_stride, out_ids);
  return pkv::cuda_status(cudaGetLastError(), "argmax_kernel");
}
