// Next-token argmax over FP32 logits ("Architecture et flux d'inference" of
// the samir-vllm article: the final logits are FP32 and a GPU argmax selects
// the next token).  Result per row: the first index of the largest non-NaN
// value; 0 when every value is NaN.
//
// Few rows (fewer than two per SM): a cluster of kClusterCtas CTAs per row,
// each reducing one contiguous part; the parts' results meet in the first
// CTA's shared memory (distributed shared memory) after a cluster barrier.
// Many rows: one CTA per row.  Inside a CTA each thread keeps the best
// (value, index) of a strided share (16-byte streaming loads, four in flight,
// when the part is 16-byte aligned); warp shuffles, then one shared-memory
// round, reduce the
// pairs under the same total order (larger value first, then lower index,
// NaN last), which is associative and commutative, so the result does not
// depend on the reduction order.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "pkv.h"

namespace pkv {
namespace {

constexpr int kArgThreads = 512;
static_assert(kArgThreads % 64 == 0 && kArgThreads <= 1024, "warps reduced by one warp");
constexpr int kClusterCtas = 8;

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

// Four consecutive elements starting at index `base`, later in this thread's
// share than everything it has seen: their largest non-NaN value m (fmaxf
// ignores a NaN operand) replaces the best only if it is strictly larger --
// an equal value seen before has the lower index -- or if nothing non-NaN
// was seen yet; then the first of the four equal to m is the index.
__device__ __forceinline__ void take4(const float4& v, int base, float& bv, int& bi) {
  const float m = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
  if (bi < 0 ? m == m : m > bv) {
    bi = base + (v.x == m ? 0 : v.y == m ? 1 : v.z == m ? 2 : 3);
    bv = m;
  }
}

// Best (value, index) of elements [lo, hi) of `row`, reduced over the CTA;
// valid in thread 0.  Each thread walks its share in increasing index order,
// four 16-byte loads in flight at a time.
__device__ void cta_best(const float* __restrict__ row, int lo, int hi, float& bv, int& bi) {
  bv = 0.f;
  bi = -1;
  int i = lo + threadIdx.x;
  if (((reinterpret_cast<uintptr_t>(row + lo)) & 15u) == 0) {
    const int n4 = (hi - lo) / 4;
    const float4* r4 = reinterpret_cast<const float4*>(row + lo);
    int k = threadIdx.x;
    for (; k + 3 * kArgThreads < n4; k += 4 * kArgThreads) {
      float4 a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = __ldcs(r4 + k + u * kArgThreads);
#pragma unroll
      for (int u = 0; u < 4; ++u) take4(a[u], lo + 4 * (k + u * kArgThreads), bv, bi);
    }
    for (; k < n4; k += kArgThreads) take4(__ldcs(r4 + k), lo + 4 * k, bv, bi);
    i = lo + 4 * n4 + threadIdx.x;
  }
  for (; i < hi; i += kArgThreads) take(__ldcs(row + i), i, bv, bi);
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
    for (int o = kArgThreads / 64; o > 0; o >>= 1) {
      const float ov = __shfl_down_sync(0xffffffffu, bv, o);
      const int oi = __shfl_down_sync(0xffffffffu, bi, o);
      take(ov, oi, bv, bi);
    }
  }
}

__global__ void __launch_bounds__(kArgThreads) argmax_kernel(const float* __restrict__ x, int vocab,
                                                             long long stride,
                                                             int32_t* __restrict__ out) {
  float bv;
  int bi;
  cta_best(x + (size_t)blockIdx.x * (size_t)stride, 0, vocab, bv, bi);
  if (threadIdx.x == 0) out[blockIdx.x] = bi < 0 ? 0 : bi;
}

// Cluster of kClusterCtas CTAs per row (cluster dimension set at launch).
__global__ void __launch_bounds__(kArgThreads) argmax_cluster_kernel(const float* __restrict__ x,
                                                                     int vocab, long long stride,
                                                                     int32_t* __restrict__ out) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ float part_v[kClusterCtas];
  __shared__ int part_i[kClusterCtas];
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.x / kClusterCtas;
  // part boundaries on multiples of 4 elements
  const int per = ((vocab + kClusterCtas - 1) / kClusterCtas + 3) & ~3;
  const int lo = min(vocab, rank * per), hi = min(vocab, lo + per);
  float bv;
  int bi;
  cta_best(x + (size_t)row * (size_t)stride, lo, hi, bv, bi);
  if (threadIdx.x == 0) {
    float* rv = cluster.map_shared_rank(part_v, 0);
    int* ri = cluster.map_shared_rank(part_i, 0);
    rv[rank] = bv;
    ri[rank] = bi;
  }
  cluster.sync();  // every part is in the first CTA's shared memory
  if (rank == 0 && threadIdx.x == 0) {
    float v = 0.f;
    int i = -1;
    for (int r = 0; r < kClusterCtas; ++r) take(part_v[r], part_i[r], v, i);
    out[row] = i < 0 ? 0 : i;
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows < 2 * pkv::sm_count(dev) && vocab >= 64 * pkv::kClusterCtas &&
      (long long)rows * pkv::kClusterCtas <= 0x7fffffffll) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = pkv::kClusterCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows * pkv::kClusterCtas));
    cfg.blockDim = dim3(pkv::kArgThreads);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return pkv::cuda_status(cudaLaunchKernelEx(&cfg, pkv::argmax_cluster_kernel, logits, vocab,
                                               row_stride, out_ids),
                            "cudaLaunchKernelEx(argmax cluster)");
  }
  pkv::argmax_kernel<<<rows, pkv::kArgThreads, 0, st>>>(logits, vocab, row_stride, out_ids);
  return pkv::cuda_status(cudaGetLastError(), "argmax_kernel");
}
