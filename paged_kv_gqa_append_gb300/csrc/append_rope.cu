// Fused RoPE + paged KV append for sm_103a.
//
// Source: samir-vllm article, section "Gestion de la KV cache et strategies de
// batching": during decode each new token is added at its absolute RoPE
// position, into the 16-token pages that the sequence's per-layer block table
// lists.  The rotation convention (half-split pairs, fp32 operation order,
// bf16 nearest-even) is the library's reading of what the pages leave open.
//
// One CTA per token, one warp per KV head; lane i rotates the pair
// (i, i + 32).  Each (token, head) writes one 128-byte K row and one 128-byte
// V row of a page: the kernel moves 4 KiB per token and is bound by launch
// latency, not bandwidth.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "i8_layout.cuh"
#include "internal.h"
#include "pkv.h"
#include "ptx.cuh"
#include "quant.cuh"
#include "rope.cuh"

namespace pkv {

struct AppendParams {
  const uint16_t* k;          // [T][8][64]
  const uint16_t* v;          // [T][8][64]
  const int32_t* positions;   // [T]
  const int32_t* token_seq;   // [T] or null
  const int32_t* block_tables;
  const float* cos;           // [max_pos][32]
  const float* sin;
  const uint16_t* q_in;       // [T][32][64] or null
  uint16_t* q_out;
  uint16_t* pool;             // [num_pages][2][8][16][64]
  int T, num_seqs, bt_stride, max_blocks, num_pages, max_pos;
  int* d_err;
};

__global__ void __launch_bounds__(256) kv_append_rope_kernel(const AppendParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const int g = threadIdx.x >> 5;  // KV head
  const int lane = threadIdx.x & 31;
  const int s = p.token_seq ? __ldg(p.token_seq + t) : t;
  const int pos = __ldg(p.positions + t);
  bool ok = s >= 0 && s < p.num_seqs && pos >= 0 && pos < p.max_pos &&
            (pos / PKV_PAGE_TOKENS) < p.max_blocks;
  int page = -1;
  if (ok) {
    page = __ldg(p.block_tables + (size_t)s * p.bt_stride + pos / PKV_PAGE_TOKENS);
    ok = page >= 0 && page < p.num_pages;
  }
  if (!ok) {
    if (threadIdx.x == 0) report_error(p.d_err, PKV_ERR_DEVICE_INDEX);
    if (p.q_out) {
      for (int hh = 0; hh < 4; ++hh) {
        uint16_t* qo = p.q_out + ((size_t)t * PKV_NUM_Q_HEADS + g * 4 + hh) * 64;
        qo[lane] = 0;
        qo[lane + 32] = 0;
      }
    }
    return;
  }
  const int slot = pos % PKV_PAGE_TOKENS;
  const float c = __ldg(p.cos + (size_t)pos * PKV_ROPE_PAIRS + lane);
  const float sn = __ldg(p.sin + (size_t)pos * PKV_ROPE_PAIRS + lane);

  // K: rotate and scatter into pool[page][0][g][slot][:]
  const uint16_t* kr = p.k + ((size_t)t * PKV_NUM_KV_HEADS + g) * 64;
  uint16_t* kdst = p.pool + ((((size_t)page * 2 + 0) * PKV_NUM_KV_HEADS + g) * PKV_PAGE_TOKENS + slot) * 64;
  uint16_t r0, r1;
  rope_pair(kr[lane], kr[lane + 32], c, sn, r0, r1);
  kdst[lane] = r0;
  kdst[lane + 32] = r1;

  // V: copied bit for bit into pool[page][1][g][slot][:]
  const uint32_t* vr = reinterpret_cast<const uint32_t*>(p.v + ((size_t)t * PKV_NUM_KV_HEADS + g) * 64);
  uint32_t* vdst = reinterpret_cast<uint32_t*>(
      p.pool + ((((size_t)page * 2 + 1) * PKV_NUM_KV_HEADS + g) * PKV_PAGE_TOKENS + slot) * 64);
  vdst[lane] = vr[lane];

  // q: the 4 query heads of this group, same rotation
  if (p.q_in) {
    for (int hh = 0; hh < 4; ++hh) {
      const size_t row = ((size_t)t * PKV_NUM_Q_HEADS + g * 4 + hh) * 64;
      const uint16_t* qi = p.q_in + row;
      uint16_t q0, q1;
      rope_pair(qi[lane], qi[lane + 32], c, sn, q0, q1);
      __syncwarp();  // q_out may alias q_in: all reads of the row before any write
      p.q_out[row + lane] = q0;
      p.q_out[row + lane + 32] = q1;
    }
  }
}

// ---------------------------------------------------------------------------
// INT8 K/V pages (the "INT8 K/V" storage mode of a request's KV cache in
// "Lifecycle and Memory Model", section "Per-request / handle-owned memory").
// Each (token, head) row of K (rotated and rounded to bf16 exactly as above)
// and of V is quantised on its own: amax = max |x|, scale = amax / 127 and
// code = round-half-even(x / scale) in [-127, 127], both divisions IEEE fp32;
// amax == 0 gives scale 0 and zero codes.  A (page, head) is one 2176-byte
// block of the pool in the format of i8_layout.cuh (codes as code + 128; K
// codes row-major; V codes in slot pairs; scales in the decode's lane
// order).  Same grid as the bf16 append: one CTA per token, one warp per KV
// head, lane i holding dims i and i + 32.
// ---------------------------------------------------------------------------
struct AppendI8Params {
  const uint16_t* k;          // [T][8][64] bf16
  const uint16_t* v;          // [T][8][64] bf16
  const int32_t* positions;   // [T]
  const int32_t* token_seq;   // [T] or null
  const int32_t* block_tables;
  const float* cos;           // [max_pos][32]
  const float* sin;
  const uint16_t* q_in;       // [T][32][64] or null
  uint16_t* q_out;
  uint8_t* pool;              // [num_pages][8][2176]
  int T, num_seqs, bt_stride, max_blocks, num_pages, max_pos;
  int* d_err;
};

__global__ void __launch_bounds__(256) kv_append_rope_int8_kernel(const AppendI8Params p) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const int g = threadIdx.x >> 5;  // KV head
  const int lane = threadIdx.x & 31;
  const int s = p.token_seq ? __ldg(p.token_seq + t) : t;
  const int pos = __ldg(p.positions + t);
  bool ok = s >= 0 && s < p.num_seqs && pos >= 0 && pos < p.max_pos &&
            (pos / PKV_PAGE_TOKENS) < p.max_blocks;
  int page = -1;
  if (ok) {
    page = __ldg(p.block_tables + (size_t)s * p.bt_stride + pos / PKV_PAGE_TOKENS);
    ok = page >= 0 && page < p.num_pages;
  }
  if (!ok) {
    if (threadIdx.x == 0) report_error(p.d_err, PKV_ERR_DEVICE_INDEX);
    if (p.q_out) {
      for (int hh = 0; hh < 4; ++hh) {
        uint16_t* qo = p.q_out + ((size_t)t * PKV_NUM_Q_HEADS + g * 4 + hh) * 64;
        qo[lane] = 0;
        qo[lane + 32] = 0;
      }
    }
    return;
  }
  const int slot = pos % PKV_PAGE_TOKENS;
  const float c = __ldg(p.cos + (size_t)pos * PKV_ROPE_PAIRS + lane);
  const float sn = __ldg(p.sin + (size_t)pos * PKV_ROPE_PAIRS + lane);
  uint8_t* blk = p.pool + ((size_t)page * PKV_NUM_KV_HEADS + g) * PKV_I8_BLOCK_BYTES;

  // K: rotate (bf16 result, as in the bf16 cache), quantise, store
  const uint16_t* kr = p.k + ((size_t)t * PKV_NUM_KV_HEADS + g) * 64;
  uint16_t r0, r1;
  rope_pair(kr[lane], kr[lane + 32], c, sn, r0, r1);
  int8_t k0, k1;
  const float ks = quantize_pair(__uint_as_float((uint32_t)r0 << 16), __uint_as_float((uint32_t)r1 << 16),
                                 k0, k1);
  blk[i8_k_byte(slot, lane)] = i8_code_byte(k0);
  blk[i8_k_byte(slot, lane + 32)] = i8_code_byte(k1);

  // V: quantise the bf16 row
  const uint16_t* vr = p.v + ((size_t)t * PKV_NUM_KV_HEADS + g) * 64;
  int8_t v0, v1;
  const float vs = quantize_pair(__uint_as_float((uint32_t)vr[lane] << 16),
                                 __uint_as_float((uint32_t)vr[lane + 32] << 16), v0, v1);
  blk[i8_v_byte(slot, lane)] = i8_code_byte(v0);
  blk[i8_v_byte(slot, lane + 32)] = i8_code_byte(v1);
  if (lane == 0) {
    *reinterpret_cast<float*>(blk + i8_k_scale_byte(slot)) = ks;
    *reinterpret_cast<float*>(blk + i8_v_scale_byte(slot)) = vs;
  }

  // q: the 4 query heads of this group, rotated as in the bf16 append
  if (p.q_in) {
    for (int hh = 0; hh < 4; ++hh) {
      const size_t row = ((size_t)t * PKV_NUM_Q_HEADS + g * 4 + hh) * 64;
      const uint16_t* qi = p.q_in + row;
      uint16_t q0, q1;
      rope_pair(qi[lane], qi[lane + 32], c, sn, q0, q1);
      __syncwarp();
      p.q_out[row + lane] = q0;
      p.q_out[row + lane + 32] = q1;
    }
  }
}

}  // namespace pkv

using namespace pkv;

extern "C" int kv_append_rope(const void* k, const void* v, const int32_t* positions,
                              const int32_t* token_seq, int T, const int32_t* block_tables,
                              int num_seqs, int bt_row_stride, int max_blocks, void* kv_pool,
                              int num_pages, const float* rope_cos, const float* rope_sin,
                              int max_pos, const void* q_in, void* q_out, int* d_err,
                              void* stream) {
  if (T < 0 || num_seqs < 1 || max_blocks < 1 || bt_row_stride < max_blocks || num_pages < 1 ||
      max_pos < 1)
    return PKV_ERR_INVALID_ARGUMENT;
  if (T == 0) return PKV_OK;
  if (!k || !v || !positions || !block_tables || !kv_pool || !rope_cos || !rope_sin)
    return PKV_ERR_INVALID_ARGUMENT;
  if ((q_in == nullptr) != (q_out == nullptr)) return PKV_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(kv_pool) | reinterpret_cast<uintptr_t>(q_in) |
       reinterpret_cast<uintptr_t>(q_out)) & 3u)
    return PKV_ERR_MISALIGNED;
  if (T > (1 << 30) || (long long)num_pages * PKV_PAGE_ELEMS >= (1ll << 40))
    return PKV_ERR_UNSUPPORTED_SHAPE;
  int dev = 0;
  int rc = bind_stream_device(stream, &dev);
  if (rc != PKV_OK) return rc;

  AppendParams p;
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.positions = positions;
  p.token_seq = token_seq;
  p.block_tables = block_tables;
  p.cos = rope_cos;
  p.sin = rope_sin;
  p.q_in = static_cast<const uint16_t*>(q_in);
  p.q_out = static_cast<uint16_t*>(q_out);
  p.pool = static_cast<uint16_t*>(kv_pool);
  p.T = T;
  p.num_seqs = num_seqs;
  p.bt_stride = bt_row_stride;
  p.max_blocks = max_blocks;
  p.num_pages = num_pages;
  p.max_pos = max_pos;
  p.d_err = d_err;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T);
  cfg.blockDim = dim3(256);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kv_append_rope_kernel, p), "cudaLaunchKernelEx(append)");
}

extern "C" int kv_append_rope_int8(const void* k, const void* v, const int32_t* positions,
                                   const int32_t* token_seq, int T, const int32_t* block_tables,
                                   int num_seqs, int bt_row_stride, int max_blocks,
                                   void* kv_pool, int num_pages,
                                   const float* rope_cos, const float* rope_sin, int max_pos,
                                   const void* q_in, void* q_out, int* d_err, void* stream) {
  if (T < 0 || num_seqs < 1 || max_blocks < 1 || bt_row_stride < max_blocks || num_pages < 1 ||
      max_pos < 1)
    return PKV_ERR_INVALID_ARGUMENT;
  if (T == 0) return PKV_OK;
  if (!k || !v || !positions || !block_tables || !kv_pool || !rope_cos || !rope_sin)
    return PKV_ERR_INVALID_ARGUMENT;
  if ((q_in == nullptr) != (q_out == nullptr)) return PKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(k) || !aligned16(v) || !aligned16(kv_pool) ||
      ((reinterpret_cast<uintptr_t>(q_in) | reinterpret_cast<uintptr_t>(q_out)) & 3u))
    return PKV_ERR_MISALIGNED;
  if (T > (1 << 30) || (long long)num_pages * PKV_PAGE_ELEMS >= (1ll << 40))
    return PKV_ERR_UNSUPPORTED_SHAPE;
  int dev = 0;
  int rc = bind_stream_device(stream, &dev);
  if (rc != PKV_OK) return rc;

  AppendI8Params p;
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.positions = positions;
  p.token_seq = token_seq;
  p.block_tables = block_tables;
  p.cos = rope_cos;
  p.sin = rope_sin;
  p.q_in = static_cast<const uint16_t*>(q_in);
  p.q_out = static_cast<uint16_t*>(q_out);
  p.pool = static_cast<uint8_t*>(kv_pool);
  p.T = T;
  p.num_seqs = num_seqs;
  p.bt_stride = bt_row_stride;
  p.max_blocks = max_blocks;
  p.num_pages = num_pages;
  p.max_pos = max_pos;
  p.d_err = d_err;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T);
  cfg.blockDim = dim3(256);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kv_append_rope_int8_kernel, p),
                     "cudaLaunchKernelEx(append int8)");
}

// The same T tokens appended into every layer of a request: the prompt of a
// newly admitted sequence ("Gestion de la KV cache et strategies de
// batching": a request's pages are written layer by layer as it enters the
// batch).  One host call for the L copies and L launches a serving loop
// would otherwise make one by one.
extern "C" int kv_append_rope_layers(const void* const* k, const void* const* v, int num_layers,
                                     int src_host, void* stage, size_t stage_bytes,
                                     const int32_t* positions, const int32_t* token_seq, int T,
                                     const int32_t* block_tables, long long bt_layer_stride,
                                     int num_seqs, int bt_row_stride, int max_blocks,
                                     void* kv_pool, int num_pages, int int8, const float* rope_cos,
                                     const float* rope_sin, int max_pos, int* d_err, void* stream) {
  // every check of every layer first: a call that is refused enqueues nothing
  if (num_layers < 0 || T < 0 || (src_host != 0 && src_host != 1) || (int8 != 0 && int8 != 1) ||
      bt_layer_stride < 0 || num_seqs < 1 || max_blocks < 1 || bt_row_stride < max_blocks ||
      num_pages < 1 || max_pos < 1)
    return PKV_ERR_INVALID_ARGUMENT;
  if (num_layers == 0 || T == 0) return PKV_OK;
  if (!k || !v || !block_tables || !positions || !kv_pool || !rope_cos || !rope_sin)
    return PKV_ERR_INVALID_ARGUMENT;
  if (bt_layer_stride < (long long)num_seqs * bt_row_stride) return PKV_ERR_INVALID_ARGUMENT;
  if (T > (1 << 30)) return PKV_ERR_UNSUPPORTED_SHAPE;
  const uintptr_t amask = int8 ? 15u : 3u;  // the alignment each append wants of k, v and the pool
  if (reinterpret_cast<uintptr_t>(kv_pool) & amask) return PKV_ERR_MISALIGNED;
  const size_t rows = (size_t)T * PKV_NUM_KV_HEADS * PKV_HEAD_DIM * 2;  // bytes of k (or v) per layer
  for (int l = 0; l < num_layers; ++l) {
    if (!k[l] || !v[l]) return PKV_ERR_INVALID_ARGUMENT;
    if (!src_host && ((reinterpret_cast<uintptr_t>(k[l]) | reinterpret_cast<uintptr_t>(v[l])) & amask))
      return PKV_ERR_MISALIGNED;
  }
  if (src_host) {
    if (!stage || stage_bytes < 2 * rows) return PKV_ERR_INVALID_ARGUMENT;
    if (!aligned16(stage)) return PKV_ERR_MISALIGNED;
    int dev = 0;  // the copies below go to the stream's device
    const int rb = bind_stream_device(stream, &dev);
    if (rb != PKV_OK) return rb;
  }
  int rc = PKV_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* sk = static_cast<uint8_t*>(stage);
  for (int l = 0; l < num_layers; ++l) {
    const void* kl = k[l];
    const void* vl = v[l];
    if (src_host) {  // the stage is reused by every layer: stream order keeps the launches apart
      rc = cuda_status(cudaMemcpyAsync(sk, kl, rows, cudaMemcpyHostToDevice, st), "cudaMemcpyAsync(k)");
      if (rc == PKV_OK)
        rc = cuda_status(cudaMemcpyAsync(sk + rows, vl, rows, cudaMemcpyHostToDevice, st),
                         "cudaMemcpyAsync(v)");
      if (rc != PKV_OK) return rc;
      kl = sk;
      vl = sk + rows;
    }
    const int32_t* bt = block_tables + l * bt_layer_stride;
    rc = int8 ? kv_append_rope_int8(kl, vl, positions, token_seq, T, bt, num_seqs, bt_row_stride,
                                    max_blocks, kv_pool, num_pages, rope_cos, rope_sin, max_pos,
                                    nullptr, nullptr, d_err, stream)
              : kv_append_rope(kl, vl, positions, token_seq, T, bt, num_seqs, bt_row_stride,
                               max_blocks, kv_pool, num_pages, rope_cos, rope_sin, max_pos, nullptr,
                               nullptr, d_err, stream);
    if (rc != PKV_OK) return rc;
  }
  return PKV_OK;
}
