// Paged causal GQA prefill: attention of each sequence's newest tokens (a
// prompt, or a chunk of one after a cached prefix) over the sequence's own
// pages.
//
// "Gestion de la KV cache et strategies de batching" (samir-vllm article):
// attention reads only the sequence's pages, and a token at absolute
// position p sees the positions up to its own.  Sequence s holds
// n = seq_lens[s] tokens; its queries are the last q_len = cu_q[s+1] - cu_q[s]
// of them, at positions n - q_len .. n - 1.
//
// Work unit = (query block of 32 tokens, KV head g, sequence s), one CTA.
// Its 128 query rows (32 tokens x the 4 query heads of g) share every K/V
// page they read: a producer warp streams the pages [0, last position / 16]
// through a 4-stage TMA ring (one {64, 16, 1, 2} box = K then V tile), and
// 8 consumer warps each own 16 rows (4 tokens x 4 heads) of bf16 mma.sync
// m16n8k16 with fp32 accumulation, per-row causal masks and an online
// softmax in base 2 (the same arithmetic as the decode kernel, with all 16
// mma rows real).  Blocks are scheduled longest (latest tokens) first.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "internal.h"
#include "pkv.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kPfWarps = 8;                    // consumer warps
constexpr int kPfTokens = 4 * kPfWarps;        // query tokens per CTA
constexpr int kPfStages = 4;
constexpr int kPfStageBytes = 4096;            // K tile + V tile of one (page, head)
constexpr int kPfThreads = (kPfWarps + 1) * 32;
constexpr uint64_t kPfWaitNs = 2000000000ull;  // 2 s per wait
constexpr float kLog2e = 1.4426950408889634f;

struct PrefillParams {
  const uint16_t* q;             // [T][32][64] bf16, rotated
  const int32_t* cu_q;           // [S + 1]
  const int32_t* block_tables;   // [S][bt_stride]
  const int32_t* seq_lens;       // [S]
  uint16_t* out;                 // [T][32][64] bf16
  int num_tokens;                // T
  int bt_stride, max_blocks, num_pages, num_seqs;
  float sl2;                     // scale * log2(e)
  int* d_err;
};

// Zero this CTA's share of the rows of sequence s (head group g): rows
// t = blockIdx.x * kPfTokens + k * gridDim.x * kPfTokens, 32 at a time.
__device__ void zero_rows(const PrefillParams& p, int r0, int q_len, int g) {
  const int per_row = 4 * 64 / 8;  // uint4 per (token, head group)
  for (int base = blockIdx.x * kPfTokens; base < q_len; base += gridDim.x * kPfTokens) {
    const int cnt = min(kPfTokens, q_len - base) * per_row;
    for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
      const int t = base + i / per_row, c = i % per_row;
      uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)(r0 + t) * PKV_NUM_Q_HEADS + g * 4) * 64);
      dst[c] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

__global__ void __launch_bounds__(kPfThreads, 2)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap, const PrefillParams p) {
  __shared__ __align__(1024) uint8_t tiles[kPfStages * kPfStageBytes];
  __shared__ __align__(8) uint64_t full[kPfStages], empty[kPfStages];
  __shared__ int bad_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, g = blockIdx.y;
  const int qb = (int)gridDim.x - 1 - (int)blockIdx.x;  // latest (longest) blocks first

  pdl_wait();  // the pages (appended by the previous kernel) and q are ready
  pdl_launch_dependents();
  const int r0 = __ldg(p.cu_q + s), r1 = __ldg(p.cu_q + s + 1), q_len = r1 - r0;
  const int n = __ldg(p.seq_lens + s);
  if (r0 < 0 || r1 > p.num_tokens || q_len < 0) {  // rows outside q/out: touch nothing
    if (blockIdx.x == 0 && g == 0 && threadIdx.x == 0) report_error(p.d_err, PKV_ERR_DEVICE_INDEX);
    return;
  }
  if (q_len == 0) return;
  const int n_pages_seq = (n + PKV_PAGE_TOKENS - 1) / PKV_PAGE_TOKENS;
  // the sequence must fit its table and the grid, and hold its queries
  bool bad = q_len > n || n > PKV_PAGE_TOKENS * p.max_blocks || q_len > (int)gridDim.x * kPfTokens;
  if (threadIdx.x == 0) bad_flag = 0;
  __syncthreads();
  if (!bad && warp == 0) {  // every needed page id of the sequence, as the definition reads them
    int any = 0;
    for (int j = lane; j < n_pages_seq; j += 32) {
      const int pid = __ldg(p.block_tables + (size_t)s * p.bt_stride + j);
      any |= (pid < 0 || pid >= p.num_pages);
    }
    if (__any_sync(0xffffffffu, any) && lane == 0) bad_flag = 1;
  }
  __syncthreads();
  bad = bad || bad_flag;
  if (bad) {
    if (blockIdx.x == 0 && g == 0 && threadIdx.x == 0) report_error(p.d_err, PKV_ERR_DEVICE_INDEX);
    zero_rows(p, r0, q_len, g);
    return;
  }
  const int t0 = qb * kPfTokens;
  if (t0 >= q_len) return;
  const int t_end = min(t0 + kPfTokens, q_len);
  const int pos0 = n - q_len;                      // position of query token 0
  const int n_pages = (pos0 + t_end - 1) / PKV_PAGE_TOKENS + 1;
  const int n_active = (t_end - t0 + 3) / 4;       // consumer warps with tokens

  if (threadIdx.x == 0) {
    for (int st = 0; st < kPfStages; ++st) {
      mbar_init(smem_u32(&full[st]), 1);
      mbar_init(smem_u32(&empty[st]), (uint32_t)n_active);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kPfWarps) {
    // ---------------- producer ---------------------------------------------
    // page ids 32 at a time, the next batch read one batch ahead
    const int32_t* row = p.block_tables + (size_t)s * p.bt_stride;
    int cur = lane < n_pages ? __ldg(row + lane) : -1;
    int nxt = 32 + lane < n_pages ? __ldg(row + 32 + lane) : -1;
    for (int j = 0; j < n_pages; ++j) {
      if ((j & 31) == 0 && j > 0) {
        cur = nxt;
        nxt = j + 32 + lane < n_pages ? __ldg(row + j + 32 + lane) : -1;
      }
      const int pid = __shfl_sync(0xffffffffu, cur, j & 31);
      const int st = j % kPfStages;
      bool ok = true;
      if (lane == 0 && j >= kPfStages)
        ok = mbar_wait_bounded(smem_u32(&empty[st]), (uint32_t)((j / kPfStages - 1) & 1), kPfWaitNs);
      if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
        if (lane == 0) report_error(p.d_err, PKV_ERR_TIMEOUT);
        return;  // consumers time out on the pages never issued
      }
      if (lane == 0) {
        const uint32_t bar = smem_u32(&full[st]);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, kPfStageBytes);
        tma_load_4d(smem_u32(tiles + st * kPfStageBytes), &tmap, 0, 0, g, pid * 2, bar);
      }
      __syncwarp();
    }
    // wait (bounded) for the last copies to land before the CTA may exit
    if (lane == 0)
      for (int j = max(0, n_pages - kPfStages); j < n_pages; ++j)
        (void)mbar_wait_bounded(smem_u32(&full[j % kPfStages]), (uint32_t)((j / kPfStages) & 1), kPfWaitNs);
    return;
  }
  if (warp >= n_active) return;

  // ---------------- consumers ----------------------------------------------
  const int gq = lane >> 2, tig = lane & 3, mi = lane >> 3, rr = lane & 7;
  const int hl = gq & 3;
  const int tw0 = t0 + 4 * warp;
  // this lane's two rows: tokens tA (rows 0..7) and tB (rows 8..15), head 4g + hl
  const int tA = tw0 + (gq >> 2), tB = tw0 + 2 + (gq >> 2);
  const bool vA = tA < t_end, vB = tB < t_end;
  const int pA = vA ? pos0 + tA : -1, pB = vB ? pos0 + tB : -1;
  const int p_w = pos0 + min(tw0 + 3, t_end - 1);   // this warp's last position

  uint32_t qa[4][4];
  {
    const uint32_t* qrA = reinterpret_cast<const uint32_t*>(
        p.q + ((size_t)(r0 + (vA ? tA : 0)) * PKV_NUM_Q_HEADS + g * 4 + hl) * 64);
    const uint32_t* qrB = reinterpret_cast<const uint32_t*>(
        p.q + ((size_t)(r0 + (vB ? tB : 0)) * PKV_NUM_Q_HEADS + g * 4 + hl) * 64);
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      qa[kc][0] = vA ? __ldg(qrA + kc * 8 + tig) : 0u;
      qa[kc][1] = vB ? __ldg(qrB + kc * 8 + tig) : 0u;
      qa[kc][2] = vA ? __ldg(qrA + kc * 8 + 4 + tig) : 0u;
      qa[kc][3] = vB ? __ldg(qrB + kc * 8 + 4 + tig) : 0u;
    }
  }
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  bool timed_out = false;

  for (int j = 0; j < n_pages; ++j) {
    const int st = j % kPfStages;
    if (!mbar_wait_bounded(smem_u32(&full[st]), (uint32_t)((j / kPfStages) & 1), kPfWaitNs)) {
      if (lane == 0) report_error(p.d_err, PKV_ERR_TIMEOUT);
      timed_out = true;
      break;
    }
    const int kp0 = j * PKV_PAGE_TOKENS;
    if (kp0 <= p_w) {
      const uint32_t sK = smem_u32(tiles + st * kPfStageBytes), sV = sK + 2048;
      // ---- S = Q K^T for keys kp0 .. kp0 + 15 --------------------------------
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t krow = sK + (uint32_t)((8 * (mi >> 1) + rr) * 128);
#pragma unroll
      for (int kc = 0; kc < 4; ++kc) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(krow + ((((2 * kc) + (mi & 1)) ^ rr) << 4), b0, b1, b2, b3);
        mma_bf16_16816_full(s0, qa[kc][0], qa[kc][1], qa[kc][2], qa[kc][3], b0, b1);
        mma_bf16_16816_full(s1, qa[kc][0], qa[kc][1], qa[kc][2], qa[kc][3], b2, b3);
      }
      // keys of this lane: kp0 + 2 tig, +1 (s0) and kp0 + 8 + 2 tig, +1 (s1)
      const int k0 = kp0 + 2 * tig;
      float xA0 = (k0 <= pA) ? s0[0] * p.sl2 : -INFINITY;
      float xA1 = (k0 + 1 <= pA) ? s0[1] * p.sl2 : -INFINITY;
      float xA2 = (k0 + 8 <= pA) ? s1[0] * p.sl2 : -INFINITY;
      float xA3 = (k0 + 9 <= pA) ? s1[1] * p.sl2 : -INFINITY;
      float xB0 = (k0 <= pB) ? s0[2] * p.sl2 : -INFINITY;
      float xB1 = (k0 + 1 <= pB) ? s0[3] * p.sl2 : -INFINITY;
      float xB2 = (k0 + 8 <= pB) ? s1[2] * p.sl2 : -INFINITY;
      float xB3 = (k0 + 9 <= pB) ? s1[3] * p.sl2 : -INFINITY;
      float pmA = fmaxf(fmaxf(xA0, xA1), fmaxf(xA2, xA3));
      float pmB = fmaxf(fmaxf(xB0, xB1), fmaxf(xB2, xB3));
      pmA = fmaxf(pmA, __shfl_xor_sync(0xffffffffu, pmA, 1));
      pmA = fmaxf(pmA, __shfl_xor_sync(0xffffffffu, pmA, 2));
      pmB = fmaxf(pmB, __shfl_xor_sync(0xffffffffu, pmB, 1));
      pmB = fmaxf(pmB, __shfl_xor_sync(0xffffffffu, pmB, 2));
      const float mnA = fmaxf(mA, pmA), mnB = fmaxf(mB, pmB);
      // a row with no key yet (mn = -inf) gets weights 0 and keeps alpha = 1
      const float alA = (mA == mnA) ? 1.f : exp2f(mA - mnA);
      const float alB = (mB == mnB) ? 1.f : exp2f(mB - mnB);
      auto w = [](float x, float mn) { return x == -INFINITY ? 0.f : (x == mn ? 1.f : exp2f(x - mn)); };
      const uint32_t pa0 = pack_bf16x2(w(xA0, mnA), w(xA1, mnA));
      const uint32_t pa1 = pack_bf16x2(w(xB0, mnB), w(xB1, mnB));
      const uint32_t pa2 = pack_bf16x2(w(xA2, mnA), w(xA3, mnA));
      const uint32_t pa3 = pack_bf16x2(w(xB2, mnB), w(xB3, mnB));
      mA = mnA;
      mB = mnB;
      // the denominator uses the same bf16-rounded weights as the PV product
      lA = lA * alA + ((bf16lo_to_f32(pa0) + bf16hi_to_f32(pa0)) + (bf16lo_to_f32(pa2) + bf16hi_to_f32(pa2)));
      lB = lB * alB + ((bf16lo_to_f32(pa1) + bf16hi_to_f32(pa1)) + (bf16lo_to_f32(pa3) + bf16hi_to_f32(pa3)));
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        o[i][0] *= alA;
        o[i][1] *= alA;
        o[i][2] *= alB;
        o[i][3] *= alB;
      }
      // ---- O += P V (V rows past the sequence's end may hold any bits) -------
      uint32_t m01 = 0xFFFFFFFFu, m89 = 0xFFFFFFFFu;
      const int valid = n - kp0;
      if (valid < PKV_PAGE_TOKENS) {
        const int t0k = 2 * tig;
        m01 = ((t0k < valid) ? 0x0000FFFFu : 0u) | ((t0k + 1 < valid) ? 0xFFFF0000u : 0u);
        m89 = ((t0k + 8 < valid) ? 0x0000FFFFu : 0u) | ((t0k + 9 < valid) ? 0xFFFF0000u : 0u);
      }
      const uint32_t vrow = sV + (uint32_t)((8 * (mi & 1) + rr) * 128);
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(vrow + ((((2 * pp) + (mi >> 1)) ^ rr) << 4), v0, v1, v2, v3);
        v0 &= m01;
        v2 &= m01;
        v1 &= m89;
        v3 &= m89;
        mma_bf16_16816_full(o[2 * pp], pa0, pa1, pa2, pa3, v0, v1);
        mma_bf16_16816_full(o[2 * pp + 1], pa0, pa1, pa2, pa3, v2, v3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
  }
  if (timed_out) return;

  // ---- normalise and store the rows of this warp ---------------------------
  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  if (vA) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + ((size_t)(r0 + tA) * PKV_NUM_Q_HEADS + g * 4 + hl) * 64) + tig;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      dst[4 * i] = pack_bf16x2(__fdiv_rn(o[i][0], lA), __fdiv_rn(o[i][1], lA));
  }
  if (vB) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + ((size_t)(r0 + tB) * PKV_NUM_Q_HEADS + g * 4 + hl) * 64) + tig;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      dst[4 * i] = pack_bf16x2(__fdiv_rn(o[i][2], lB), __fdiv_rn(o[i][3], lB));
  }
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int paged_gqa_prefill(const void* q, int num_tokens, const int32_t* cu_q,
                                 const void* kv_pool, int num_pages, const int32_t* block_tables,
                                 int bt_row_stride, int max_blocks, const int32_t* seq_lens,
                                 int num_seqs, int max_q_len, void* out, float scale, int* d_err,
                                 void* stream) {
  if (num_seqs < 0 || num_tokens < 0 || num_pages < 1 || max_blocks < 1 ||
      bt_row_stride < max_blocks || max_q_len < 0)
    return PKV_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0 || max_q_len == 0 || num_tokens == 0) return PKV_OK;
  if (!q || !cu_q || !kv_pool || !block_tables || !seq_lens || !out) return PKV_ERR_INVALID_ARGUMENT;
  if (!isfinite(scale)) return PKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(cu_q) & 3u))
    return PKV_ERR_MISALIGNED;
  const long long blocks_x = ((long long)max_q_len + kPfTokens - 1) / kPfTokens;
  if (num_seqs > 65535 || blocks_x > (1ll << 30) || (long long)num_pages * 16 * 8 * 2 >= (1ll << 31) ||
      (long long)max_blocks * PKV_PAGE_TOKENS >= (1ll << 24))
    return PKV_ERR_UNSUPPORTED_SHAPE;
  int dev = 0;
  int rc = bind_stream_device(stream, &dev);
  if (rc != PKV_OK) return rc;
  CUtensorMap map;
  rc = make_pool_map(&map, kv_pool, num_pages);
  if (rc != PKV_OK) return rc;

  PrefillParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.q = static_cast<const uint16_t*>(q);
  prm.cu_q = cu_q;
  prm.block_tables = block_tables;
  prm.seq_lens = seq_lens;
  prm.out = static_cast<uint16_t*>(out);
  prm.num_tokens = num_tokens;
  prm.bt_stride = bt_row_stride;
  prm.max_blocks = max_blocks;
  prm.num_pages = num_pages;
  prm.num_seqs = num_seqs;
  prm.sl2 = scale * kLog2e;
  prm.d_err = d_err;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks_x, PKV_NUM_KV_HEADS, (unsigned)num_seqs);
  cfg.blockDim = dim3(kPfThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, paged_prefill_kernel, map, prm),
                     "cudaLaunchKernelEx(prefill)");
}
