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
// Two implementations of the same contract:
//  * tcgen05 (default): one CTA per (32 query tokens, KV head, sequence) =
//    an M = 128 tile of query rows (token-major, the 4 query heads of the
//    group inside); keys in blocks of 64 (4 pages).  S = Q K^T and O += P V
//    run on the 5th-generation tensor cores with Q, S, P and O in tensor
//    memory (Q loaded once by the softmax warps as the A operand of S; P
//    written over the first half of its own S buffer as the A operand of
//    P V); K and V tiles arrive by TMA in 128-byte-swizzled shared memory
//    (V is the MN-major B operand as stored).  Two producer warps stream K
//    and V through their own 4-stage rings; S = Q K^T (into one of two S
//    buffers) and O += P V are issued by threads of two different warps; a
//    warpgroup runs the softmax with one thread per row (the row max and
//    sum need no shuffles).  O is rescaled in tensor memory only when a
//    row's running max grows by more than 8 (in log2 units) -- softmax does
//    not depend on the subtracted constant, and the weights stay below 2^8.
//  * mma.sync (comparison arm, below): the same units on the legacy tensor path.
//
// mma.sync arm: work unit = (query block of 32 tokens, KV head g, sequence s), one CTA.
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
constexpr uint32_t kPfWaitUs = 2000000u;  // 2 s per wait (in us)
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
        ok = mbar_wait_bounded(smem_u32(&empty[st]), (uint32_t)((j / kPfStages - 1) & 1), kPfWaitUs);
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
        (void)mbar_wait_bounded(smem_u32(&full[j % kPfStages]), (uint32_t)((j / kPfStages) & 1), kPfWaitUs);
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
    if (!mbar_wait_bounded(smem_u32(&full[st]), (uint32_t)((j / kPfStages) & 1), kPfWaitUs)) {
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

// ---------------------------------------------------------------------------
// tcgen05 prefill.
//
// Pipeline per 64-key block b (S buffers alternate with b & 1, K and V stages
// rotate with b % 4):
//   producer warp 0: K(b) -> K stage               (after S(b - 4) read it)
//   producer warp 2: V(b) -> V stage               (after P V(b - 4) read it)
//   S thread:        S(b) = Q K^T -> S buffer b & 1 once K(b) has landed and
//                    P V(b - 2) has read that buffer's P
//   P V thread:      O += P(b) V(b) once P(b) is written
//   softmax:         S(b) -> row max -> P(b) (bf16) over the first half of
//                    S buffer b & 1, row sums in registers
// Q, S, P and O live in tensor memory; shared memory only feeds K and V to
// the tensor cores (its bandwidth bounds small-N MMAs reading it).  S and P V
// are issued by threads of different warps: one thread issues an MMA every
// ~100 cycles whatever its N, so a single issuer of both would bound a
// 64-key block at 8 issue slots.  Each K copy has three blocks of time to
// land (copies take microseconds when every SM streams); page ids are read
// one block ahead.  Every barrier is used per buffer, so a waiter is never
// two phases behind its barrier.
// ---------------------------------------------------------------------------
constexpr int kTcRows = 128;                   // 32 tokens x 4 query heads
constexpr int kTcKeys = 64;                    // keys per block (4 pages)
constexpr int kTcPages = kTcKeys / PKV_PAGE_TOKENS;
constexpr int kTcKStages = 4;
constexpr int kTcVStages = 4;
constexpr int kTcThreads = 256;                // w0 K TMA, w1 S MMA, w2 V TMA, w3 P V MMA, w4-7 softmax
constexpr uint32_t kTmemCols = 256;            // S0 [0, 64), S1 [64, 128), O [128, 192), Q [192, 224)
constexpr uint32_t kTmemO = 128;
constexpr uint32_t kTmemQ = 192;               // 64 bf16 per row = 32 columns (P likewise, over S)
constexpr float kLazyRescale = 8.f;            // log2 units

struct TcSmem {
  static constexpr int kKV = kTcKeys * 128;              // 8 KB: 64 keys of 128 B
  static constexpr int kK = 0;                           // [kTcKStages] K stages
  static constexpr int kV = kK + kTcKStages * kKV;       // [kTcVStages] V stages
  static constexpr int kBars = kV + kTcVStages * kKV;
  // kfull, kempty [kTcKStages]; vfull, vempty [kTcVStages]; sfull, pfull, odone
  // [2] each; qready; drain [2] (each MMA thread's last commit)
  static constexpr int kNumBars = 2 * kTcKStages + 2 * kTcVStages + 3 * 2 + 3;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kBytes = kTmemSlot + 8;
};

// (y0, y1) = (a0 * b + c, a1 * b + c) by one packed fp32 FMA, each rounded once.
__device__ __forceinline__ void fma2(float a0, float a1, float b, float c, float& y0, float& y1) {
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %4};\n\t"
      "mov.b64 c, {%5, %5};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (s0, s1) += (e0, e1) by one packed fp32 add.
__device__ __forceinline__ void add2(float& s0, float& s1, float e0, float e1) {
  asm("{\n\t.reg .b64 s, e;\n\t"
      "mov.b64 s, {%0, %1};\n\t"
      "mov.b64 e, {%2, %3};\n\t"
      "add.rn.f32x2 s, s, e;\n\t"
      "mov.b64 {%0, %1}, s;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(e0), "f"(e1));
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Page ids of key block b (4 pages; 0 past the sequence's last page).
__device__ __forceinline__ void block_page_ids(const int32_t* row, int b, int n_pages, int (&ids)[kTcPages]) {
#pragma unroll
  for (int k = 0; k < kTcPages; ++k) {
    const int j = b * kTcPages + k;
    ids[k] = j < n_pages ? __ldg(row + j) : 0;
  }
}

__global__ void __launch_bounds__(kTcThreads, 2)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ int bad_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, g = blockIdx.y;
  const int qb = (int)gridDim.x - 1 - (int)blockIdx.x;  // latest (longest) blocks first

  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + TcSmem::kBars;
  const uint32_t kfull = bars, kempty = kfull + 8 * kTcKStages, vfull = kempty + 8 * kTcKStages,
                 vempty = vfull + 8 * kTcVStages;
  const uint32_t sfull = vempty + 8 * kTcVStages, pfull = sfull + 16, odone = sfull + 32,
                 qready = sfull + 48, drain = sfull + 56;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + TcSmem::kTmemSlot);

  // set-up that reads no global memory runs before the dependency wait
  if (threadIdx.x == 0) {
    for (int k = 0; k < kTcKStages; ++k) {
      mbar_init(kfull + 8 * k, 1);
      mbar_init(kempty + 8 * k, 1);
    }
    for (int k = 0; k < kTcVStages; ++k) {
      mbar_init(vfull + 8 * k, 1);
      mbar_init(vempty + 8 * k, 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(sfull + 8 * k, 1);
      mbar_init(pfull + 8 * k, kTcRows);
      mbar_init(odone + 8 * k, 1);
    }
    mbar_init(qready, kTcRows);
    mbar_init(drain, 1);
    mbar_init(drain + 8, 1);
    fence_mbar_init();
    bad_flag = 0;
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_wait();
  pdl_launch_dependents();
  const int r0 = __ldg(p.cu_q + s), r1 = __ldg(p.cu_q + s + 1), q_len = r1 - r0;
  const int n = __ldg(p.seq_lens + s);
  const int n_pages_seq = (n + PKV_PAGE_TOKENS - 1) / PKV_PAGE_TOKENS;
  const bool rows_ok = r0 >= 0 && r1 <= p.num_tokens && q_len >= 0;  // else touch no rows
  const bool some = rows_ok && q_len > 0;
  bool bad = some && (q_len > n || n > PKV_PAGE_TOKENS * p.max_blocks ||
                      q_len > (int)gridDim.x * kPfTokens);
  if (some && !bad && warp == 0) {
    int any = 0;
    for (int j = lane; j < n_pages_seq; j += 32) {
      const int pid = __ldg(p.block_tables + (size_t)s * p.bt_stride + j);
      any |= (pid < 0 || pid >= p.num_pages);
    }
    if (__any_sync(0xffffffffu, any) && lane == 0) bad_flag = 1;
  }
  __syncthreads();
  bad = bad || bad_flag;
  if ((!rows_ok || bad) && blockIdx.x == 0 && g == 0 && threadIdx.x == 0)
    report_error(p.d_err, PKV_ERR_DEVICE_INDEX);
  if (some && bad) zero_rows(p, r0, q_len, g);
  const int t0 = qb * kPfTokens;
  const bool run = some && !bad && t0 < q_len;
  const int t_end = min(t0 + kPfTokens, q_len);
  const int pos0 = n - q_len;
  const int nb = run ? (pos0 + t_end - 1) / kTcKeys + 1 : 0;  // key blocks [0, nb)
  bool failed = false;

  if (!run) {
  } else if (warp == 0 || warp == 2) {
    // ---------------- producers: warp 0 K tiles, warp 2 V tiles ----------
    // (one lane each, in separate warps: two lanes of one warp would
    // reconverge after every wait, tying each K copy to a V stage)
    if (lane == 0) {
      const int kv = warp == 2;
      const uint32_t full = kv ? vfull : kfull, empty = kv ? vempty : kempty;
      const uint32_t dst0 = sbase + (kv ? TcSmem::kV : TcSmem::kK);
      const int nst = kv ? kTcVStages : kTcKStages;
      const int32_t* row = p.block_tables + (size_t)s * p.bt_stride;
      int ids[kTcPages];
      block_page_ids(row, 0, n_pages_seq, ids);
      int issued = 0;
      for (int b = 0; b < nb; ++b) {
        const int st = b % nst;
        int next[kTcPages];
        block_page_ids(row, b + 1, n_pages_seq, next);
        if (b >= nst && !mbar_wait_bounded(empty + 8 * st, (uint32_t)((b / nst - 1) & 1), kPfWaitUs)) {
          report_error(p.d_err, PKV_ERR_TIMEOUT);
          break;
        }
        const int jn = min(kTcPages, n_pages_seq - b * kTcPages);
        mbar_arrive_expect_tx(full + 8 * st, (uint32_t)(jn * 2048));
#pragma unroll
        for (int pg = 0; pg < kTcPages; ++pg)
          if (pg < jn)
            tma_load_4d(dst0 + st * TcSmem::kKV + pg * 2048, &tmap, 0, 0, g, ids[pg] * 2 + kv,
                        full + 8 * st);
#pragma unroll
        for (int pg = 0; pg < kTcPages; ++pg) ids[pg] = next[pg];
        issued = b + 1;
      }
      // no copy may still be landing when the CTA exits (its consumers
      // normally saw every one; after a timeout they may not have)
      bool landed = true;
      for (int b = max(0, issued - nst); b < issued; ++b)
        landed = landed && mbar_wait_bounded(full + 8 * (b % nst), (uint32_t)((b / nst) & 1), kPfWaitUs);
      if (!landed) report_error(p.d_err, PKV_ERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ---------------- S = Q K^T issuer ------------------------------------
    if (lane == 0) {
      const uint32_t id_s = umma_idesc_bf16(kTcRows, kTcKeys, 0);
      bool ok = mbar_wait_bounded(qready, 0, kPfWaitUs);
      for (int b = 0; b < nb && ok; ++b) {
        const int st = b % kTcKStages, sb = b & 1;
        // S buffer sb holds P(b - 2) until P V(b - 2) is done
        if (!mbar_wait_bounded(kfull + 8 * st, (uint32_t)((b / kTcKStages) & 1), kPfWaitUs) ||
            (b >= 2 && !mbar_wait_bounded(odone + 8 * sb, (uint32_t)((b / 2 - 1) & 1), kPfWaitUs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sK = sbase + TcSmem::kK + st * TcSmem::kKV;
#pragma unroll
        for (int k = 0; k < 4; ++k)  // 16 dims (8 columns of Q) per step
          umma_bf16_ta(tmem + 64 * sb, tmem + kTmemQ + 8 * k, umma_desc_sw128(sK + 32 * k, 16, 1024),
                       id_s, k > 0);
        umma_commit(sfull + 8 * sb);
        umma_commit(kempty + 8 * st);  // the K stage may be refilled once S(b) is done
      }
      // every MMA issued here is complete before tensor memory is freed
      umma_commit(drain);
      if (!mbar_wait_bounded(drain, 0, kPfWaitUs)) ok = false;
      if (!ok) report_error(p.d_err, PKV_ERR_TIMEOUT);
    }
  } else if (warp == 3) {
    // ---------------- O += P V issuer -------------------------------------
    if (lane == 0) {
      const uint32_t id_o = umma_idesc_bf16(kTcRows, 64, 1);
      bool ok = true;
      for (int b = 0; b < nb; ++b) {
        const int st = b % kTcVStages, sb = b & 1;
        if (!mbar_wait_bounded(pfull + 8 * sb, (uint32_t)((b / 2) & 1), kPfWaitUs) ||
            !mbar_wait_bounded(vfull + 8 * st, (uint32_t)((b / kTcVStages) & 1), kPfWaitUs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tP = tmem + 64 * sb;  // P(b) over the first half of S buffer sb
        const uint32_t sV = sbase + TcSmem::kV + st * TcSmem::kKV;
#pragma unroll
        for (int k = 0; k < 4; ++k)  // 16 keys (8 columns of P) per step; V is MN-major (16 rows = 2048 B)
          umma_bf16_ta(tmem + kTmemO, tP + 8 * k, umma_desc_sw128(sV + 2048 * k, 8192, 1024), id_o,
                       (b > 0 || k > 0));
        umma_commit(odone + 8 * sb);
        umma_commit(vempty + 8 * st);
      }
      umma_commit(drain + 8);
      if (!mbar_wait_bounded(drain + 8, 0, kPfWaitUs)) ok = false;
      if (!ok) report_error(p.d_err, PKV_ERR_TIMEOUT);
    }
  } else if (warp >= 4) {
    // ---------------- softmax: thread = row ------------------------------
    const int i = threadIdx.x - 128;               // TMEM lane = query row
    const uint32_t lane_base = (uint32_t)(32 * (warp - 4)) << 16;
    const int tok = t0 + (i >> 2);
    const bool valid = tok < t_end;
    const int p_i = valid ? pos0 + tok : -1;
    float m_used = -INFINITY;
    float l_run = 0.f;  // row sum of the bf16 weights, relative to m_used
    // every wait is decided warp-wide: the tensor-memory loads are warp-collective
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, kPfWaitUs));
    };
    {  // this row of Q (zeros past the chunk) into tensor memory: the A operand of S
      uint32_t w[32];
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + ((size_t)(r0 + (valid ? tok : 0)) * PKV_NUM_Q_HEADS + g * 4 + (i & 3)) * 64);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 x = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        w[4 * c] = x.x, w[4 * c + 1] = x.y, w[4 * c + 2] = x.z, w[4 * c + 3] = x.w;
      }
      tmem_st32_nowait(tmem + lane_base + kTmemQ, w);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(qready);
    }
    for (int b = 0; b < nb; ++b) {
      const int st = b % kTcVStages, sb = b & 1;
      if (!wait_all(sfull + 8 * sb, (uint32_t)((b / 2) & 1))) {
        failed = true;
        break;
      }
      tc_fence_after();
      float v[64];
      tmem_ld64(tmem + lane_base + 64 * sb, v);
      // keys k0 + c with c > lim are after this row's position (or past the
      // sequence): their scores become -inf, their weights 0
      const int k0 = b * kTcKeys, lim = p_i - k0;
      if (!__all_sync(0xffffffffu, lim >= kTcKeys - 1)) {
#pragma unroll
        for (int c = 0; c < 64; ++c) v[c] = c <= lim ? v[c] : -INFINITY;
      }
      // the block's row max of the raw scores (scale * log2 e > 0, so it is
      // applied once to the max)
      float t[22];
#pragma unroll
      for (int c = 0; c < 21; ++c) t[c] = fmax3(v[3 * c], v[3 * c + 1], v[3 * c + 2]);
      t[21] = v[63];
#pragma unroll
      for (int c = 0; c < 7; ++c) t[c] = fmax3(t[3 * c], t[3 * c + 1], t[3 * c + 2]);
      const float rmx = fmax3(fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]), fmaxf(t[6], t[21]));
      const float mx = rmx * p.sl2;
      // (P V(b - 2), the last reader of S buffer sb, finished before S(b) was issued)
      const bool grow = mx > m_used + kLazyRescale || (m_used == -INFINITY && mx > -INFINITY);
      if (__any_sync(0xffffffffu, grow && m_used > -INFINITY)) {
        // O is rescaled: every P V so far (the last is P V(b - 1)) must be done
        if (b >= 1 && !wait_all(odone + 8 * ((b - 1) & 1), (uint32_t)(((b - 1) / 2) & 1))) {
          failed = true;
          break;
        }
        tc_fence_after();
        const float alpha = (grow && m_used > -INFINITY) ? exp2f(m_used - mx) : 1.f;
#pragma unroll 1
        for (int c = 0; c < 64; c += 8) tmem_scale8(tmem + lane_base + kTmemO + c, alpha);
        l_run *= alpha;
      }
      if (grow) m_used = mx;
      // weights 2^(x sl2 - m_used) (two per packed fp32 FMA), rounded to bf16
      // and packed two per column (even key low); their fp32 sum (two per
      // packed add); a row with nothing visible yet keeps m_used = -inf and
      // gets zeros
      const float nm = m_used == -INFINITY ? 0.f : -m_used;
      uint32_t pk[32];
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float y0, y1;
        fma2(v[2 * c], v[2 * c + 1], p.sl2, nm, y0, y1);
        const float e0 = ex2_approx(y0), e1 = ex2_approx(y1);
        pk[c] = pack_bf16x2(e0, e1);
        add2(ls0, ls1, e0, e1);
      }
      l_run += ls0 + ls1;
      tmem_st32_nowait(tmem + lane_base + 64 * sb, pk);
      // keys past the sequence's end: their V rows may hold any bits; zero
      // them once this block's V tiles have landed
      const int zero_from = max(0, n - k0);
      if (zero_from < kTcKeys) {
        if (!wait_all(vfull + 8 * st, (uint32_t)((b / kTcVStages) & 1))) {
          failed = true;
          break;
        }
        uint8_t* vst = smem + TcSmem::kV + st * TcSmem::kKV;
        for (int idx = i; idx < (kTcKeys - zero_from) * 8; idx += kTcRows)
          *reinterpret_cast<uint4*>(vst + (zero_from + idx / 8) * 128 + (idx & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();  // P and any rescale of O are in tensor memory
      mbar_arrive(pfull + 8 * sb);
    }
    const int lb = nb - 1;
    if (!failed && wait_all(odone + 8 * (lb & 1), (uint32_t)((lb / 2) & 1))) {
      tc_fence_after();
      const float l = l_run;
      uint4* dst = reinterpret_cast<uint4*>(
          p.out + ((size_t)(r0 + (valid ? tok : 0)) * PKV_NUM_Q_HEADS + g * 4 + (i & 3)) * 64);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float o[32];
        tmem_ld32(tmem + lane_base + kTmemO + 32 * h, o);  // every lane: warp-collective
        if (valid) {
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8)
            dst[4 * h + c8] =
                make_uint4(pack_bf16x2(__fdiv_rn(o[8 * c8], l), __fdiv_rn(o[8 * c8 + 1], l)),
                           pack_bf16x2(__fdiv_rn(o[8 * c8 + 2], l), __fdiv_rn(o[8 * c8 + 3], l)),
                           pack_bf16x2(__fdiv_rn(o[8 * c8 + 4], l), __fdiv_rn(o[8 * c8 + 5], l)),
                           pack_bf16x2(__fdiv_rn(o[8 * c8 + 6], l), __fdiv_rn(o[8 * c8 + 7], l)));
        }
      }
    } else if (!failed) {
      failed = true;
    }
    if (failed && i == 0) report_error(p.d_err, PKV_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int paged_gqa_prefill_ex(const void* q, int num_tokens, const int32_t* cu_q,
                                    const void* kv_pool, int num_pages, const int32_t* block_tables,
                                    int bt_row_stride, int max_blocks, const int32_t* seq_lens,
                                    int num_seqs, int max_q_len, void* out, float scale, int* d_err,
                                    void* stream, int compute) {
  if (compute != PKV_COMPUTE_TENSOR && compute != PKV_PREFILL_MMA_SYNC) return PKV_ERR_INVALID_ARGUMENT;
  if (num_seqs < 0 || num_tokens < 0 || num_pages < 1 || max_blocks < 1 ||
      bt_row_stride < max_blocks || max_q_len < 0)
    return PKV_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0 || max_q_len == 0 || num_tokens == 0) return PKV_OK;
  if (!q || !cu_q || !kv_pool || !block_tables || !seq_lens || !out) return PKV_ERR_INVALID_ARGUMENT;
  if (!isfinite(scale) || !(scale > 0.f)) return PKV_ERR_INVALID_ARGUMENT;
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
  rc = compute == PKV_COMPUTE_TENSOR ? make_pool_tile_map(&map, kv_pool, num_pages)
                                     : make_pool_map(&map, kv_pool, num_pages);
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
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (compute == PKV_PREFILL_MMA_SYNC) {
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = 0;
    return cuda_status(cudaLaunchKernelEx(&cfg, paged_prefill_kernel, map, prm),
                       "cudaLaunchKernelEx(prefill mma.sync)");
  }
  static bool attr_set[64] = {false};
  const size_t smem = (size_t)TcSmem::kBytes + 1024;
  if (dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  if (!attr_set[dev]) {  // benign race: every caller sets the same value
    const cudaError_t e = cudaFuncSetAttribute(paged_prefill_tc_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(prefill)");
    attr_set[dev] = true;
  }
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  return cuda_status(cudaLaunchKernelEx(&cfg, paged_prefill_tc_kernel, map, prm),
                     "cudaLaunchKernelEx(prefill tcgen05)");
}

extern "C" int paged_gqa_prefill(const void* q, int num_tokens, const int32_t* cu_q,
                                 const void* kv_pool, int num_pages, const int32_t* block_tables,
                                 int bt_row_stride, int max_blocks, const int32_t* seq_lens,
                                 int num_seqs, int max_q_len, void* out, float scale, int* d_err,
                                 void* stream) {
  return paged_gqa_prefill_ex(q, num_tokens, cu_q, kv_pool, num_pages, block_tables, bt_row_stride,
                              max_blocks, seq_lens, num_seqs, max_q_len, out, scale, d_err, stream,
                              PKV_COMPUTE_TENSOR);
}
