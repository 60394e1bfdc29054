// Paged GQA decode attention for sm_103a, one kernel per call.
//
// Source of the computation: samir-vllm article, section "Gestion de la KV
// cache et strategies de batching" (paged attention reads only the current
// sequence's pages and accumulates weighted V without a contiguous prefix or
// stored scores) and section "Architecture et flux d'inference" (grouped-query
// attention, BF16 tensors, FP32 reductions).
//
// Work decomposition (GB300-specific, not from the pages):
//   * A unit is one (sequence s, KV head g, logical page j): 2 KiB of K plus
//     2 KiB of V, contiguous in the head-major page layout.  Units are ordered
//     (s, g, j); a segment is the run of units of one (s, g).  Every CTA
//     rebuilds the per-sequence page prefix from seq_lens in shared memory (no
//     host synchronisation for variable lengths), takes the contiguous unit
//     range [c*U/NC, (c+1)*U/NC) and cuts it into kWarps contiguous warp
//     ranges, so the load is even for any length mix.
//   * Each warp is an independent pipeline: lane 0 issues TMA loads of the K
//     and V tiles (128-byte swizzle) kStages units ahead, one mbarrier per
//     stage.  Per unit the 4 query heads of the group share the page: scores
//     S = Q K^T and O += P V run on the tensor cores as bf16 mma.sync
//     m16n8k16 with fp32 accumulation (heads padded 4 -> 16 rows), or, in the
//     comparison variant, as fp32 FMA.  Online softmax in base 2, scale folded.
//   * Segment ends: a segment inside one warp range is normalised and stored
//     as bf16 by that warp.  Otherwise the warps deposit (o, m, l) records in
//     shared memory and, after one CTA barrier, the first warp of the segment
//     merges them.  A segment that lies inside the CTA range is then stored;
//     one that crosses CTA ranges is written as a CTA partial at index
//     8*s + g + c (unique: both terms grow along the unit order), counted in
//     with an atomic, and the CTA that arrives last merges the partials with a
//     log-sum-exp combine and resets the counter.  No CTA ever waits on
//     another.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <algorithm>
#include <mutex>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "i8_layout.cuh"
#include "internal.h"
#include "pkv.h"
#include "ptx.cuh"
#include "quant.cuh"
#include "rope.cuh"

namespace pkv {

constexpr int kTileBytes = 2048;     // 16 tokens x 64 dims bf16
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kRecordBytes = 4 * 64 * 4 + 4 * 8;  // o[4][64] fp32 + (m, l)[4]
constexpr int kMaxCtasPerSm = 8;     // workspace is sized for this many CTAs per SM
constexpr int kMaxSeqs = 4096;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per stage wait
constexpr uint32_t kWaitLimitUs = 2000000u;
constexpr long long kEvictFirstBytes = 64ll << 20;  // K/V bytes from which page copies evict first (L2: 129 MB)
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  const uint16_t* q;              // [S][32][64] bf16
  const int32_t* block_tables;    // [S][bt_stride]
  const int32_t* seq_lens;        // [S]
  uint8_t* pool_i8;               // INT8 pages: [num_pages][8][2176] bytes, else null
  uint16_t* out;                  // [S][32][64] bf16
  int bt_stride, max_blocks, num_pages, num_seqs;
  float sl2;                      // scale * log2(e)
  int* d_err;
  uint32_t* ws_cnt;               // [8 S] CTA arrivals per segment; zero between calls
  int32_t* ws_prefix;             // [S + 1] page prefix (separate-combine mode)
  int combine_mode;               // 0: last CTA merges; 1: boundary kernel merges
  float2* ws_ml;                  // [npart][4] (m, l); l < 0 marks a bad segment
  float* ws_o;                    // [npart][4][64]
  // Fused decode step (paged_gqa_decode_append): sequence s's new token sits
  // at position seq_lens[s] - 1; q holds the un-rotated query.
  const uint16_t* k_new;          // [S][8][64] bf16
  const uint16_t* v_new;          // [S][8][64] bf16
  const float* rope_cos;          // [max_pos][32]
  const float* rope_sin;          // [max_pos][32]
  uint16_t* q_out;                // [S][32][64] rotated q, or null
  uint16_t* pool;                 // the pool, writable (same memory as the TMA map)
  int max_pos;
  // 1: block tables, lengths and K/V pages are not written by the previous
  // kernel in the stream, so they are read (and the first pages staged)
  // before waiting for it; everything else still waits.
  int early;
  uint32_t wait_us;  // limit of each bounded wait in us (drains of copies in flight keep kWaitLimitUs)
  int kv_evict_first;  // 1: page copies under the L2 evict-first policy
  int expire_first;  // 1: warp 0 of CTA 0 waits on a barrier nothing completes (timeout test)
};

// One (o, m, l) record: unnormalised o[4][64] and (m, l) for the 4 heads of a
// KV group; l < 0 marks a segment that touched a bad page.
struct Record {
  float* o;
  float2* ml;
};

template <int kWarps, int kStages, int kStageB = kStageBytes, int kTokB = 0>
struct SmemLayout {
  static_assert(kStages * kStageB >= kRecordBytes, "slot 1 lives in the warp's own stages");
  static constexpr int kTiles = kWarps * kStages * kStageB;
  static constexpr int kBars = kTiles;                                 // u64 [kWarps][kStages]
  static constexpr int kPid = kBars + kWarps * kStages * 8;            // int [kWarps][kStages]
  static constexpr int kCnt = kPid + kWarps * kStages * 4;             // int [kWarps + 1]
  static constexpr int kSlots = kCnt + (((kWarps + 1) * 4 + 15) / 16) * 16;  // Record [kWarps]
  static constexpr int kTok = kSlots + kWarps * kRecordBytes;          // per-warp new-token area
  static constexpr int kPrefix = kTok + kWarps * kTokB;                 // int [S + 1], then len [S]
  static size_t bytes(int num_seqs) { return 1024 + kPrefix + 4 * (size_t)(2 * num_seqs + 1); }
  // Slot 0 (dedicated) holds the warp's record for a segment that began
  // before its range; slot 1 holds the record for a segment that runs past
  // its range, written after the warp's last page, in its own idle tiles.
  __device__ static Record slot(uint8_t* smem, int warp, int which) {
    uint8_t* base = which == 0 ? smem + kSlots + warp * kRecordBytes
                               : smem + warp * kStages * kStageB;
    return Record{reinterpret_cast<float*>(base), reinterpret_cast<float2*>(base + 1024)};
  }
};

__device__ __forceinline__ Record global_record(const struct DecodeParams& p, uint32_t idx) {
  return Record{p.ws_o + (size_t)idx * 256, p.ws_ml + (size_t)idx * 4};
}

// ---------------------------------------------------------------------------
// Unit cursor: walks (s, g, j) in unit order, skipping empty sequences.
// ---------------------------------------------------------------------------
struct Cursor {
  int s, g, j, np;
};

__device__ __forceinline__ void cursor_seek(Cursor& c, uint32_t u, const int32_t* prefix, int S) {
  int lo = 0, hi = S - 1;  // largest s with 8 * prefix[s] <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (8u * (uint32_t)prefix[mid] <= u) lo = mid; else hi = mid - 1;
  }
  c.s = lo;
  c.np = prefix[lo + 1] - prefix[lo];
  const uint32_t r = u - 8u * (uint32_t)prefix[lo];
  c.g = (int)(r / (uint32_t)c.np);
  c.j = (int)(r % (uint32_t)c.np);
}

__device__ __forceinline__ void cursor_next(Cursor& c, const int32_t* prefix, int S) {
  if (++c.j < c.np) return;
  c.j = 0;
  if (++c.g < 8) return;
  c.g = 0;
  do { ++c.s; } while (c.s < S && prefix[c.s + 1] == prefix[c.s]);
  if (c.s < S) c.np = prefix[c.s + 1] - prefix[c.s];
}

// First unit of the segment that contains the cursor's unit.
__device__ __forceinline__ uint32_t seg_base(const Cursor& c, const int32_t* prefix) {
  return 8u * (uint32_t)prefix[c.s] + (uint32_t)c.g * (uint32_t)c.np;
}

// Page ids of unit u, which covers logical pages kP*j .. kP*j + kP - 1 of its
// (sequence, head): .x the first, .y the second when kP == 2.  -1: an entry
// outside the pool (in .x, for the unit); -2: u is past the end of this
// warp's range; -3 (.y only): the sequence ends before the second page.
template <int kP>
__device__ __forceinline__ int2 unit_pages(uint32_t u, uint32_t u_end, const int32_t* prefix,
                                           const int32_t* lens, const DecodeParams& p) {
  if (u >= u_end) return make_int2(-2, -2);
  Cursor c;
  cursor_seek(c, u, prefix, p.num_seqs);
  const int32_t* row = p.block_tables + (size_t)c.s * p.bt_stride + kP * c.j;
  const int a = __ldg(row);
  bool ok = a >= 0 && a < p.num_pages;
  int b = -3;
  if (kP == 2 && 2 * c.j + 1 < (lens[c.s] + PKV_PAGE_TOKENS - 1) / PKV_PAGE_TOKENS) {
    b = __ldg(row + 1);
    ok = ok && b >= 0 && b < p.num_pages;
  }
  return ok ? make_int2(a, b) : make_int2(-1, -1);
}

// Units of a sequence (kP pages each), or 0 (and an error) for a length
// outside [0, max_len].
template <int kP = 1>
__device__ __forceinline__ int seq_pages(int n, int max_len, bool* bad) {
  if (n < 0 || n > max_len) {
    *bad = true;
    return 0;
  }
  return (n + kP * PKV_PAGE_TOKENS - 1) / (kP * PKV_PAGE_TOKENS);
}

// Block-wide exclusive prefix of pages over all sequences into prefix[0..S],
// if `nz` is given of non-empty sequences into nz[0..S], and if `lens` is
// given a copy of seq_lens[0..S); returns the number of sequences without
// pages (empty or invalid length).
template <int kWarps, bool kAppend, int kP = 1>
__device__ int build_prefix(const DecodeParams& p, int32_t* prefix, int32_t* nz = nullptr,
                            int32_t* lens = nullptr) {
  // with a fused append the new token's position must also lie in the table
  const int max_len = kAppend ? min(PKV_PAGE_TOKENS * p.max_blocks, p.max_pos)
                              : PKV_PAGE_TOKENS * p.max_blocks;
  __shared__ int warp_tot[kWarps], warp_nz[kWarps];
  __shared__ int n_empty;
  if (threadIdx.x == 0) n_empty = 0;
  const int S = p.num_seqs;
  const int nthr = kWarps * 32;
  const int per = (S + nthr - 1) / nthr;
  const int lo = threadIdx.x * per, hi = min(S, lo + per);
  bool bad = false;
  int sum = 0, cnt = 0;
  for (int s = lo; s < hi; ++s) {
    const int len = __ldg(p.seq_lens + s);
    if (lens) lens[s] = len;
    const int np = seq_pages<kP>(len, max_len, &bad);
    sum += np;
    cnt += (np > 0);
  }
  if (bad && blockIdx.x == 0) report_error(p.d_err, PKV_ERR_DEVICE_INDEX);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = sum, incl_nz = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    const int w = __shfl_up_sync(0xffffffffu, incl_nz, o);
    if (lane >= o) {
      incl += v;
      incl_nz += w;
    }
  }
  if (lane == 31) {
    warp_tot[warp] = incl;
    warp_nz[warp] = incl_nz;
  }
  __syncthreads();
  int base = 0, base_nz = 0;
  for (int w = 0; w < warp; ++w) {
    base += warp_tot[w];
    base_nz += warp_nz[w];
  }
  int run = base + incl - sum, run_nz = base_nz + incl_nz - cnt;
  int empties = 0;
  for (int s = lo; s < hi; ++s) {
    prefix[s] = run;
    if (nz) nz[s] = run_nz;
    const int np = seq_pages<kP>(lens ? lens[s] : __ldg(p.seq_lens + s), max_len, &bad);
    empties += (np == 0);
    run += np;
    run_nz += (np > 0);
  }
  if (threadIdx.x == nthr - 1) {
    prefix[S] = run;
    if (nz) nz[S] = run_nz;
  }
  if (empties) atomicAdd(&n_empty, empties);
  __syncthreads();
  return n_empty;
}

// Owner of unit u when U units are cut into N ranges [k*U/N, (k+1)*U/N): the
// largest k with floor(k*U/N) <= u.
__device__ __forceinline__ uint32_t owner_of(uint32_t u, uint32_t U, uint32_t N) {
  return (uint32_t)((((uint64_t)u + 1) * N - 1) / U);
}
__device__ __forceinline__ uint32_t range_start(uint32_t k, uint32_t U, uint32_t N) {
  return (uint32_t)(((uint64_t)k * U) / N);
}
// The same owner for the kN warp ranges of a CTA (kN a compile-time count):
// the number of k in 1 .. kN-1 whose range starts at or before u -- the
// starts never decrease -- with no division by the runtime size U.
template <int kN>
__device__ __forceinline__ int warp_owner(uint32_t u, uint32_t U) {
  int j = 0;
#pragma unroll
  for (int k = 1; k < kN; ++k) j += range_start(k, U, kN) <= u;
  return j;
}

// ---------------------------------------------------------------------------
// Merging records.  Lane (hh = lane/8, r = lane%8) keeps head hh, dims
// 4r .. 4r+3 (acc[0..3]) and 32+4r .. 32+4r+3 (acc[4..7]): a quarter-warp's
// 16-byte reads of a record row then cover 128 contiguous bytes, free of
// bank conflicts.  Records are combined by the log-sum-exp rule
//   M = max_k m_k,  o = sum_k 2^(m_k - M) o_k,  l = sum_k 2^(m_k - M) l_k.
// ---------------------------------------------------------------------------
struct MergeAcc {
  float acc[8];
  float M, L;
  bool bad;

  // byte offsets of this lane's two dim groups in a record's o[4][64]
  __device__ static __forceinline__ uint32_t off0(int lane) { return (uint32_t)((lane >> 3) * 256 + (lane & 7) * 16); }
  static constexpr uint32_t kOff1 = 128;  // + 32 dims

  __device__ __forceinline__ void init() {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    M = -INFINITY;
    L = 0.f;
    bad = false;
  }

  // Online form, one record at a time (the dynamic schedule's merges):
  //   M' = max(M, m);  acc = acc 2^(M - M') + o 2^(m - M');  L likewise.
  __device__ __forceinline__ void add(float2 ml, float4 o0, float4 o1) {
    if (ml.y < 0.f) {
      bad = true;
      return;
    }
    const float Mn = fmaxf(M, ml.x);
    const float a = (M == Mn) ? 1.f : exp2f(M - Mn);
    const float b = (ml.x == Mn) ? 1.f : exp2f(ml.x - Mn);
    const float ov[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = acc[i] * a + b * ov[i];
    L = L * a + b * ml.y;
    M = Mn;
  }

  // record in shared memory
  __device__ __forceinline__ void add_shared(const Record& r, int lane) {
    const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const uint8_t*>(r.o) + off0(lane));
    add(r.ml[lane >> 3], src[0], src[kOff1 / 16]);
  }

  // Merge of records 0 .. n-1 (n <= kN; record k at addr(k), skipped when
  // !live(k)) in two passes, every load of a pass in flight at once: lane
  // (hh, r) reads (m, l) of head hh of records r, r + 8, ..., the 8 lanes of
  // a head reduce the largest m, each lane turns its (m, l) into weights
  // 2^(m - M), and every lane then adds w o over all records for its dims,
  // the weight of record k coming from lane (hh, k % 8) by a shuffle.  The
  // sums run in a fixed order, so the result does not depend on timing.
  // Shared-memory records (kGlobal false) are addressed by 32-bit shared
  // addresses; records of other CTAs (kGlobal) by pointers, read through L2.
  template <int kN, bool kGlobal, class Addr, class Live>
  __device__ __forceinline__ void merge_records(int n, Addr addr, Live live, int lane) {
    static_assert(kN % 8 == 0 && kN <= 32, "records in groups of 8, at most 32");
    constexpr int kG = kN / 8;
    const int hh = lane >> 3, r8 = lane & 7;
    float mk[kG], lk[kG];
    bool bd = false;
#pragma unroll
    for (int i = 0; i < kG; ++i) {
      const int k = r8 + 8 * i;
      mk[i] = -INFINITY;
      lk[i] = 0.f;
      if (k < n && live(k)) {
        const float2 ml = ld_ml(addr(k), hh);
        if (ml.y < 0.f) {
          bd = true;
        } else {
          mk[i] = ml.x;
          lk[i] = ml.y;
        }
      }
    }
    float Mx = mk[0];
#pragma unroll
    for (int i = 1; i < kG; ++i) Mx = fmaxf(Mx, mk[i]);
    Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, 1));
    Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, 2));
    Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, 4));
    bad = bad || __any_sync(0xffffffffu, bd);
    float wk[kG], Ls = 0.f;
#pragma unroll
    for (int i = 0; i < kG; ++i) {
      wk[i] = mk[i] == -INFINITY ? 0.f : (mk[i] == Mx ? 1.f : exp2f(mk[i] - Mx));
      Ls += wk[i] * lk[i];
    }
#pragma unroll
    for (int k = 0; k < kN; ++k) {
      const float w = __shfl_sync(0xffffffffu, wk[k >> 3], (lane & ~7) | (k & 7));
      if (k < n && live(k)) {  // a bad or vanishing record has weight 0 and finite o
        float4 o0, o1;
        ld_o(addr(k), lane, o0, o1);
        acc[0] += w * o0.x; acc[1] += w * o0.y; acc[2] += w * o0.z; acc[3] += w * o0.w;
        acc[4] += w * o1.x; acc[5] += w * o1.y; acc[6] += w * o1.z; acc[7] += w * o1.w;
      }
    }
    Ls += __shfl_xor_sync(0xffffffffu, Ls, 1);
    Ls += __shfl_xor_sync(0xffffffffu, Ls, 2);
    Ls += __shfl_xor_sync(0xffffffffu, Ls, 4);
    L = Ls;
    M = Mx;
  }

  // (m, l) of head hh and this lane's o groups of a record: in shared memory
  // (32-bit address of the record) or written by another CTA (read via L2).
  __device__ static __forceinline__ float2 ld_ml(uint32_t rec, int hh) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(rec + 1024u + 8u * hh));
    return v;
  }
  __device__ static __forceinline__ float2 ld_ml(const Record& r, int hh) { return __ldcg(r.ml + hh); }
  __device__ static __forceinline__ void ld_o(uint32_t rec, int lane, float4& o0, float4& o1) {
    const uint32_t a = rec + off0(lane);
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(o0.x), "=f"(o0.y), "=f"(o0.z), "=f"(o0.w) : "r"(a));
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(o1.x), "=f"(o1.y), "=f"(o1.z), "=f"(o1.w) : "r"(a + kOff1));
  }
  __device__ static __forceinline__ void ld_o(const Record& r, int lane, float4& o0, float4& o1) {
    const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const uint8_t*>(r.o) + off0(lane));
    o0 = __ldcg(src);
    o1 = __ldcg(src + kOff1 / 16);
  }

  // Merge of any number of records written by other CTAs, eight at a time
  // with merge_records, and the groups combined by the log-sum-exp rule.
  template <class Rec>
  __device__ __forceinline__ void merge_global(int n, Rec rec, int lane) {
    if (n <= 8) {
      merge_records<8, true>(n, rec, [](int) { return true; }, lane);
      return;
    }
    for (int k0 = 0; k0 < n; k0 += 8) {
      MergeAcc part;
      part.init();
      part.merge_records<8, true>(min(8, n - k0), [&](int k) { return rec(k0 + k); },
                                  [](int) { return true; }, lane);
      bad = bad || part.bad;
      if (part.L > 0.f) {
        add(make_float2(part.M, part.L), make_float4(part.acc[0], part.acc[1], part.acc[2], part.acc[3]),
            make_float4(part.acc[4], part.acc[5], part.acc[6], part.acc[7]));
      }
    }
  }

  __device__ __forceinline__ void store_record(const Record& r, int lane) const {
    float4* dst = reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(r.o) + off0(lane));
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[kOff1 / 16] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    if ((lane & 7) == 0) r.ml[lane >> 3] = make_float2(M, bad ? -1.f : L);
  }

  __device__ __forceinline__ void store_output(const DecodeParams& p, int s, int g, int lane) const {
    const int hh = lane >> 3, r8 = lane & 7;
    const bool ok = !bad && L > 0.f;
    uint32_t packed[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      packed[i] = pack_bf16x2(ok ? __fdiv_rn(acc[2 * i], L) : 0.f, ok ? __fdiv_rn(acc[2 * i + 1], L) : 0.f);
    uint16_t* dst = p.out + ((size_t)s * PKV_NUM_Q_HEADS + g * 4 + hh) * 64 + 4 * r8;
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
    *reinterpret_cast<uint2*>(dst + 32) = make_uint2(packed[2], packed[3]);
  }
};

// ---------------------------------------------------------------------------
// Tensor-core page compute (bf16 mma.sync m16n8k16, fp32 accumulate).
// Lane (gq = lane/4, tig = lane%4).  Rows of A are query heads (rows 0..3 real,
// 4..15 zero), so only lanes 0..15 carry results.  S = Q K^T has N = tokens
// (two 8-token tiles per page, K = 64 dims in 4 chunks); O += P V has N = dims
// (8 tiles), K = 16 tokens.  The C layout of S is the A layout of P, so the
// probabilities never leave registers.
// ---------------------------------------------------------------------------
// 2^x by the hardware approximation (results below 2^-126 flush to zero):
// ex2(0) is 1 and ex2(-inf) is 0, so no special cases are needed here.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct NewToken;
template <int kP>
struct NewTokenI8;

// Stage contents of a bf16 page unit: the K tile then the V tile of one
// (page, head), one 4-D TMA box with the 128-byte swizzle.
struct Bf16Pages {
  using Token = NewToken;
  static constexpr int kTokenBytes = 0;  // the new token lives in registers
  static constexpr bool kBf16Pages = true;
  static constexpr int kPagesPerUnit = 1;
  static constexpr int kStageBytes = pkv::kStageBytes;
  static constexpr int kVOffset = kTileBytes;
  __device__ static __forceinline__ void copy(uint32_t dst, const CUtensorMap* map,
                                              const DecodeParams& p, int g, int2 pid, uint32_t bar) {
    mbar_arrive_expect_tx(bar, kStageBytes);
    if (p.kv_evict_first)  // K tile, then V tile
      tma_load_4d_ef(dst, map, 0, 0, g, pid.x * 2, bar);
    else
      tma_load_4d(dst, map, 0, 0, g, pid.x * 2, bar);
  }
};

struct MmaState : Bf16Pages {
  // at most 128 registers per thread: 16 warps of work per SM
  __host__ __device__ static constexpr int min_blocks(int warps) { return warps >= 16 ? 1 : 16 / warps; }
  uint32_t qa[4][2];  // Q A-fragments per 16-dim chunk: (row gq, k 2tig..) and (k 8+2tig..)
  float o[8][2];      // O accumulators per 8-dim tile (row lane/4; rows 8..15 are padding)
  float m, l;         // running max (log2 units) and per-lane partial denominator

  // Q fragments of query heads 4g..4g+3.  With kAppend the query is rotated
  // here at position `pos` (dims d < 32 and d + 32 sit in the same lane:
  // fragments kc and kc + 2), and written to q_out when `write_q`.
  template <bool kAppend>
  __device__ __forceinline__ void load_q(const DecodeParams& p, int s, int g, int pos,
                                         bool write_q, int lane) {
    const size_t row0 = ((size_t)s * PKV_NUM_Q_HEADS + g * 4) * 64;
    load_q_rows<kAppend, false>(p, p.q + row0, p.rope_cos + (size_t)pos * PKV_ROPE_PAIRS,
                                p.rope_sin + (size_t)pos * PKV_ROPE_PAIRS, row0, write_q, lane);
  }

  // The same from rows at `qsrc` (4 heads x 64, global or, with kStaged,
  // shared memory) and the cos/sin rows `cr`, `sr` of the new position;
  // q_out rows start at element `row0`.
  template <bool kAppend, bool kStaged>
  __device__ __forceinline__ void load_q_rows(const DecodeParams& p, const uint16_t* qsrc,
                                              const float* cr, const float* sr, size_t row0,
                                              bool write_q, int lane) {
    const int gq = lane >> 2, tig = lane & 3;
    if (gq < 4) {
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qsrc + gq * 64);
#pragma unroll
      for (int kc = 0; kc < 4; ++kc) {
        qa[kc][0] = kStaged ? qrow[kc * 8 + tig] : __ldg(qrow + kc * 8 + tig);
        qa[kc][1] = kStaged ? qrow[kc * 8 + 4 + tig] : __ldg(qrow + kc * 8 + 4 + tig);
      }
      if (kAppend) {
#pragma unroll
        for (int kc = 0; kc < 2; ++kc) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int d = 16 * kc + 8 * h + 2 * tig;
            const float2* cp = reinterpret_cast<const float2*>(cr + d);
            const float2* sp = reinterpret_cast<const float2*>(sr + d);
            const float2 c = kStaged ? *cp : __ldg(cp);
            const float2 sn = kStaged ? *sp : __ldg(sp);
            const uint32_t lo = qa[kc][h], hi = qa[kc + 2][h];
            uint16_t a0, b0, a1, b1;
            rope_pair((uint16_t)(lo & 0xFFFFu), (uint16_t)(hi & 0xFFFFu), c.x, sn.x, a0, b0);
            rope_pair((uint16_t)(lo >> 16), (uint16_t)(hi >> 16), c.y, sn.y, a1, b1);
            qa[kc][h] = (uint32_t)a0 | ((uint32_t)a1 << 16);
            qa[kc + 2][h] = (uint32_t)b0 | ((uint32_t)b1 << 16);
          }
        }
        if (write_q && p.q_out != nullptr) {
          uint32_t* qo = reinterpret_cast<uint32_t*>(p.q_out + row0 + gq * 64);
#pragma unroll
          for (int kc = 0; kc < 4; ++kc) {
            qo[kc * 8 + tig] = qa[kc][0];
            qo[kc * 8 + 4 + tig] = qa[kc][1];
          }
        }
      }
    } else {
#pragma unroll
      for (int kc = 0; kc < 4; ++kc) qa[kc][0] = qa[kc][1] = 0u;
    }
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int n = 0; n < 8; ++n) o[n][0] = o[n][1] = 0.f;
    m = -INFINITY;
    l = 0.f;
  }

  __device__ __forceinline__ void page(uint32_t sK, uint32_t sV, int valid, float sl2, int lane) {
    const int tig = lane & 3, mi = lane >> 3, r = lane & 7;
    // ---- S = Q K^T -------------------------------------------------------
    float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};
    const uint32_t krow = sK + (uint32_t)((8 * (mi >> 1) + r) * 128);
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(krow + ((((2 * kc) + (mi & 1)) ^ r) << 4), b0, b1, b2, b3);
      mma_bf16_16816(s0, qa[kc][0], qa[kc][1], b0, b1);
      mma_bf16_16816(s1, qa[kc][0], qa[kc][1], b2, b3);
    }
    // ---- online softmax (base 2) ------------------------------------------
    const int t0 = 2 * tig;
    float x0 = s0[0] * sl2, x1 = s0[1] * sl2, x2 = s1[0] * sl2, x3 = s1[1] * sl2;
    if (valid < PKV_PAGE_TOKENS) {
      x0 = (t0 < valid) ? x0 : -INFINITY;
      x1 = (t0 + 1 < valid) ? x1 : -INFINITY;
      x2 = (t0 + 8 < valid) ? x2 : -INFINITY;
      x3 = (t0 + 9 < valid) ? x3 : -INFINITY;
    }
    float pm = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 1));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 2));
    const float mn = fmaxf(m, pm);
    // hardware 2^x: exact at 0 (the row maximum weighs exactly 1, and a
    // one-token context returns V exactly), 0 at -inf (masked tokens)
    const float alpha = ex2_approx(m - mn);
    const float p0 = ex2_approx(x0 - mn);
    const float p1 = ex2_approx(x1 - mn);
    const float p2 = ex2_approx(x2 - mn);
    const float p3 = ex2_approx(x3 - mn);
    m = mn;
    const uint32_t pa0 = pack_bf16x2(p0, p1);  // P[gq][2tig, 2tig+1]
    const uint32_t pa2 = pack_bf16x2(p2, p3);  // P[gq][8+2tig, 9+2tig]
    // the denominator uses the same bf16-rounded weights as the PV product
    l = l * alpha + ((bf16lo_to_f32(pa0) + bf16hi_to_f32(pa0)) +
                     (bf16lo_to_f32(pa2) + bf16hi_to_f32(pa2)));
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      o[n][0] *= alpha;
      o[n][1] *= alpha;
    }
    // ---- O += P V ----------------------------------------------------------
    uint32_t m01 = 0xFFFFFFFFu, m89 = 0xFFFFFFFFu;
    if (valid < PKV_PAGE_TOKENS) {  // zero V rows past the end (they may hold NaN bits)
      m01 = ((t0 < valid) ? 0x0000FFFFu : 0u) | ((t0 + 1 < valid) ? 0xFFFF0000u : 0u);
      m89 = ((t0 + 8 < valid) ? 0x0000FFFFu : 0u) | ((t0 + 9 < valid) ? 0xFFFF0000u : 0u);
    }
    const uint32_t vrow = sV + (uint32_t)((8 * (mi & 1) + r) * 128);
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      uint32_t v0, v1, v2, v3;
      ldsm_x4_t(vrow + ((((2 * pp) + (mi >> 1)) ^ r) << 4), v0, v1, v2, v3);
      v0 &= m01; v2 &= m01; v1 &= m89; v3 &= m89;
      mma_bf16_16816(o[2 * pp], pa0, pa2, v0, v1);
      mma_bf16_16816(o[2 * pp + 1], pa0, pa2, v2, v3);
    }
  }

  __device__ __forceinline__ float total_l() const {
    float lt = l;
    lt += __shfl_xor_sync(0xffffffffu, lt, 1);
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
    return lt;
  }

  __device__ __forceinline__ void write_record(const Record& r, bool bad, int lane) {
    const int gq = lane >> 2, tig = lane & 3;
    const float lt = total_l();
    if (gq < 4) {
      float* o_dst = r.o + gq * 64 + 2 * tig;
#pragma unroll
      for (int n = 0; n < 8; ++n)
        *reinterpret_cast<float2*>(o_dst + 8 * n) = make_float2(o[n][0], o[n][1]);
      if (tig == 0) r.ml[gq] = make_float2(m, bad ? -1.f : lt);
    }
  }

  // A segment that one warp covers alone: normalise and store bf16 directly.
  __device__ __forceinline__ void write_output(const DecodeParams& p, int s, int g, bool bad,
                                               int lane) {
    const int gq = lane >> 2, tig = lane & 3;
    const float lt = total_l();
    if (gq < 4) {
      const bool ok = !bad && lt > 0.f;
      uint32_t* dst =
          reinterpret_cast<uint32_t*>(p.out + ((size_t)s * PKV_NUM_Q_HEADS + g * 4 + gq) * 64) + tig;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const float lo = ok ? __fdiv_rn(o[n][0], lt) : 0.f;
        const float hi = ok ? __fdiv_rn(o[n][1], lt) : 0.f;
        dst[4 * n] = pack_bf16x2(lo, hi);
      }
    }
  }
};

// ---------------------------------------------------------------------------
// CUDA-core page compute (fp32 FMA), the comparison variant.
// Lane (t8 = lane/4, qd = lane%4): tokens t8 and t8+8 of the page, dims
// [16 qd, 16 qd + 16).  Scores are reduced over the 4 lanes of a quad; the
// output accumulates per lane and is reduced over t8 once per segment.
// ---------------------------------------------------------------------------
struct FmaState : Bf16Pages {
  __host__ __device__ static constexpr int min_blocks(int) { return 1; }
  float qf[4][16];
  float o[4][16];
  float m[4], l[4];

  template <bool kAppend>
  __device__ __forceinline__ void load_q(const DecodeParams& p, int s, int g, int, bool, int lane) {
    static_assert(!kAppend, "the fused append runs on the tensor-core path only");
    const int qd = lane & 3;
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + ((size_t)s * PKV_NUM_Q_HEADS + g * 4 + hh) * 64 + 16 * qd);
      const uint4 a = __ldg(src), b = __ldg(src + 1);
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        qf[hh][2 * i] = bf16lo_to_f32(w[i]);
        qf[hh][2 * i + 1] = bf16hi_to_f32(w[i]);
      }
    }
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
#pragma unroll
      for (int d = 0; d < 16; ++d) o[hh][d] = 0.f;
      m[hh] = -INFINITY;
      l[hh] = 0.f;
    }
  }

  __device__ __forceinline__ static void load_row16(uint32_t tile, int t, int qd, float (&f)[16]) {
    uint4 a, b;
    const uint32_t row = tile + (uint32_t)(t * 128);
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w)
                 : "r"(row + (((2 * qd) ^ (t & 7)) << 4)));
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "r"(row + (((2 * qd + 1) ^ (t & 7)) << 4)));
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f[2 * i] = bf16lo_to_f32(w[i]);
      f[2 * i + 1] = bf16hi_to_f32(w[i]);
    }
  }

  __device__ __forceinline__ void page(uint32_t sK, uint32_t sV, int valid, float sl2, int lane) {
    const int t8 = lane >> 2, qd = lane & 3;
    float x[2][4];
#pragma unroll
    for (int ps = 0; ps < 2; ++ps) {
      float kf[16];
      load_row16(sK, t8 + 8 * ps, qd, kf);
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        float acc = 0.f;
#pragma unroll
        for (int d = 0; d < 16; ++d) acc = fmaf(qf[hh][d], kf[d], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        x[ps][hh] = (t8 + 8 * ps < valid) ? acc * sl2 : -INFINITY;
      }
    }
    float pr[2][4];
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      float pm = fmaxf(x[0][hh], x[1][hh]);
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
      const float mn = fmaxf(m[hh], pm);
      const float alpha = (m[hh] == mn) ? 1.f : exp2f(m[hh] - mn);
      pr[0][hh] = (x[0][hh] == mn) ? 1.f : exp2f(x[0][hh] - mn);
      pr[1][hh] = (x[1][hh] == mn) ? 1.f : exp2f(x[1][hh] - mn);
      m[hh] = mn;
      l[hh] = l[hh] * alpha + (pr[0][hh] + pr[1][hh]);
#pragma unroll
      for (int d = 0; d < 16; ++d) o[hh][d] *= alpha;
    }
#pragma unroll
    for (int ps = 0; ps < 2; ++ps) {
      if (t8 + 8 * ps < valid) {  // rows past the end may hold NaN bits: never touch them
        float vf[16];
        load_row16(sV, t8 + 8 * ps, qd, vf);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh)
#pragma unroll
          for (int d = 0; d < 16; ++d) o[hh][d] = fmaf(pr[ps][hh], vf[d], o[hh][d]);
      }
    }
  }

  // Sum o and l over the 8 token lanes (t8) that share a dim quarter.
  __device__ __forceinline__ void reduce_tokens(float (&lt)[4]) {
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      float v = l[hh];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      lt[hh] = v;
#pragma unroll
      for (int d = 0; d < 16; ++d) {
        float x = o[hh][d];
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        x += __shfl_xor_sync(0xffffffffu, x, 8);
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        o[hh][d] = x;
      }
    }
  }

  __device__ __forceinline__ void write_record(const Record& r, bool bad, int lane) {
    const int t8 = lane >> 2, qd = lane & 3;
    float lt[4];
    reduce_tokens(lt);
    if (t8 == 0) {
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        float4* dst = reinterpret_cast<float4*>(r.o + hh * 64 + 16 * qd);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_float4(o[hh][4 * i], o[hh][4 * i + 1], o[hh][4 * i + 2], o[hh][4 * i + 3]);
        if (qd == 0) r.ml[hh] = make_float2(m[hh], bad ? -1.f : lt[hh]);
      }
    }
  }

  __device__ __forceinline__ void write_output(const DecodeParams& p, int s, int g, bool bad,
                                               int lane) {
    const int t8 = lane >> 2, qd = lane & 3;
    float lt[4];
    reduce_tokens(lt);
    if (t8 == 0) {
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const bool ok = !bad && lt[hh] > 0.f;
        uint32_t* dst = reinterpret_cast<uint32_t*>(
            p.out + ((size_t)s * PKV_NUM_Q_HEADS + g * 4 + hh) * 64 + 16 * qd);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float lo = ok ? __fdiv_rn(o[hh][2 * i], lt[hh]) : 0.f;
          const float hi = ok ? __fdiv_rn(o[hh][2 * i + 1], lt[hh]) : 0.f;
          dst[i] = pack_bf16x2(lo, hi);
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------
// INT8 pages (kv_append_rope_int8).  A (page, head) is one contiguous
// 2176-byte block of the pool in the format of i8_layout.cuh, so one bulk
// copy per page brings everything a unit needs (a unit is two consecutive
// pages of a (sequence, head)).
//
// The page's 16 tokens are the M of the MMAs (m16n8k16, fp16 operands, fp32
// accumulation) and the group's 4 query heads the N (of 8): S^T = K q'^T and
// O^T += V^T P'^T, four MMAs each per page, every accumulator a full
// four-register fragment updated in place.  P' leaves S^T in accumulator
// layout (lane (g8, c) holds tokens g8 and g8 + 8 of heads 2c and 2c + 1);
// one movmatrix transpose per 8 x 8 half turns it into the B fragment of
// P'^T.  Lanes with c >= 2 carry the 4 padding heads (zero rows of q).
//
// Codes enter the MMAs as h = 1024 + byte = code + 1152: one byte permute
// makes two such fp16 (bits 0x64bb) of stored bytes, and the constant is
// taken out of the results instead of out of every operand.  Every score of
// head r carries 1152 sum_d q'_rd, so the S accumulators start at minus
// that; every element of O^T's column r carries 1152 sum_j P'_rj, which one
// more MMA per page (A = ones) accumulates beside O (rescaled with it), and
// O - 1152 * that is the result.  The cancellation costs about ten of fp32's
// 24 bits in the worst case here (2048 near-uniform weights), far below the
// bf16 output's rounding.  fp16 operands need ranges kept in check:
//   * q is multiplied by a power of two per segment so that its largest
//     |value| lies in [2^14, 2^15) (exact: a bf16 value times a power of two
//     fits fp16's 11 significant bits), and the score scale divided by it;
//   * the V scale of token j multiplies its probability, and the product is
//     divided by 2^E, E the exponent of the largest V scale of the unit, so
//     P' = p_j s_j 2^-E < 2 before its rounding to fp16; O is kept in units
//     of 2^E of the latest unit and rescaled with the softmax factors when E
//     changes.
// Scores: x_j = (q' . code_j) s_K,j scale log2(e) / 2^e_q, online softmax in
// base 2 per head as for bf16 pages; the denominator sums the fp32
// probabilities.
//
// Fragments, lane (g8 = lane / 4, c = lane % 4): in S^T's k step kt the MMA
// k indices {2c, 2c+1, 2c+8, 2c+9} are dims 16c + 4kt + {0, 1, 2, 3} (q's
// dims permuted the same way, which leaves q.k unchanged), so the lane's A
// fragments are bytes 16c .. 16c+15 of K rows g8 and g8 + 8; its B
// fragments are q' of head g8.  In O^T's m-tile m the rows are dims 16m + g8
// and 16m + g8 + 8 and the k indices tokens, so the A fragments are dims
// g8 + 8j of the token pairs (2c, 2c+1) and (2c+8, 2c+9), one 16-byte chunk
// each.  O^T's fragment of tile m holds dims 16m + g8 (elements 0, 1) and
// 16m + g8 + 8 (2, 3) of heads 2c (0, 2) and 2c + 1 (1, 3).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
// D += A B (m16n8k16, fp16 operands, fp32 accumulation), all four fragments.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// 2^k as a float for a biased exponent k clamped to the normal range.
__device__ __forceinline__ float pow2_biased(int k) {
  return __int_as_float(min(max(k, 1), 254) << 23);
}

// Rotation of the q words of an INT8-page decode lane (dims d and d + 32 sit
// in lanes c and c ^ 2 of a row) by the cos/sin pairs `rc`, `rs` (pairs
// 16 (c % 2) .. + 15 of the position's row), and their store to q_out when
// `write_q`.
__device__ __forceinline__ void rotate_q_i8(const DecodeParams& p, uint32_t (&w)[8],
                                         const float4 (&rc)[4], const float4 (&rs)[4], size_t row,
                                         bool write_q, int lane) {
  const int gq = lane >> 2, c = lane & 3;
  // Each lane makes only its own dims: own * cos + partner' * sin with
  // partner' = -partner for d < 32 (x_d cos - x_(d+32) sin) and partner for
  // d >= 32 (x_(d-32) sin + x_d cos).  The products and the sum are rounded
  // separately, as in rope_pair (the sign is exact, the sum commutes).
  const uint32_t pflip = c < 2 ? 0x80008000u : 0u;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t o = __shfl_xor_sync(0xffffffffu, w[k], 2) ^ pflip;  // the partner dims (d +- 32)
    if (gq < 4) {
      const float4 cq = rc[k >> 1], sq = rs[k >> 1];
      const float c0 = (k & 1) ? cq.z : cq.x, c1 = (k & 1) ? cq.w : cq.y;
      const float s0 = (k & 1) ? sq.z : sq.x, s1 = (k & 1) ? sq.w : sq.y;
      const float r0 = __fadd_rn(__fmul_rn(__uint_as_float(w[k] << 16), c0),
                                 __fmul_rn(__uint_as_float(o << 16), s0));
      const float r1 = __fadd_rn(__fmul_rn(__uint_as_float(w[k] & 0xFFFF0000u), c1),
                                 __fmul_rn(__uint_as_float(o & 0xFFFF0000u), s1));
      w[k] = pack_bf16x2(r0, r1);
    }
  }
  if (write_q && p.q_out != nullptr && gq < 4) {
    uint4* dst = reinterpret_cast<uint4*>(p.q_out + row);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

template <int kP>
struct MmaI8State {
  static_assert(kP == 1 || kP == 2, "one or two pages per unit");
  using Token = NewTokenI8<kP>;
  static constexpr int kTokenBytes = 4 * 128;  // the new token's K, V, cos and sin rows, per warp
  static constexpr bool kBf16Pages = false;
  static constexpr int kPagesPerUnit = kP;
  static constexpr int kBlock = PKV_I8_BLOCK_BYTES;     // one (page, head): 2176 bytes
  static constexpr int kStageBytes = kBlock * kP;        // a multiple of 16
  static constexpr int kVOffset = 1024;                  // V codes (unused: the block is one piece)
  __host__ __device__ static constexpr int min_blocks(int warps) { return warps >= 16 ? 1 : 16 / warps; }
  uint32_t qb[4][2];  // B fragments of q'^T per k step: head g8, dims 16c + 4kt + {0, 1} / {2, 3}
  float o[4][4];      // O^T + 1152 o1 in units of 2^(ev - 127) (fragment layout above)
  float o1[4];        // sum of P' of heads 2c, 2c + 1 (twice), same units
  float m0, m1;       // running max of heads 2c, 2c + 1 (log2 units)
  float l0, l1;       // their partial denominators over the lane's tokens
  float sl2q;         // scale * log2(e) / (q's power-of-two factor)
  float nc0, nc1;     // -1152 sum_d q'_d of heads 2c, 2c + 1: the S accumulators' start
  int ev;             // biased exponent of O's unit

  // The unit's pages: pid.x, and pid.y when kP == 2 and the sequence has it.
  __device__ static __forceinline__ void copy(uint32_t dst, const CUtensorMap* map,
                                              const DecodeParams& p, int g, int2 pid, uint32_t bar) {
    const bool two = kP == 2 && pid.y >= 0;
    mbar_arrive_expect_tx(bar, (two ? 2 : 1) * kBlock);
    const uint8_t* b0 = p.pool_i8 + ((size_t)pid.x * PKV_NUM_KV_HEADS + g) * kBlock;
    const uint8_t* b1 = p.pool_i8 + ((size_t)pid.y * PKV_NUM_KV_HEADS + g) * kBlock;
    if (p.kv_evict_first) {
      bulk_load_ef(dst, b0, kBlock, bar);
      if (two) bulk_load_ef(dst + kBlock, b1, kBlock, bar);
    } else {
      bulk_load(dst, b0, kBlock, bar);
      if (two) bulk_load(dst + kBlock, b1, kBlock, bar);
    }
  }

  // q rows of heads 4g..4g+3; with kAppend rotated at position `pos` first
  // (dims d and d + 32 sit in lanes c and c ^ 2 of a row) and, when
  // `write_q`, stored to q_out.
  template <bool kAppend>
  __device__ __forceinline__ void load_q(const DecodeParams& p, int s, int g, int pos, bool write_q,
                                         int lane) {
    const int gq = lane >> 2, c = lane & 3;
    uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    const size_t row = ((size_t)s * PKV_NUM_Q_HEADS + g * 4 + gq) * 64 + 16 * c;
    // the position's cos/sin pairs, requested together with q (not after it)
    float4 rc[4], rs[4];
    if (kAppend) {
      const size_t t = (size_t)pos * PKV_ROPE_PAIRS + 16 * (c & 1);
      const float4* cr = reinterpret_cast<const float4*>(p.rope_cos + t);
      const float4* sr = reinterpret_cast<const float4*>(p.rope_sin + t);
#pragma unroll
      for (int j = 0; j < 4; ++j) rc[j] = __ldg(cr + j), rs[j] = __ldg(sr + j);
    }
    if (gq < 4) {  // words 8c .. 8c+7 of the row: dims 16c .. 16c+15
      const uint4* src = reinterpret_cast<const uint4*>(p.q + row);
      const uint4 a = __ldg(src), b = __ldg(src + 1);
      w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    }
    if (kAppend) rotate_q_i8(p, w, rc, rs, row, write_q, lane);
    // largest |q| of the group (4 heads) -> factor 2^(14 - e), 2^e <= max < 2^(e+1)
    uint32_t amax = 0u;
#pragma unroll
    for (int k = 0; k < 8; ++k) amax = max(amax, max((w[k] << 16) & 0x7FFFFFFFu, w[k] & 0x7FFF0000u));
    amax = __reduce_max_sync(0xffffffffu, amax);
    // biased exponent of the largest |q|, clamped so that both factors stay normal
    const int eb = min(max((int)(amax >> 23), 15), 267);
    const float f = amax ? pow2_biased(268 - eb) : 1.f;
    sl2q = p.sl2 * (amax ? pow2_biased(eb - 14) : 1.f);
    float qsum = 0.f;  // of head gq's q' (exact products; the lane's 16 dims, then the row)
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      const float a0 = bf16lo_to_f32(w[2 * kt]) * f, a1 = bf16hi_to_f32(w[2 * kt]) * f;
      const float a2 = bf16lo_to_f32(w[2 * kt + 1]) * f, a3 = bf16hi_to_f32(w[2 * kt + 1]) * f;
      qb[kt][0] = pack_f16x2(a0, a1);
      qb[kt][1] = pack_f16x2(a2, a3);
      qsum += (a0 + a1) + (a2 + a3);
    }
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
    // heads 2c and 2c + 1 sit in lanes 8c and 8c + 4 (zero rows for c >= 2)
    nc0 = -1152.f * __shfl_sync(0xffffffffu, qsum, 8 * c);
    nc1 = -1152.f * __shfl_sync(0xffffffffu, qsum, 8 * c + 4);
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int m = 0; m < 4; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
    o1[0] = o1[1] = o1[2] = o1[3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
    ev = 127;
  }

  // One unit: kP page blocks at `base`, `valid` tokens (1 .. 16 kP) counted
  // from the unit's first token.  A missing second page (valid <= 16) is
  // computed from whatever its buffer holds, all of it masked: codes are
  // finite whatever their bits, and its scores and V scales are replaced.
  __device__ __forceinline__ void page(uint32_t base, uint32_t, int valid, float, int lane) {
    const int g8 = lane >> 2, c = lane & 3;
    constexpr uint32_t kMagic = 0x64646464u;  // high bytes of the fp16 1024 + byte
    const uint32_t koff = 64u * g8 + 16u * c;                                 // K row g8 (g8 + 8: +512)
    const uint32_t voff = 1024u + 128u * c + 16u * (uint32_t)(g8 ^ (2 * c));  // pair c (c + 4: +512)
    const uint32_t soff = 2048u + 16u * g8;                                   // scales of g8, g8 + 8
    // ---- S^T = h q'^T (accumulators start at -1152 sum q') and the scores ----
    float x[kP][4];   // tokens g8 (0, 1) and g8 + 8 (2, 3) of heads 2c (0, 2) and 2c + 1 (1, 3)
    float sv[kP][2];  // V scales of tokens g8, g8 + 8
#pragma unroll
    for (int pg = 0; pg < kP; ++pg) {
      const uint32_t blk = base + kBlock * pg;
      float s[4] = {nc0, nc1, nc0, nc1};
      const uint4 ka = lds128(blk + koff), kb = lds128(blk + koff + 512u);
      const uint32_t kaw[4] = {ka.x, ka.y, ka.z, ka.w}, kbw[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
      for (int kt = 0; kt < 4; ++kt)
        mma_f16_16816(s, __byte_perm(kaw[kt], kMagic, 0x4140), __byte_perm(kbw[kt], kMagic, 0x4140),
                      __byte_perm(kaw[kt], kMagic, 0x4342), __byte_perm(kbw[kt], kMagic, 0x4342),
                      qb[kt][0], qb[kt][1]);
      const uint4 sc = lds128(blk + soff);  // K scales of g8, g8 + 8, then their V scales
      const float fa = __uint_as_float(sc.x) * sl2q, fb = __uint_as_float(sc.y) * sl2q;
      x[pg][0] = s[0] * fa;
      x[pg][1] = s[1] * fa;
      x[pg][2] = s[2] * fb;
      x[pg][3] = s[3] * fb;
      sv[pg][0] = __uint_as_float(sc.z);
      sv[pg][1] = __uint_as_float(sc.w);
    }
    // tokens past the end: no score, and their scales may hold any bits
    if (valid < kP * PKV_PAGE_TOKENS) {
#pragma unroll
      for (int pg = 0; pg < kP; ++pg)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const bool live = pg * PKV_PAGE_TOKENS + g8 + 8 * j < valid;
          x[pg][2 * j] = live ? x[pg][2 * j] : -INFINITY;
          x[pg][2 * j + 1] = live ? x[pg][2 * j + 1] : -INFINITY;
          sv[pg][j] = live ? sv[pg][j] : 0.f;
        }
    }
    // ---- online softmax (base 2) per head over the unit's tokens -------------
    float pm0 = fmaxf(x[0][0], x[0][2]), pm1 = fmaxf(x[0][1], x[0][3]), vm = fmaxf(sv[0][0], sv[0][1]);
#pragma unroll
    for (int pg = 1; pg < kP; ++pg) {
      pm0 = fmaxf(pm0, fmaxf(x[pg][0], x[pg][2]));
      pm1 = fmaxf(pm1, fmaxf(x[pg][1], x[pg][3]));
      vm = fmaxf(vm, fmaxf(sv[pg][0], sv[pg][1]));
    }
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {  // the 8 lanes of this c hold all 16 rows
      pm0 = fmaxf(pm0, __shfl_xor_sync(0xffffffffu, pm0, sh));
      pm1 = fmaxf(pm1, __shfl_xor_sync(0xffffffffu, pm1, sh));
      vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, sh));
    }
    const float mn0 = fmaxf(m0, pm0), mn1 = fmaxf(m1, pm1);
    const int evn = vm > 0.f ? (__float_as_int(vm) >> 23) : ev;  // O's unit from this unit on
    // (mn is finite: every unit has a live token; m - mn is -inf on the first unit)
    const float as0 = ex2_approx(m0 - mn0), as1 = ex2_approx(m1 - mn1);
    const float ue = pow2_biased(127 + ev - evn);
    const float al0 = as0 * ue, al1 = as1 * ue;
    const float vinv = pow2_biased(254 - evn);  // 2^-(evn - 127)
    m0 = mn0;
    m1 = mn1;
    ev = evn;
    uint32_t pk[kP][2];  // P' (fp16) of tokens g8 + 8j, heads 2c (low) and 2c + 1
    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
    for (int pg = 0; pg < kP; ++pg)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float p0 = ex2_approx(x[pg][2 * j] - mn0), p1 = ex2_approx(x[pg][2 * j + 1] - mn1);
        const float wv = sv[pg][j] * vinv;
        ls0 += p0;
        ls1 += p1;
        pk[pg][j] = pack_f16x2(p0 * wv, p1 * wv);
      }
    l0 = l0 * as0 + ls0;
    l1 = l1 * as1 + ls1;
    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {  // most units change neither max nor unit
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        o[m][0] *= al0;
        o[m][1] *= al1;
        o[m][2] *= al0;
        o[m][3] *= al1;
      }
      o1[0] *= al0;
      o1[1] *= al1;
      o1[2] *= al0;
      o1[3] *= al1;
    }
    // ---- O^T += h^T P'^T, per page, and the ones row -------------------------
#pragma unroll
    for (int pg = 0; pg < kP; ++pg) {
      const uint32_t b0 = movmatrix_trans(pk[pg][0]), b1 = movmatrix_trans(pk[pg][1]);  // tokens 0-7, 8-15
      const uint32_t sV = base + kBlock * pg + voff;
      const uint4 va = lds128(sV), vb = lds128(sV + 512u);  // pairs c and c + 4
      const uint32_t vaw[4] = {va.x, va.y, va.z, va.w}, vbw[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
      for (int m = 0; m < 4; ++m)  // word m: dims g8 + 16m and g8 + 16m + 8 of both tokens
        mma_f16_16816(o[m], __byte_perm(vaw[m], kMagic, 0x4140), __byte_perm(vaw[m], kMagic, 0x4342),
                      __byte_perm(vbw[m], kMagic, 0x4140), __byte_perm(vbw[m], kMagic, 0x4342), b0, b1);
      mma_f16_16816(o1, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, b0, b1);  // A = 1
    }
  }

  // The denominators of heads 2c and 2c + 1 (all 16 rows of every page).
  __device__ __forceinline__ void totals(float& lt0, float& lt1) const {
    lt0 = l0;
    lt1 = l1;
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, sh);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, sh);
    }
  }

  __device__ __forceinline__ void write_record(const Record& r, bool bad, int lane) {
    const int g8 = lane >> 2, c = lane & 3;
    float lt0, lt1;
    totals(lt0, lt1);
    if (c < 2) {
      const float u = pow2_biased(ev);  // O's unit
      const float cb0 = 1152.f * o1[0], cb1 = 1152.f * o1[1];  // the codes' offset in O
      float* r0 = r.o + (2 * c) * 64 + g8;  // head 2c; head 2c + 1 at +64
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        r0[16 * m] = (o[m][0] - cb0) * u;
        r0[64 + 16 * m] = (o[m][1] - cb1) * u;
        r0[16 * m + 8] = (o[m][2] - cb0) * u;
        r0[64 + 16 * m + 8] = (o[m][3] - cb1) * u;
      }
      if (g8 == 0) {
        r.ml[2 * c] = make_float2(m0, bad ? -1.f : lt0);
        r.ml[2 * c + 1] = make_float2(m1, bad ? -1.f : lt1);
      }
    }
  }

  __device__ __forceinline__ void write_output(const DecodeParams& p, int s, int g, bool bad,
                                               int lane) {
    const int g8 = lane >> 2, c = lane & 3;
    float lt0, lt1;
    totals(lt0, lt1);
    if (c < 2) {
      const bool ok0 = !bad && lt0 > 0.f, ok1 = !bad && lt1 > 0.f;
      const float u = pow2_biased(ev);
      const float cb0 = 1152.f * o1[0], cb1 = 1152.f * o1[1];
      uint16_t* d0 = p.out + ((size_t)s * PKV_NUM_Q_HEADS + g * 4 + 2 * c) * 64 + g8;  // head 2c + 1: +64
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float v0 = ok0 ? __fdiv_rn((o[m][2 * j] - cb0) * u, lt0) : 0.f;
          const float v1 = ok1 ? __fdiv_rn((o[m][2 * j + 1] - cb1) * u, lt1) : 0.f;
          const uint32_t b = pack_bf16x2(v0, v1);
          d0[16 * m + 8 * j] = (uint16_t)(b & 0xFFFFu);
          d0[64 + 16 * m + 8 * j] = (uint16_t)(b >> 16);
        }
    }
  }
};

// ---------------------------------------------------------------------------
// Fused append: the warp that owns a sequence's last page writes the new
// token's rotated K row and its V row into the staged tiles (so its own
// attention sees them) and into the pool.  Lane l rotates the pair
// (l, l + 32) and moves V dims (2l, 2l + 1).  Shared-memory element (row, d)
// of a tile is at row*128 + (((d / 8) ^ (row % 8)) * 16) + (d % 8) * 2.
// ---------------------------------------------------------------------------
struct NewToken {
  uint16_t k0, k1;
  uint32_t v;
  float c, s;

  __device__ __forceinline__ void load(const DecodeParams& p, int seq, int g, int pos, int lane,
                                       uint32_t = 0) {
    const uint16_t* kr = p.k_new + ((size_t)seq * PKV_NUM_KV_HEADS + g) * 64;
    k0 = __ldg(kr + lane);
    k1 = __ldg(kr + lane + 32);
    v = __ldg(reinterpret_cast<const uint32_t*>(p.v_new + ((size_t)seq * PKV_NUM_KV_HEADS + g) * 64) +
              lane);
    c = __ldg(p.rope_cos + (size_t)pos * PKV_ROPE_PAIRS + lane);
    s = __ldg(p.rope_sin + (size_t)pos * PKV_ROPE_PAIRS + lane);
  }

  // The unit staged at sK holds the token's page: insert at position pos.
  __device__ __forceinline__ void insert_at(const DecodeParams& p, uint32_t sK, int pid, int,
                                            int g, int pos, int lane, uint32_t) const {
    insert(p, sK, sK + kTileBytes, pid, g, pos % PKV_PAGE_TOKENS, lane);
  }

  __device__ __forceinline__ void insert(const DecodeParams& p, uint32_t sK, uint32_t sV, int pid,
                                         int g, int slot, int lane) const {
    uint16_t r0, r1;
    rope_pair(k0, k1, c, s, r0, r1);
    const uint32_t sw = (uint32_t)(slot & 7), low = (uint32_t)(lane & 7) * 2;
    const uint32_t rk = sK + (uint32_t)slot * 128;
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(rk + ((((uint32_t)lane >> 3) ^ sw) << 4) + low),
                 "h"(r0) : "memory");
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(rk + (((((uint32_t)lane >> 3) + 4) ^ sw) << 4) + low),
                 "h"(r1) : "memory");
    const uint32_t dv = 2u * (uint32_t)lane;
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(sV + (uint32_t)slot * 128 + (((dv >> 3) ^ sw) << 4) +
                                                  (dv & 7) * 2),
                 "r"(v) : "memory");
    uint16_t* kg = p.pool + ((((size_t)pid * 2 + 0) * PKV_NUM_KV_HEADS + g) * PKV_PAGE_TOKENS + slot) * 64;
    kg[lane] = r0;
    kg[lane + 32] = r1;
    uint32_t* vg = reinterpret_cast<uint32_t*>(
        p.pool + ((((size_t)pid * 2 + 1) * PKV_NUM_KV_HEADS + g) * PKV_PAGE_TOKENS + slot) * 64);
    vg[lane] = v;
  }
};

// Fused append on INT8 pages: the warp that owns a sequence's last unit
// rotates the new token's K (rounded to bf16), quantises its K and V rows as
// kv_append_rope_int8 does (lane l holds dims l and l + 32), and writes codes
// and scales into the staged block of the token's page -- so its own
// attention sees them -- and into the pool.
template <int kP>
struct NewTokenI8 {
  // Nothing is held in registers, which the page loop needs, and nothing
  // waits at the segment's start: the token's K row, V row and the cos and
  // sin rows of its position (128 bytes each) are copied into the warp's
  // area in shared memory by cp.async (one 16-byte piece per lane), and are
  // rotated and quantised at the page that receives the token.
  static constexpr uint32_t kK = 0, kV = 128, kCos = 256, kSin = 384;

  __device__ __forceinline__ void load(const DecodeParams& p, int s, int g, int pos, int lane,
                                    uint32_t area) {
    const int part = lane >> 3, piece = lane & 7;
    const size_t row = ((size_t)s * PKV_NUM_KV_HEADS + g) * 64;
    const void* src = part == 0 ? static_cast<const void*>(p.k_new + row)
                    : part == 1 ? static_cast<const void*>(p.v_new + row)
                    : static_cast<const void*>((part == 2 ? p.rope_cos : p.rope_sin) +
                                               (size_t)pos * PKV_ROPE_PAIRS);
    cp_async16(area + 128u * (uint32_t)part + 16u * (uint32_t)piece,
               static_cast<const uint8_t*>(src) + 16 * piece);
    cp_async_commit();
  }

  // The unit staged at `base` (first page id `pid`) of sequence `seq` holds
  // position pos.
  __device__ __forceinline__ void insert_at(const DecodeParams& p, uint32_t base, int pid, int seq,
                                            int g, int pos, int lane, uint32_t area) const {
    cp_async_wait_all();
    __syncwarp();  // every lane's piece has landed
    uint16_t kd0, kd1, vd0, vd1;
    float c, sn;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(kd0) : "r"(area + kK + 2u * lane) : "memory");
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(kd1) : "r"(area + kK + 2u * (lane + 32)) : "memory");
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(vd0) : "r"(area + kV + 2u * lane) : "memory");
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(vd1) : "r"(area + kV + 2u * (lane + 32)) : "memory");
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(c) : "r"(area + kCos + 4u * lane) : "memory");
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sn) : "r"(area + kSin + 4u * lane) : "memory");
    uint16_t r0, r1;
    rope_pair(kd0, kd1, c, sn, r0, r1);
    int8_t k0, k1, v0, v1;
    const float ks = quantize_pair(__uint_as_float((uint32_t)r0 << 16),
                                   __uint_as_float((uint32_t)r1 << 16), k0, k1);
    const float vs = quantize_pair(__uint_as_float((uint32_t)vd0 << 16),
                                   __uint_as_float((uint32_t)vd1 << 16), v0, v1);
    const int lp = pos / PKV_PAGE_TOKENS, slot = pos % PKV_PAGE_TOKENS;
    const int pg = kP == 2 ? (lp & 1) : 0;  // the token's page within the unit
    const int page = pg == 0 ? pid : __ldg(p.block_tables + (size_t)seq * p.bt_stride + lp);
    const uint32_t blk = base + (uint32_t)(PKV_I8_BLOCK_BYTES * pg);
    uint8_t* gblk = p.pool_i8 + ((size_t)page * PKV_NUM_KV_HEADS + g) * PKV_I8_BLOCK_BYTES;
    const uint32_t k0o = i8_k_byte(slot, lane), k1o = i8_k_byte(slot, lane + 32);
    const uint32_t v0o = i8_v_byte(slot, lane), v1o = i8_v_byte(slot, lane + 32);
    const uint16_t b0 = i8_code_byte(k0), b1 = i8_code_byte(k1), b2 = i8_code_byte(v0),
                   b3 = i8_code_byte(v1);
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(blk + k0o), "h"(b0) : "memory");
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(blk + k1o), "h"(b1) : "memory");
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(blk + v0o), "h"(b2) : "memory");
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(blk + v1o), "h"(b3) : "memory");
    gblk[k0o] = (uint8_t)b0;
    gblk[k1o] = (uint8_t)b1;
    gblk[v0o] = (uint8_t)b2;
    gblk[v1o] = (uint8_t)b3;
    if (lane == 0) {
      const uint32_t kso = i8_k_scale_byte(slot), vso = i8_v_scale_byte(slot);
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(blk + kso), "f"(ks) : "memory");
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(blk + vso), "f"(vs) : "memory");
      *reinterpret_cast<float*>(gblk + kso) = ks;
      *reinterpret_cast<float*>(gblk + vso) = vs;
    }
  }
};

// ---------------------------------------------------------------------------
// A segment whose records come from several CTAs: store this CTA's merged
// record, count it in, and let the CTA that arrives last merge all of them.
// CTA c owns units [c*U/NC, (c+1)*U/NC); when U >= NC every CTA owns some
// units, so the CTAs touching the segment are c0..c1, else each owns at most
// one unit and the record of unit base + k comes from owner_of(base + k).
// ---------------------------------------------------------------------------
// Count this CTA's record of segment (s, g) in (it is already stored at
// record 8s + g + c) and, if it is the last one, merge all of them.
__device__ __noinline__ void cross_cta_arrive(const DecodeParams& p, int s, int g, uint32_t base,
                                              uint32_t np, uint32_t U, uint32_t NC, int lane) {
  const uint32_t sg = 8u * (uint32_t)s + (uint32_t)g;
  if (p.combine_mode == 1) return;  // merged by the boundary kernel after this grid
  __threadfence();
  __syncwarp();
  uint32_t old = 0;
  if (lane == 0) old = atomicAdd(p.ws_cnt + sg, 1u);
  old = __shfl_sync(0xffffffffu, old, 0);
  const bool dense = U >= NC;
  const uint32_t c0 = owner_of(base, U, NC);
  const uint32_t P = dense ? owner_of(base + np - 1, U, NC) - c0 + 1 : np;
  if (old != P - 1) return;
  __threadfence();  // every other record of this segment is now visible
  MergeAcc t;
  t.init();
  t.merge_global(
      (int)P,
      [&](int k) {
        const uint32_t ck = dense ? c0 + (uint32_t)k : owner_of(base + (uint32_t)k, U, NC);
        return global_record(p, sg + ck);
      },
      lane);
  t.store_output(p, s, g, lane);
  if (lane == 0) p.ws_cnt[sg] = 0u;  // ready for the next call
}

__device__ __forceinline__ void cross_cta_merge(const DecodeParams& p, const MergeAcc& mine, int s,
                                                int g, uint32_t base, uint32_t np, uint32_t U,
                                                uint32_t NC, uint32_t c, int lane) {
  mine.store_record(global_record(p, 8u * (uint32_t)s + (uint32_t)g + c), lane);
  cross_cta_arrive(p, s, g, base, np, U, NC, lane);
}

// A segment that several warps of this CTA cover, once every covering warp
// has written its record to shared memory: merge the records and store the
// output, or hand the CTA's record on to the cross-CTA merge.  CTA c owns
// units [a, b), split evenly over kWarps warps.  (Called out of line from the
// bf16-page kernels, whose page loop needs the registers, and inline from
// the INT8-page ones, where the call's saved registers spill instead.)
template <class Smem, int kWarps>
__device__ __forceinline__ void finalise_segment(const DecodeParams& p, uint8_t* smem, int s, int g,
                                                 uint32_t base, uint32_t np, uint32_t a, uint32_t b,
                                                 uint32_t U, uint32_t NC, uint32_t c, int lane) {
  const uint32_t last = base + np - 1;
  const uint32_t lo = max(base, a), hi = min(last, b - 1), n_cta = b - a;
  const int j0 = warp_owner<kWarps>(lo - a, n_cta), j1 = warp_owner<kWarps>(hi - a, n_cta);
  // the records of the covering warps j0 .. j1 with non-empty ranges: warp
  // j0's is in slot 1 if the segment starts in its range, every other one in
  // slot 0 (the segment began before the warp's range)
  const bool first_own = base >= a + range_start(j0, n_cta, kWarps);
  MergeAcc m;
  m.init();
  m.merge_records<(kWarps + 7) / 8 * 8, false>(
      j1 - j0 + 1,
      [&](int k) { return smem_u32(Smem::slot(smem, j0 + k, (k == 0 && first_own) ? 1 : 0).o); },
      [&](int k) { return range_start(j0 + k + 1, n_cta, kWarps) > range_start(j0 + k, n_cta, kWarps); },
      lane);
  if (base >= a && last < b)
    m.store_output(p, s, g, lane);
  else
    cross_cta_merge(p, m, s, g, base, np, U, NC, c, lane);
}

template <class Smem, int kWarps>
__device__ __noinline__ void finalise_segment_call(const DecodeParams& p, uint8_t* smem, int s, int g,
                                                   uint32_t base, uint32_t np, uint32_t a, uint32_t b,
                                                   uint32_t U, uint32_t NC, uint32_t c, int lane) {
  finalise_segment<Smem, kWarps>(p, smem, s, g, base, np, a, b, U, NC, c, lane);
}

// ---------------------------------------------------------------------------
// The decode kernel.
// ---------------------------------------------------------------------------
template <class State, int kWarps, int kStages, bool kAppend>
__global__ void __launch_bounds__(kWarps * 32, State::min_blocks(kWarps))
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ DecodeParams p) {
  constexpr int kStageB = State::kStageBytes;
  constexpr int kP = State::kPagesPerUnit;  // pages per unit (and per pipeline stage)
  using Smem = SmemLayout<kWarps, kStages, kStageB, State::kTokenBytes>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + Smem::kPrefix);
  int32_t* slen = prefix + (p.num_seqs + 1);
  int* spid = reinterpret_cast<int*>(smem + Smem::kPid);
  // per crossing segment: covering warps counted in (key: the warp where it
  // starts, or kWarps for the one that began before the CTA's range)
  int* seg_cnt = reinterpret_cast<int*>(smem + Smem::kCnt);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.num_seqs;
  if (threadIdx.x <= kWarps) seg_cnt[threadIdx.x] = 0;  // ordered by build_prefix's barriers

  // Without `early` everything waits for the previous kernel here.  With it,
  // only reads of q and the new token, and every global write, wait (below).
  if (!p.early) pdl_wait();
  const int n_empty = build_prefix<kWarps, kAppend, kP>(p, prefix, nullptr, slen);
  pdl_launch_dependents();

  const uint32_t U = 8u * (uint32_t)prefix[S];
  const uint32_t NC = gridDim.x, c = blockIdx.x;
  const uint32_t a = range_start(c, U, NC), b = range_start(c + 1, U, NC);
  const uint32_t u0 = a + range_start(warp, b - a, kWarps);
  const uint32_t u1 = a + range_start(warp + 1, b - a, kWarps);
  const int n_units = (int)(u1 - u0);

  if (n_units > 0) {
    const uint32_t tiles = smem_u32(smem) + warp * kStages * kStageB;
    const uint32_t bars = smem_u32(smem + Smem::kBars) + warp * kStages * 8;
    int* my_pid = spid + warp * kStages;
    if (lane == 0) {
      for (int st = 0; st < kStages; ++st) mbar_init(bars + 8 * st, 1);
      fence_mbar_init();
    }
    __syncwarp();

    // Page ids of the next 64 units, one per lane in two chunks.
    int2 pidA = unit_pages<kP>(u0 + lane, u1, prefix, slen, p);
    int2 pidB = unit_pages<kP>(u0 + 32 + lane, u1, prefix, slen, p);
    int chunk_base = 0;
    Cursor ci;
    cursor_seek(ci, u0, prefix, S);
    // the first unit's cursor and length, kept for the page loop: after the
    // dependency wait the q load is then the first thing the warp issues
    const Cursor c0 = ci;
    const int seg_len0 = slen[ci.s];
    int iv = 0;
    bool timed_out = false;

    auto issue = [&](int stage) {
      const int rel = iv - chunk_base;
      const int2 mine = rel < 32 ? pidA : pidB;
      int2 pid;
      pid.x = __shfl_sync(0xffffffffu, mine.x, rel & 31);
      pid.y = kP == 2 ? __shfl_sync(0xffffffffu, mine.y, rel & 31) : -3;
      if (lane == 0) {
        my_pid[stage] = pid.x;
        const uint32_t bar = bars + 8 * stage;
        if (pid.x >= 0) {
          fence_proxy_async_smem();
          State::copy(tiles + stage * kStageB, &tmap, p, ci.g, pid, bar);
        } else {
          mbar_arrive(bar);  // keep the phase sequence of this stage intact
        }
      }
      cursor_next(ci, prefix, S);
      ++iv;
      if (iv - chunk_base == 32) {
        pidA = pidB;
        chunk_base += 32;
        pidB = unit_pages<kP>(u0 + chunk_base + 32 + lane, u1, prefix, slen, p);
      }
    };

    for (int st = 0; st < kStages && iv < n_units; ++st) issue(st);
    __syncwarp();
    if (p.early) pdl_wait();

    State st;
    Cursor cc = c0;
    st.reset();
    int seg_len = seg_len0;
    typename State::Token tok;
    // this warp's new-token area in shared memory (states that keep the token there)
    auto tok_area = [&]() { return smem_u32(smem + Smem::kTok) + (uint32_t)(warp * State::kTokenBytes); };
    auto enter_segment = [&]() {
      const uint32_t base = seg_base(cc, prefix);
      // this warp rotates q (and stores it if it owns the segment's first
      // page) and, if it owns the last page, brings in the new token
      st.template load_q<kAppend>(p, cc.s, cc.g, seg_len - 1, base >= u0, lane);
      if (kAppend && base + (uint32_t)cc.np - 1 < u1) tok.load(p, cc.s, cc.g, seg_len - 1, lane, tok_area());
    };
    enter_segment();
    bool seg_bad = false;

    // A segment that crosses warp ranges: this warp's record is in its slot;
    // count it in, and the last of the CTA's covering warps merges them all
    // at once (no CTA-wide barrier) and finalises the segment -- after its own
    // last page, if it still has pages to stream (fin_* below).
    int fin_s = -1, fin_g = 0;
    uint32_t fin_base = 0, fin_np = 0;
    auto finalise = [&](int s, int g, uint32_t base, uint32_t np) {
      if constexpr (State::kBf16Pages)
        finalise_segment_call<Smem, kWarps>(p, smem, s, g, base, np, a, b, U, NC, c, lane);
      else
        finalise_segment<Smem, kWarps>(p, smem, s, g, base, np, a, b, U, NC, c, lane);
    };
    auto count_in = [&](int s, int g, uint32_t base, uint32_t np, bool more) {
      const uint32_t last = base + np - 1;
      const uint32_t lo = max(base, a), hi = min(last, b - 1), n_cta = b - a;
      const int j0 = warp_owner<kWarps>(lo - a, n_cta), j1 = warp_owner<kWarps>(hi - a, n_cta);
      int total = 0;
      for (int j = j0; j <= j1; ++j) total += range_start(j + 1, n_cta, kWarps) > range_start(j, n_cta, kWarps);
      int old = 0;
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();  // the record before the count
        old = atomicAdd(seg_cnt + (base < a ? kWarps : j0), 1);
      }
      old = __shfl_sync(0xffffffffu, old, 0);
      if (old + 1 != total) return;
      __threadfence_block();
      if (more) {  // keep streaming; finalise after this warp's last page
        fin_s = s;
        fin_g = g;
        fin_base = base;
        fin_np = np;
      } else {
        finalise(s, g, base, np);
      }
    };

    // the timeout test: the first warp waits on a barrier that nothing
    // arrives on instead of its first page (whose copy is drained below)
    if (p.expire_first && blockIdx.x == 0 && warp == 0) {
      __shared__ __align__(8) uint64_t never_bar;
      if (lane == 0) {
        mbar_init(smem_u32(&never_bar), 1);
        fence_mbar_init();
      }
      __syncwarp();
      if (!mbar_wait_bounded(smem_u32(&never_bar), 0u, p.wait_us)) {
        timed_out = true;
        if (lane == 0) report_error(p.d_err, PKV_ERR_TIMEOUT);
      }
    }
    for (int uc = 0; uc < n_units; ++uc) {
      const int stage = uc % kStages;
      const uint32_t parity = (uint32_t)(uc / kStages) & 1u;
      const int pid = my_pid[stage];
      if (!timed_out) {
        if (!mbar_wait_bounded(bars + 8 * stage, parity, p.wait_us)) {
          timed_out = true;
          if (lane == 0) report_error(p.d_err, PKV_ERR_TIMEOUT);
        }
      }
      if (timed_out) {
        seg_bad = true;
      } else if (pid >= 0) {
        const int valid = min(kP * PKV_PAGE_TOKENS, seg_len - kP * PKV_PAGE_TOKENS * cc.j);
        const uint32_t sK = tiles + stage * kStageB;
        if (kAppend && cc.j == cc.np - 1) {  // the page that receives the new token
          tok.insert_at(p, sK, pid, cc.s, cc.g, seg_len - 1, lane, tok_area());
          __syncwarp();
        }
        st.page(sK, sK + State::kVOffset, valid, p.sl2, lane);
      } else {
        seg_bad = true;
        if (lane == 0) report_error(p.d_err, PKV_ERR_DEVICE_INDEX);
      }
      __syncwarp();
      if (!timed_out && iv < n_units) issue(stage);
      const bool seg_end = (cc.j == cc.np - 1) || (uc == n_units - 1);
      if (seg_end) {
        const uint32_t base = seg_base(cc, prefix), last = base + (uint32_t)cc.np - 1;
        const bool before = base < u0, after = last >= u1;
        if (!before && !after) {
          st.write_output(p, cc.s, cc.g, seg_bad, lane);
        } else if (!timed_out) {  // after a timeout the segment is left unfinished
          st.write_record(Smem::slot(smem, warp, before ? 0 : 1), seg_bad, lane);
          count_in(cc.s, cc.g, base, (uint32_t)cc.np, uc + 1 < n_units);
        }
        st.reset();
        seg_bad = false;
      }
      cursor_next(cc, prefix, S);
      if (seg_end && uc + 1 < n_units) {
        seg_len = slen[cc.s];
        enter_segment();
      }
      __syncwarp();
    }
    if (fin_s >= 0 && !timed_out) finalise(fin_s, fin_g, fin_base, fin_np);
    if (timed_out) {
      // Drain whatever this warp still has in flight before leaving (bounded).
      for (int u = max(0, iv - kStages); u < iv; ++u) {
        const int stage = u % kStages;
        (void)mbar_wait_bounded(bars + 8 * stage, (uint32_t)(u / kStages) & 1u, kWaitLimitUs);
      }
    }
    // a new token's rows copied into shared memory for a page never reached
    // (an error or a timeout skipped it) must land before the CTA exits
    if (kAppend && !State::kBf16Pages) cp_async_wait_all();
  } else if (p.early) {
    pdl_wait();
  }
  if (p.combine_mode == 1 && blockIdx.x == 0)
    for (int i = threadIdx.x; i <= S; i += blockDim.x) p.ws_prefix[i] = prefix[i];
  if (n_empty > 0) {
    // Sequences without pages get a zero output (16-byte stores, grid-strided).
    const uint32_t per_seq = PKV_NUM_Q_HEADS * 64 / 8;
    const uint32_t total = (uint32_t)S * per_seq;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += gridDim.x * blockDim.x) {
      const int s = (int)(i / per_seq);
      if (prefix[s + 1] == prefix[s]) {
        reinterpret_cast<uint4*>(p.out)[i] = make_uint4(0u, 0u, 0u, 0u);
        if (kAppend && p.q_out != nullptr)
          reinterpret_cast<uint4*>(p.q_out)[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Dynamic schedule (opts.schedule = 1).  CTA c owns the unit range [a, b) as
// in the static schedule, but its warps take units one at a time from a
// shared counter, each through its own two-stage TMA pipeline, instead of
// fixed sub-ranges: the warps of a CTA finish together however unevenly
// memory serves them.  Units are taken in this order: the part of the
// segment that began in the previous CTA (block F), the part of the segment
// that runs on into the next CTA (block E), then the inner segments.  The
// records of the two shared segments are therefore complete, and merged
// across CTAs, while the inner segments still stream.
//
// A warp keeps one online-softmax state while the units it takes stay in one
// segment.  When it moves on it stores the segment (it took all of the CTA's
// units of it) or writes its (o, m, l) record into one of its two
// shared-memory record slots and counts it in with one 64-bit atomic add on
// the segment's word (units in the low half, the slot's bit in the high
// half); the record that completes the count makes its writer merge every
// listed record, free their slots and finalise the segment (store, or record
// + cross-CTA arrival).  No warp waits for another's merge.  Word e serves
// the segments of order e, e + kSeg, ... in turn -- a segment one warp
// covers alone takes its turn too -- and a slot is reused only once its last
// record has been merged, so a warp only ever waits for an older segment,
// and the oldest open segment never waits.
//
// Warps claim chunks of consecutive units, large first and shrinking to single
// units at the end (guided self-scheduling: remaining / (2 x warps)), so a
// segment gets few contributors and the CTA still ends evenly.  Per warp and
// stage one mbarrier covers the K and V tiles (TMA), the q rows of the KV
// group when the unit starts a new segment for that warp, and, for the fused
// append, the cos/sin rows of the new position and (on the page that
// receives it) the new token's K and V rows.  Page ids and (s, g) of the
// CTA's units are resolved once, into shared memory, before the pipeline
// starts.
// ---------------------------------------------------------------------------
constexpr int kDynWarps = 16;
constexpr int kDynStages = 2;
constexpr int kSeg = 64;  // segment words, reused in segment order
// staged rows per warp and stage: q (4 heads, 512 B) | k_new | v_new | cos | sin
constexpr int kSideQ = 0, kSideK = 512, kSideV = 640, kSideCos = 768, kSideSin = 896;
constexpr int kSideBytes = 1024;

struct SegWord {
  unsigned long long word;  // units counted in (low 32 bits) | record-slot bits (high 32)
  int tag;                  // order of the one segment that may use the word now
  int pad;
};

struct DynSmem {
  static constexpr int kThreads = kDynWarps * 32;
  static constexpr int kSlots = kDynWarps * kDynStages;
  static constexpr int kSide = kSlots * kStageBytes;  // tiles first (1024-aligned)
  static constexpr int kBars = kSide + kSlots * kSideBytes;
  static constexpr int kMeta = kBars + kSlots * 8;
  static constexpr int kRecs = kMeta + kSlots * 16;             // Record [2][kDynWarps]
  static constexpr int kBusy = kRecs + 2 * kDynWarps * kRecordBytes;  // int [2 kDynWarps]
  static constexpr int kSegs = kBusy + 2 * kDynWarps * 4;
  static constexpr int kCtl = kSegs + kSeg * (int)sizeof(SegWord);
  static constexpr int kPrefix = kCtl + 64;  // prefix[S + 1] | nz[S + 1] | len[S]
  __host__ __device__ static size_t table_off(int S) { return ((size_t)kPrefix + 4 * (3 * (size_t)S + 2) + 15) & ~(size_t)15; }
  __host__ __device__ static size_t bytes(int S, int n_cap) { return 1024 + table_off(S) + 8 * (size_t)n_cap; }
  // record slot `bit` = warp + kDynWarps * slot
  __device__ static Record rec(uint8_t* smem, int bit) {
    uint8_t* base = smem + kRecs + bit * kRecordBytes;
    return Record{reinterpret_cast<float*>(base), reinterpret_cast<float2*>(base + 1024)};
  }
};
static_assert(DynSmem::kRecs % 16 == 0 && kRecordBytes % 16 == 0 && DynSmem::kSegs % 16 == 0,
              "aligned records");

// Spin (one lane, bounded) until `pred()`; false after about limit_ns.
template <class Pred>
__device__ __forceinline__ bool spin_until(Pred pred, uint32_t limit_us) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (pred()) return true;
    if ((it & 255u) == 255u) {
      const uint64_t now = global_timer_ns();
      if (t0 == 0) t0 = now;
      else if (now - t0 > (uint64_t)limit_us * 1000ull) return false;
    }
  }
}

template <bool kAppend>
__global__ void __launch_bounds__(DynSmem::kThreads, 1)
    paged_decode_dyn_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ DecodeParams p,
                            int n_cap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int S = p.num_seqs;
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + DynSmem::kPrefix);
  int32_t* nz = prefix + (S + 1);
  int32_t* slen = nz + (S + 1);
  int2* ptab = reinterpret_cast<int2*>(smem + DynSmem::table_off(S));  // {page id, 8 s + g}
  int* ctl = reinterpret_cast<int*>(smem + DynSmem::kCtl);  // [0] next unit, [1] error
  const uint32_t ctl_addr = smem_u32(ctl);
  volatile int* vctl = ctl;
  SegWord* segw = reinterpret_cast<SegWord*>(smem + DynSmem::kSegs);
  volatile int* busy = reinterpret_cast<volatile int*>(smem + DynSmem::kBusy);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot0 = warp * kDynStages;
  int4* my_meta = reinterpret_cast<int4*>(smem + DynSmem::kMeta) + slot0;
  const uint32_t tiles0 = smem_u32(smem) + slot0 * kStageBytes;
  uint8_t* side0 = smem + DynSmem::kSide + slot0 * kSideBytes;
  const uint32_t bars0 = smem_u32(smem + DynSmem::kBars) + slot0 * 8;

  // shared-memory set-up (made visible by the barriers inside build_prefix)
  if (lane == 0) {
    for (int st = 0; st < kDynStages; ++st) mbar_init(bars0 + 8 * st, 1);
    fence_mbar_init();
  }
  for (int e = threadIdx.x; e < kSeg; e += blockDim.x) {
    segw[e].word = 0ull;
    segw[e].tag = e;
  }
  if (threadIdx.x < 2 * kDynWarps) busy[threadIdx.x] = 0;
  if (threadIdx.x == 0) ctl[0] = ctl[1] = 0;

  // Without `early` everything waits for the previous kernel here; with it,
  // reads of q and the new token, and every global write, wait (below).
  if (!p.early) pdl_wait();
  const int n_empty = build_prefix<kDynWarps, kAppend>(p, prefix, nz, slen);
  pdl_launch_dependents();

  const uint32_t U = 8u * (uint32_t)prefix[S];
  const uint32_t NC = gridDim.x, c = blockIdx.x;
  const uint32_t a = range_start(c, U, NC), b = range_start(c + 1, U, NC);
  int n = (int)(b - a);
  if (n > n_cap) {  // cannot happen for lengths the prefix accepts; never index past the table
    if (threadIdx.x == 0) report_error(p.d_err, PKV_ERR_DEVICE_INDEX);
    n = 0;
  }
  // blocks F and E (the segments shared with the neighbouring CTAs) first
  int F = 0, E = 0, rank0 = 0, rlast = 0;
  if (n > 0) {
    Cursor ca, cb;
    cursor_seek(ca, a, prefix, S);
    cursor_seek(cb, b - 1, prefix, S);
    const uint32_t base_a = seg_base(ca, prefix), last_a = base_a + (uint32_t)ca.np - 1;
    const uint32_t base_b = seg_base(cb, prefix), last_b = base_b + (uint32_t)cb.np - 1;
    if (base_a < a) F = (int)(min(last_a, b - 1) - a + 1);
    if (last_b >= b && base_b >= a) E = (int)(b - base_b);
    rank0 = 8 * nz[ca.s] + ca.g;
    rlast = 8 * nz[cb.s] + cb.g - rank0;
  }
  auto unit_of = [&](int q) -> uint32_t {
    if (q < F) return a + (uint32_t)q;
    if (q < F + E) return b - (uint32_t)E + (uint32_t)(q - F);
    return a + (uint32_t)(q - E);
  };
  // order of segment (s, g) among the CTA's segments as they are taken
  auto order_of = [&](int s, int g) -> int {
    const int nat = 8 * nz[s] + g - rank0;
    if (E > 0 && nat == rlast) return F > 0 ? 1 : 0;
    if (F > 0 && nat == 0) return 0;
    return nat + (E > 0 ? 1 : 0);
  };
  for (int q = threadIdx.x; q < n; q += blockDim.x) {
    Cursor cu;
    cursor_seek(cu, unit_of(q), prefix, S);
    const int pid = __ldg(p.block_tables + (size_t)cu.s * p.bt_stride + cu.j);
    ptab[q] = make_int2((pid >= 0 && pid < p.num_pages) ? pid : -1, (cu.s << 3) | cu.g);
  }
  __syncthreads();

  // ---- per-warp pipeline ----------------------------------------------------
  int last_seg = -1;   // 8 s + g of the last unit this warp staged
  uint32_t ph = 0;     // bit st: parity of the next phase of stage st
  uint32_t armed = 0;  // bit st: stage st has been armed at least once
  bool failed = false;
  int cq = 0, ce = 0;  // rest of the warp's current chunk: [cq, ce)

  // next unit for this warp: from its chunk, else a new chunk of
  // max(1, remaining / (2 x warps)) units (n when none is left)
  auto claim = [&]() -> int {
    if (cq < ce) return cq++;
    int q0 = n, sz = 0;
    if (lane == 0) {
      for (int it = 0; it < (1 << 16); ++it) {
        const int cur = ld_shared_volatile(ctl_addr);
        if (cur >= n) break;
        const int want = max(1, (n - cur) / (2 * kDynWarps));
        if (atom_cas_shared(ctl_addr, cur, cur + want) == cur) {
          q0 = cur;
          sz = want;
          break;
        }
      }
    }
    q0 = __shfl_sync(0xffffffffu, q0, 0);
    sz = __shfl_sync(0xffffffffu, sz, 0);
    cq = q0 + 1;
    ce = q0 + sz;
    return q0;
  };
  // The q / new-token / rope rows of a staged unit (lane 0).
  auto stage_rows = [&](int stage, int s, int g, bool need_q, bool is_last, int pid) {
    const uint32_t sd = smem_u32(side0 + stage * kSideBytes), bar = bars0 + 8 * stage;
    if (need_q)
      bulk_load(sd + kSideQ, p.q + ((size_t)s * PKV_NUM_Q_HEADS + g * 4) * 64, 512, bar);
    if (kAppend && (need_q || is_last)) {
      const size_t r = (size_t)(slen[s] - 1) * PKV_ROPE_PAIRS;
      bulk_load(sd + kSideCos, p.rope_cos + r, 128, bar);
      bulk_load(sd + kSideSin, p.rope_sin + r, 128, bar);
    }
    if (kAppend && is_last && pid >= 0) {
      const size_t r = ((size_t)s * PKV_NUM_KV_HEADS + g) * 64;
      bulk_load(sd + kSideK, p.k_new + r, 128, bar);
      bulk_load(sd + kSideV, p.v_new + r, 128, bar);
    }
  };
  // Table entry of unit q and its sequence's page prefix, read ahead of use.
  struct Ahead {
    int q, pid, seg, p0, p1;
  };
  auto look_ahead = [&](int q) -> Ahead {
    Ahead h;
    h.q = q;
    h.pid = -1;
    h.seg = h.p0 = h.p1 = 0;
    if (q < n) {  // entries past n were never written
      const int2 te = ptab[q];
      h.pid = te.x;
      h.seg = te.y;
      h.p0 = prefix[te.y >> 3];
      h.p1 = prefix[(te.y >> 3) + 1];
    }
    return h;
  };
  // Stage a unit: the tiles now; the q / new-token / rope rows now unless
  // `defer` (they may depend on the previous kernel).
  auto stage_unit = [&](int stage, const Ahead& h, bool defer) {
    if (h.q >= n) {
      if (lane == 0) my_meta[stage] = make_int4(-1, 0, 0, -1);
      __syncwarp();
      return;
    }
    const int q = h.q, pid = h.pid, seg = h.seg, ss = h.seg >> 3, gg = h.seg & 7;
    const int np = h.p1 - h.p0;
    const int jj = (int)(unit_of(q) - (8u * (uint32_t)h.p0 + (uint32_t)(gg * np)));
    const bool need_q = seg != last_seg;
    last_seg = seg;
    const bool is_last = kAppend && jj == np - 1;
    const uint32_t bytes = (pid >= 0 ? kStageBytes : 0) + (need_q ? 512 : 0) +
                           (kAppend && (need_q || is_last) ? 256 : 0) +
                           (kAppend && is_last && pid >= 0 ? 256 : 0);
    if (lane == 0) {
      my_meta[stage] = make_int4(q, ss, gg | (need_q << 3) | (is_last << 4) | (jj << 5), pid);
      const uint32_t bar = bars0 + 8 * stage;
      fence_proxy_async_smem();  // the stage was last read (and patched) by generic accesses
      if (bytes == 0) {
        mbar_arrive(bar);
      } else {
        mbar_arrive_expect_tx(bar, bytes);
        if (pid >= 0) {
          const uint32_t dst = tiles0 + stage * kStageBytes;
          if (p.kv_evict_first)  // K tile, then V tile
            tma_load_4d_ef(dst, &tmap, 0, 0, gg, pid * 2, bar);
          else
            tma_load_4d(dst, &tmap, 0, 0, gg, pid * 2, bar);
        }
        if (!defer) stage_rows(stage, ss, gg, need_q, is_last, pid);
      }
    }
    ph ^= 1u << stage;
    armed |= 1u << stage;
    __syncwarp();
  };

  MmaState st;
  st.reset();
  int cs = 0, cg = 0, clen = 0, m_units = 0, lorder = 0;
  uint32_t sbase = 0, snp = 1;
  bool seg_bad = false;

  int next_slot = 0;
  // Leave the current segment; false if a bounded wait gave up.
  auto flush = [&]() -> bool {
    if (m_units == 0) return true;
    const uint32_t last = sbase + snp - 1;
    const int n_x = (int)(min(last, b - 1) - max(sbase, a) + 1);
    const bool inside = sbase >= a && last < b;
    const int units = m_units;
    const bool bad = seg_bad;
    m_units = 0;
    seg_bad = false;
    SegWord& E = segw[lorder % kSeg];
    volatile int* tag = &E.tag;
    int got = 0;
    if (units == n_x) {
      // this warp took every unit the CTA has of the segment: no record, but
      // the word still passes through this segment's turn, in order
      if (lane == 0) {
        got = spin_until([&] { return *tag == lorder; }, p.wait_us);
        if (got) *tag = lorder + kSeg;
      }
      got = __shfl_sync(0xffffffffu, got, 0);
      if (got) {
        if (inside) {
          st.write_output(p, cs, cg, bad, lane);
        } else {
          st.write_record(global_record(p, 8u * (uint32_t)cs + (uint32_t)cg + c), bad, lane);
          cross_cta_arrive(p, cs, cg, sbase, snp, U, NC, lane);
        }
      }
      st.reset();
      return got != 0;
    }
    // a record slot of this warp whose last record has been merged
    const int bit = warp + kDynWarps * next_slot;
    next_slot ^= 1;
    if (lane == 0) got = spin_until([&] { return busy[bit] == 0; }, p.wait_us);
    got = __shfl_sync(0xffffffffu, got, 0);
    if (!got) {
      st.reset();
      return false;
    }
    st.write_record(DynSmem::rec(smem, bit), bad, lane);
    st.reset();
    __syncwarp();
    uint32_t lo = 0, hi = 0;
    if (lane == 0) {
      busy[bit] = 1;
      got = spin_until([&] { return *tag == lorder; }, p.wait_us);
      if (got) {
        __threadfence_block();  // the record before the count
        const unsigned long long old = atom_add_shared_u64(
            smem_u32(&E.word), (unsigned long long)units | (1ull << (32 + bit)));
        lo = (uint32_t)old;
        hi = (uint32_t)(old >> 32);
      }
    }
    got = __shfl_sync(0xffffffffu, got, 0);
    if (!got) return false;
    lo = __shfl_sync(0xffffffffu, lo, 0) + (uint32_t)units;
    hi = __shfl_sync(0xffffffffu, hi, 0) | (1u << bit);
    if ((int)lo != n_x) return true;
    // this record completes the segment: merge every record listed
    __threadfence_block();
    MergeAcc t;
    t.init();
    for (uint32_t mm = hi; mm != 0; mm &= mm - 1) t.add_shared(DynSmem::rec(smem, __ffs(mm) - 1), lane);
    __syncwarp();
    __threadfence_block();  // the reads before the slots are handed back
    if ((hi >> lane) & 1u) busy[lane] = 0;
    if (lane == 0) {
      E.word = 0ull;
      __threadfence_block();
      *tag = lorder + kSeg;
    }
    if (inside) {
      t.store_output(p, cs, cg, lane);
    } else {
      t.store_record(global_record(p, 8u * (uint32_t)cs + (uint32_t)cg + c), lane);
      cross_cta_arrive(p, cs, cg, sbase, snp, U, NC, lane);
    }
    return true;
  };

  // prologue: two units in flight (tiles only before the wait with `early`)
  for (int stg = 0; stg < kDynStages; ++stg) stage_unit(stg, look_ahead(claim()), p.early != 0);
  if (p.early) {
    pdl_wait();
    if (lane == 0)
      for (int stg = 0; stg < kDynStages; ++stg) {
        const int4 mt = my_meta[stg];
        if (mt.x >= 0) stage_rows(stg, mt.y, mt.z & 7, (mt.z >> 3) & 1, (mt.z >> 4) & 1, mt.w);
      }
    __syncwarp();
  }

  if (p.expire_first && blockIdx.x == 0 && warp == 0) {
    // the timeout test: a barrier nothing arrives on, before the first unit
    // (whether or not this warp claimed one; the drain below waits only for
    // the stages it armed)
    __shared__ __align__(8) uint64_t never_bar;
    if (lane == 0) {
      mbar_init(smem_u32(&never_bar), 1);
      fence_mbar_init();
    }
    __syncwarp();
    if (!mbar_wait_bounded(smem_u32(&never_bar), 0u, p.wait_us)) {
      failed = true;
      if (lane == 0) {
        atomicOr(ctl + 1, 1);
        report_error(p.d_err, PKV_ERR_TIMEOUT);
      }
    }
  }
  for (int k = 0; !failed; ++k) {
    const int stage = k % kDynStages;
    const int4 mt = my_meta[stage];
    if (mt.x < 0 || vctl[1] != 0) break;
    // the next unit of this warp's chunk, read before the page is computed (a
    // new chunk is claimed only after it, so claims do not run ahead)
    const bool in_chunk = cq < ce;
    const Ahead nxt = look_ahead(in_chunk ? cq++ : n);
    if (!mbar_wait_bounded(bars0 + 8 * stage, ((ph >> stage) & 1u) ^ 1u, p.wait_us)) {
      failed = true;
      if (lane == 0) {
        atomicOr(ctl + 1, 1);
        report_error(p.d_err, PKV_ERR_TIMEOUT);
      }
      break;
    }
    const int s = mt.y, g = mt.z & 7, j = mt.z >> 5, pid = mt.w;
    const bool need_q = (mt.z >> 3) & 1, is_last = (mt.z >> 4) & 1;
    const uint8_t* sd = side0 + stage * kSideBytes;
    if (need_q) {  // a new segment for this warp
      if (!flush()) {
        failed = true;
        if (lane == 0) {
          atomicOr(ctl + 1, 1);
          report_error(p.d_err, PKV_ERR_TIMEOUT);
        }
        break;
      }
      cs = s;
      cg = g;
      clen = slen[s];
      snp = (uint32_t)(prefix[s + 1] - prefix[s]);
      sbase = 8u * (uint32_t)prefix[s] + (uint32_t)g * snp;
      lorder = order_of(s, g);
      st.template load_q_rows<kAppend, true>(
          p, reinterpret_cast<const uint16_t*>(sd + kSideQ),
          reinterpret_cast<const float*>(sd + kSideCos), reinterpret_cast<const float*>(sd + kSideSin),
          ((size_t)s * PKV_NUM_Q_HEADS + g * 4) * 64, j == 0, lane);
    }
    if (pid >= 0) {
      const uint32_t sK = tiles0 + stage * kStageBytes;
      if (kAppend && is_last) {  // the new token, staged next to the tiles
        NewToken tok;
        tok.k0 = reinterpret_cast<const uint16_t*>(sd + kSideK)[lane];
        tok.k1 = reinterpret_cast<const uint16_t*>(sd + kSideK)[lane + 32];
        tok.v = reinterpret_cast<const uint32_t*>(sd + kSideV)[lane];
        tok.c = reinterpret_cast<const float*>(sd + kSideCos)[lane];
        tok.s = reinterpret_cast<const float*>(sd + kSideSin)[lane];
        tok.insert(p, sK, sK + kTileBytes, pid, g, (clen - 1) % PKV_PAGE_TOKENS, lane);
        __syncwarp();
      }
      st.page(sK, sK + kTileBytes, min(PKV_PAGE_TOKENS, clen - PKV_PAGE_TOKENS * j), p.sl2, lane);
    } else {
      seg_bad = true;
      if (lane == 0) report_error(p.d_err, PKV_ERR_DEVICE_INDEX);
    }
    ++m_units;
    __syncwarp();
    stage_unit(stage, in_chunk ? nxt : look_ahead(claim()), false);
  }
  if (!failed && vctl[1] == 0) {
    if (!flush() && lane == 0) {
      atomicOr(ctl + 1, 1);
      report_error(p.d_err, PKV_ERR_TIMEOUT);
    }
  } else {
    // after a timeout: wait (bounded) for this warp's copies still in flight
    for (int stg = 0; stg < kDynStages; ++stg)
      if ((armed >> stg) & 1u)
        (void)mbar_wait_bounded(bars0 + 8 * stg, ((ph >> stg) & 1u) ^ 1u, kWaitLimitUs);
  }

  if (p.combine_mode == 1 && blockIdx.x == 0)
    for (int i = threadIdx.x; i <= S; i += blockDim.x) p.ws_prefix[i] = prefix[i];
  if (n_empty > 0) {
    const uint32_t per_seq = PKV_NUM_Q_HEADS * 64 / 8;
    const uint32_t total = (uint32_t)S * per_seq;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += gridDim.x * blockDim.x) {
      const int s = (int)(i / per_seq);
      if (prefix[s + 1] == prefix[s]) {
        reinterpret_cast<uint4*>(p.out)[i] = make_uint4(0u, 0u, 0u, 0u);
        if (kAppend && p.q_out != nullptr)
          reinterpret_cast<uint4*>(p.q_out)[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Separate-combine mode: one warp per CTA boundary c (1 <= c < NC) merges the
// segment that first crosses it, after the decode grid has finished.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) paged_decode_boundary_kernel(const __grid_constant__ DecodeParams p,
                                                                    uint32_t NC) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const uint32_t c = blockIdx.x * 8u + (threadIdx.x >> 5) + 1u;
  if (c >= NC) return;
  const int S = p.num_seqs;
  const int32_t* prefix = p.ws_prefix;
  const uint32_t U = 8u * (uint32_t)prefix[S];
  if (U == 0) return;
  const uint32_t bc = range_start(c, U, NC);
  if (bc == 0 || bc >= U) return;
  Cursor cs;
  cursor_seek(cs, bc, prefix, S);
  const uint32_t base = seg_base(cs, prefix), np = (uint32_t)cs.np;
  if (!(base < bc) || c != owner_of(base, U, NC) + 1u) return;
  const uint32_t sg = 8u * (uint32_t)cs.s + (uint32_t)cs.g;
  const bool dense = U >= NC;
  const uint32_t c0 = owner_of(base, U, NC);
  const uint32_t P = dense ? owner_of(base + np - 1, U, NC) - c0 + 1 : np;
  MergeAcc t;
  t.init();
  t.merge_global(
      (int)P,
      [&](int k) {
        const uint32_t ck = dense ? c0 + (uint32_t)k : owner_of(base + (uint32_t)k, U, NC);
        return global_record(p, sg + ck);
      },
      lane);
  t.store_output(p, cs.s, cs.g, lane);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
struct WorkspaceLayout {
  size_t cnt, prefix, ml, o, total;
  int npart;
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// [cnt: u32 x 8S][prefix: i32 x (S+1)][ml: float2 x 4 x npart][o: float x 256 x npart] with
// npart = 8S + the most CTAs a launch can use (record index 8s + g + c).
static WorkspaceLayout workspace_layout(int num_seqs, int num_sms) {
  WorkspaceLayout w;
  w.npart = 8 * num_seqs + num_sms * kMaxCtasPerSm;
  w.cnt = 0;
  w.prefix = align256(4 * (size_t)8 * num_seqs);
  w.ml = w.prefix + align256(4 * (size_t)(num_seqs + 1));
  w.o = w.ml + align256((size_t)w.npart * 4 * sizeof(float2));
  w.total = w.o + (size_t)w.npart * 4 * 64 * sizeof(float);
  return w;
}

template <class State, int kWarps, int kStages, bool kAppend>
static int setup_kernel(int device, size_t smem, int* occ) {
  static std::mutex mu;
  static int configured[64] = {0};
  static int cached_occ[64] = {0};
  static size_t cached_smem[64] = {0};
  static int max_dyn_smem[64] = {0};
  std::lock_guard<std::mutex> lock(mu);
  auto kern = paged_decode_kernel<State, kWarps, kStages, kAppend>;
  if (device < 0 || device >= 64) {
    set_last_error("paged_gqa_decode", "device index out of range");
    return PKV_ERR_CUDA;
  }
  if (!configured[device]) {
    // opt-in limit per block minus this kernel's static shared memory
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess) return cuda_status(e, "cudaDeviceGetAttribute(smem optin)");
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncGetAttributes(decode)");
    const int max_dyn = optin - (int)fa.sharedSizeBytes;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(decode)");
    max_dyn_smem[device] = max_dyn;
    configured[device] = 1;
  }
  if ((long long)smem > max_dyn_smem[device]) return PKV_ERR_UNSUPPORTED_SHAPE;
  if (cached_smem[device] != smem) {
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kWarps * 32, smem);
    if (e != cudaSuccess) return cuda_status(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    cached_smem[device] = smem;
    cached_occ[device] = n;
  }
  *occ = cached_occ[device];
  return PKV_OK;
}

// A segment split between two CTAs costs a record hand-off through global
// memory at the end of the launch: about as long as streaming kCrossUnits
// more units per CTA (measured on the 32 x 2048 batch).  With every sequence
// at the length bound there are 8 S segments of `pages_bound` units each; if
// the CTAs can hold k whole segments each (k dividing 8 S) at a load within
// kCrossUnits of the even split, take that grid of 8 S / k CTAs instead.
constexpr long long kCrossUnits = 64;
static long long whole_segment_grid(long long nc, int num_seqs, long long pages_bound) {
  const long long n_seg = 8ll * num_seqs;
  if (nc < 2 || pages_bound < 1 || n_seg <= nc) return nc;
  const long long k = (n_seg + nc - 1) / nc;
  if (n_seg % k != 0) return nc;
  if (k * pages_bound * nc > n_seg * pages_bound + kCrossUnits * nc) return nc;
  return n_seg / k;
}

template <class State, int kWarps, int kStages, bool kAppend = false>
static int launch_decode(const DecodeParams& prm, const CUtensorMap& map, int device, int num_sms,
                         int max_seq_len, int min_units, int ctas_per_sm, cudaStream_t stream,
                         bool one_segment = false) {
  const size_t smem =
      SmemLayout<kWarps, kStages, State::kStageBytes, State::kTokenBytes>::bytes(prm.num_seqs);
  constexpr int kP = State::kPagesPerUnit;
  int occ = 0;
  int rc = setup_kernel<State, kWarps, kStages, kAppend>(device, smem, &occ);
  if (rc != PKV_OK) return rc;
  if (occ < 1) return PKV_ERR_UNSUPPORTED_SHAPE;
  occ = min(occ, kMaxCtasPerSm);
  if (ctas_per_sm > 0) occ = min(occ, ctas_per_sm);
  const long long pages_bound = max_seq_len > 0 ? (max_seq_len + 16 * kP - 1) / (16 * kP) : 0;
  const long long u_bound = 8ll * prm.num_seqs * pages_bound;  // (units of kP pages)
  long long nc = (long long)num_sms * occ;
  const long long want = (u_bound + (long long)kWarps * min_units - 1) / ((long long)kWarps * min_units);
  if (want < nc) nc = want;
  if (nc < 1) nc = 1;
  if (occ == 1) nc = whole_segment_grid(nc, prm.num_seqs, pages_bound);
  else if (one_segment && 8ll * prm.num_seqs <= (long long)num_sms * occ) nc = 8ll * prm.num_seqs;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nc);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e =
      cudaLaunchKernelEx(&cfg, paged_decode_kernel<State, kWarps, kStages, kAppend>, map, prm);
  if (e != cudaSuccess || prm.combine_mode != 1 || nc < 2) return cuda_status(e, "cudaLaunchKernelEx(decode)");
  cfg.gridDim = dim3((unsigned)((nc - 1 + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, paged_decode_boundary_kernel, prm, (uint32_t)nc);
  return cuda_status(e, "cudaLaunchKernelEx(boundary)");
}

template <bool kAppend>
static int launch_decode_dyn(const DecodeParams& prm, const CUtensorMap& map, int device,
                             int num_sms, int max_seq_len, int min_units, cudaStream_t stream) {
  static std::mutex mu;
  static int max_dyn[64] = {0};
  auto kern = paged_decode_dyn_kernel<kAppend>;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64) return PKV_ERR_CUDA;
    if (max_dyn[device] == 0) {
      int optin = 0;
      cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
      if (e != cudaSuccess) return cuda_status(e, "cudaDeviceGetAttribute(smem optin)");
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return cuda_status(e, "cudaFuncGetAttributes(dyn)");
      const int m = optin - (int)fa.sharedSizeBytes;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, m);
      if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(dyn)");
      max_dyn[device] = m;
    }
  }
  const long long pages_bound = max_seq_len > 0 ? (max_seq_len + 15) / 16 : 0;
  const long long u_bound = 8ll * prm.num_seqs * pages_bound;
  long long nc = num_sms;
  const long long per = (long long)kDynWarps * (min_units > 0 ? min_units : 1);
  const long long want = (u_bound + per - 1) / per;
  if (want < nc) nc = want;
  if (nc < 1) nc = 1;
  nc = whole_segment_grid(nc, prm.num_seqs, pages_bound);
  // page-id table: the most units any CTA can own for lengths the kernel accepts
  const long long max_len = kAppend ? std::min<long long>(16ll * prm.max_blocks, prm.max_pos)
                                    : 16ll * prm.max_blocks;
  const long long units_max = 8ll * prm.num_seqs * ((max_len + 15) / 16);
  const long long n_cap = (units_max + nc - 1) / nc + 1;
  const long long smem = (long long)DynSmem::bytes(prm.num_seqs, 0) + 8 * n_cap;
  if (smem > max_dyn[device]) return PKV_ERR_UNSUPPORTED_SHAPE;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nc);
  cfg.blockDim = dim3(DynSmem::kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, map, prm, (int)n_cap), "cudaLaunchKernelEx(dyn)");
}

}  // namespace pkv

using namespace pkv;

extern "C" size_t paged_gqa_decode_workspace_bytes(int num_seqs) {
  if (num_seqs < 0) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  const int sms = sm_count(dev);
  if (sms <= 0) return 0;
  return workspace_layout(num_seqs, sms).total;
}

namespace pkv {

// New-token inputs of the fused decode step.
struct AppendArgs {
  const void* k_new;
  const void* v_new;
  const float* rope_cos;
  const float* rope_sin;
  int max_pos;
  void* q_out;
};

int decode_check_args(const void* q, const void* kv_pool, int num_pages,
                      const int32_t* block_tables, int bt_row_stride, int max_blocks,
                      const int32_t* seq_lens, int num_seqs, const void* out, float scale) {
  if (num_seqs < 0 || num_pages < 1 || max_blocks < 1 || bt_row_stride < max_blocks)
    return PKV_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !kv_pool || !block_tables || !seq_lens || !out) return PKV_ERR_INVALID_ARGUMENT;
  if (!isfinite(scale)) return PKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return PKV_ERR_MISALIGNED;
  if (num_seqs > kMaxSeqs || (long long)num_pages * 16 * 8 * 2 >= (1ll << 31) ||
      (long long)max_blocks * PKV_PAGE_TOKENS >= (1ll << 24))
    return PKV_ERR_UNSUPPORTED_SHAPE;
  return PKV_OK;
}

static int decode_entry(const void* q, const void* kv_pool, int num_pages,
                        const int32_t* block_tables, int bt_row_stride, int max_blocks,
                        const int32_t* seq_lens, int num_seqs, int max_seq_len, void* out,
                        float scale, void* workspace, size_t workspace_bytes, int* d_err,
                        void* stream, const pkv_decode_opts* opts, const AppendArgs* app,
                        bool int8 = false, int bound_dev = -1) {
  // bound_dev >= 0: the caller has bound `stream`'s device (bind_stream_device) and passes it
  if (num_seqs < 0 || num_pages < 1 || max_blocks < 1 || bt_row_stride < max_blocks)
    return PKV_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !kv_pool || !block_tables || !seq_lens || !out || !workspace)
    return PKV_ERR_INVALID_ARGUMENT;
  if (!isfinite(scale)) return PKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(out) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return PKV_ERR_MISALIGNED;
  if (app) {
    if (!app->k_new || !app->v_new || !app->rope_cos || !app->rope_sin || app->max_pos < 1)
      return PKV_ERR_INVALID_ARGUMENT;
    if (!aligned16(app->k_new) || !aligned16(app->v_new) || !aligned16(app->rope_cos) ||
        !aligned16(app->rope_sin) || !aligned16(app->q_out))
      return PKV_ERR_MISALIGNED;
  }
  if (num_seqs > kMaxSeqs || (long long)num_pages * 16 * 8 * 2 >= (1ll << 31) ||
      (long long)max_blocks * PKV_PAGE_TOKENS >= (1ll << 24))
    return PKV_ERR_UNSUPPORTED_SHAPE;
  const int compute = opts ? opts->compute : PKV_COMPUTE_TENSOR;
  const int min_units = (opts && opts->min_units_per_warp > 0) ? opts->min_units_per_warp : 2;
  const int ctas_per_sm = opts ? opts->ctas_per_sm : 0;
  const int stages = (opts && opts->stages > 0) ? opts->stages : 2;
  // A problem that the default launch would give to at most four CTAs (a
  // few short sequences) is latency-bound: there 8 warps per CTA, fewer
  // warps to merge per sequence, answer sooner (one 37-token sequence:
  // 10.3 -> 8.2 us).  INT8 pages keep their own default.
  const long long units_hint = max_seq_len > 0 ? 8ll * num_seqs * ((max_seq_len + 15) / 16) : -1;
  const bool tiny = units_hint >= 0 && units_hint <= 4ll * 16 * 2 && !int8;
  // Between one and two (sequence, KV head) segments per SM at the length
  // bound (19 .. 38 sequences on a 152-SM GB300): 8-warp CTAs, two to an SM,
  // one segment each -- no segment is split between CTAs, and the next
  // launch's CTAs find free slots while this one's last CTAs finish (batch
  // 32 x 2048 fused step: 26.8 -> 26.1 us/layer; on INT8 pages 20.6 -> 19.1).
  const long long pages_hint = max_seq_len > 0 ? (max_seq_len + 15) / 16 : 0;
  const int sms_hint = [&] {
    int d = bound_dev;
    if (d < 0 && cudaGetDevice(&d) != cudaSuccess) return 0;
    return sm_count(d);
  }();
  const bool seg_pairs = !tiny && compute == PKV_COMPUTE_TENSOR && sms_hint > 0 &&
                         !(opts && (opts->warps_per_cta > 0 || opts->stages > 0 ||
                                    opts->ctas_per_sm > 0 || opts->min_units_per_warp > 0 ||
                                    opts->combine == 1)) &&
                         8ll * num_seqs >= sms_hint && 8ll * num_seqs <= 2ll * sms_hint &&
                         pages_hint >= 16;
  const int warps = (opts && opts->warps_per_cta > 0) ? opts->warps_per_cta : ((tiny || seg_pairs) ? 8 : 16);
  if (compute != PKV_COMPUTE_TENSOR && compute != PKV_COMPUTE_FMA) return PKV_ERR_INVALID_ARGUMENT;
  if (opts && (opts->wait_limit_ns < 0 || (opts->expire_first_wait != 0 && opts->expire_first_wait != 1)))
    return PKV_ERR_INVALID_ARGUMENT;
  if (app && compute != PKV_COMPUTE_TENSOR) return PKV_ERR_INVALID_ARGUMENT;
  const int cfg = warps * 100 + stages;
  // INT8 pages: static schedule, tensor cores, two pages per stage by default
  const int cfg8 = warps * 100 + ((opts && opts->stages > 0) ? opts->stages : 2);
  if (opts && (opts->schedule < 0 || opts->schedule > 2)) return PKV_ERR_INVALID_ARGUMENT;
  if (int8 && (compute != PKV_COMPUTE_TENSOR || (opts && (opts->schedule == 1 || opts->combine == 1)) ||
               (cfg8 != 1604 && cfg8 != 1602 && cfg8 != 804 && cfg8 != 802) || (app && cfg8 != 1602 && cfg8 != 802)))
    return PKV_ERR_INVALID_ARGUMENT;
  if (!int8 && compute == PKV_COMPUTE_TENSOR && cfg != 1602 && cfg != 1603 && cfg != 802 &&
      cfg != 804 && cfg != 402 && cfg != 404)
    return PKV_ERR_INVALID_ARGUMENT;
  if (!int8 && app && cfg != 1602 && cfg != 802 && cfg != 402) return PKV_ERR_INVALID_ARGUMENT;

  int dev = bound_dev;
  int rc = PKV_OK;
  if (dev < 0) {
    rc = bind_stream_device(stream, &dev);
    if (rc != PKV_OK) return rc;
  }
  const int sms = sm_count(dev);
  if (sms <= 0) return PKV_ERR_CUDA;
  const WorkspaceLayout wl = workspace_layout(num_seqs, sms);
  if (workspace_bytes < wl.total) return PKV_ERR_WORKSPACE_TOO_SMALL;

  CUtensorMap map;  // INT8 pages are copied by plain bulk copies: no map
  if (int8)
    memset(&map, 0, sizeof(map));
  else
    rc = make_pool_map(&map, kv_pool, num_pages);
  if (rc != PKV_OK) return rc;

  DecodeParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.q = static_cast<const uint16_t*>(q);
  prm.block_tables = block_tables;
  prm.seq_lens = seq_lens;
  prm.pool_i8 = int8 ? static_cast<uint8_t*>(const_cast<void*>(kv_pool)) : nullptr;
  prm.out = static_cast<uint16_t*>(out);
  prm.bt_stride = bt_row_stride;
  prm.max_blocks = max_blocks;
  prm.num_pages = num_pages;
  prm.num_seqs = num_seqs;
  prm.sl2 = scale * kLog2e;
  prm.d_err = d_err;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  prm.ws_cnt = reinterpret_cast<uint32_t*>(ws + wl.cnt);
  prm.ws_prefix = reinterpret_cast<int32_t*>(ws + wl.prefix);
  prm.combine_mode = (opts && opts->combine == 1) ? 1 : 0;
  prm.early = (opts && opts->early_kv == 1) ? 1 : 0;
  const uint64_t wait_ns = (opts && opts->wait_limit_ns > 0) ? (uint64_t)opts->wait_limit_ns : kWaitLimitNs;
  prm.wait_us = (uint32_t)std::min<uint64_t>(std::max<uint64_t>(wait_ns / 1000ull, 1ull), 0xFFFFFFFFull);
  prm.expire_first = (opts && opts->expire_first_wait == 1) ? 1 : 0;
  // At most this many K/V bytes can be read (at the length bound): from half
  // of the L2 up the pages go through it under the evict-first policy, so
  // that q, the tables and the records stay resident (batch 32 x 2048 fused
  // step: 25.6 -> 24.95 us/layer); smaller sets keep the default policy and
  // can stay in L2 for the next read.
  {
    const long long pages = std::min<long long>(
        max_seq_len > 0 ? (max_seq_len + PKV_PAGE_TOKENS - 1) / PKV_PAGE_TOKENS : max_blocks, max_blocks);
    const long long kv_bytes =
        (long long)num_seqs * PKV_NUM_KV_HEADS * pages * (int8 ? PKV_I8_BLOCK_BYTES : kStageBytes);
    prm.kv_evict_first = kv_bytes >= kEvictFirstBytes ? 1 : 0;
  }
  prm.ws_ml = reinterpret_cast<float2*>(ws + wl.ml);
  prm.ws_o = reinterpret_cast<float*>(ws + wl.o);
  if (app) {
    prm.k_new = static_cast<const uint16_t*>(app->k_new);
    prm.v_new = static_cast<const uint16_t*>(app->v_new);
    prm.rope_cos = app->rope_cos;
    prm.rope_sin = app->rope_sin;
    prm.max_pos = app->max_pos;
    prm.q_out = static_cast<uint16_t*>(app->q_out);
    prm.pool = static_cast<uint16_t*>(const_cast<void*>(kv_pool));
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int ms = max_seq_len;
  if (int8) {  // stages 2: two pages per stage; stages 4: one page per stage
    if (app) return cfg8 == 802 ? launch_decode<MmaI8State<2>, 8, 2, true>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st, seg_pairs)
                                : launch_decode<MmaI8State<2>, 16, 2, true>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st);
    switch (cfg8) {
      case 1604: return launch_decode<MmaI8State<1>, 16, 4>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st);
      case 804: return launch_decode<MmaI8State<1>, 8, 4>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st);
      case 802: return launch_decode<MmaI8State<2>, 8, 2>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st, seg_pairs);
      default: return launch_decode<MmaI8State<2>, 16, 2>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st);
    }
  }
  int schedule = opts ? opts->schedule : PKV_SCHEDULE_AUTO;
  if (schedule == PKV_SCHEDULE_AUTO) {
    // long per-SM ranges: the dynamic schedule evens out the warps' ends
    const long long pages_bound = ms > 0 ? (ms + 15) / 16 : 0;
    const long long units = 8ll * num_seqs * pages_bound;
    schedule = (units >= (long long)PKV_DYNAMIC_MIN_UNITS * sms && min_units == 2 &&
                (!opts || (opts->warps_per_cta == 0 && opts->stages == 0 && opts->ctas_per_sm == 0)))
                   ? PKV_SCHEDULE_DYNAMIC : PKV_SCHEDULE_STATIC;
  }
  if (schedule == PKV_SCHEDULE_DYNAMIC && compute == PKV_COMPUTE_TENSOR) {
    const int rc2 = app ? launch_decode_dyn<true>(prm, map, dev, sms, ms, min_units, st)
                        : launch_decode_dyn<false>(prm, map, dev, sms, ms, min_units, st);
    if (rc2 != PKV_ERR_UNSUPPORTED_SHAPE) return rc2;  // too many sequences: static schedule
  }
  if (app) {
    switch (cfg) {
      case 802: return launch_decode<MmaState, 8, 2, true>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st, seg_pairs);
      case 402: return launch_decode<MmaState, 4, 2, true>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st);
      default: return launch_decode<MmaState, 16, 2, true>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st);
    }
  }
  if (compute == PKV_COMPUTE_FMA)
    return launch_decode<FmaState, 4, 4>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st);
  switch (cfg) {
    case 1603: return launch_decode<MmaState, 16, 3>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st);
    case 802: return launch_decode<MmaState, 8, 2>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st, seg_pairs);
    case 804: return launch_decode<MmaState, 8, 4>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st);
    case 402: return launch_decode<MmaState, 4, 2>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st);
    case 404: return launch_decode<MmaState, 4, 4>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st);
    default: return launch_decode<MmaState, 16, 2>(prm, map, dev, sms, ms, min_units, ctas_per_sm, st);
  }
}

}  // namespace pkv

extern "C" int paged_gqa_decode_ex(const void* q, const void* kv_pool, int num_pages,
                                   const int32_t* block_tables, int bt_row_stride, int max_blocks,
                                   const int32_t* seq_lens, int num_seqs, int max_seq_len,
                                   void* out, float scale, void* workspace,
                                   size_t workspace_bytes, int* d_err, void* stream,
                                   const pkv_decode_opts* opts) {
  return decode_entry(q, kv_pool, num_pages, block_tables, bt_row_stride, max_blocks, seq_lens,
                      num_seqs, max_seq_len, out, scale, workspace, workspace_bytes, d_err, stream,
                      opts, nullptr);
}

extern "C" int paged_gqa_decode_append(const void* q, const void* k_new, const void* v_new,
                                       const float* rope_cos, const float* rope_sin, int max_pos,
                                       void* kv_pool, int num_pages, const int32_t* block_tables,
                                       int bt_row_stride, int max_blocks, const int32_t* seq_lens,
                                       int num_seqs, int max_seq_len, void* q_out, void* out,
                                       float scale, void* workspace, size_t workspace_bytes,
                                       int* d_err, void* stream, const pkv_decode_opts* opts) {
  const AppendArgs app{k_new, v_new, rope_cos, rope_sin, max_pos, q_out};
  return decode_entry(q, kv_pool, num_pages, block_tables, bt_row_stride, max_blocks, seq_lens,
                      num_seqs, max_seq_len, out, scale, workspace, workspace_bytes, d_err, stream,
                      opts, &app);
}

extern "C" int paged_gqa_decode(const void* q, const void* kv_pool, int num_pages,
                                const int32_t* block_tables, int bt_row_stride, int max_blocks,
                                const int32_t* seq_lens, int num_seqs, int max_seq_len, void* out,
                                float scale, void* workspace, size_t workspace_bytes, int* d_err,
                                void* stream) {
  return paged_gqa_decode_ex(q, kv_pool, num_pages, block_tables, bt_row_stride, max_blocks,
                             seq_lens, num_seqs, max_seq_len, out, scale, workspace,
                             workspace_bytes, d_err, stream, nullptr);
}

extern "C" int paged_gqa_decode_append_int8(const void* q, const void* k_new, const void* v_new,
                                            const float* rope_cos, const float* rope_sin,
                                            int max_pos, void* kv_pool, int num_pages,
                                            const int32_t* block_tables, int bt_row_stride,
                                            int max_blocks, const int32_t* seq_lens, int num_seqs,
                                            int max_seq_len, void* q_out, void* out, float scale,
                                            void* workspace, size_t workspace_bytes, int* d_err,
                                            void* stream, const pkv_decode_opts* opts) {
  const AppendArgs app{k_new, v_new, rope_cos, rope_sin, max_pos, q_out};
  return decode_entry(q, kv_pool, num_pages, block_tables, bt_row_stride, max_blocks, seq_lens,
                      num_seqs, max_seq_len, out, scale, workspace, workspace_bytes, d_err, stream,
                      opts, &app, true);
}

extern "C" int paged_gqa_decode_int8_ex(const void* q, const void* kv_pool, int num_pages,
                                        const int32_t* block_tables, int bt_row_stride,
                                        int max_blocks, const int32_t* seq_lens, int num_seqs,
                                        int max_seq_len, void* out, float scale, void* workspace,
                                        size_t workspace_bytes, int* d_err, void* stream,
                                        const pkv_decode_opts* opts) {
  return decode_entry(q, kv_pool, num_pages, block_tables, bt_row_stride, max_blocks, seq_lens,
                      num_seqs, max_seq_len, out, scale, workspace, workspace_bytes, d_err, stream,
                      opts, nullptr, true);
}

extern "C" int paged_gqa_decode_int8(const void* q, const void* kv_pool, int num_pages,
                                     const int32_t* block_tables, int bt_row_stride, int max_blocks,
                                     const int32_t* seq_lens, int num_seqs, int max_seq_len,
                                     void* out, float scale, void* workspace,
                                     size_t workspace_bytes, int* d_err, void* stream) {
  return paged_gqa_decode_int8_ex(q, kv_pool, num_pages, block_tables, bt_row_stride, max_blocks,
                                  seq_lens, num_seqs, max_seq_len, out, scale, workspace,
                                  workspace_bytes, d_err, stream, nullptr);
}

extern "C" int paged_gqa_decode_append_layers(
    const void* q, const void* k_new, const void* v_new, void* q_out, void* out, int num_layers,
    int num_seqs, const float* rope_cos, const float* rope_sin, int max_pos, void* kv_pool,
    int num_pages, int int8, const int32_t* block_tables, long long bt_layer_stride,
    int bt_row_stride, int max_blocks, const int32_t* seq_lens, int max_seq_len, float scale,
    void* workspace, size_t workspace_bytes, int* d_err, void* stream, int early_kv,
    const void* host_stage, void* dev_stage, size_t stage_bytes) {
  if (num_layers < 0 || num_seqs < 0 || bt_layer_stride < 0 || (int8 != 0 && int8 != 1) ||
      (early_kv != 0 && early_kv != 1))
    return PKV_ERR_INVALID_ARGUMENT;
  if ((host_stage == nullptr) != (dev_stage == nullptr) || (host_stage && stage_bytes == 0))
    return PKV_ERR_INVALID_ARGUMENT;
  if (num_layers == 0 || num_seqs == 0) return PKV_OK;
  if (!q || !k_new || !v_new || !out || !block_tables) return PKV_ERR_INVALID_ARGUMENT;
  if (bt_layer_stride < (long long)num_seqs * bt_row_stride) return PKV_ERR_INVALID_ARGUMENT;
  int rc = decode_check_args(q, kv_pool, num_pages, block_tables, bt_row_stride, max_blocks,
                             seq_lens, num_seqs, out, scale);
  if (rc != PKV_OK) return rc;
  int dev = 0;  // bound once for the copy and every layer's launch
  rc = bind_stream_device(stream, &dev);
  if (rc != PKV_OK) return rc;
  if (host_stage) {
    rc = cuda_status(cudaMemcpyAsync(dev_stage, host_stage, stage_bytes, cudaMemcpyHostToDevice,
                                     static_cast<cudaStream_t>(stream)),
                     "cudaMemcpyAsync(step block)");
    if (rc != PKV_OK) return rc;
  }
  const size_t qb = (size_t)num_seqs * PKV_NUM_Q_HEADS * PKV_HEAD_DIM * 2;
  const size_t kb = (size_t)num_seqs * PKV_NUM_KV_HEADS * PKV_HEAD_DIM * 2;
  const uint8_t* q8 = static_cast<const uint8_t*>(q);
  const uint8_t* k8 = static_cast<const uint8_t*>(k_new);
  const uint8_t* v8 = static_cast<const uint8_t*>(v_new);
  uint8_t* o8 = static_cast<uint8_t*>(out);
  uint8_t* qo8 = static_cast<uint8_t*>(q_out);
  for (int l = 0; l < num_layers; ++l) {
    pkv_decode_opts opts;
    memset(&opts, 0, sizeof(opts));
    opts.schedule = PKV_SCHEDULE_AUTO;
    opts.early_kv = (early_kv && l > 0) ? 1 : 0;
    const AppendArgs app{k8 + l * kb, v8 + l * kb, rope_cos, rope_sin, max_pos,
                         qo8 ? qo8 + l * qb : nullptr};
    rc = decode_entry(q8 + l * qb, kv_pool, num_pages, block_tables + l * bt_layer_stride,
                      bt_row_stride, max_blocks, seq_lens, num_seqs, max_seq_len, o8 + l * qb,
                      scale, workspace, workspace_bytes, d_err, stream, &opts, &app, int8 != 0, dev);
    if (rc != PKV_OK) return rc;
  }
  return PKV_OK;
}
