/*
 * pkv.h - paged GQA decode attention and fused RoPE + paged KV append
 *         for NVIDIA GB300 (sm_103a).  Plain C ABI.
 *
 * What the calls compute comes from the samir-vllm article (techfi24,
 * "samir-vllm implemente l'inference Llama 3.2 1B en C++/CUDA"):
 *   - section "Gestion de la KV cache et strategies de batching": a shared KV
 *     pool of 16-token physical pages, one block table per sequence and per
 *     layer, each new token's K/V written at its absolute RoPE position, and
 *     paged attention that reads only the sequence's own pages, accumulating
 *     weighted V without a contiguous prefix or stored scores; admission
 *     credit and explicit rejection of oversize requests;
 *   - section "Architecture et flux d'inference": grouped-query attention,
 *     BF16 storage with FP32 reductions.
 * Shapes are Llama-3.2-1B's ("2. Weight Loading and GPU Buffer Design",
 * section "Preallocating the 16 compute buffers": 32 query heads,
 * KV_DIM 512, hidden 2048), i.e. 8 KV heads of dimension 64, group size 4.
 *
 * Conventions shared by every call
 *   - Ownership: the caller owns every buffer (pool, tables, q/k/v, outputs,
 *     workspace, error word, stream).  No call allocates device memory or
 *     keeps per-call state; the library holds only a per-thread cache of TMA
 *     descriptors (host memory).  Model-owned vs caller-owned memory follows
 *     the split of "Lifecycle and Memory Model" (TinyLoop C++ API), sections
 *     "Model-owned memory" and "Per-request / handle-owned memory".
 *   - Pointers named d_* or documented as "device" are device addresses;
 *     "host" pointers are ordinary CPU memory.  bf16 tensors are passed as
 *     void* to keep CUDA headers out of this file.
 *   - Asynchrony: GPU calls only enqueue work on `stream` (a cudaStream_t,
 *     NULL = legacy default stream) and return at once.  The return value
 *     reports host-side checks (null pointers, alignment, sizes, launch
 *     errors) only.  Problems the kernels find in the data (a page id
 *     outside the pool, a position beyond the table) are written to the
 *     caller's device error word *d_err: the first code wins (atomic
 *     compare-and-swap from 0), the offending token or sequence is skipped
 *     (its output rows are written as zeros) and no kernel ever traps.
 *   - Thread safety: calls are re-entrant; concurrent calls on different
 *     streams need distinct workspaces and outputs ("Lifecycle and Memory
 *     Model", section "Mutable state and thread-safety implications").
 *     The scheduler object (pkv_sched_*) is not thread-safe.
 *   - Device selection: a call runs on the device that owns `stream`
 *     (the current device for the default stream).  While `stream` is being
 *     captured into a CUDA graph the stream cannot be queried, so the device
 *     made current by the last uncaptured call on this thread is used: run
 *     each call once before capturing it (which also does the one-time
 *     kernel set-up outside the capture).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Fixed layer topology (compile-time in the kernels). */
#define PKV_NUM_Q_HEADS 32
#define PKV_NUM_KV_HEADS 8
#define PKV_GROUP 4
#define PKV_HEAD_DIM 64
#define PKV_ROPE_PAIRS 32
#define PKV_PAGE_TOKENS 16
#define PKV_PAGE_ELEMS (2 * PKV_NUM_KV_HEADS * PKV_PAGE_TOKENS * PKV_HEAD_DIM)
#define PKV_PAGE_BYTES (2 * PKV_PAGE_ELEMS) /* 32768 */
/* INT8 pages: one block per (page, KV head) = K codes [16][64] int8, V codes
 * [16][64] int8, K scales [16] float, V scales [16] float. */
#define PKV_I8_BLOCK_BYTES (2 * PKV_PAGE_TOKENS * PKV_HEAD_DIM + 2 * PKV_PAGE_TOKENS * 4) /* 2176 */
#define PKV_I8_PAGE_BYTES (PKV_NUM_KV_HEADS * PKV_I8_BLOCK_BYTES)                       /* 17408 */

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARGUMENT = 1,   /* null pointer, negative size, bad stride  */
  PKV_ERR_MISALIGNED = 2,         /* a buffer is not 16-byte aligned          */
  PKV_ERR_UNSUPPORTED_SHAPE = 3,  /* size outside what the kernels support    */
  PKV_ERR_WORKSPACE_TOO_SMALL = 4,
  PKV_ERR_CUDA = 5,               /* CUDA runtime/launch error                 */
  PKV_ERR_DEVICE_INDEX = 6,       /* device word: bad page id / position / row */
  PKV_ERR_POOL_EXHAUSTED = 7,     /* scheduler: not enough free pages now      */
  PKV_ERR_REQUEST_TOO_LARGE = 8,  /* scheduler: credit exceeds the whole pool  */
  PKV_ERR_TIMEOUT = 9             /* device word: a bounded wait gave up       */
} pkv_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* pkv_status_string(int status);

/* Description of the last PKV_ERR_CUDA raised on the calling thread (the
 * failing CUDA call and its error string); "" if none.  Static per-thread
 * storage, valid until the next failing call on that thread. */
const char* pkv_last_error(void);

/* Library version as 10000*major + 100*minor + patch. */
int pkv_version(void);

/* ------------------------------------------------------------------------
 * RoPE tables (host-side set-up, run once, like the frequency table the
 * tiny-vllm engine builds at start-up: "2. Weight Loading and GPU Buffer
 * Design", section "What else is set up in the initialization block").
 * ---------------------------------------------------------------------- */

/* inv_freq[i] = theta^(-2i/64), i < 32.  inv_freq: host double[32] (out). */
int pkv_rope_inv_freq_plain(double* inv_freq, double theta);

/* Llama 3 frequency scaling of the plain table: components with wavelength
 * 2*pi/f below original_max_pos/high_freq_factor are kept, above
 * original_max_pos/low_freq_factor divided by `factor`, blended linearly in
 * between.  inv_freq: host double[32] (out). */
int pkv_rope_inv_freq_llama3(double* inv_freq, double theta, double factor,
                             double low_freq_factor, double high_freq_factor,
                             int original_max_pos);

/* host_cos/host_sin: host float[max_pos][32] (out);
 * cos[p][i] = (float)cos((double)p * inv_freq[i]), same for sin.
 * The caller copies the tables to the device for kv_append_rope. */
int pkv_rope_table_fill(float* host_cos, float* host_sin, int max_pos, const double* inv_freq);

/* ------------------------------------------------------------------------
 * kv_append_rope - write T new tokens' K/V into their pages.
 *
 * For token t of block-table row s = token_seq[t] (or t when token_seq is
 * NULL) at absolute position p = positions[t]: K of every KV head g is
 * rotated by RoPE at position p (pairs (i, i+32), fp32 operations in the
 * order r0 = x0*c - x1*s, r1 = x0*s + x1*c, each rounded to nearest, then
 * rounded to bf16 nearest-even) and written to slot p % 16 of page
 * block_tables[s * bt_row_stride + p / 16]; V is copied bit for bit.
 * If q_in is given, the 32 query heads of token t are rotated the same way
 * into q_out (q_out may equal q_in).  Tokens of one call must address
 * distinct (row, position) pairs.
 *
 *   k, v          device bf16 [T][8][64]
 *   positions     device int32 [T]
 *   token_seq     device int32 [T] or NULL
 *   block_tables  device int32 [num_seqs][bt_row_stride], first max_blocks
 *                 entries of each row used; -1 = no page
 *   kv_pool       device bf16 [num_pages][2 (K,V)][8][16][64], 32 KiB/page
 *   rope_cos/sin  device float [max_pos][32] (see pkv_rope_table_fill)
 *   q_in, q_out   device bf16 [T][32][64], or both NULL
 *   d_err         device int32, first device-detected error code (or NULL)
 * A token whose row, position or page id is out of range writes nothing,
 * gets a zero q_out row and sets *d_err = PKV_ERR_DEVICE_INDEX.
 * Returns PKV_OK or a host-side error (nothing is launched then).
 * ---------------------------------------------------------------------- */
int kv_append_rope(const void* k, const void* v, const int32_t* positions,
                   const int32_t* token_seq, int T,
                   const int32_t* block_tables, int num_seqs, int bt_row_stride, int max_blocks,
                   void* kv_pool, int num_pages,
                   const float* rope_cos, const float* rope_sin, int max_pos,
                   const void* q_in, void* q_out,
                   int* d_err, void* stream);

/* ------------------------------------------------------------------------
 * paged_gqa_decode - one decode step of grouped-query attention over
 * each sequence's own pages.
 *
 * For sequence s with n = seq_lens[s] tokens (positions [0, n), including
 * the token just appended) and query head h (KV head g = h / 4):
 *     x_j = scale * q[s][h] . K_j[g],   out[s][h] = sum_j softmax(x)_j V_j[g]
 * K_j/V_j are read from slot j % 16 of page block_tables[s][j / 16].
 * Loads are bf16, all arithmetic fp32 (exponentials in base 2), output
 * rounded to bf16 nearest-even.  Work is split into page ranges spread
 * evenly over the GPU (flash-decoding); the partial (o, m, l) triples of a
 * sequence split across warps go to the workspace and the last warp to
 * finish merges them with a log-sum-exp combine (one kernel launch).
 *
 *   q             device bf16 [num_seqs][32][64] (already rotated)
 *   kv_pool       device bf16 pool as in kv_append_rope, 16-byte aligned
 *   block_tables  device int32 [num_seqs][bt_row_stride]
 *   seq_lens      device int32 [num_seqs]
 *   max_seq_len   host upper bound of seq_lens (sizes the grid; a larger
 *                 actual length is still handled correctly; 0: none, then
 *                 16 max_blocks).  The bound also picks the L2 policy of the
 *                 page copies: when num_seqs x 8 heads x its pages reach
 *                 64 MiB of K/V, half of the L2, the pages are copied under
 *                 the evict-first policy; below that, the default policy
 *                 leaves them in L2 for the next read
 *   out           device bf16 [num_seqs][32][64]
 *   workspace     device memory of at least
 *                 paged_gqa_decode_workspace_bytes(num_seqs) bytes, 16-byte
 *                 aligned and zero-filled before its first use.  Each call
 *                 leaves it zero-filled again (per-segment arrival counters
 *                 are reset by the warp that merges the segment), so one
 *                 workspace serves any number of calls in stream order;
 *                 calls that may run at the same time need distinct
 *                 workspaces.  After a PKV_ERR_TIMEOUT, zero it again.
 * seq_len 0 gives a zero output.  A negative seq_len, seq_len above
 * 16 * max_blocks, or a needed page id outside [0, num_pages) gives a zero
 * output for that sequence and sets *d_err = PKV_ERR_DEVICE_INDEX.
 * ---------------------------------------------------------------------- */
size_t paged_gqa_decode_workspace_bytes(int num_seqs);

int paged_gqa_decode(const void* q, const void* kv_pool, int num_pages,
                     const int32_t* block_tables, int bt_row_stride, int max_blocks,
                     const int32_t* seq_lens, int num_seqs, int max_seq_len,
                     void* out, float scale,
                     void* workspace, size_t workspace_bytes,
                     int* d_err, void* stream);

/* Tuning / comparison knobs for paged_gqa_decode_ex (NULL = defaults). */
typedef enum pkv_compute {
  PKV_COMPUTE_TENSOR = 0, /* scores and P*V on the tensor cores (bf16 mma, fp32 accumulate) */
  PKV_COMPUTE_FMA = 1     /* same pipeline, fp32 FMA on the CUDA cores (comparison arm)     */
} pkv_compute;

typedef struct pkv_decode_opts {
  int compute;            /* pkv_compute                                             */
  int min_units_per_warp; /* 0 = default (2): fewer CTAs for small batches           */
  int ctas_per_sm;        /* 0 = as many as fit (at most 8)                          */
  int stages;             /* pages in flight per warp: 0 = default (2), 2 or 4       */
  int warps_per_cta;      /* 0 = default: 16, or 8 on bf16 pages when max_seq_len
                             bounds the problem to at most 128 (sequence, head,
                             page) units; else 16 (2 or 3 stages), 8 or 4      */
  int combine;            /* segments split across CTAs: 0 = the last CTA merges
                             them in the same kernel, 1 = a second kernel merges
                             them after the first (programmatic dependent launch) */
  int schedule;           /* 0 = static: each warp a fixed contiguous sub-range;
                             1 = dynamic: warps claim chunks of the CTA's range
                             from a shared counter (large first, single pages at
                             the end) and the CTA's shared segments go first.
                             Falls back to 0 when its page table does not fit in
                             shared memory (tensor path only);
                             2 = automatic: dynamic when the length bound gives
                             every SM at least PKV_DYNAMIC_MIN_UNITS units of
                             (sequence, KV head, page) -- long ranges, where
                             evening out the warps pays for the claims -- else
                             static.  Calls without options use 2.             */
  int early_kv;           /* 1 = the caller guarantees that block_tables, seq_lens
                             and the K/V pages this call reads are not written by
                             the kernel enqueued just before it on the stream:
                             the call then reads them, and stages its first pages,
                             while that kernel is still finishing (programmatic
                             dependent launch); q, the new token and all writes
                             still wait for it.  0 = everything waits (default). */
  long long wait_limit_ns; /* limit of every bounded wait inside the kernel (a page's
                             copy, a shared-memory turn): 0 = the default of 2 s;
                             when one runs out the kernel sets *d_err =
                             PKV_ERR_TIMEOUT, waits (2 s at most) for its own copies
                             still in flight and returns; the outputs are then
                             undefined and the workspace must be zeroed again      */
  int expire_first_wait;  /* test of that path: 1 = the first warp of the first CTA
                             waits on a barrier nothing completes instead of its
                             first page, so its wait runs out after wait_limit_ns
                             (no fault, no hang: the bounded-wait contract above) */
} pkv_decode_opts;

/* Work per SM from which the automatic schedule is the dynamic one (on
 * GB300 the dynamic schedule is 3-4 % faster from 96 sequences of 2048 tokens
 * on, 512 units per SM and more; at 32 sequences the static one is 13 %
 * faster). */
#define PKV_DYNAMIC_MIN_UNITS 512
#define PKV_SCHEDULE_STATIC 0
#define PKV_SCHEDULE_DYNAMIC 1
#define PKV_SCHEDULE_AUTO 2

/* paged_gqa_decode with explicit options; same contract otherwise. */
int paged_gqa_decode_ex(const void* q, const void* kv_pool, int num_pages,
                        const int32_t* block_tables, int bt_row_stride, int max_blocks,
                        const int32_t* seq_lens, int num_seqs, int max_seq_len,
                        void* out, float scale,
                        void* workspace, size_t workspace_bytes,
                        int* d_err, void* stream, const pkv_decode_opts* opts);

/* ------------------------------------------------------------------------
 * paged_gqa_decode_noalloc - paged_gqa_decode for callers that cannot
 * allocate device memory.  (No counterpart on the source pages: it exists
 * for integration, not for the method.)
 *
 * Some callers cannot call cudaMalloc at all: a plug-in inside a host
 * program that owns the whole device-memory budget, or a serving loop that
 * may not allocate after start-up.  This entry point takes the same inputs
 * and outputs as paged_gqa_decode but no workspace: it uses a fixed array of
 * PKV_NOALLOC_WORKSPACE_BYTES in the library's own device memory, which each
 * GPU that loads the library holds until the process exits.  It allocates
 * nothing and calls no allocating routine.
 *   - Limit: paged_gqa_decode_workspace_bytes(num_seqs) must fit in the
 *     array (on a 152-SM GB300: up to 343 sequences per call); larger
 *     batches return PKV_ERR_WORKSPACE_TOO_SMALL and pkv_last_error() says
 *     why.
 *   - Arguments are checked (as paged_gqa_decode checks them) before
 *     anything touches the device or the array.
 *   - Each call made outside stream capture looks up the array's device
 *     address (with the stream's device current), so a device reset does not
 *     leave a stale address behind.  A call made while `stream` is being
 *     captured reuses the address of the last uncaptured call on the current
 *     device: make the first call on each device before any capture (a first
 *     call under capture returns PKV_ERR_CUDA), and make the captured
 *     stream's device current.
 *   - Every call on a device shares the array: calls whose kernels may run
 *     at the same time on the GPU race with each other.  Each call clears the
 *     part that must start at zero (on `stream`) before its kernel runs.
 * ---------------------------------------------------------------------- */
#define PKV_NOALLOC_WORKSPACE_BYTES (4 * 1024 * 1024)

int paged_gqa_decode_noalloc(const void* q, const void* kv_pool, int num_pages,
                             const int32_t* block_tables, int bt_row_stride, int max_blocks,
                             const int32_t* seq_lens, int num_seqs, int max_seq_len,
                             void* out, float scale, int* d_err, void* stream);

/* ------------------------------------------------------------------------
 * paged_gqa_decode_append - one decode step with the KV append fused in.
 *
 * Same result as kv_append_rope(k_new, v_new, positions = seq_lens - 1,
 * token_seq = NULL, ..., q_in = q, q_out) followed by
 * paged_gqa_decode(q_out, ...), in one kernel: for every sequence s with
 * n = seq_lens[s] >= 1, the new token sits at position p = n - 1; its K is
 * rotated at p and written with its V into slot p % 16 of page
 * block_tables[s][p / 16] (bytes identical to kv_append_rope), q[s] is
 * rotated at p into q_out (if q_out is not NULL), and attention runs over
 * positions [0, n) with the rotated query.  The warp that owns the page of
 * the new token inserts it into its staged copy of that page, so no second
 * pass over memory is needed ("Gestion de la KV cache et strategies de
 * batching": each new token is written at its absolute RoPE position and
 * attention reads only the sequence's pages).
 *
 *   q             device bf16 [num_seqs][32][64], NOT rotated
 *   k_new, v_new  device bf16 [num_seqs][8][64]
 *   rope_cos/sin  device float [max_pos][32]
 *   kv_pool       device bf16 pool, written (the new token) and read
 *   q_out         device bf16 [num_seqs][32][64] or NULL
 * Other arguments as paged_gqa_decode.  seq_len 0 appends nothing and gives
 * zero outputs; seq_len above max_pos or 16 * max_blocks, or a bad page id,
 * gives zero outputs for that sequence and sets *d_err.  Tensor-core path
 * only (opts->compute must be PKV_COMPUTE_TENSOR); warps_per_cta 16, 8 or 4
 * with 2 stages.
 * ---------------------------------------------------------------------- */
int paged_gqa_decode_append(const void* q, const void* k_new, const void* v_new,
                            const float* rope_cos, const float* rope_sin, int max_pos,
                            void* kv_pool, int num_pages,
                            const int32_t* block_tables, int bt_row_stride, int max_blocks,
                            const int32_t* seq_lens, int num_seqs, int max_seq_len,
                            void* q_out, void* out, float scale,
                            void* workspace, size_t workspace_bytes,
                            int* d_err, void* stream, const pkv_decode_opts* opts);

/* ------------------------------------------------------------------------
 * INT8 K/V pages - the "INT8 K/V" storage mode of a request's KV cache
 * ("Lifecycle and Memory Model", TinyLoop C++ API, section "Per-request /
 * handle-owned memory", RuntimeKVCache).  The page names the mode only; the
 * scheme here is the library's reading of it for a cache written one token
 * at a time: every (token, KV head) row of K and of V -- 64 values -- is
 * quantised on its own, symmetrically, with one fp32 scale:
 *     amax = max_d |x_d|,  scale = amax / 127,
 *     code_d = round-half-even(x_d / scale) in [-127, 127]
 * (both divisions IEEE fp32; amax == 0 gives scale 0 and zero codes), where
 * x is the row the bf16 cache would hold (K rotated and rounded to bf16 as in
 * kv_append_rope, V as given).  A code stands for code * scale.  Rows must be
 * finite.  Pages keep the bf16 pool's block tables and 16 tokens; a page of
 * the INT8 pool is 8 blocks of PKV_I8_BLOCK_BYTES, one per KV head:
 *   kv_pool  device bytes [num_pages][8][2176], 17408 bytes/page, 16-byte
 *            aligned, caller-owned; one contiguous copy brings a unit.  The
 *            block of (page, head), in this library's format:
 *            - a code c is stored as the byte c + 128 (an all-0x80 block
 *              holds zero codes);
 *            - bytes 0..1023, K codes: slot t, dim d at 64 t + d;
 *            - bytes 1024..2047, V codes by slot pairs: slot t is member
 *              t % 2 of pair p = t / 2, and dim d of a pair is the byte
 *              pair at 1024 + 128 p + 16 ((d % 8) ^ (2 (p % 4)))
 *              + 2 (d / 8) + member;
 *            - bytes 2048..2175, float scales (little-endian) in groups of
 *              four: group j = 0..7 at 2048 + 16 j holds the K scales of
 *              slots j and j + 8, then their V scales.
 *            (So each shared-memory read of the decode is one
 *            conflict-free 16-byte load: two K rows, one scale group, and
 *            eight dims of a slot pair.)
 * ---------------------------------------------------------------------- */

/* kv_append_rope_layers: the same T tokens appended into each of num_layers
 * layers -- a newly admitted request's prompt, whose pages are written layer
 * by layer ("Gestion de la KV cache et strategies de batching", samir-vllm
 * article) -- in one host call: for layer l, kv_append_rope (int8 = 0; bf16
 * pool) or kv_append_rope_int8 (int8 = 1; INT8 pool) of k[l], v[l] with the
 * tables at block_tables + l * bt_layer_stride, no q rotation.
 *   k, v       arrays (host memory, num_layers entries) of pointers to
 *              [T][8][64] bf16 rows: device memory with src_host = 0; host
 *              memory with src_host = 1, copied first into `stage` by
 *              cudaMemcpyAsync on `stream` (pinned memory for an
 *              asynchronous copy; other host memory works, synchronously).
 *              The host rows must stay unchanged until those copies have run.
 *   stage      with src_host = 1: caller-owned device memory of at least
 *              2 * T * 1024 bytes, 16-byte aligned, reused by every layer in
 *              stream order; unused with src_host = 0.
 *   positions, token_seq, T, num_seqs, bt_row_stride, max_blocks, kv_pool,
 *   num_pages, rope_cos, rope_sin, max_pos, d_err, stream: as for
 *   kv_append_rope (every layer uses the same positions and token_seq).
 * Errors: the host checks of kv_append_rope for each layer, and
 * PKV_ERR_INVALID_ARGUMENT for a null array entry, num_layers < 0,
 * bt_layer_stride < num_seqs * bt_row_stride, or a missing or short stage;
 * a layer that fails returns at once, the layers before it stay enqueued. */
int kv_append_rope_layers(const void* const* k, const void* const* v, int num_layers, int src_host,
                          void* stage, size_t stage_bytes, const int32_t* positions,
                          const int32_t* token_seq, int T, const int32_t* block_tables,
                          long long bt_layer_stride, int num_seqs, int bt_row_stride,
                          int max_blocks, void* kv_pool, int num_pages, int int8,
                          const float* rope_cos, const float* rope_sin, int max_pos, int* d_err,
                          void* stream);

/* kv_append_rope into INT8 pages: the arguments, ordering and error rules of
 * kv_append_rope, with kv_pool the INT8 pool.  The rotated q (when q_in is
 * given) stays bf16.  k, v and kv_pool must be 16-byte aligned, q_in/q_out
 * 4-byte aligned. */
int kv_append_rope_int8(const void* k, const void* v, const int32_t* positions,
                        const int32_t* token_seq, int T,
                        const int32_t* block_tables, int num_seqs, int bt_row_stride,
                        int max_blocks, void* kv_pool, int num_pages,
                        const float* rope_cos, const float* rope_sin, int max_pos,
                        const void* q_in, void* q_out, int* d_err, void* stream);

/* paged_gqa_decode over INT8 pages: the same arguments, workspace
 * (paged_gqa_decode_workspace_bytes) and error rules, with kv_pool the INT8
 * pool.  Attention is over the dequantised values: scores
 * scale * q . (code_K * scale_K), weights applied to code_V * scale_V.
 * Codes enter fp16 tensor-core MMAs exactly (fp32 accumulation); q is scaled
 * by a power of two per (sequence, KV head) so that its largest |value| lies
 * in [2^14, 2^15) (exact), the K scale multiplies each fp32 score, and each
 * probability times its V scale, divided by a power of two that puts the
 * largest V scale of its two-page block in [1, 2), is rounded to fp16 for
 * the P V product.  Output bf16. */
int paged_gqa_decode_int8(const void* q, const void* kv_pool, int num_pages,
                          const int32_t* block_tables, int bt_row_stride, int max_blocks,
                          const int32_t* seq_lens, int num_seqs, int max_seq_len,
                          void* out, float scale,
                          void* workspace, size_t workspace_bytes,
                          int* d_err, void* stream);

/* paged_gqa_decode_int8 with tuning options: compute must be
 * PKV_COMPUTE_TENSOR, schedule and combine 0; (warps_per_cta, stages) one of
 * (16, 2) (the default: two pages per stage), (16, 4) or (8, 4) (one page
 * per stage); other fields as paged_gqa_decode_ex. */
int paged_gqa_decode_int8_ex(const void* q, const void* kv_pool, int num_pages,
                             const int32_t* block_tables, int bt_row_stride, int max_blocks,
                             const int32_t* seq_lens, int num_seqs, int max_seq_len,
                             void* out, float scale,
                             void* workspace, size_t workspace_bytes,
                             int* d_err, void* stream, const pkv_decode_opts* opts);

/* paged_gqa_decode_append on INT8 pages: for sequence s with n = seq_lens[s]
 * its new token (k_new[s], v_new[s]) is rotated and quantised exactly as
 * kv_append_rope_int8 does and written at position n - 1, q is rotated there
 * (into q_out when given), and attention covers [0, n) including the new
 * token -- one kernel.  Arguments, error rules and the early_kv option as
 * paged_gqa_decode_append, with kv_pool the INT8 pool; opts may be NULL, and
 * otherwise must select the default configuration (warps 0 or 16, stages 0
 * or 2, compute PKV_COMPUTE_TENSOR, schedule and combine 0). */
int paged_gqa_decode_append_int8(const void* q, const void* k_new, const void* v_new,
                                 const float* rope_cos, const float* rope_sin, int max_pos,
                                 void* kv_pool, int num_pages,
                                 const int32_t* block_tables, int bt_row_stride, int max_blocks,
                                 const int32_t* seq_lens, int num_seqs, int max_seq_len,
                                 void* q_out, void* out, float scale,
                                 void* workspace, size_t workspace_bytes,
                                 int* d_err, void* stream, const pkv_decode_opts* opts);

/* ------------------------------------------------------------------------
 * paged_gqa_decode_append_layers - one decode step of every layer in one
 * call: the batched decode of the samir-vllm article ("Gestion de la KV
 * cache et strategies de batching": each step appends every active
 * sequence's token at its absolute position and attends over its pages),
 * for all layers of the model in layer order.
 *
 * If host_stage is given, first one host->device copy of stage_bytes from
 * host_stage (pinned host memory, caller-owned; it must stay unchanged until
 * the copy has run on `stream`) to dev_stage (device) is enqueued: the block
 * tables and lengths of the step may live there (pkv_sched_pack_step).  Then
 * for l = 0 .. num_layers-1 exactly the call
 *   paged_gqa_decode_append(q + l Q, k_new + l K, v_new + l K, rope_cos,
 *       rope_sin, max_pos, kv_pool, num_pages,
 *       block_tables + l * bt_layer_stride, bt_row_stride, max_blocks,
 *       seq_lens, num_seqs, max_seq_len, q_out ? q_out + l Q : NULL,
 *       out + l Q, scale, workspace, workspace_bytes, d_err, stream, &opts)
 * (paged_gqa_decode_append_int8 when int8 = 1) with Q = num_seqs*32*64 and
 * K = num_seqs*8*64 bf16 elements and default options, except that with
 * early_kv = 1 the layers l >= 1 take opts.early_kv = 1: the layers' block
 * tables must then name disjoint pages, as the layers of a paged cache do.
 *   q, out, q_out   device bf16 [num_layers][num_seqs][32][64] (q_out or NULL)
 *   k_new, v_new    device bf16 [num_layers][num_seqs][8][64]
 *   block_tables    device int32, layer l at + l * bt_layer_stride elements
 *                   (bt_layer_stride >= num_seqs * bt_row_stride)
 * Returns the first non-zero status of a layer's call (later layers are then
 * not launched) or of the copy; PKV_OK otherwise.
 * ---------------------------------------------------------------------- */
int paged_gqa_decode_append_layers(const void* q, const void* k_new, const void* v_new,
                                   void* q_out, void* out, int num_layers, int num_seqs,
                                   const float* rope_cos, const float* rope_sin, int max_pos,
                                   void* kv_pool, int num_pages, int int8,
                                   const int32_t* block_tables, long long bt_layer_stride,
                                   int bt_row_stride, int max_blocks, const int32_t* seq_lens,
                                   int max_seq_len, float scale, void* workspace,
                                   size_t workspace_bytes, int* d_err, void* stream,
                                   int early_kv, const void* host_stage, void* dev_stage,
                                   size_t stage_bytes);

/* ------------------------------------------------------------------------
 * paged_gqa_prefill - causal GQA attention of each sequence's newest tokens
 * over its own pages: a whole prompt, or a chunk of one after a cached
 * prefix ("Gestion de la KV cache et strategies de batching": attention
 * reads only the sequence's pages; a token at position p sees positions
 * up to its own).
 *
 * Sequence s holds n = seq_lens[s] tokens in its pages (already written,
 * e.g. by kv_append_rope earlier on the stream); its queries are the last
 * q_len = cu_q[s+1] - cu_q[s] of them, at positions n - q_len .. n - 1, and
 * are rows cu_q[s] .. cu_q[s+1] - 1 of q and out:
 *   out[t][h] = sum_{j <= p_t} softmax_j(scale * q[t][h] . K_j[h/4]) V_j[h/4].
 *
 *   q           device bf16 [num_tokens][32][64], rotated
 *   cu_q        device int32 [num_seqs + 1], row offsets (cu_q[0] = 0)
 *   kv_pool     device bf16 pool (read only), num_pages pages
 *   block_tables, bt_row_stride, max_blocks, seq_lens: as paged_gqa_decode
 *   max_q_len   host upper bound of every q_len (sizes the grid)
 *   out         device bf16 [num_tokens][32][64]
 *   scale       positive and finite (the kernel takes the row max of the
 *               unscaled scores), else PKV_ERR_INVALID_ARGUMENT
 * tcgen05 MMAs (bf16 operands, fp32 accumulation in tensor memory) and an
 * online softmax, one CTA per (32 query tokens, KV head, sequence);
 * deterministic.  A sequence whose
 * rows fall outside [0, num_tokens) or whose q_len is negative is left
 * untouched; one with q_len > n, q_len > max_q_len, n above
 * 16 * max_blocks or a needed page id outside [0, num_pages) gets zero
 * rows; both set *d_err = PKV_ERR_DEVICE_INDEX.  No workspace.
 * ---------------------------------------------------------------------- */
int paged_gqa_prefill(const void* q, int num_tokens, const int32_t* cu_q,
                      const void* kv_pool, int num_pages,
                      const int32_t* block_tables, int bt_row_stride, int max_blocks,
                      const int32_t* seq_lens, int num_seqs, int max_q_len,
                      void* out, float scale, int* d_err, void* stream);

/* paged_gqa_prefill with the compute path chosen: PKV_COMPUTE_TENSOR (the
 * default: tcgen05 MMAs with S and O in tensor memory, 64-key blocks) or
 * PKV_PREFILL_MMA_SYNC (bf16 mma.sync with register accumulators, the
 * comparison arm).  Same contract and results within the same tolerance. */
#define PKV_PREFILL_MMA_SYNC 2
int paged_gqa_prefill_ex(const void* q, int num_tokens, const int32_t* cu_q,
                         const void* kv_pool, int num_pages,
                         const int32_t* block_tables, int bt_row_stride, int max_blocks,
                         const int32_t* seq_lens, int num_seqs, int max_q_len,
                         void* out, float scale, int* d_err, void* stream, int compute);

/* ------------------------------------------------------------------------
 * pkv_argmax_f32 - next-token selection ("Architecture et flux
 * d'inference": the final logits are FP32 and a GPU argmax selects the next
 * token).  out_ids[r] = the first index of the largest non-NaN value of row
 * r (NaN orders below every number, -inf included); 0 when every value of
 * the row is NaN.
 *   logits      device float [rows][row_stride], vocab <= row_stride used
 *   out_ids     device int32 [rows]
 * One CTA per row; deterministic.  Host-side checks only (no device error).
 * ---------------------------------------------------------------------- */
int pkv_argmax_f32(const float* logits, int rows, int vocab, long long row_stride,
                   int32_t* out_ids, void* stream);

/* Wait for `stream`, then copy the device error word to *code_out (host).
 * If `clear` is non-zero the word is reset to 0 afterwards. */
int pkv_read_device_error(int* d_err, void* stream, int clear, int* code_out);

/* ------------------------------------------------------------------------
 * Continuous-batching scheduler (host only): FIFO admission by credit and
 * on-demand page allocation.  From the samir-vllm article, section
 * "Gestion de la KV cache et strategies de batching": a request is admitted
 * once its page budget is available; credit = prompt_tokens +
 * allowed_new_tokens - 1 tokens rounded up to 16-token pages, per layer; a
 * request whose budget exceeds the pool is rejected with an explicit error.
 * Rules the article leaves open: strict FIFO (the head blocks the queue);
 * a request fits when credit <= free pages - pages still reserved by running
 * requests; pages come from a LIFO free stack that starts [N-1 ... 0] (page
 * 0 first); a finished request pushes back its pages layer by layer in
 * logical order; a new request takes the lowest free slot (block-table row).
 * ---------------------------------------------------------------------- */
typedef struct pkv_sched pkv_sched;

/* Pages reserved for a request: num_layers * ceil((prompt + new - 1) / 16). */
int pkv_credit_pages(int prompt_tokens, int allowed_new_tokens, int num_layers);

/* NULL on invalid sizes or allocation failure (fail closed, as load_model
 * does in "Lifecycle and Memory Model", section "Internal allocation
 * phases"). */
pkv_sched* pkv_sched_create(int num_pages, int num_layers, int max_blocks, int max_slots);
void pkv_sched_destroy(pkv_sched* s);

/* Batching mode ("Gestion de la KV cache et strategies de batching": two
 * modes): 0 = continuous (default), admit whenever the head of the queue
 * fits; 1 = static, admit only when no request is running, i.e. wait for
 * the current group to finish, then admit the FIFO prefix that fits. */
int pkv_sched_set_mode(pkv_sched* s, int mode);

/* Queue a request; *req_id (host, out) gets its id.  Returns
 * PKV_ERR_REQUEST_TOO_LARGE (not queued) if its credit exceeds the pool or
 * its length exceeds max_blocks pages. */
int pkv_sched_submit(pkv_sched* s, int prompt_tokens, int allowed_new_tokens, int* req_id);

/* Admit queued requests in FIFO order while the head fits.  Writes up to
 * max_out admitted ids to admitted (host) and their count to *n_admitted. */
int pkv_sched_admit(pkv_sched* s, int* admitted, int max_out, int* n_admitted);

/* Make every layer of a running request hold pages for positions
 * [0, new_len).  PKV_ERR_POOL_EXHAUSTED if that would exceed its credit. */
int pkv_sched_grow(pkv_sched* s, int req_id, int new_len);

/* Release a running request's pages and slot. */
int pkv_sched_finish(pkv_sched* s, int req_id);

/* Host side of one decode step of the continuous batch: every running
 * request, in admission order (= id order), grows by one token as
 * pkv_sched_grow(id, length + 1) would, where length is the largest length
 * it was grown to.  ids (host int32[max_out], out) gets the batch's request
 * ids in that order, lens (host int32[max_out], out) their lengths after the
 * step, *batch their count.  All or nothing: if any request cannot take its
 * token (PKV_ERR_POOL_EXHAUSTED) nothing changes; PKV_ERR_INVALID_ARGUMENT
 * if more than max_out requests run. */
int pkv_sched_begin_step(pkv_sched* s, int32_t* ids, int32_t* lens, int max_out, int* batch);

/* Bytes of a step block for `batch` rows of lengths at most max_len: the
 * lengths [batch] int32, then at the next 16-byte boundary the block tables
 * [num_layers][batch][P] int32 with P = max(1, ceil(max_len / 16)). */
size_t pkv_sched_step_bytes(const pkv_sched* s, int batch, int max_len);

/* Write the step block of requests ids[0 .. batch) (running, lengths at most
 * max_len) into `block` (host memory of at least pkv_sched_step_bytes
 * bytes): their current lengths and, per layer, their page ids padded with
 * -1.  Layer l's tables then start at element offset l * batch * P of the
 * tables part, rows of P entries: the block_tables / seq_lens arguments of
 * paged_gqa_decode_append_layers once the block is on the device. */
int pkv_sched_pack_step(const pkv_sched* s, const int32_t* ids, int batch, int max_len,
                        void* block, size_t bytes);

/* Copy one request's block table for `layer` (host int32[max_blocks], -1
 * padded) and report its slot (may be NULL). */
int pkv_sched_block_table(const pkv_sched* s, int req_id, int layer, int32_t* row, int* slot);

/* Counters: free pages, pages still reserved by running requests, queued
 * requests, running requests (any may be NULL). */
int pkv_sched_stats(const pkv_sched* s, int* free_pages, int* reserved_pages,
                    int* queued, int* running);

/* Allocation log: number of page grants so far, and grant i as
 * (request, layer, logical page, page id). */
int pkv_sched_event_count(const pkv_sched* s);
int pkv_sched_event(const pkv_sched* s, int i, int* req_id, int* layer, int* logical, int* page);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
