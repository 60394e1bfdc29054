"""Paged KV append and paged GQA decode attention (oracle; test infrastructure only).

What the path computes, from the samir-vllm article ("Gestion de la KV cache et
strategies de batching"):
  * the KV cache is a shared pool of physical pages of 16 tokens holding K and
    V; each sequence has one block table per layer listing its pages;
  * during decode every new token's K/V is written at its absolute RoPE
    position;
  * paged attention reads only the current sequence's pages and accumulates the
    weighted V, without building a contiguous prefix or storing the scores.
and from "Architecture et flux d'inference" of the same article: grouped-query
attention, BF16 tensors with FP32 reductions.  The model constants (32 query
heads, KV_DIM 512 -> 8 KV heads of 64) are from "2. Weight Loading and GPU
Buffer Design", section "Preallocating the 16 compute buffers"; the block table
starts out all -1 (section "What else is set up in the initialization block").

Readings taken where the pages are silent (the CUDA library follows the same
contract):
  * page layout pool[page][K=0,V=1][kv_head][slot][dim], 32 KiB per page;
  * query head h reads KV head h // 4;
  * seq_len counts the just-appended token: attend to positions [0, seq_len);
  * seq_len == 0 gives a zero output; a negative seq_len, one above
    16 * max_blocks, or a page id outside [0, num_pages) for a needed page,
    gives a zero output for that sequence and raises the error flag;
  * an append token with a bad sequence, position or page id writes nothing,
    zeroes its rotated-q row (when q is rotated) and raises the error flag.

The oracle may gather a sequence's pages into a contiguous array: the
"no contiguous prefix" constraint describes the GPU kernel, not the result.
"""
from __future__ import annotations

import math

import numpy as np

from . import bf16, rope

NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
GROUP = NUM_Q_HEADS // NUM_KV_HEADS
HEAD_DIM = 64
PAGE_TOKENS = 16


def new_pool(num_pages: int, fill_bits: int = 0) -> np.ndarray:
    """A pool of bf16 bit patterns [num_pages][2][8][16][64]."""
    return np.full((num_pages, 2, NUM_KV_HEADS, PAGE_TOKENS, HEAD_DIM), fill_bits, dtype=np.uint16)


def locate(block_table_row, pos: int, num_pages: int, max_blocks: int):
    """(page, slot) holding absolute position `pos`, or None when invalid."""
    if pos < 0 or pos // PAGE_TOKENS >= max_blocks:
        return None
    page = int(block_table_row[pos // PAGE_TOKENS])
    if page < 0 or page >= num_pages:
        return None
    return page, pos % PAGE_TOKENS


def append_rope(pool, k_bits, v_bits, positions, token_seq, block_tables, cos, sin,
                q_bits=None, inplace=False):
    """Write T new tokens into the pool.  Returns (pool', q_rot or None, error_flag).

    pool:          uint16 [N][2][8][16][64] (a copy is returned, or the pool
                   itself is written when inplace=True)
    k_bits/v_bits: uint16 [T][8][64]
    positions:     [T] absolute positions; token_seq: [T] rows of block_tables
                   (None: token t belongs to row t)
    block_tables:  [S][max_blocks] page ids for this layer
    cos/sin:       fp32 [max_pos][32]
    q_bits:        optional uint16 [T][32][64], rotated at the same positions
    Tokens are applied in order, so a later duplicate (same row and position)
    would overwrite an earlier one.
    """
    out = pool if inplace else np.array(pool, copy=True)
    num_pages = out.shape[0]
    S, max_blocks = block_tables.shape
    max_pos = cos.shape[0]
    T = k_bits.shape[0]
    q_rot = None if q_bits is None else np.zeros_like(q_bits)
    err = False
    for t in range(T):
        s = t if token_seq is None else int(token_seq[t])
        p = int(positions[t])
        if s < 0 or s >= S or p < 0 or p >= max_pos:
            err = True
            continue
        where = locate(block_tables[s], p, num_pages, max_blocks)
        if where is None:
            err = True
            continue
        page, slot = where
        out[page, 0, :, slot, :] = rope.rotate_bf16(k_bits[t], cos[p], sin[p])   # all 8 heads
        out[page, 1, :, slot, :] = v_bits[t]
        if q_bits is not None:
            for h in range(NUM_Q_HEADS):
                q_rot[t, h] = rope.rotate_bf16(q_bits[t, h], cos[p], sin[p])
    return out, q_rot, err


def gather(pool, block_table_row, n: int):
    """K, V of positions [0, n) as float64 [n][8][64]; None if a page id is bad."""
    num_pages = pool.shape[0]
    K = np.empty((n, NUM_KV_HEADS, HEAD_DIM))
    V = np.empty((n, NUM_KV_HEADS, HEAD_DIM))
    for j in range((n + PAGE_TOKENS - 1) // PAGE_TOKENS):
        page = int(block_table_row[j])
        if page < 0 or page >= num_pages:
            return None
        lo, hi = j * PAGE_TOKENS, min(n, (j + 1) * PAGE_TOKENS)
        # pool[page][kv][head][slot][dim] -> [slot][head][dim]
        K[lo:hi] = bf16.to_f64(pool[page, 0, :, :hi - lo, :]).transpose(1, 0, 2)
        V[lo:hi] = bf16.to_f64(pool[page, 1, :, :hi - lo, :]).transpose(1, 0, 2)
    return K, V


def attend(qh, K, V, scale: float):
    """softmax(scale * K qh) weighted sum of V, all FP64 (one head, one sequence)."""
    x = scale * (K @ qh)
    w = np.exp(x - x.max())
    return (w @ V) / w.sum()


def decode(q_bits, pool, block_tables, seq_lens, scale: float):
    """Decode-step GQA attention over each sequence's own pages.

    q_bits: uint16 [S][32][64]; block_tables: [S][max_blocks]; seq_lens: [S].
    Returns (out float64 [S][32][64], error_flag).
    """
    S = q_bits.shape[0]
    max_blocks = block_tables.shape[1]
    out = np.zeros((S, NUM_Q_HEADS, HEAD_DIM))
    err = False
    q = bf16.to_f64(q_bits)
    for s in range(S):
        n = int(seq_lens[s])
        if n < 0 or n > PAGE_TOKENS * max_blocks:
            err = True
            continue
        if n == 0:
            continue
        kv = gather(pool, block_tables[s], n)
        if kv is None:
            err = True
            continue
        K, V = kv
        for h in range(NUM_Q_HEADS):
            g = h // GROUP
            out[s, h] = attend(q[s, h], K[:, g, :], V[:, g, :], scale)
    return out, err


def prefill(q_bits, cu_q, pool, block_tables, seq_lens, scale: float):
    """Causal GQA attention of each sequence's newest tokens over its own pages.

    From the samir-vllm article ("Gestion de la KV cache et strategies de
    batching"): attention reads only the sequence's pages; a token at
    absolute position p sees the positions up to its own.  Sequence s holds
    n = seq_lens[s] tokens in its pages; its queries are the last
    q_len = cu_q[s+1] - cu_q[s] of them, at positions n - q_len .. n - 1,
    rows cu_q[s] .. cu_q[s+1] - 1 of q (a whole prompt is q_len == n; a chunk
    after a cached prefix has q_len < n).

    q_bits: uint16 [T][32][64] (rotated); cu_q: [S + 1]; block_tables:
    [S][max_blocks]; seq_lens: [S].  Returns (out float64 [T][32][64],
    error_flag).  The rows of a sequence with q_len < 0 or q_len > n, an n
    outside [0, 16 * max_blocks] or a bad needed page id stay zero and raise
    the flag.
    """
    T = q_bits.shape[0]
    S = len(seq_lens)
    max_blocks = block_tables.shape[1]
    out = np.zeros((T, NUM_Q_HEADS, HEAD_DIM))
    err = False
    q = bf16.to_f64(q_bits)
    for s in range(S):
        n = int(seq_lens[s])
        r0, r1 = int(cu_q[s]), int(cu_q[s + 1])
        q_len = r1 - r0
        if q_len < 0 or q_len > n or n > PAGE_TOKENS * max_blocks:
            err = True
            continue
        if q_len == 0:
            continue
        kv = gather(pool, block_tables[s], n)
        if kv is None:
            err = True
            continue
        K, V = kv
        for i in range(q_len):
            p = n - q_len + i
            for h in range(NUM_Q_HEADS):
                g = h // GROUP
                out[r0 + i, h] = attend(q[r0 + i, h], K[:p + 1, g, :], V[:p + 1, g, :], scale)
    return out, err


def decode_step(pool, q_bits, k_bits, v_bits, block_tables, seq_lens, cos, sin, scale: float):
    """One decode step: append each sequence's new token, then attend.

    For sequence s with n = seq_lens[s]:
      * n == 0: nothing is appended; output and rotated query are zero;
      * n < 0, or n beyond the RoPE table or 16 * max_blocks: the same, and
        the error flag is raised;
      * otherwise q_bits[s] is rotated at position n - 1 (returned in q_rot);
        the new token (k_bits[s], v_bits[s]) is appended at n - 1 through
        append_rope, which raises the flag and writes nothing if the page for
        n - 1 is outside the pool; attention over [0, n) uses the rotated
        query, and a needed page outside the pool gives a zero output and
        raises the flag (decode's rule).
    Returns (pool', q_rot [S][32][64] bits, out float64 [S][32][64], err).
    """
    S = q_bits.shape[0]
    lens = np.asarray(seq_lens)
    max_len = min(cos.shape[0], PAGE_TOKENS * block_tables.shape[1])
    q_rot = np.zeros_like(q_bits)
    out = np.zeros((S, NUM_Q_HEADS, HEAD_DIM))
    err = False
    valid = []
    for s in range(S):
        n = int(lens[s])
        if n == 0:
            continue
        if n < 0 or n > max_len:
            err = True
            continue
        valid.append(s)
        for h in range(NUM_Q_HEADS):
            q_rot[s, h] = rope.rotate_bf16(q_bits[s, h], cos[n - 1], sin[n - 1])
        pool, _, e = append_rope(pool, k_bits[s:s + 1], v_bits[s:s + 1], [n - 1], [s],
                                 block_tables, cos, sin)
        err |= e
    for s in valid:
        o, e = decode(q_rot[s:s + 1], pool, block_tables[s:s + 1], [int(lens[s])], scale)
        err |= e
        out[s] = o[0]
    return pool, q_rot, out, err


def decode_one(q_bits_sh, pool, block_table_row, n: int, scale: float, h: int):
    """One (sequence, query head) output, for sampled checks at full size."""
    kv = gather(pool, block_table_row, n)
    if kv is None:
        raise ValueError("bad page id")
    K, V = kv
    g = h // GROUP
    return attend(bf16.to_f64(q_bits_sh), K[:, g, :], V[:, g, :], scale)


# ---------------------------------------------------------------------------
# Split form: the same result reached by independent partial softmaxes over
# disjoint token ranges and a log-sum-exp combine.
# ---------------------------------------------------------------------------

def partial(qh, K, V, scale: float, lo: int, hi: int):
    """Unnormalised partial (o, m, l) over tokens [lo, hi); empty -> m = -inf."""
    if hi <= lo:
        return np.zeros(V.shape[-1]), -math.inf, 0.0
    x = scale * (K[lo:hi] @ qh)
    m = float(x.max())
    p = np.exp(x - m)
    return p @ V[lo:hi], m, float(p.sum())


def combine(parts):
    """o = sum_r e^{m_r - M} o_r / sum_r e^{m_r - M} l_r with M = max_r m_r."""
    live = [(o, m, l) for (o, m, l) in parts if m != -math.inf]
    if not live:
        return np.zeros_like(parts[0][0])
    M = max(m for _, m, _ in live)
    num = sum(math.exp(m - M) * o for o, m, _ in live)
    den = sum(math.exp(m - M) * l for _, m, l in live)
    return num / den


def attend_split(qh, K, V, scale: float, bounds):
    """attend() through partials over [b_0, b_1), [b_1, b_2), ... and combine()."""
    parts = [partial(qh, K, V, scale, lo, hi) for lo, hi in zip(bounds[:-1], bounds[1:])]
    return combine(parts)
