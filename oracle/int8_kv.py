"""INT8 K/V pages: quantised paged append and paged GQA decode over them.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``).

Source: "Lifecycle and Memory Model" (TinyLoop C++ API), section
"Per-request / handle-owned memory": a request's RuntimeKVCache keeps its
layers as FP16 K/V or as INT8 K/V, among other storage modes.  The page does
not say how the 8-bit values are formed.  Reading taken here (the plainest
one for a cache that grows one token at a time, where a row, once written,
never changes):

  * every (token, KV head) row of K and every such row of V -- 64 values --
    is quantised on its own, symmetrically, with one fp32 scale:
        amax    = max_d |x_d|
        scale   = fp32(amax / 127)
        code_d  = round-half-even(fp32(x_d / scale)), kept in [-127, 127]
    and a row with amax == 0 gets scale 0 and codes 0;
  * x is the row the bf16 cache would hold: K rotated at its position and
    rounded to bf16 exactly as ``paged_kv.append_rope`` does, V as given;
  * the value a code stands for is code * scale (exact in FP64);
  * decode is the bf16 definition (``paged_kv.attend``) applied to those
    values: nothing else about attention changes.

Logical arrays (the page geometry of the bf16 pool, one byte per element):
  codes   int8    [num_pages][2 (K, V)][8 heads][16 slots][64 dims]
  scales  float32 [num_pages][2 (K, V)][8 heads][16 slots]
The pool the library reads and writes holds them as bytes, one 2176-byte
block per (page, head), so a page is 8 x 2176 = 17408 bytes (``pack_pages``
/ ``unpack_pages``).  This byte format is the library's own (the page says
nothing of storage); it is defined here by ``block_positions``:
  * a code is stored as the byte code + 128 (1 .. 255 for codes in
    [-127, 127]);
  * K codes, bytes 0 .. 1023: slot t, dim d at 64 t + d;
  * V codes, bytes 1024 .. 2047, by slot pairs: slot t is member t % 2 of
    pair p = t // 2, and dim d of a pair is the byte pair at
        1024 + 128 p + 16 ((d % 8) ^ (2 (p % 4))) + 2 (d // 8) + member;
  * scales, bytes 2048 .. 2175, little-endian fp32 in groups of four:
    group j = 0..7 at 2048 + 16 j holds the K scales of slots j and j + 8,
    then their V scales.

fp32 emulation: each division is done in FP64 and rounded once to fp32.  For
+, -, *, / a binary64 intermediate followed by rounding to binary32 gives the
correctly rounded binary32 result (53 >= 2*24 + 2; Figueroa, "When is double
rounding innocuous?", 1995), so these are the IEEE fp32 divisions.

Parity status: pinned by ``tests/test_oracle_int8.py`` (integer rows,
power-of-two scaling, the half-step error bound, ties, brute-force nearest
code, a sentinel scan of the append, and the decode against a float64
library attention over the dequantised pages).
"""
from __future__ import annotations

import numpy as np

from . import bf16, rope
from .paged_kv import GROUP, HEAD_DIM, NUM_KV_HEADS, NUM_Q_HEADS, PAGE_TOKENS, attend, locate

QMAX = 127
BLOCK_BYTES = 2 * PAGE_TOKENS * HEAD_DIM + 2 * PAGE_TOKENS * 4   # 2176 per (page, head)


def quantize_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Symmetric 8-bit codes and fp32 scales of rows of 64 values (last axis).

    x: values exactly representable in fp32 (here: bf16 values), [..., 64].
    Returns (codes int8 [..., 64], scales float32 [...]).  Each row is
    quantised on its own, by the steps of the module docstring.
    """
    x = np.asarray(x, dtype=np.float64)
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / QMAX).astype(np.float32)                       # fp32(amax / 127)
    zero = scale == 0                                              # amax == 0 (see below)
    den = np.where(zero, 1.0, scale.astype(np.float64))[..., None]
    q = (x / den).astype(np.float32)                               # fp32(x_d / scale)
    codes = np.clip(np.rint(q), -QMAX, QMAX)                       # ties to even
    codes = np.where(zero[..., None], 0.0, codes)
    return codes.astype(np.int8), scale


def quantize_row(x) -> tuple[np.ndarray, np.float32]:
    """``quantize_rows`` of a single row: (codes int8 [64], scale float32)."""
    codes, scale = quantize_rows(np.asarray(x, dtype=np.float64)[None, :])
    return codes[0], np.float32(scale[0])


def dequantize(codes, scales) -> np.ndarray:
    """code * scale in FP64; scales broadcast over the last (dim) axis."""
    return np.asarray(codes, np.float64) * np.asarray(scales, np.float64)[..., None]


def new_pools(num_pages: int, code_fill: int = 0, scale_fill: float = 0.0):
    """(codes int8 [N][2][8][16][64], scales float32 [N][2][8][16])."""
    codes = np.full((num_pages, 2, NUM_KV_HEADS, PAGE_TOKENS, HEAD_DIM), code_fill, dtype=np.int8)
    scales = np.full((num_pages, 2, NUM_KV_HEADS, PAGE_TOKENS), scale_fill, dtype=np.float32)
    return codes, scales


def append_rope_int8(codes, scales, k_bits, v_bits, positions, token_seq, block_tables, cos, sin,
                     q_bits=None, inplace=False):
    """Write T new tokens into the INT8 pools.  Returns (codes', scales', q_rot or None, err).

    Arguments as ``paged_kv.append_rope``; the pools are those of
    ``new_pools``.  The K row of each head is rotated and rounded to bf16 as
    in the bf16 cache, then quantised; the V row is quantised from its bf16
    values.  q (when given) is rotated as in the bf16 append and not
    quantised.  A token with a bad row, position or page id writes nothing,
    gets a zero q row and raises the flag.
    """
    c_out = codes if inplace else np.array(codes, copy=True)
    s_out = scales if inplace else np.array(scales, copy=True)
    num_pages = c_out.shape[0]
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
        k_rot = rope.rotate_bf16(k_bits[t], cos[p], sin[p])          # [8][64] bf16 bits
        for g in range(NUM_KV_HEADS):
            c_out[page, 0, g, slot], s_out[page, 0, g, slot] = quantize_row(bf16.to_f64(k_rot[g]))
            c_out[page, 1, g, slot], s_out[page, 1, g, slot] = quantize_row(bf16.to_f64(v_bits[t, g]))
        if q_bits is not None:
            for h in range(NUM_Q_HEADS):
                q_rot[t, h] = rope.rotate_bf16(q_bits[t, h], cos[p], sin[p])
    return c_out, s_out, q_rot, err


def gather_int8(codes, scales, block_table_row, n: int):
    """Dequantised K, V of positions [0, n) as float64 [n][8][64]; None on a bad page id."""
    num_pages = codes.shape[0]
    K = np.empty((n, NUM_KV_HEADS, HEAD_DIM))
    V = np.empty((n, NUM_KV_HEADS, HEAD_DIM))
    for j in range((n + PAGE_TOKENS - 1) // PAGE_TOKENS):
        page = int(block_table_row[j])
        if page < 0 or page >= num_pages:
            return None
        lo, hi = j * PAGE_TOKENS, min(n, (j + 1) * PAGE_TOKENS)
        k = dequantize(codes[page, 0, :, :hi - lo, :], scales[page, 0, :, :hi - lo])   # [8][slot][64]
        v = dequantize(codes[page, 1, :, :hi - lo, :], scales[page, 1, :, :hi - lo])
        K[lo:hi] = k.transpose(1, 0, 2)
        V[lo:hi] = v.transpose(1, 0, 2)
    return K, V


def decode_int8(q_bits, codes, scales, block_tables, seq_lens, scale: float):
    """Decode-step GQA attention over INT8 pages; the rules of ``paged_kv.decode``.

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
        kv = gather_int8(codes, scales, block_tables[s], n)
        if kv is None:
            err = True
            continue
        K, V = kv
        for h in range(NUM_Q_HEADS):
            g = h // GROUP
            out[s, h] = attend(q[s, h], K[:, g, :], V[:, g, :], scale)
    return out, err


def decode_one_int8(q_bits_sh, codes, scales, block_table_row, n: int, scale: float, h: int):
    """One (sequence, query head) output, for sampled checks at full size."""
    kv = gather_int8(codes, scales, block_table_row, n)
    if kv is None:
        raise ValueError("bad page id")
    K, V = kv
    g = h // GROUP
    return attend(bf16.to_f64(q_bits_sh), K[:, g, :], V[:, g, :], scale)


def quantize_pool(pool_bits):
    """INT8 pools holding what ``append_rope_int8`` would store for every row of
    a bf16 pool (pool bits [N][2][8][16][64]); for building test inputs."""
    return quantize_rows(bf16.to_f64(pool_bits))


def block_positions():
    """Byte positions inside a (page, head) block, from the rules of the module
    docstring: (k [16][64], v [16][64], k_scale [16], v_scale [16]) -- the
    byte of each code, and the first byte of each fp32 scale."""
    k = np.empty((PAGE_TOKENS, HEAD_DIM), np.int64)
    v = np.empty((PAGE_TOKENS, HEAD_DIM), np.int64)
    ks = np.empty(PAGE_TOKENS, np.int64)
    vs = np.empty(PAGE_TOKENS, np.int64)
    for t in range(PAGE_TOKENS):
        pair, member = t // 2, t % 2
        ks[t] = 2048 + 16 * (t % 8) + 4 * (t // 8)
        vs[t] = ks[t] + 8
        for d in range(HEAD_DIM):
            k[t, d] = 64 * t + d
            v[t, d] = 1024 + 128 * pair + 16 * ((d % 8) ^ (2 * (pair % 4))) + 2 * (d // 8) + member
    return k, v, ks, vs


def pack_pages(codes, scales) -> np.ndarray:
    """Logical (codes, scales) -> the pool's bytes, uint8 [N][8][2176], in the
    block format of the module docstring."""
    codes = np.asarray(codes, np.int8)
    scales = np.asarray(scales, np.float32)
    N = codes.shape[0]
    kpos, vpos, kspos, vspos = block_positions()
    out = np.zeros((N, NUM_KV_HEADS, BLOCK_BYTES), np.uint8)
    biased = (codes.astype(np.int16) + 128).astype(np.uint8)       # code + 128
    out[:, :, kpos] = biased[:, 0]
    out[:, :, vpos] = biased[:, 1]
    for kv, pos in ((0, kspos), (1, vspos)):
        sb = np.ascontiguousarray(scales[:, kv].astype('<f4')).view(np.uint8).reshape(
            N, NUM_KV_HEADS, PAGE_TOKENS, 4)
        for j in range(4):
            out[:, :, pos + j] = sb[..., j]
    return out


def unpack_pages(pool_bytes):
    """The pool's bytes uint8 [N][8][2176] -> logical (codes, scales)."""
    b = np.ascontiguousarray(np.asarray(pool_bytes, np.uint8))
    N = b.shape[0]
    kpos, vpos, kspos, vspos = block_positions()
    codes = np.empty((N, 2, NUM_KV_HEADS, PAGE_TOKENS, HEAD_DIM), np.int8)
    scales = np.empty((N, 2, NUM_KV_HEADS, PAGE_TOKENS), np.float32)
    codes[:, 0] = (b[:, :, kpos].astype(np.int16) - 128).astype(np.int8)
    codes[:, 1] = (b[:, :, vpos].astype(np.int16) - 128).astype(np.int8)
    for kv, pos in ((0, kspos), (1, vspos)):
        sb = np.stack([b[:, :, pos + j] for j in range(4)], axis=-1)  # [N][8][16][4]
        scales[:, kv] = np.ascontiguousarray(sb).view('<f4')[..., 0]
    return codes, scales


def decode_step_int8(codes, scales, q_bits, k_bits, v_bits, block_tables, seq_lens, cos, sin,
                     scale: float):
    """One decode step on INT8 pages: append each sequence's new token, then attend.

    The rules of ``paged_kv.decode_step`` with the INT8 append and decode: for
    sequence s with n = seq_lens[s], n == 0 does nothing (zero output and
    rotated query); n < 0 or n beyond the RoPE table or 16 * max_blocks
    raises the flag and does nothing; otherwise q is rotated at n - 1, the
    token (k, v) is appended at n - 1 by ``append_rope_int8`` (nothing written
    and the flag raised if that page is outside the pool), and attention
    covers [0, n) (zero output and the flag for a bad needed page).
    Returns (codes', scales', q_rot bits [S][32][64], out float64 [S][32][64], err).
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
        codes, scales, _, e = append_rope_int8(codes, scales, k_bits[s:s + 1], v_bits[s:s + 1],
                                               [n - 1], [s], block_tables, cos, sin)
        err |= e
    for s in valid:
        o, e = decode_int8(q_rot[s:s + 1], codes, scales, block_tables[s:s + 1], [int(lens[s])], scale)
        err |= e
        out[s] = o[0]
    return codes, scales, q_rot, out, err
