"""Seeded synthetic inputs for paged GQA decode and KV append.

This module only draws random numbers and lays out block tables; it holds none
of the attention, RoPE or rounding arithmetic.  Both the CUDA path (through its
tests, ``bench.py`` and ``__graft_entry__.smoke``) and the FP64 oracle take
their inputs from here, so the two sides see the same values.

Shapes follow the Llama-3.2-1B attention layer that the serving engines on the
source pages are built around ("2. Weight Loading and GPU Buffer Design",
section "Preallocating the 16 compute buffers": 32 query heads, KV_DIM 512,
hidden 2048 -> head_dim 64, 8 KV heads) and the paged pool of the samir-vllm
article (section "Gestion de la KV cache et strategies de batching": 16-token
physical pages, one block table per sequence and per layer).

Pool layout (shared contract of every consumer):
    pool[num_pages][2][8][16][64] bf16,   index 0 = K, 1 = V
    block_tables[L][S][M] int32, M = 128 (2048 / 16), -1 = unused
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 64
PAGE_TOKENS = 16
MAX_CONTEXT = 2048
MAX_BLOCKS = MAX_CONTEXT // PAGE_TOKENS
PAGE_ELEMS = 2 * NUM_KV_HEADS * PAGE_TOKENS * HEAD_DIM  # 16384 bf16 = 32 KiB
DEFAULT_SCALE = 1.0 / 8.0  # 1/sqrt(64), exact in fp32

# Llama-3.2's published RoPE settings; the pages do not print the frequency table.
ROPE_THETA = 500000.0
ROPE_LLAMA3 = dict(factor=32.0, low_freq_factor=1.0, high_freq_factor=4.0,
                   original_max_pos=8192)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (a view, no arithmetic)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def normal_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    """N(0,1) samples rounded to bf16 by torch, on the generator's device."""
    dev = gen.device
    return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)


def cpu_gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


@dataclasses.dataclass
class DecodeCase:
    """One decode batch: shapes, lengths and page placement for every layer."""
    name: str
    seed: int
    num_layers: int
    seq_lens: np.ndarray          # [S] int32, includes the just-appended token
    num_pages: int
    block_tables: np.ndarray      # [L][S][MAX_BLOCKS] int32, -1 = unused
    scale: float = DEFAULT_SCALE
    outlier_frac: float = 0.0     # fraction of (token, KV head) keys scaled by 8

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.num_seqs else 0

    def kv_bytes_per_layer(self) -> int:
        """Algorithmic K+V bytes one decode layer reads (valid tokens only)."""
        return int(self.seq_lens.astype(np.int64).sum()) * NUM_KV_HEADS * HEAD_DIM * 2 * 2


def _tables_from_permutation(perm: np.ndarray, lens: np.ndarray, num_layers: int) -> np.ndarray:
    """Hand out consecutive chunks of `perm` to (layer, seq) in order."""
    S = lens.shape[0]
    bt = np.full((num_layers, S, MAX_BLOCKS), -1, dtype=np.int32)
    cur = 0
    for l in range(num_layers):
        for s in range(S):
            n = (int(lens[s]) + PAGE_TOKENS - 1) // PAGE_TOKENS
            bt[l, s, :n] = perm[cur:cur + n]
            cur += n
    assert cur <= perm.shape[0]
    return bt


def case_single(seed: int = 0) -> DecodeCase:
    """One sequence, one layer, 37 tokens in pages 16+16+5 of an 8-page pool."""
    lens = np.array([37], dtype=np.int32)
    ids = np.random.default_rng(seed).permutation(8)[:3].astype(np.int32)
    bt = np.full((1, 1, MAX_BLOCKS), -1, dtype=np.int32)
    bt[0, 0, :3] = ids
    return DecodeCase("single_seq_ctx37", seed, 1, lens, 8, bt)


def case_mixed(seed: int = 1, batch: int = 8) -> DecodeCase:
    """Batch 8, one layer, lengths uniform in [1, 2048], 1024-page shuffled pool."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, MAX_CONTEXT + 1, size=batch).astype(np.int32)
    num_pages = 1024
    perm = rng.permutation(num_pages).astype(np.int32)
    return DecodeCase("mixed_b8_ctx1-2048", seed, 1, lens, num_pages,
                      _tables_from_permutation(perm, lens, 1))


def case_uniform(seed: int, batch: int, layers: int, ctx: int = MAX_CONTEXT,
                 outlier_frac: float = 0.0, name: str | None = None) -> DecodeCase:
    """`batch` sequences x `layers` layers, every context `ctx`, pool exactly full."""
    rng = np.random.default_rng(seed)
    lens = np.full(batch, ctx, dtype=np.int32)
    pages_per = (ctx + PAGE_TOKENS - 1) // PAGE_TOKENS
    num_pages = batch * layers * pages_per
    perm = rng.permutation(num_pages).astype(np.int32)
    return DecodeCase(name or f"uniform_b{batch}_l{layers}_ctx{ctx}", seed, layers, lens,
                      num_pages, _tables_from_permutation(perm, lens, layers),
                      outlier_frac=outlier_frac)


def case_batch32(seed: int = 2) -> DecodeCase:
    """Batch 32 x 16 layers x 2048 context: 65536 pages = 2 GiB pool."""
    return case_uniform(seed, 32, 16, name="decode_b32_l16_ctx2048")


def case_stress(seed: int = 4) -> DecodeCase:
    """Batch 256 x 16 layers x 2048 context: 524288 pages = 16 GiB, 1% outlier keys x8."""
    return case_uniform(seed, 256, 16, outlier_frac=0.01, name="stress_b256_l16_ctx2048")


def fill_pool(case: DecodeCase, device="cpu", chunk_pages: int = 8192) -> torch.Tensor:
    """Whole pool N(0,1) bf16 (unused slots included), outlier keys scaled by 8.

    Drawn in chunks from one generator seeded with the case seed, so the same
    seed on the same device always yields the same pool.
    """
    gen = torch.Generator(device=device).manual_seed(case.seed)
    pool = torch.empty((case.num_pages, 2, NUM_KV_HEADS, PAGE_TOKENS, HEAD_DIM),
                       dtype=torch.bfloat16, device=device)
    for p0 in range(0, case.num_pages, chunk_pages):
        p1 = min(case.num_pages, p0 + chunk_pages)
        pool[p0:p1] = normal_bf16((p1 - p0, 2, NUM_KV_HEADS, PAGE_TOKENS, HEAD_DIM), gen)
    if case.outlier_frac > 0:
        # Outliers are chosen among all key vectors (page, head, slot) of the pool.
        n_vec = case.num_pages * NUM_KV_HEADS * PAGE_TOKENS
        n_out = int(round(case.outlier_frac * n_vec))
        idx = torch.randperm(n_vec, generator=gen, device=device)[:n_out]
        page, vec = idx // (NUM_KV_HEADS * PAGE_TOKENS), idx % (NUM_KV_HEADS * PAGE_TOKENS)
        kv = pool.view(case.num_pages, 2, NUM_KV_HEADS * PAGE_TOKENS, HEAD_DIM)
        kv[page, 0, vec] = kv[page, 0, vec] * 8              # x8 is exact in bf16
    return pool


I8_BLOCK_BYTES = 2 * PAGE_TOKENS * HEAD_DIM + 2 * PAGE_TOKENS * 4   # 2176


def fill_pool_int8(case: DecodeCase, device="cpu", chunk_pages: int = 8192) -> torch.Tensor:
    """An INT8 pool for the same geometry: uint8 [N][8][2176], per (page, KV
    head) 1024 K code bytes, 1024 V code bytes, 16 K scales, 16 V scales
    (the block format of include/pkv.h).

    Codes are N(0, 42^2) samples rounded and clipped to [-127, 127], stored as
    code + 128, and scales uniform on [0.015, 0.025) -- about max|x| / 127 for
    rows of 64 N(0,1) values, so that code * scale is close to N(0,1) -- drawn
    in chunks from one generator seeded with the case seed.  Every code and
    every scale is drawn on its own, so the bytes are filled in storage order
    (which slot and dim a byte stands for does not change the law).  The
    case's outlier fraction of key scales get 8x their value: the INT8 image
    of a key row scaled by 8.
    """
    gen = torch.Generator(device=device).manual_seed(case.seed + 5000)
    N = case.num_pages
    scales = 0.015 + 0.01 * torch.rand((N, 2, NUM_KV_HEADS, PAGE_TOKENS), generator=gen,
                                       device=device)
    if case.outlier_frac > 0:
        n_vec = N * NUM_KV_HEADS * PAGE_TOKENS
        n_out = int(round(case.outlier_frac * n_vec))
        idx = torch.randperm(n_vec, generator=gen, device=device)[:n_out]
        page, vec = idx // (NUM_KV_HEADS * PAGE_TOKENS), idx % (NUM_KV_HEADS * PAGE_TOKENS)
        sv = scales.view(N, 2, NUM_KV_HEADS * PAGE_TOKENS)
        sv[page, 0, vec] = sv[page, 0, vec] * 8
    pool = torch.empty((N, NUM_KV_HEADS, I8_BLOCK_BYTES), dtype=torch.uint8, device=device)
    for p0 in range(0, N, chunk_pages):
        p1 = min(N, p0 + chunk_pages)
        g = torch.randn((p1 - p0, 2, NUM_KV_HEADS, PAGE_TOKENS * HEAD_DIM), generator=gen,
                        device=device)
        codes = ((g * 42.0).round().clamp(-127, 127) + 128).to(torch.uint8)       # code + 128
        pool[p0:p1, :, 0:1024] = codes[:, 0]
        pool[p0:p1, :, 1024:2048] = codes[:, 1]
        sc = scales[p0:p1].contiguous().view(torch.uint8)          # [n][2][8][64] bytes
        pool[p0:p1, :, 2048:2112] = sc[:, 0]
        pool[p0:p1, :, 2112:2176] = sc[:, 1]
    return pool


def _i8_scale_words(t: int) -> tuple:
    """Word indices (of a block's 544) of slot t's K and V scales, in the block
    format of include/pkv.h: group t % 8 of four words at word 512 + 4 (t % 8)
    holds the K scales of slots t % 8 and t % 8 + 8, then their V scales."""
    k = 512 + 4 * (t % 8) + t // 8
    return k, k + 2


def garbage_fill_unused_int8(pool: torch.Tensor, case: DecodeCase, layer: int) -> None:
    """Overwrite the scales of the unused tail slots of each sequence's last
    page with NaN / +Inf bits (codes are finite whatever their bits)."""
    for s in range(case.num_seqs):
        n = int(case.seq_lens[s])
        if n % PAGE_TOKENS == 0 or n == 0:
            continue
        page = int(case.block_tables[layer, s, n // PAGE_TOKENS])
        words = pool[page].view(torch.int32)                      # [8][544]
        for t in range(n % PAGE_TOKENS, PAGE_TOKENS):
            kw, vw = _i8_scale_words(t)
            words[:, kw] = 0x7FC00000                             # K scale: NaN
            words[:, vw] = 0x7F800000                             # V scale: +Inf


def fill_queries(case: DecodeCase, device="cpu") -> torch.Tensor:
    """q[L][S][32][64] bf16 ~ N(0,1) (already rotated; rotation-invariant law)."""
    gen = torch.Generator(device=device).manual_seed(case.seed + 1000)
    return normal_bf16((case.num_layers, case.num_seqs, NUM_Q_HEADS, HEAD_DIM), gen)


def fill_new_kv(case: DecodeCase, device="cpu"):
    """New token K/V per layer [L][S][8][64] bf16 ~ N(0,1), appended at seq_len-1."""
    gen = torch.Generator(device=device).manual_seed(case.seed + 2000)
    k = normal_bf16((case.num_layers, case.num_seqs, NUM_KV_HEADS, HEAD_DIM), gen)
    v = normal_bf16((case.num_layers, case.num_seqs, NUM_KV_HEADS, HEAD_DIM), gen)
    return k, v


def new_positions(case: DecodeCase) -> np.ndarray:
    """Absolute position of each sequence's new token (the last one)."""
    return (case.seq_lens.astype(np.int32) - 1).clip(min=0)


def garbage_fill_unused(pool: torch.Tensor, case: DecodeCase, layer: int) -> None:
    """Overwrite the unused tail slots of each sequence's last page with NaN/Inf bits.

    A kernel that reads past seq_len would then produce non-finite output.
    """
    bits = pool.view(torch.int16)
    for s in range(case.num_seqs):
        n = int(case.seq_lens[s])
        if n % PAGE_TOKENS == 0 or n == 0:
            continue
        page = int(case.block_tables[layer, s, n // PAGE_TOKENS])
        bits[page, 0, :, n % PAGE_TOKENS:, :] = 0x7FC0  # NaN
        bits[page, 1, :, n % PAGE_TOKENS:, 0::2] = 0x7F80  # +Inf
        bits[page, 1, :, n % PAGE_TOKENS:, 1::2] = -64  # 0xFFC0 = -NaN


# ---------------------------------------------------------------------------
# Continuous batching mix (64 requests, geometric prompts, 128 decode steps).
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class ContinuousCase:
    name: str
    seed: int
    prompt_lens: np.ndarray   # [R] int32, in [1, 1920]
    decode_steps: int         # 128
    num_layers: int           # 16
    num_pages: int            # 128 MiB / 32 KiB = 4096

    @property
    def allowed_new_tokens(self) -> int:
        # The prefill yields the first new token; each decode step appends one
        # token's K/V, so KV length reaches prompt + decode_steps.
        return self.decode_steps + 1


def case_continuous(seed: int = 3, requests: int = 64, mean_prompt: float = 300.0,
                    decode_steps: int = 128, num_layers: int = 16,
                    pool_mib: int = 128) -> ContinuousCase:
    rng = np.random.default_rng(seed)
    p = rng.geometric(1.0 / mean_prompt, size=requests)
    p = np.clip(p, 1, MAX_CONTEXT - decode_steps).astype(np.int32)
    num_pages = pool_mib * 1024 * 1024 // (PAGE_ELEMS * 2)
    return ContinuousCase("continuous_r64_geo300", seed, p, decode_steps, num_layers, num_pages)


def request_kv(case_seed: int, req: int, layer: int, first_pos: int, n: int):
    """K, V [n][8][64] bf16 for positions first_pos..first_pos+n-1 of one request/layer.

    Each (request, layer) owns a generator, and positions are drawn in order,
    so the prompt block and later single-token draws never overlap: the
    stream for (req, layer) is consumed at offsets that depend only on pos.
    """
    gen = cpu_gen(hash_seed(case_seed, req, layer, first_pos))
    k = normal_bf16((n, NUM_KV_HEADS, HEAD_DIM), gen)
    v = normal_bf16((n, NUM_KV_HEADS, HEAD_DIM), gen)
    return k, v


def request_q(case_seed: int, req: int, layer: int, pos: int):
    gen = cpu_gen(hash_seed(case_seed, req, layer, pos) ^ 0x5A5A5A5A)
    return normal_bf16((NUM_Q_HEADS, HEAD_DIM), gen)


def hash_seed(*parts: int) -> int:
    """Deterministic 63-bit mix of small integers (splitmix64 finaliser)."""
    h = 0x9E3779B97F4A7C15
    for x in parts:
        h ^= (int(x) + 0x9E3779B97F4A7C15 + ((h << 6) & 0xFFFFFFFFFFFFFFFF) + (h >> 2)) & 0xFFFFFFFFFFFFFFFF
        z = h
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        h = z ^ (z >> 31)
    return h & 0x7FFFFFFFFFFFFFFF


def pages_needed(tokens: int) -> int:
    return (tokens + PAGE_TOKENS - 1) // PAGE_TOKENS if tokens > 0 else 0


__all__ = [n for n in dir() if not n.startswith("_")]
assert math.isclose(DEFAULT_SCALE, 1 / math.sqrt(HEAD_DIM))
