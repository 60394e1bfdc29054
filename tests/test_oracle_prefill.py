"""Pins for the oracle's paged causal prefill attention (CPU only).

Checked against: the decode definition for a one-token chunk (decode is pinned
on its own in test_oracle_paged.py), torch's scaled_dot_product_attention in
FP64 on a contiguous copy (causal for a whole prompt, an explicit
bottom-right mask for a chunk after a cached prefix), causality (K/V after a
query's position never change its row), the first position returning V
exactly, a 50-digit mpmath brute force, and the error contract.
"""
import numpy as np
import pytest
import torch

from oracle import bf16, paged_kv as P
from tests.test_oracle_paged import contiguous_kv, rand_bits, random_paged

SCALE = 0.125


def prompt_case(rng, lens, q_lens):
    pool, bt, _ = random_paged(rng, lens)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = rand_bits(rng, (int(cu[-1]), 32, 64))
    return pool, bt, q, cu


def sdpa_rows(q_bits, pool, row, n, q_len):
    """torch SDPA on a contiguous FP64 copy, queries at positions n-q_len..n-1."""
    K, V = contiguous_kv(pool, row, n)
    qt = torch.from_numpy(bf16.to_f64(q_bits)).permute(1, 0, 2)[None]         # [1][32][q][64]
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(4, 0)[None]   # [1][32][n][64]
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(4, 0)[None]
    pos = torch.arange(n - q_len, n)[:, None]
    mask = torch.arange(n)[None, :] <= pos                                     # bottom-right causal
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=SCALE)
    return o[0].permute(1, 0, 2).numpy()


def test_one_token_chunk_is_decode():
    rng = np.random.default_rng(10)
    lens = [1, 17, 40, 300]
    pool, bt, q, cu = prompt_case(rng, lens, [1, 1, 1, 1])
    got, err = P.prefill(q, cu, pool, bt, np.array(lens), SCALE)
    ref, err2 = P.decode(q, pool, bt, np.array(lens), SCALE)
    assert not err and not err2
    np.testing.assert_array_equal(got, ref)


def test_whole_prompt_matches_causal_sdpa():
    rng = np.random.default_rng(11)
    lens = [5, 16, 33]
    pool, bt, q, cu = prompt_case(rng, lens, lens)
    got, err = P.prefill(q, cu, pool, bt, np.array(lens), SCALE)
    assert not err
    for s, n in enumerate(lens):
        K, V = contiguous_kv(pool, bt[s], n)
        qt = torch.from_numpy(bf16.to_f64(q[cu[s]:cu[s + 1]])).permute(1, 0, 2)[None]
        kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(4, 0)[None]
        vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(4, 0)[None]
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=SCALE)
        np.testing.assert_allclose(got[cu[s]:cu[s + 1]], o[0].permute(1, 0, 2).numpy(),
                                   rtol=0, atol=1e-12)


def test_chunk_after_prefix_matches_masked_sdpa():
    rng = np.random.default_rng(12)
    lens, q_lens = [40, 50, 17], [7, 50, 16]
    pool, bt, q, cu = prompt_case(rng, lens, q_lens)
    got, err = P.prefill(q, cu, pool, bt, np.array(lens), SCALE)
    assert not err
    for s, (n, ql) in enumerate(zip(lens, q_lens)):
        ref = sdpa_rows(q[cu[s]:cu[s + 1]], pool, bt[s], n, ql)
        np.testing.assert_allclose(got[cu[s]:cu[s + 1]], ref, rtol=0, atol=1e-12)


def test_causality_later_keys_never_matter():
    rng = np.random.default_rng(13)
    n = 37
    pool, bt, q, cu = prompt_case(rng, [n], [n])
    base, _ = P.prefill(q, cu, pool, bt, np.array([n]), SCALE)
    cut = 20  # overwrite K and V of positions > cut
    pool2 = pool.copy()
    for j in range(cut + 1, n):
        page, slot = int(bt[0, j // 16]), j % 16
        pool2[page, :, :, slot, :] = rand_bits(rng, (2, 8, 64), 5.0)
    got, _ = P.prefill(q, cu, pool2, bt, np.array([n]), SCALE)
    np.testing.assert_array_equal(got[:cut + 1], base[:cut + 1])
    assert not np.array_equal(got[cut + 1:], base[cut + 1:])


def test_first_position_returns_v():
    rng = np.random.default_rng(14)
    n = 20
    pool, bt, q, cu = prompt_case(rng, [n], [n])
    got, _ = P.prefill(q, cu, pool, bt, np.array([n]), SCALE)
    page = int(bt[0, 0])
    for h in range(32):
        np.testing.assert_array_equal(got[0, h], bf16.to_f64(pool[page, 1, h // 4, 0, :]))


def test_mpmath_brute_force_tiny_prompt():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    rng = np.random.default_rng(15)
    n = 3
    pool, bt, q, cu = prompt_case(rng, [n], [n])
    got, _ = P.prefill(q, cu, pool, bt, np.array([n]), SCALE)
    K, V = contiguous_kv(pool, bt[0], n)
    qf = bf16.to_f64(q)
    for i in range(n):
        for h in (0, 5, 31):
            g = h // 4
            xs = [mp.mpf(SCALE) * mp.fsum(mp.mpf(float(qf[i, h, d])) * mp.mpf(float(K[j, g, d]))
                                           for d in range(64)) for j in range(i + 1)]
            m = max(xs)
            w = [mp.e ** (x - m) for x in xs]
            den = mp.fsum(w)
            for d in (0, 17, 63):
                ref = mp.fsum(w[j] * mp.mpf(float(V[j, g, d])) for j in range(i + 1)) / den
                assert abs(float(ref) - got[i, h, d]) < 1e-13


def test_error_contract():
    rng = np.random.default_rng(16)
    lens, q_lens = [10, 20, 30], [10, 25, 5]          # second: q_len > n
    pool, bt, q, cu = prompt_case(rng, lens, q_lens)
    bt[2, 1] = pool.shape[0] + 4                       # third: a bad needed page
    got, err = P.prefill(q, cu, pool, bt, np.array(lens), SCALE)
    assert err
    assert np.any(got[cu[0]:cu[1]] != 0)
    assert np.all(got[cu[1]:] == 0)
    # an empty chunk is fine and touches nothing
    cu0 = np.array([0, 0], np.int32)
    got0, err0 = P.prefill(q[:0], cu0, pool, bt[:1], np.array([10]), SCALE)
    assert got0.shape == (0, 32, 64) and not err0
