"""Pins for the oracle's paged append and paged decode attention (CPU only).

The decode definition is checked against closed forms (one token, identical
keys, two tokens, constant V), linearity, page-permutation invariance, torch's
scaled_dot_product_attention on a contiguous FP64 copy, and a 50-digit mpmath
brute force; the append is checked by a brute-force scan of a sentinel pool;
the page geometry against the sizes the pages print (tests/golden/).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import bf16, paged_kv as P, rope

rng_global = np.random.default_rng(1234)


def rand_bits(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def random_paged(rng, lens, num_pages=None, extra_pages=3):
    """Random pool + tables holding sequences of the given lengths."""
    lens = np.asarray(lens)
    need = sum((int(n) + 15) // 16 for n in lens)
    num_pages = num_pages or need + extra_pages
    pool = rand_bits(rng, (num_pages, 2, 8, 16, 64))
    perm = rng.permutation(num_pages)
    bt = np.full((len(lens), 128), -1, np.int32)
    cur = 0
    for s, n in enumerate(lens):
        k = (int(n) + 15) // 16
        bt[s, :k] = perm[cur:cur + k]
        cur += k
    q = rand_bits(rng, (len(lens), 32, 64))
    return pool, bt, q


def contiguous_kv(pool, row, n):
    """K, V [n][8][64] read position by position (independent of P.gather)."""
    K = np.empty((n, 8, 64))
    V = np.empty((n, 8, 64))
    for j in range(n):
        page, slot = int(row[j // 16]), j % 16
        K[j] = bf16.to_f64(pool[page, 0, :, slot, :])
        V[j] = bf16.to_f64(pool[page, 1, :, slot, :])
    return K, V


# ------------------------------------------------------------ closed forms --

def test_one_token_returns_v_exactly():
    rng = np.random.default_rng(0)
    pool, bt, q = random_paged(rng, [1, 1])
    out, err = P.decode(q, pool, bt, [1, 1], 0.125)
    assert not err
    for s in range(2):
        for h in range(32):
            v = bf16.to_f64(pool[bt[s, 0], 1, h // 4, 0, :])
            assert np.array_equal(out[s, h], v)


def test_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(1)
    n = 37
    pool, bt, q = random_paged(rng, [n])
    for j in range(n):
        pool[bt[0, j // 16], 0, :, j % 16, :] = pool[bt[0, 0], 0, :, 0, :]
    out, _ = P.decode(q, pool, bt, [n], 0.125)
    _, V = contiguous_kv(pool, bt[0], n)
    for h in range(32):
        assert np.allclose(out[0, h], V[:, h // 4, :].mean(axis=0), rtol=0, atol=1e-14)


def test_two_tokens_sigmoid_closed_form():
    rng = np.random.default_rng(2)
    pool, bt, q = random_paged(rng, [2])
    out, _ = P.decode(q, pool, bt, [2], 0.125)
    K, V = contiguous_kv(pool, bt[0], 2)
    qf = bf16.to_f64(q[0])
    for h in range(32):
        g = h // 4
        x0, x1 = 0.125 * (qf[h] @ K[0, g]), 0.125 * (qf[h] @ K[1, g])
        sig = 1.0 / (1.0 + math.exp(-(x0 - x1)))
        assert np.allclose(out[0, h], sig * V[0, g] + (1 - sig) * V[1, g], rtol=0, atol=1e-14)


def test_constant_v_gives_constant():
    rng = np.random.default_rng(3)
    lens = [5, 16, 33]
    pool, bt, q = random_paged(rng, lens)
    c = rand_bits(rng, (8, 64))
    for s, n in enumerate(lens):
        for j in range(n):
            pool[bt[s, j // 16], 1, :, j % 16, :] = c
    out, _ = P.decode(q, pool, bt, lens, 0.125)
    for s in range(3):
        for h in range(32):
            assert np.allclose(out[s, h], bf16.to_f64(c[h // 4]), rtol=0, atol=1e-14)


def test_linear_in_v():
    rng = np.random.default_rng(4)
    n = 50
    K = rng.standard_normal((n, 64))
    V1, V2 = rng.standard_normal((n, 64)), rng.standard_normal((n, 64))
    qh = rng.standard_normal(64)
    a, b = 0.7, -1.3
    lhs = P.attend(qh, K, a * V1 + b * V2, 0.125)
    rhs = a * P.attend(qh, K, V1, 0.125) + b * P.attend(qh, K, V2, 0.125)
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-13)


# ------------------------------------------------------------- invariants ---

def test_page_permutation_invariance():
    rng = np.random.default_rng(5)
    lens = [37, 1, 300, 16, 17]
    pool, bt, q = random_paged(rng, lens, extra_pages=10)
    out1, _ = P.decode(q, pool, bt, lens, 0.125)
    # move every page to a new physical id and rewrite the tables accordingly
    N = pool.shape[0]
    perm = rng.permutation(N)
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2, _ = P.decode(q, pool2, bt2, lens, 0.125)
    assert np.array_equal(out1, out2)


def test_paged_equals_contiguous_sdpa():
    rng = np.random.default_rng(6)
    lens = [1, 15, 16, 17, 31, 32, 129, 700]
    pool, bt, q = random_paged(rng, lens)
    scale = 0.125
    out, err = P.decode(q, pool, bt, lens, scale)
    assert not err
    for s, n in enumerate(lens):
        K, V = contiguous_kv(pool, bt[s], n)
        Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(4, dim=0)   # [32][n][64]
        Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(4, dim=0)
        qt = torch.from_numpy(bf16.to_f64(q[s]))[:, None, :]                    # [32][1][64]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)[:, 0, :]
        assert np.allclose(out[s], ref.numpy(), rtol=0, atol=1e-12)


def test_gqa_mapping_is_h_div_4():
    rng = np.random.default_rng(7)
    pool, bt, q = random_paged(rng, [20])
    # make KV heads clearly different: V of head g is the constant g
    for j in range(20):
        for g in range(8):
            pool[bt[0, j // 16], 1, g, j % 16, :] = bf16.from_f32_rne(np.full(64, float(g), np.float32))
    out, _ = P.decode(q, pool, bt, [20], 0.125)
    for h in range(32):
        assert np.allclose(out[0, h], h // 4, atol=1e-14)


def test_mpmath_brute_force():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    rng = np.random.default_rng(8)
    for n in (1, 2, 3, 4):
        pool, bt, q = random_paged(rng, [n])
        out, _ = P.decode(q, pool, bt, [n], 0.125)
        K, V = contiguous_kv(pool, bt[0], n)
        qf = bf16.to_f64(q[0])
        for h in (0, 5, 31):
            g = h // 4
            xs = [mp.mpf(0.125) * mp.fsum(mp.mpf(qf[h, d]) * mp.mpf(K[j, g, d]) for d in range(64))
                  for j in range(n)]
            es = [mp.exp(x) for x in xs]
            den = mp.fsum(es)
            for d in range(64):
                o = mp.fsum(es[j] * mp.mpf(V[j, g, d]) for j in range(n)) / den
                assert abs(float(o) - out[0, h, d]) <= 1e-13


def test_split_combine_identity():
    rng = np.random.default_rng(9)
    n = 777
    K = rng.standard_normal((n, 64)) * 2
    V = rng.standard_normal((n, 64))
    qh = rng.standard_normal(64)
    ref = P.attend(qh, K, V, 0.125)
    for _ in range(20):
        cuts = np.sort(rng.choice(np.arange(0, n + 1), size=rng.integers(1, 12), replace=True))
        bounds = [0] + [int(c) for c in cuts] + [n]
        assert np.allclose(P.attend_split(qh, K, V, 0.125, bounds), ref, rtol=0, atol=1e-12)


def test_tail_garbage_is_never_read():
    rng = np.random.default_rng(10)
    lens = [5, 37]
    pool, bt, q = random_paged(rng, lens)
    clean, _ = P.decode(q, pool, bt, lens, 0.125)
    for s, n in enumerate(lens):
        page = bt[s, n // 16]
        pool[page, :, :, n % 16:, :] = 0x7FC0          # NaN in unused slots
    dirty, _ = P.decode(q, pool, bt, lens, 0.125)
    assert np.array_equal(clean, dirty)


def test_error_contract():
    rng = np.random.default_rng(11)
    lens = [20, 0, 40]
    pool, bt, q = random_paged(rng, lens)
    ok, err = P.decode(q, pool, bt, lens, 0.125)
    assert not err and np.all(ok[1] == 0)
    bt_bad = bt.copy()
    bt_bad[2, 1] = pool.shape[0]          # out of range page in a needed block
    out, err = P.decode(q, pool, bt_bad, lens, 0.125)
    assert err and np.all(out[2] == 0) and np.array_equal(out[0], ok[0])
    out, err = P.decode(q, pool, bt, [20, 0, 16 * 128 + 1], 0.125)
    assert err and np.all(out[2] == 0)
    out, err = P.decode(q, pool, bt, [20, -1, 40], 0.125)
    assert err and np.all(out[1] == 0) and np.array_equal(out[2], ok[2])


# ------------------------------------------------------------------ append --

def test_append_sentinel_brute_force():
    rng = np.random.default_rng(12)
    S, N, T = 3, 12, 40
    SENT = 0xABCD
    pool0 = P.new_pool(N, SENT)
    perm = rng.permutation(N)
    bt = np.full((S, 8), -1, np.int32)
    bt[0, :3], bt[1, :2], bt[2, :4] = perm[:3], perm[3:5], perm[5:9]
    caps = [48, 32, 64]
    # distinct (seq, pos) pairs
    pairs = set()
    while len(pairs) < T:
        s = int(rng.integers(0, S))
        pairs.add((s, int(rng.integers(0, caps[s]))))
    pairs = sorted(pairs, key=lambda _: rng.random())
    seqs = np.array([p[0] for p in pairs], np.int32)
    pos = np.array([p[1] for p in pairs], np.int32)
    k, v, q = rand_bits(rng, (T, 8, 64)), rand_bits(rng, (T, 8, 64)), rand_bits(rng, (T, 32, 64))
    f = rope.inv_freq_llama3()
    cos, sin = rope.table(f, 64)
    pool, qrot, err = P.append_rope(pool0, k, v, pos, seqs, bt, cos, sin, q)
    assert not err
    # brute force: walk every element of the pool and find who (if anyone) owns it
    for page in range(N):
        for slot in range(16):
            owners = [t for t in range(T)
                      if bt[seqs[t], pos[t] // 16] == page and pos[t] % 16 == slot]
            assert len(owners) <= 1
            if not owners:
                assert np.all(pool[page, :, :, slot, :] == SENT)
                continue
            t = owners[0]
            assert np.array_equal(pool[page, 1, :, slot, :], v[t])
            exact = rope.rotate_exact(bf16.to_f64(k[t]), pos[t], f)
            got = bf16.to_f64(pool[page, 0, :, slot, :])
            assert np.all(np.abs(got - exact) <= 2.0 ** -8 * np.abs(exact) + 1e-5)
    for t in range(T):
        exact = rope.rotate_exact(bf16.to_f64(q[t]), pos[t], f)
        assert np.all(np.abs(bf16.to_f64(qrot[t]) - exact) <= 2.0 ** -8 * np.abs(exact) + 1e-5)


def test_append_then_decode_one_token_is_v():
    rng = np.random.default_rng(13)
    pool0 = P.new_pool(4, 0x7FC0)              # NaN everywhere else
    bt = np.array([[2, -1]], np.int32)
    k, v = rand_bits(rng, (1, 8, 64)), rand_bits(rng, (1, 8, 64))
    cos, sin = rope.table(rope.inv_freq_llama3(), 16)
    pool, _, err = P.append_rope(pool0, k, v, [0], None, bt, cos, sin)
    q = rand_bits(rng, (1, 32, 64))
    out, err2 = P.decode(q, pool, bt, [1], 0.125)
    assert not err and not err2
    for h in range(32):
        assert np.array_equal(out[0, h], bf16.to_f64(v[0, h // 4]))


def test_append_error_contract():
    rng = np.random.default_rng(14)
    pool0 = P.new_pool(4, 0x1111)
    bt = np.array([[0, 1], [2, 9]], np.int32)   # page 9 does not exist
    cos, sin = rope.table(rope.inv_freq_llama3(), 32)
    k, v, q = rand_bits(rng, (4, 8, 64)), rand_bits(rng, (4, 8, 64)), rand_bits(rng, (4, 32, 64))
    # token 0 ok; 1: bad page; 2: bad seq row; 3: position beyond table
    pool, qrot, err = P.append_rope(pool0, k, v, [3, 20, 0, 40], [0, 1, 5, 0], bt, cos, sin, q)
    assert err
    assert np.array_equal(pool[0, 1, :, 3, :], v[0])
    untouched = np.ones(pool.shape, bool)
    untouched[0, :, :, 3, :] = False
    assert np.all(pool[untouched] == 0x1111)
    assert np.all(qrot[1:] == 0) and np.any(qrot[0] != 0)


def test_workload_shapes():
    c = W.case_single()
    assert list(c.block_tables[0, 0, :3]) == list(np.random.default_rng(0).permutation(8)[:3])
    c3 = W.case_batch32()
    assert c3.num_pages == 65536 and c3.num_pages * W.PAGE_ELEMS * 2 == 2 * 2 ** 30
    ids = c3.block_tables[c3.block_tables >= 0]
    assert ids.size == 65536 and np.unique(ids).size == 65536
    c5 = W.case_stress()
    assert c5.num_pages * W.PAGE_ELEMS * 2 == 16 * 2 ** 30


def test_decode_step_is_append_then_decode():
    """The step equals the two-call composition when every index is valid,
    and isolates a bad sequence (zero output, flag) when one is not."""
    rng = np.random.default_rng(15)
    lens = np.array([1, 16, 17, 0, 50], np.int32)
    pool, bt, q = random_paged(rng, lens, extra_pages=4)
    k, v = rand_bits(rng, (5, 8, 64)), rand_bits(rng, (5, 8, 64))
    cos, sin = rope.table(rope.inv_freq_llama3(), 64)
    p1, qr, out, err = P.decode_step(pool, q, k, v, bt, lens, cos, sin, 0.125)
    assert not err
    live = np.nonzero(lens)[0]
    p2, qr2, e2 = P.append_rope(pool, k[live], v[live], lens[live] - 1, live, bt, cos, sin, q[live])
    assert not e2 and np.array_equal(p1, p2) and np.array_equal(qr[live], qr2)
    assert np.all(qr[3] == 0) and np.all(out[3] == 0)
    qf = np.zeros_like(q)
    qf[live] = qr2
    ref, _ = P.decode(qf, p2, bt, lens, 0.125)
    assert np.array_equal(out, ref)
    # a length past the 64-entry table: that sequence only is rejected
    lens_bad = lens.copy()
    lens_bad[4] = 65
    bt_big = bt.copy()
    bt_big[4, 4] = bt[4, 3]
    _, qr3, out3, err3 = P.decode_step(pool, q, k, v, bt_big, lens_bad, cos, sin, 0.125)
    assert err3 and np.all(out3[4] == 0) and np.all(qr3[4] == 0)
    assert np.array_equal(out3[:3], out[:3])


def test_page_geometry_matches_the_printed_sizes():
    # sizes the pages print (tests/golden/page_geometry.json, cited there)
    with open(os.path.join(os.path.dirname(__file__), "golden", "page_geometry.json")) as f:
        g = json.load(f)
    pool1 = P.new_pool(1)
    page_bytes = pool1.nbytes
    assert page_bytes * g["kv_cache_pages"] == g["kv_cache_bytes"]     # 65536 pages fill 2 GiB
    k_row = pool1[0, 0, :, 0, :].nbytes            # one token's K over every KV head
    assert k_row == g["kv_dim"] * 2
    assert g["max_prompt_len"] * k_row == g["prefill_k_temp_bytes"]
    assert g["decode_batch_slots"] * k_row == g["decode_k_batch_bytes"]
    assert P.PAGE_TOKENS == g["page_tokens"] == pool1.shape[3]
    assert g["default_pool_mib"] * 2 ** 20 // page_bytes == W.case_continuous().num_pages == 4096
