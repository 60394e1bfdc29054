"""Pins for the oracle's INT8 K/V pages (CPU only).

Quantisation is checked against closed forms (integer rows, power-of-two
scaling, ties to even, zero rows), the half-step error bound, and a
brute-force nearest-code search in exact rational arithmetic; the append by a
brute-force scan of sentinel-filled pools; the decode against torch's float64
scaled_dot_product_attention over pages dequantised position by position, and
against the one-token and identical-key closed forms.
"""
from fractions import Fraction

import numpy as np
import torch

from oracle import bf16, int8_kv as I, paged_kv as P, rope

from test_oracle_paged import rand_bits, random_paged


def bf16_row(rng, scale=1.0):
    return bf16.to_f64(rand_bits(rng, (64,), scale))


# --------------------------------------------------------------- quantise ---

def test_integer_row_is_its_own_code():
    # max |x| = 127 gives scale exactly 1, so the codes are the values
    rng = np.random.default_rng(0)
    x = rng.integers(-127, 128, 64).astype(np.float64)
    x[5] = -127.0
    codes, scale = I.quantize_row(x)
    assert scale == np.float32(1.0)
    assert np.array_equal(codes.astype(np.float64), x)


def test_power_of_two_scaling_keeps_codes():
    rng = np.random.default_rng(1)
    x = bf16_row(rng)
    c0, s0 = I.quantize_row(x)
    for k in (-20, -3, 1, 7, 30):
        c, s = I.quantize_row(x * 2.0 ** k)
        assert np.array_equal(c, c0)
        assert float(s) == float(s0) * 2.0 ** k


def test_ties_round_to_even():
    x = np.zeros(64)
    x[0] = 127.0
    x[1:9] = [2.5, 3.5, -2.5, -3.5, 0.5, 1.5, 126.5, -0.5]
    codes, scale = I.quantize_row(x)
    assert scale == np.float32(1.0)
    assert list(codes[1:9]) == [2, 4, -2, -4, 0, 2, 126, 0]


def test_zero_row():
    codes, scale = I.quantize_row(np.zeros(64))
    assert scale == 0.0 and np.all(codes == 0)
    x = np.zeros(64)
    x[17] = -2.0 ** -100
    codes, scale = I.quantize_row(x)
    assert codes[17] == -127 and np.count_nonzero(codes) == 1


def test_error_bound_and_range():
    rng = np.random.default_rng(2)
    for trial in range(300):
        x = bf16_row(rng, scale=float(2.0 ** rng.integers(-10, 10)))
        codes, scale = I.quantize_row(x)
        s = float(scale)
        amax = np.max(np.abs(x))
        assert abs(s - amax / 127) <= 2.0 ** -24 * amax / 127
        assert codes.min() >= -127 and codes.max() <= 127
        i = int(np.argmax(np.abs(x)))
        assert int(codes[i]) == (127 if x[i] > 0 else -127)
        err = np.abs(x - codes.astype(np.float64) * s)
        assert np.all(err <= 0.5 * s * (1 + 2.0 ** -16))


def test_brute_force_nearest_code():
    # the code is the integer in [-127, 127] nearest to x / scale (exact
    # rational arithmetic), except where the quotient lies within a hair of a
    # half-integer and the fp32 rounding of the quotient decides
    rng = np.random.default_rng(3)
    checked = 0
    for _ in range(40):
        x = bf16_row(rng)
        codes, scale = I.quantize_row(x)
        sf = Fraction(float(scale))
        for d in range(64):
            qd = Fraction(float(x[d])) / sf
            frac = qd - (qd.numerator // qd.denominator)
            if abs(frac - Fraction(1, 2)) < Fraction(1, 2 ** 15):
                continue
            best = min(range(-127, 128), key=lambda c: abs(qd - c))
            assert int(codes[d]) == best
            checked += 1
    assert checked > 2500


def test_rows_are_quantised_independently():
    rng = np.random.default_rng(4)
    X = bf16.to_f64(rand_bits(rng, (5, 3, 64)))
    codes, scales = I.quantize_rows(X)
    for i in range(5):
        for j in range(3):
            c, s = I.quantize_row(X[i, j])
            assert np.array_equal(codes[i, j], c) and scales[i, j] == s


# ----------------------------------------------------------------- append ---

def test_append_sentinel_brute_force():
    rng = np.random.default_rng(12)
    S, N, T = 3, 12, 40
    codes0, scales0 = I.new_pools(N, code_fill=-128, scale_fill=-1.0)
    perm = rng.permutation(N)
    bt = np.full((S, 8), -1, np.int32)
    bt[0, :3], bt[1, :2], bt[2, :4] = perm[:3], perm[3:5], perm[5:9]
    caps = [48, 32, 64]
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
    codes, scales, qrot, err = I.append_rope_int8(codes0, scales0, k, v, pos, seqs, bt, cos, sin, q)
    assert not err
    for page in range(N):
        for slot in range(16):
            owners = [t for t in range(T)
                      if bt[seqs[t], pos[t] // 16] == page and pos[t] % 16 == slot]
            assert len(owners) <= 1
            if not owners:
                assert np.all(codes[page, :, :, slot, :] == -128)
                assert np.all(scales[page, :, :, slot] == -1.0)
                continue
            t = owners[0]
            # dequantised values are within half a step of the exact rotation / V
            exact_k = rope.rotate_exact(bf16.to_f64(k[t]), pos[t], f)
            exact_v = bf16.to_f64(v[t])
            for kv, exact in ((0, exact_k), (1, exact_v)):
                s = scales[page, kv, :, slot].astype(np.float64)
                got = codes[page, kv, :, slot, :].astype(np.float64) * s[:, None]
                bound = 0.5 * s[:, None] * (1 + 2.0 ** -16) + 2.0 ** -8 * np.abs(exact) + 1e-5
                assert np.all(np.abs(got - exact) <= bound)
    for t in range(T):
        exact = rope.rotate_exact(bf16.to_f64(q[t]), pos[t], f)
        assert np.all(np.abs(bf16.to_f64(qrot[t]) - exact) <= 2.0 ** -8 * np.abs(exact) + 1e-5)


def test_append_stores_the_bf16_cache_rows_quantised():
    # the INT8 append quantises exactly the rows the bf16 append stores
    rng = np.random.default_rng(13)
    N, T = 6, 20
    bt = np.array([rng.permutation(N)[:2]], np.int32)
    pos = rng.permutation(32)[:T].astype(np.int32)
    k, v = rand_bits(rng, (T, 8, 64)), rand_bits(rng, (T, 8, 64))
    cos, sin = rope.table(rope.inv_freq_llama3(), 32)
    pool, _, e1 = P.append_rope(P.new_pool(N), k, v, pos, np.zeros(T, np.int32), bt, cos, sin)
    codes, scales, _, e2 = I.append_rope_int8(*I.new_pools(N), k, v, pos, np.zeros(T, np.int32),
                                              bt, cos, sin)
    assert not e1 and not e2
    c_ref, s_ref = I.quantize_pool(pool)
    for t in range(T):
        page, slot = bt[0, pos[t] // 16], pos[t] % 16
        assert np.array_equal(codes[page, :, :, slot], c_ref[page, :, :, slot])
        assert np.array_equal(scales[page, :, :, slot], s_ref[page, :, :, slot])


def test_append_error_contract():
    rng = np.random.default_rng(14)
    codes0, scales0 = I.new_pools(4, code_fill=7, scale_fill=3.0)
    bt = np.array([[0, 1], [2, 9]], np.int32)
    cos, sin = rope.table(rope.inv_freq_llama3(), 32)
    k, v, q = rand_bits(rng, (4, 8, 64)), rand_bits(rng, (4, 8, 64)), rand_bits(rng, (4, 32, 64))
    codes, scales, qrot, err = I.append_rope_int8(codes0, scales0, k, v, [3, 20, 0, 40],
                                                  [0, 1, 5, 0], bt, cos, sin, q)
    assert err
    untouched = np.ones(codes.shape, bool)
    untouched[0, :, :, 3, :] = False
    assert np.all(codes[untouched] == 7)
    s_untouched = np.ones(scales.shape, bool)
    s_untouched[0, :, :, 3] = False
    assert np.all(scales[s_untouched] == 3.0)
    assert np.all(qrot[1:] == 0) and np.any(qrot[0] != 0)


# ----------------------------------------------------------------- decode ---

def test_decode_equals_sdpa_on_dequantised_pages():
    rng = np.random.default_rng(20)
    lens = [1, 15, 16, 17, 33, 300]
    pool, bt, q = random_paged(rng, lens)
    codes, scales = I.quantize_pool(pool)
    out, err = I.decode_int8(q, codes, scales, bt, lens, 0.125)
    assert not err
    for s, n in enumerate(lens):
        # dequantise position by position (independent of gather_int8)
        K = np.empty((n, 8, 64))
        V = np.empty((n, 8, 64))
        for j in range(n):
            page, slot = int(bt[s, j // 16]), j % 16
            for g in range(8):
                K[j, g] = codes[page, 0, g, slot].astype(np.float64) * float(scales[page, 0, g, slot])
                V[j, g] = codes[page, 1, g, slot].astype(np.float64) * float(scales[page, 1, g, slot])
        Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(4, dim=0)
        Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(4, dim=0)
        qt = torch.from_numpy(bf16.to_f64(q[s]))[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=0.125)[:, 0, :]
        assert np.allclose(out[s], ref.numpy(), rtol=0, atol=1e-12)


def test_one_token_returns_dequantised_v():
    rng = np.random.default_rng(21)
    pool, bt, q = random_paged(rng, [1, 1])
    codes, scales = I.quantize_pool(pool)
    out, _ = I.decode_int8(q, codes, scales, bt, [1, 1], 0.125)
    for s in range(2):
        for h in range(32):
            page = bt[s, 0]
            v = codes[page, 1, h // 4, 0].astype(np.float64) * float(scales[page, 1, h // 4, 0])
            assert np.array_equal(out[s, h], v)


def test_identical_keys_give_mean_of_dequantised_v():
    rng = np.random.default_rng(22)
    n = 40
    pool, bt, q = random_paged(rng, [n])
    codes, scales = I.quantize_pool(pool)
    for j in range(n):
        codes[bt[0, j // 16], 0, :, j % 16] = codes[bt[0, 0], 0, :, 0]
        scales[bt[0, j // 16], 0, :, j % 16] = scales[bt[0, 0], 0, :, 0]
    out, _ = I.decode_int8(q, codes, scales, bt, [n], 0.125)
    for h in range(32):
        g = h // 4
        vs = [codes[bt[0, j // 16], 1, g, j % 16].astype(np.float64) * float(scales[bt[0, j // 16], 1, g, j % 16])
              for j in range(n)]
        assert np.allclose(out[0, h], np.mean(vs, axis=0), rtol=0, atol=1e-14)


def test_page_permutation_invariance_and_errors():
    rng = np.random.default_rng(23)
    lens = [37, 0, 129]
    pool, bt, q = random_paged(rng, lens, extra_pages=6)
    codes, scales = I.quantize_pool(pool)
    out1, err = I.decode_int8(q, codes, scales, bt, lens, 0.125)
    assert not err and np.all(out1[1] == 0)
    N = codes.shape[0]
    perm = rng.permutation(N)
    c2, s2 = np.empty_like(codes), np.empty_like(scales)
    c2[perm], s2[perm] = codes, scales
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2, _ = I.decode_int8(q, c2, s2, bt2, lens, 0.125)
    assert np.array_equal(out1, out2)
    bt_bad = bt.copy()
    bt_bad[2, 3] = N
    out3, err3 = I.decode_int8(q, codes, scales, bt_bad, lens, 0.125)
    assert err3 and np.all(out3[2] == 0) and np.array_equal(out3[0], out1[0])


def test_close_to_the_bf16_cache():
    # quantisation moves each output by at most a few half-steps of V's scale
    rng = np.random.default_rng(24)
    lens = [64, 500]
    pool, bt, q = random_paged(rng, lens)
    codes, scales = I.quantize_pool(pool)
    o8, _ = I.decode_int8(q, codes, scales, bt, lens, 0.125)
    o16, _ = P.decode(q, pool, bt, lens, 0.125)
    d = np.abs(o8 - o16)
    assert d.max() < 0.05 and d.mean() < 0.01
    assert d.max() > 0          # the two caches do differ


# ------------------------------------------------------------ byte layout ---

def test_pack_pages_layout_by_hand():
    """Positions worked out by hand from the block format's rules: a code is
    the byte code + 128; slot 15 is member 1 of pair 7, whose chunk for dims
    7, 15, .., 63 is 7 ^ 6 = 1, dim 63 being its 8th; the V scale of slot 4 is
    the third word of group 4; the K scale of slot 0 the first of group 0."""
    codes, scales = I.new_pools(3)
    codes[2, 0, 5, 7, 9] = -3          # K code: page 2, head 5, slot 7, dim 9
    codes[1, 1, 0, 15, 63] = 127       # V code: page 1, head 0, slot 15, dim 63
    scales[2, 1, 5, 4] = 0.5           # V scale: page 2, head 5, slot 4
    scales[0, 0, 7, 0] = -2.0          # K scale: page 0, head 7, slot 0
    b = I.pack_pages(codes, scales)
    assert b.shape == (3, 8, 2176) and I.BLOCK_BYTES == 2176
    assert b[2, 5, 7 * 64 + 9] == 125
    assert b[1, 0, 1024 + 128 * 7 + 16 * 1 + 2 * 7 + 1] == 255
    assert bytes(b[2, 5, 2048 + 16 * 4 + 8:2048 + 16 * 4 + 12]) == np.float32(0.5).tobytes()
    assert bytes(b[0, 7, 2048:2052]) == np.float32(-2.0).tobytes()
    codes_region = b[:, :, :2048].copy()
    codes_region[2, 5, 7 * 64 + 9] = 128
    codes_region[1, 0, 1024 + 128 * 7 + 16 * 1 + 2 * 7 + 1] = 128
    assert np.all(codes_region == 128)                 # every other code is 0
    assert np.count_nonzero(b[:, :, 2048:]) == 2       # 0.5 = 0x3F000000, -2.0 = 0xC0000000


def test_block_positions_cover_the_block_once():
    k, v, ks, vs = I.block_positions()
    pos = np.concatenate([k.ravel(), v.ravel()] + [ks + j for j in range(4)] + [vs + j for j in range(4)])
    assert np.array_equal(np.sort(pos), np.arange(I.BLOCK_BYTES))
    # the pair of a V byte pair: the two slots of a pair share every dim's 2 bytes
    for d in (0, 9, 63):
        pairs = {}
        for t in range(16):
            pairs.setdefault(int(v[t, d]) // 2, []).append(t)
        assert sorted(len(x) for x in pairs.values()) == [2] * 8


def test_pack_unpack_round_trip():
    rng = np.random.default_rng(30)
    codes = rng.integers(-128, 128, (5, 2, 8, 16, 64)).astype(np.int8)
    scales = rng.standard_normal((5, 2, 8, 16)).astype(np.float32)
    c2, s2 = I.unpack_pages(I.pack_pages(codes, scales))
    assert np.array_equal(c2, codes) and np.array_equal(s2.view(np.uint32), scales.view(np.uint32))


def test_decode_step_int8_is_append_then_decode():
    """The INT8 step equals the two-call composition when every index is
    valid, and isolates a bad sequence (zero output, flag) when one is not."""
    rng = np.random.default_rng(31)
    lens = np.array([1, 16, 17, 0, 50], np.int32)
    pool, bt, q = random_paged(rng, lens, extra_pages=4)
    codes, scales = I.quantize_pool(pool)
    k, v = rand_bits(rng, (5, 8, 64)), rand_bits(rng, (5, 8, 64))
    cos, sin = rope.table(rope.inv_freq_llama3(), 64)
    c1, s1, qr, out, err = I.decode_step_int8(codes, scales, q, k, v, bt, lens, cos, sin, 0.125)
    assert not err
    live = np.nonzero(lens)[0]
    c2, s2, qr2, e2 = I.append_rope_int8(codes, scales, k[live], v[live], lens[live] - 1, live, bt,
                                         cos, sin, q[live])
    assert not e2 and np.array_equal(c1, c2) and np.array_equal(s1, s2)
    assert np.array_equal(qr[live], qr2)
    assert np.all(qr[3] == 0) and np.all(out[3] == 0)
    qf = np.zeros_like(q)
    qf[live] = qr2
    ref, _ = I.decode_int8(qf, c2, s2, bt, lens, 0.125)
    assert np.array_equal(out, ref)
    # the rotated query is the bf16 step's, and the new token's row is the
    # quantised image of the bf16 step's row
    p1, qb, _, _ = P.decode_step(pool, q, k, v, bt, lens, cos, sin, 0.125)
    assert np.array_equal(qb, qr)
    cq, sq = I.quantize_pool(p1)
    for s in live:
        page, slot = bt[s, (lens[s] - 1) // 16], (lens[s] - 1) % 16
        assert np.array_equal(c1[page, :, :, slot], cq[page, :, :, slot])
        assert np.array_equal(s1[page, :, :, slot], sq[page, :, :, slot])
    # a length past the 64-entry table: that sequence only is rejected
    lens_bad = lens.copy()
    lens_bad[4] = 65
    bt_big = bt.copy()
    bt_big[4, 4] = bt[4, 3]
    _, _, qr3, out3, err3 = I.decode_step_int8(codes, scales, q, k, v, bt_big, lens_bad, cos, sin,
                                               0.125)
    assert err3 and np.all(out3[4] == 0) and np.all(qr3[4] == 0)
    assert np.array_equal(out3[:3], out[:3])
