"""GPU parity of the INT8 K/V pages: kv_append_rope_int8 and
paged_gqa_decode_int8 through the C ABI against the FP64 oracle.

The append (codes, scales, rotated q) is compared bit for bit.  Decode outputs
(bf16) are compared with the oracle's FP64 attention over the dequantised
pages by the bf16 bar (max |err| <= 1.5e-2, mean |err| <= 1e-3) applied
beyond the bf16 output format's own rounding (see check_close_int8).  Inputs
come from workloads.py and the oracle; nothing the CUDA path computes is fed
to the oracle.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import bf16 as OB, int8_kv as OI, rope as OR
from tests._util import (cancelling_rows, bf16_to_f64, bits, check_close_int8,
                         to_dev_bf16, to_dev_i32)
from tests.test_gpu_parity import edge_case, make_case, rand_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib(cuda_device):
    from paged_kv_gqa_append_gb300 import build
    build.build()
    import paged_kv_gqa_append_gb300 as m
    return m


@pytest.fixture(scope="module")
def tables(lib, cuda_device):
    cos_d, sin_d = lib.rope_tables_device(cuda_device, 2048)
    cos_o, sin_o = OR.table(OR.inv_freq_llama3(), 2048)
    return cos_d, sin_d, cos_o, sin_o


def dev_pool(codes, scales, dev):
    """The library's INT8 pool (bytes) holding the oracle's logical arrays."""
    return torch.from_numpy(OI.pack_pages(codes, scales)).to(dev)


def host_pool(pool):
    """Logical (codes, scales) of a device INT8 pool."""
    return OI.unpack_pages(pool.cpu().numpy())


def same_pool(pool, codes, scales):
    """The device pool's bytes equal the oracle's arrays packed (bit for bit)."""
    return np.array_equal(pool.cpu().numpy(), OI.pack_pages(codes, scales))


def run_decode8(lib, dev, q_bits, codes, scales, bt, lens, scale=0.125, **kw):
    q = to_dev_bf16(q_bits, dev)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.paged_gqa_decode_int8(q, dev_pool(codes, scales, dev), to_dev_i32(bt, dev),
                              to_dev_i32(lens, dev), out, scale, d_err=err, **kw)
    return out, lib.pkv_read_device_error(err)


# ---------------------------------------------------------------- append ----

def test_int8_append_bit_exact(lib, cuda_device, tables):
    """40 tokens of 3 sequences at shuffled positions, q rotated in the same call."""
    cos_d, sin_d, cos_o, sin_o = tables
    dev = cuda_device
    rng = np.random.default_rng(40)
    S, N, T = 3, 12, 40
    codes0, scales0 = OI.new_pools(N, code_fill=-128, scale_fill=-1.0)
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
    k, v, q = rand_bits(4000, (T, 8, 64)), rand_bits(4001, (T, 8, 64)), rand_bits(4002, (T, 32, 64))
    pool_d = dev_pool(codes0, scales0, dev)
    q_out = torch.empty((T, 32, 64), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.kv_append_rope_int8(to_dev_bf16(k, dev), to_dev_bf16(v, dev), to_dev_i32(pos, dev),
                            to_dev_i32(bt, dev), pool_d, cos_d, sin_d, token_seq=to_dev_i32(seqs, dev),
                            q_in=to_dev_bf16(q, dev), q_out=q_out, d_err=err)
    assert lib.pkv_read_device_error(err) == 0
    want_c, want_s, want_q, e = OI.append_rope_int8(codes0, scales0, k, v, pos, seqs, bt, cos_o, sin_o, q)
    assert not e
    assert same_pool(pool_d, want_c, want_s)
    assert np.array_equal(bits(q_out), want_q)


def test_int8_append_special_rows(lib, cuda_device, tables):
    """Position 0 (RoPE is the identity): an integer K row with halves (ties to
    even), a zero V row (scale 0), a tiny row, and an all-negative row."""
    cos_d, sin_d, cos_o, sin_o = tables
    dev = cuda_device
    k = np.zeros((4, 8, 64), np.float32)
    v = np.zeros((4, 8, 64), np.float32)
    k[0, :, 0] = 127.0
    k[0, :, 1:9] = [2.5, 3.5, -2.5, -3.5, 0.5, 1.5, 126.5, -0.5]
    k[1] = np.random.default_rng(1).standard_normal((8, 64)) * 2.0 ** -100
    k[2] = -np.abs(np.random.default_rng(2).standard_normal((8, 64))) - 0.25
    v[1] = 1.0
    v[3] = np.random.default_rng(3).standard_normal((8, 64))
    kb = OB.from_f32_rne(k)
    vb = OB.from_f32_rne(v)
    pos = np.array([0, 16, 32, 48], np.int32)      # slot 0 of four pages, position 0 first
    bt = np.array([[0, 1, 2, 3]], np.int32)
    codes0, scales0 = OI.new_pools(4, code_fill=5, scale_fill=7.0)
    pool_d = dev_pool(codes0, scales0, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.kv_append_rope_int8(to_dev_bf16(kb, dev), to_dev_bf16(vb, dev), to_dev_i32(pos, dev),
                            to_dev_i32(bt, dev), pool_d, cos_d, sin_d,
                            token_seq=to_dev_i32(np.zeros(4, np.int32), dev), d_err=err)
    assert lib.pkv_read_device_error(err) == 0
    want_c, want_s, _, e = OI.append_rope_int8(codes0, scales0, kb, vb, pos, np.zeros(4, np.int32),
                                               bt, cos_o, sin_o)
    assert not e
    assert same_pool(pool_d, want_c, want_s)
    got_c, got_s = host_pool(pool_d)
    assert list(got_c[0, 0, 0, 0, 1:9]) == [2, 4, -2, -4, 0, 2, 126, 0]
    assert np.all(got_c[0, 1, :, 0] == 0) and np.all(got_s[0, 1, :, 0] == 0)


def test_int8_append_error_contract(lib, cuda_device, tables):
    cos_d, sin_d, cos_o, sin_o = tables
    dev = cuda_device
    codes0, scales0 = OI.new_pools(4, code_fill=7, scale_fill=3.0)
    bt = np.array([[0, 1], [2, 9]], np.int32)      # page 9 does not exist
    k, v, q = rand_bits(4010, (4, 8, 64)), rand_bits(4011, (4, 8, 64)), rand_bits(4012, (4, 32, 64))
    pos, seqs = np.array([3, 20, 0, 40], np.int32), np.array([0, 1, 5, 0], np.int32)
    pool_d = dev_pool(codes0, scales0, dev)
    q_out = torch.full((4, 32, 64), 1.0, dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.kv_append_rope_int8(to_dev_bf16(k, dev), to_dev_bf16(v, dev), to_dev_i32(pos, dev),
                            to_dev_i32(bt, dev), pool_d, cos_d[:32], sin_d[:32],
                            token_seq=to_dev_i32(seqs, dev), q_in=to_dev_bf16(q, dev), q_out=q_out,
                            d_err=err)
    assert lib.pkv_read_device_error(err) == lib.ERR_DEVICE_INDEX
    want_c, want_s, want_q, e = OI.append_rope_int8(codes0, scales0, k, v, pos, seqs, bt,
                                                    cos_o[:32], sin_o[:32], q)
    assert e
    assert same_pool(pool_d, want_c, want_s)
    assert np.array_equal(bits(q_out), want_q)


# ---------------------------------------------------------------- decode ----

def edge_case_int8():
    """The bf16 edge case's lengths and pages, quantised by the oracle, with
    NaN / +Inf scales in every unused tail slot."""
    case, _, q = edge_case()
    codes, scales = OI.quantize_pool(W.bf16_bits(W.fill_pool(case)))
    pool = torch.from_numpy(OI.pack_pages(codes, scales))
    W.garbage_fill_unused_int8(pool, case, 0)
    codes, scales = OI.unpack_pages(pool.numpy())
    return case, codes, scales, q


def test_int8_decode_edge_lengths_and_tail_garbage(lib, cuda_device):
    case, codes, scales, q = edge_case_int8()
    bt = case.block_tables[0]
    out, code = run_decode8(lib, cuda_device, q, codes, scales, bt, case.seq_lens)
    ref, err = OI.decode_int8(q, codes, scales, bt, case.seq_lens, case.scale)
    assert code == 0 and not err
    got = bf16_to_f64(out)
    check_close_int8(got, ref, "int8 edge lengths")
    assert np.all(got[8] == 0)                      # seq_len 0 -> zeros


def test_int8_decode_permutation_invariant_and_deterministic(lib, cuda_device):
    case, codes, scales, q = edge_case_int8()
    bt = case.block_tables[0]
    out1, _ = run_decode8(lib, cuda_device, q, codes, scales, bt, case.seq_lens)
    out1b, _ = run_decode8(lib, cuda_device, q, codes, scales, bt, case.seq_lens)
    assert torch.equal(out1.view(torch.int16), out1b.view(torch.int16))
    perm = np.random.default_rng(6).permutation(case.num_pages)
    c2, s2 = np.empty_like(codes), np.empty_like(scales)
    c2[perm], s2[perm] = codes, scales
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2, _ = run_decode8(lib, cuda_device, q, c2, s2, bt2, case.seq_lens)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_int8_decode_error_contract(lib, cuda_device):
    case, codes, scales, q = edge_case_int8()
    bt = case.block_tables[0].copy()
    good, code = run_decode8(lib, cuda_device, q, codes, scales, bt, case.seq_lens)
    assert code == 0
    bad_bt = bt.copy()
    bad_bt[6, 50] = case.num_pages + 3
    out, code = run_decode8(lib, cuda_device, q, codes, scales, bad_bt, case.seq_lens)
    assert code == lib.ERR_DEVICE_INDEX
    got = bits(out)
    assert np.all(got[6] == 0)
    keep = [s for s in range(len(case.seq_lens)) if s != 6]
    assert np.array_equal(got[keep], bits(good)[keep])
    lens = case.seq_lens.copy()
    lens[3], lens[4] = -1, 16 * 128 + 1
    out, code = run_decode8(lib, cuda_device, q, codes, scales, bt, lens)
    assert code == lib.ERR_DEVICE_INDEX
    ref, err = OI.decode_int8(q, codes, scales, bt, lens, case.scale)
    assert err
    got = bf16_to_f64(out)
    assert np.all(got[3] == 0) and np.all(got[4] == 0)
    check_close_int8(got, ref, "int8 sequences next to invalid lengths")


def test_int8_decode_mixed_batch8(lib, cuda_device):
    case = W.case_mixed()
    pool = W.bf16_bits(W.fill_pool(case))
    codes, scales = OI.quantize_pool(pool)
    q = W.bf16_bits(W.fill_queries(case))[0]
    bt = case.block_tables[0]
    out, code = run_decode8(lib, cuda_device, q, codes, scales, bt, case.seq_lens)
    ref, _ = OI.decode_int8(q, codes, scales, bt, case.seq_lens, case.scale)
    assert code == 0
    check_close_int8(bf16_to_f64(out), ref, "int8 mixed batch 8")


@pytest.mark.parametrize("opts", [dict(), dict(stages=4), dict(warps_per_cta=8, stages=4),
                                  dict(min_units_per_warp=1), dict(min_units_per_warp=64),
                                  dict(ctas_per_sm=1), dict(max_seq_len=2048),
                                  dict(stages=4, min_units_per_warp=1, max_seq_len=2048),
                                  dict(warps_per_cta=8, stages=4, min_units_per_warp=1)])
def test_int8_decode_work_split_variants(lib, cuda_device, opts):
    case = make_case([3, 40, 17, 700, 1, 129, 2048, 16], seed=9, extra_pages=5)
    pool = W.bf16_bits(W.fill_pool(case))
    codes, scales = OI.quantize_pool(pool)
    q = W.bf16_bits(W.fill_queries(case))[0]
    bt = case.block_tables[0]
    out, code = run_decode8(lib, cuda_device, q, codes, scales, bt, case.seq_lens, **opts)
    ref, _ = OI.decode_int8(q, codes, scales, bt, case.seq_lens, case.scale)
    assert code == 0
    check_close_int8(bf16_to_f64(out), ref, f"int8 split variant {opts}")


def test_int8_append_then_decode_matches_oracle(lib, cuda_device, tables):
    """Prompt K/V of five sequences appended into INT8 pages (one call), then
    decoded: the pages equal the oracle's bit for bit and so does nothing else
    need to (decode within tolerance)."""
    cos_d, sin_d, cos_o, sin_o = tables
    dev = cuda_device
    lens = np.array([1, 16, 33, 200, 517], np.int32)
    case = make_case(lens, seed=31, extra_pages=3)
    bt = case.block_tables[0]
    T = int(lens.sum())
    seqs = np.repeat(np.arange(len(lens), dtype=np.int32), lens)
    pos = np.concatenate([np.arange(n, dtype=np.int32) for n in lens])
    k, v = rand_bits(4020, (T, 8, 64)), rand_bits(4021, (T, 8, 64))
    q = rand_bits(4022, (len(lens), 32, 64))
    codes0, scales0 = OI.new_pools(case.num_pages)
    pool_d = dev_pool(codes0, scales0, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.kv_append_rope_int8(to_dev_bf16(k, dev), to_dev_bf16(v, dev), to_dev_i32(pos, dev),
                            to_dev_i32(bt, dev), pool_d, cos_d, sin_d,
                            token_seq=to_dev_i32(seqs, dev), d_err=err)
    want_c, want_s, _, e = OI.append_rope_int8(codes0, scales0, k, v, pos, seqs, bt, cos_o, sin_o)
    assert not e and lib.pkv_read_device_error(err) == 0
    assert same_pool(pool_d, want_c, want_s)
    out = torch.empty((len(lens), 32, 64), dtype=torch.bfloat16, device=dev)
    lib.paged_gqa_decode_int8(to_dev_bf16(q, dev), pool_d, to_dev_i32(bt, dev),
                              to_dev_i32(lens, dev), out, 0.125, d_err=err)
    assert lib.pkv_read_device_error(err) == 0
    ref, _ = OI.decode_int8(q, want_c, want_s, bt, lens, 0.125)
    check_close_int8(bf16_to_f64(out), ref, "int8 append then decode")


# ------------------------------------------------- full-size, sampled -------

def full_size_int8_check(lib, dev, case, samples, tables):
    """One bench-shaped INT8 step on every layer (append of the new token with q
    rotation, then decode) and sampled (layer, seq) outputs against the oracle."""
    cos_d, sin_d, cos_o, sin_o = tables
    pool = W.fill_pool_int8(case, device=dev)
    q_raw = W.fill_queries(case, device=dev)
    k_new, v_new = W.fill_new_kv(case, device=dev)
    pos = W.new_positions(case)
    bt_all = to_dev_i32(case.block_tables, dev)
    lens = to_dev_i32(case.seq_lens, dev)
    posd = to_dev_i32(pos, dev)
    pre = {}
    for (l, s) in samples:
        ids = case.block_tables[l, s][case.block_tables[l, s] >= 0]
        idx = torch.from_numpy(ids).to(dev).long()
        pre[(l, s)] = (ids,) + OI.unpack_pages(pool[idx].cpu().numpy())
    q_rot = torch.empty_like(q_raw)
    out = torch.empty_like(q_raw)
    ws = lib.alloc_workspace(case.num_seqs, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for l in range(case.num_layers):
        lib.kv_append_rope_int8(k_new[l], v_new[l], posd, bt_all[l], pool, cos_d, sin_d,
                                q_in=q_raw[l], q_out=q_rot[l], d_err=err)
        lib.paged_gqa_decode_int8(q_rot[l], pool, bt_all[l], lens, out[l], case.scale,
                                  workspace=ws, max_seq_len=case.max_seq_len, d_err=err)
    assert lib.pkv_read_device_error(err) == 0
    for (l, s) in samples:
        ids, c_pages, s_pages = pre[(l, s)]
        bt_local = np.full((1, 128), -1, np.int32)
        bt_local[0, :len(ids)] = np.arange(len(ids))
        kb, vb = bits(k_new[l, s:s + 1]), bits(v_new[l, s:s + 1])
        qb = bits(q_raw[l, s:s + 1])
        want_c, want_s, want_q, e = OI.append_rope_int8(c_pages, s_pages, kb, vb, pos[s:s + 1], None,
                                                        bt_local, cos_o, sin_o, qb)
        assert not e
        idx = torch.from_numpy(ids).to(dev).long()
        assert same_pool(pool[idx], want_c, want_s), f"pages of layer {l} seq {s}"
        assert np.array_equal(bits(q_rot[l, s:s + 1]), want_q)
        ref, _ = OI.decode_int8(want_q, want_c, want_s, bt_local, case.seq_lens[s:s + 1], case.scale)
        check_close_int8(bf16_to_f64(out[l, s:s + 1]), ref, f"int8 layer {l} seq {s}")


def test_int8_full_size_batch32_sampled(lib, cuda_device, tables):
    case = W.case_batch32()
    full_size_int8_check(lib, cuda_device, case, [(0, 0), (0, 31), (7, 13), (15, 5)], tables)
    torch.cuda.empty_cache()


def test_int8_full_size_stress256_sampled(lib, cuda_device, tables):
    case = W.case_stress()
    full_size_int8_check(lib, cuda_device, case, [(0, 0), (9, 77), (15, 255)], tables)
    torch.cuda.empty_cache()


# ------------------------------------------------------ fused decode step ---

def fused_case_int8(lens, seed):
    """One layer: the oracle's INT8 image of random pages holding seq_lens - 1
    tokens, room for the new token, new K/V and un-rotated q."""
    lens = np.asarray(lens, np.int32)
    case = make_case(lens, seed=seed, extra_pages=3)
    codes, scales = OI.quantize_pool(W.bf16_bits(W.fill_pool(case)))
    k = rand_bits(seed + 1, (len(lens), 8, 64))
    v = rand_bits(seed + 2, (len(lens), 8, 64))
    q = rand_bits(seed + 3, (len(lens), 32, 64))
    return case, codes, scales, q, k, v


def run_fused8(lib, dev, tables, case, codes, scales, q, k, v, lens=None, bt=None, **kw):
    cos_d, sin_d, _, _ = tables
    lens = case.seq_lens if lens is None else lens
    bt = case.block_tables[0] if bt is None else bt
    pool = dev_pool(codes, scales, dev)
    out = torch.empty((len(lens), 32, 64), dtype=torch.bfloat16, device=dev)
    q_out = torch.empty_like(out)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.paged_gqa_decode_append_int8(to_dev_bf16(q, dev), to_dev_bf16(k, dev), to_dev_bf16(v, dev),
                                     pool, to_dev_i32(bt, dev), to_dev_i32(lens, dev), out, cos_d,
                                     sin_d, 0.125, q_out=q_out, d_err=err, **kw)
    return pool, q_out, out, lib.pkv_read_device_error(err)


def test_int8_fused_step_matches_oracle(lib, cuda_device, tables):
    """The new token lands in the first or the second page of a two-page unit,
    on page boundaries, in one-page sequences and in full contexts."""
    _, _, cos_o, sin_o = tables
    lens = [1, 16, 17, 32, 33, 48, 49, 0, 700, 2048, 5, 1023]
    case, codes, scales, q, k, v = fused_case_int8(lens, 50)
    pool, q_out, out, code = run_fused8(lib, cuda_device, tables, case, codes, scales, q, k, v)
    wc, ws, wq, ref, e = OI.decode_step_int8(codes, scales, q, k, v, case.block_tables[0],
                                             case.seq_lens, cos_o, sin_o, 0.125)
    assert code == 0 and not e
    assert same_pool(pool, wc, ws), "appended pages differ from the oracle's"
    assert np.array_equal(bits(q_out), wq), "rotated q differs from the oracle's"
    got = bf16_to_f64(out)
    check_close_int8(got, ref, "fused INT8 step")
    assert np.all(got[7] == 0) and np.all(bits(q_out)[7] == 0)


@pytest.mark.parametrize("bad", ["last_page", "middle_page", "past_table"])
def test_int8_fused_step_error_contract(lib, cuda_device, tables, bad):
    _, _, cos_o, sin_o = tables
    lens = np.array([40, 17, 300, 1], np.int32)
    case, codes, scales, q, k, v = fused_case_int8(lens, 60)
    bt = case.block_tables[0].copy()
    if bad == "last_page":
        bt[2, (lens[2] - 1) // 16] = case.num_pages + 5     # the new token's page
    elif bad == "middle_page":
        bt[2, 3] = -1
    else:
        lens[2] = 16 * 128 + 1
    pool, q_out, out, code = run_fused8(lib, cuda_device, tables, case, codes, scales, q, k, v,
                                        lens=lens, bt=bt)
    wc, ws, wq, ref, e = OI.decode_step_int8(codes, scales, q, k, v, bt, lens, cos_o, sin_o, 0.125)
    assert e and code == lib.ERR_DEVICE_INDEX
    assert same_pool(pool, wc, ws)
    assert np.array_equal(bits(q_out), wq)
    got = bf16_to_f64(out)
    assert np.all(got[2] == 0)
    check_close_int8(got, ref, f"fused INT8 step next to a bad sequence ({bad})")


def test_int8_fused_full_size_batch32_sampled(lib, cuda_device, tables):
    """The bench's INT8 step (16 fused launches) at batch 32 x 2048, sampled."""
    cos_d, sin_d, cos_o, sin_o = tables
    dev = cuda_device
    case = W.case_batch32()
    pool = W.fill_pool_int8(case, device=dev)
    q_raw = W.fill_queries(case, device=dev)
    k_new, v_new = W.fill_new_kv(case, device=dev)
    bt_all = to_dev_i32(case.block_tables, dev)
    lens = to_dev_i32(case.seq_lens, dev)
    pos = to_dev_i32(W.new_positions(case), dev)
    out = torch.empty_like(q_raw)
    samples = [(0, 0), (5, 31), (15, 7)]
    pre = {}
    for (l, s) in samples:
        ids = case.block_tables[l, s][case.block_tables[l, s] >= 0]
        pre[(l, s)] = (ids,) + OI.unpack_pages(pool[torch.from_numpy(ids).to(dev).long()].cpu().numpy())
    step = lib.Int8DecodeStep(pool, bt_all, lens, pos, k_new, v_new, q_raw, out, cos_d, sin_d,
                              case.scale, max_seq_len=case.max_seq_len, use_graph=False,
                              q_rot=torch.empty_like(q_raw))
    assert step.error() == 0
    for (l, s) in samples:
        ids, c_pages, s_pages = pre[(l, s)]
        bt_local = np.full((1, 128), -1, np.int32)
        bt_local[0, :len(ids)] = np.arange(len(ids))
        wc, ws, wq, ref, e = OI.decode_step_int8(
            c_pages, s_pages, bits(q_raw[l, s:s + 1]), bits(k_new[l, s:s + 1]),
            bits(v_new[l, s:s + 1]), bt_local, case.seq_lens[s:s + 1], cos_o, sin_o, case.scale)
        assert not e
        assert same_pool(pool[torch.from_numpy(ids).to(dev).long()], wc, ws), f"layer {l} seq {s}"
        assert np.array_equal(bits(step.q_rot[l, s:s + 1]), wq)
        check_close_int8(bf16_to_f64(out[l, s:s + 1]), ref, f"fused INT8 layer {l} seq {s}")
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fused", [True, False])
def test_int8_step_graph_matches_eager_and_oracle(lib, cuda_device, tables, fused):
    """Int8DecodeStep over 3 layers (fused: with the layer overlap), replayed
    from its CUDA graph and run eagerly: identical bits, and equal to the
    oracle's INT8 step layer by layer."""
    cos_d, sin_d, cos_o, sin_o = tables
    case = W.case_uniform(7, batch=4, layers=3, ctx=300, name="i8_step_small")
    case.seq_lens[:] = [300, 17, 129, 256]
    dev = cuda_device
    pool0 = W.fill_pool_int8(case, device=dev)
    q = W.fill_queries(case, device=dev)
    k, v = W.fill_new_kv(case, device=dev)
    pos = torch.from_numpy(W.new_positions(case)).to(dev)
    bt = torch.from_numpy(case.block_tables).to(dev)
    lens = torch.from_numpy(case.seq_lens).to(dev)
    outs = []
    for use_graph in (False, True):
        pool = pool0.clone()
        out = torch.empty_like(q)
        step = lib.Int8DecodeStep(pool, bt, lens, pos, k, v, q, out, cos_d, sin_d, case.scale,
                                  max_seq_len=300, use_graph=use_graph, fused=fused,
                                  q_rot=torch.empty_like(q))
        step.run()
        assert step.error() == 0
        outs.append((bits(out), pool.cpu().numpy(), bits(step.q_rot)))
    assert all(np.array_equal(a, b) for a, b in zip(outs[0], outs[1]))
    # the decode-only graph of the step (layers >= 1 staging early) over the
    # step's pool and rotated q gives the step's output bit for bit
    if fused:
        out_step = out.clone()
        g = step.partial_graph(False, True)
        g.replay()
        assert step.error() == 0
        assert torch.equal(out.view(torch.int16), out_step.view(torch.int16))
    # without a q_rot buffer the fused step keeps no rotated queries; the rest is the same
    pool = pool0.clone()
    out = torch.empty_like(q)
    step = lib.Int8DecodeStep(pool, bt, lens, pos, k, v, q, out, cos_d, sin_d, case.scale,
                              max_seq_len=300, fused=fused)
    assert (step.q_rot is None) == bool(fused)
    step.run()
    assert step.error() == 0
    assert np.array_equal(bits(out), outs[1][0]) and np.array_equal(pool.cpu().numpy(), outs[1][1])
    out_b, pool_b, qrot_b = outs[1]
    codes, scales = OI.unpack_pages(pool0.cpu().numpy())
    for l in range(case.num_layers):
        codes, scales, want_q, ref, e = OI.decode_step_int8(
            codes, scales, bits(q[l]), bits(k[l]), bits(v[l]), case.block_tables[l], case.seq_lens,
            cos_o, sin_o, case.scale)
        assert not e
        assert np.array_equal(qrot_b[l], want_q)
        check_close_int8(OB.to_f64(out_b[l]), ref, f"INT8 step layer {l}")
    assert np.array_equal(pool_b, OI.pack_pages(codes, scales))


def ragged24(seed):
    """24 lengths in [1, 2048] with the edges 1, 16, 17 and 2048 among them."""
    lens = np.random.default_rng(seed).integers(1, 2049, size=24).astype(np.int32)
    lens[:4] = [1, 16, 17, 2048]
    return lens


def test_int8_decode_one_segment_pairs_ragged(lib, cuda_device):
    """24 sequences at a length bound of 2048: the default launch takes 8-warp
    CTAs, two per SM, one (sequence, KV head) segment each; ragged lengths put
    one-page, partial and full segments side by side."""
    case = make_case(ragged24(64), seed=64, extra_pages=9)
    pool = W.bf16_bits(W.fill_pool(case))
    codes, scales = OI.quantize_pool(pool)
    q = W.bf16_bits(W.fill_queries(case))[0]
    bt = case.block_tables[0]
    out, code = run_decode8(lib, cuda_device, q, codes, scales, bt, case.seq_lens, max_seq_len=2048)
    ref, _ = OI.decode_int8(q, codes, scales, bt, case.seq_lens, case.scale)
    assert code == 0
    check_close_int8(bf16_to_f64(out), ref, "int8, 24 ragged sequences, one segment per CTA")


def test_int8_fused_one_segment_pairs_ragged(lib, cuda_device, tables):
    """The fused INT8 step on the same grid: pages, rotated q and outputs."""
    _, _, cos_o, sin_o = tables
    case, codes, scales, q, k, v = fused_case_int8(ragged24(65), 65)
    pool, q_out, out, code = run_fused8(lib, cuda_device, tables, case, codes, scales, q, k, v,
                                        max_seq_len=2048)
    wc, ws, wq, ref, e = OI.decode_step_int8(codes, scales, q, k, v, case.block_tables[0],
                                             case.seq_lens, cos_o, sin_o, 0.125)
    assert code == 0 and not e
    assert same_pool(pool, wc, ws), "appended pages differ from the oracle's"
    assert np.array_equal(bits(q_out), wq), "rotated q differs from the oracle's"
    check_close_int8(bf16_to_f64(out), ref, "fused INT8 step, 24 ragged sequences")


@pytest.mark.parametrize("shape", ["ragged24", "mixed12"])
def test_int8_rotations_round_separately_on_cancelling_pairs(lib, cuda_device, tables, shape):
    """q and new K rows whose pairs nearly cancel under the rotation (a fused
    multiply-add gives other bits there): the fused INT8 step's rotated q and
    quantised K, and the INT8 append kernel's, are the oracle's bit for bit.
    24 ragged sequences take the one-segment 8-warp grid, 12 mixed ones the
    default 16-warp CTAs."""
    cos_d, sin_d, cos_o, sin_o = tables
    dev = cuda_device
    lens = ragged24(67) if shape == "ragged24" else \
        np.array([2, 16, 17, 32, 33, 48, 49, 700, 2048, 5, 1023, 100], np.int32)
    case, codes, scales, _, _, v = fused_case_int8(lens, 67)
    S = len(lens)
    pos = (case.seq_lens - 1).astype(np.int32)
    q = cancelling_rows(670, pos, 32, cos_o, sin_o)
    k = cancelling_rows(671, pos, 8, cos_o, sin_o)
    bt = case.block_tables[0]
    pool, q_out, out, code = run_fused8(lib, dev, tables, case, codes, scales, q, k, v,
                                        max_seq_len=2048)
    wc, ws, wq, ref, e = OI.decode_step_int8(codes, scales, q, k, v, bt, case.seq_lens, cos_o,
                                             sin_o, 0.125)
    assert code == 0 and not e
    assert np.array_equal(bits(q_out), wq), "fused INT8 step: rotated q"
    assert same_pool(pool, wc, ws), "fused INT8 step: appended pages"
    check_close_int8(bf16_to_f64(out), ref, "fused INT8 step on cancelling pairs")
    seqs = np.arange(S, dtype=np.int32)
    want_c, want_s, want_q, e = OI.append_rope_int8(codes, scales, k, v, pos, seqs, bt, cos_o,
                                                    sin_o, q)
    assert not e
    pool_d = dev_pool(codes, scales, dev)
    q_out = torch.empty((S, 32, 64), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.kv_append_rope_int8(to_dev_bf16(k, dev), to_dev_bf16(v, dev), to_dev_i32(pos, dev),
                            to_dev_i32(bt, dev), pool_d, cos_d, sin_d, token_seq=to_dev_i32(seqs, dev),
                            q_in=to_dev_bf16(q, dev), q_out=q_out, d_err=err)
    assert lib.pkv_read_device_error(err) == 0
    assert np.array_equal(bits(q_out), want_q), "INT8 append kernel: rotated q"
    assert same_pool(pool_d, want_c, want_s), "INT8 append kernel: appended pages"
