"""GPU parity: the sm_103a kernels through the C ABI against the FP64 oracle.

Append and page indexing are compared bit for bit; decode outputs (bf16) are
compared with the oracle's FP64 result within max |err| <= 1.5e-2 and
mean |err| <= 1e-3 (q/k/v ~ N(0,1)).  Inputs come from the seeded generators
in workloads.py; the oracle never sees a value produced by the CUDA path.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import bf16 as OB, paged_kv as OP, rope as OR
from tests._util import (cancelling_rows, bf16_to_f64, bits, check_close, to_dev_bf16, to_dev_i32)

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def lib(cuda_device):
    from paged_kv_gqa_append_gb300 import build
    build.build()
    import paged_kv_gqa_append_gb300 as m
    return m


@pytest.fixture(scope="module")
def tables(lib, cuda_device):
    """(device cos, device sin) from the library, (host cos, host sin) from the oracle."""
    cos_d, sin_d = lib.rope_tables_device(cuda_device, 2048)
    cos_o, sin_o = OR.table(OR.inv_freq_llama3(), 2048)
    return cos_d, sin_d, cos_o, sin_o


def rand_bits(seed, shape):
    return W.bf16_bits(W.normal_bf16(shape, W.cpu_gen(seed)))


def run_decode(lib, dev, q_bits, pool_bits, bt, lens, scale=0.125, **kw):
    q = to_dev_bf16(q_bits, dev)
    pool = to_dev_bf16(pool_bits, dev)
    btd = to_dev_i32(bt, dev)
    ld = to_dev_i32(lens, dev)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.paged_gqa_decode(q, pool, btd, ld, out, scale, d_err=err, **kw)
    code = lib.pkv_read_device_error(err)
    return out, code


# ---------------------------------------------------------------- append ----

def test_append_single_sequence_bit_exact(lib, cuda_device, tables):
    """37 raw tokens of one sequence appended at positions 0..36, then decoded."""
    cos_d, sin_d, cos_o, sin_o = tables
    case = W.case_single()
    pool0 = OP.new_pool(case.num_pages, 0x7FC0)                # NaN everywhere
    k, v = rand_bits(3000, (37, 8, 64)), rand_bits(3001, (37, 8, 64))
    q = rand_bits(3002, (37, 32, 64))
    pos = np.arange(37, dtype=np.int32)
    seqs = np.zeros(37, np.int32)
    bt = case.block_tables[0]
    want_pool, want_q, err = OP.append_rope(pool0, k, v, pos, seqs, bt, cos_o, sin_o, q)
    assert not err
    pool = to_dev_bf16(pool0, cuda_device)
    qd, qo = to_dev_bf16(q, cuda_device), torch.empty(37, 32, 64, dtype=torch.bfloat16, device=cuda_device)
    errd = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    lib.kv_append_rope(to_dev_bf16(k, cuda_device), to_dev_bf16(v, cuda_device),
                       to_dev_i32(pos, cuda_device), to_dev_i32(bt, cuda_device), pool, cos_d, sin_d,
                       token_seq=to_dev_i32(seqs, cuda_device), q_in=qd, q_out=qo, d_err=errd)
    assert lib.pkv_read_device_error(errd) == 0
    assert np.array_equal(bits(pool), want_pool)
    assert np.array_equal(bits(qo), want_q)
    # decode the last token's query over the 37 appended tokens
    qlast = want_q[36:37]
    out, code = run_decode(lib, cuda_device, qlast, want_pool, bt, [37])
    ref, _ = OP.decode(qlast, want_pool, bt, [37], case.scale)
    assert code == 0
    check_close(bf16_to_f64(out), ref, "single sequence after append")


def test_append_many_sequences_bit_exact_inplace_q(lib, cuda_device, tables):
    cos_d, sin_d, cos_o, sin_o = tables
    rng = np.random.default_rng(11)
    S, N, T = 6, 64, 500
    pool0 = OP.new_pool(N, 0x1234)
    perm = rng.permutation(N).astype(np.int32)
    bt = np.full((S, 128), -1, np.int32)
    caps = [160, 16, 33, 300, 1, 129]     # 639 distinct (row, position) pairs >= T
    assert sum(caps) >= T
    cur = 0
    for s, c in enumerate(caps):
        n = (c + 15) // 16
        bt[s, :n] = perm[cur:cur + n]
        cur += n
    pairs = set()
    while len(pairs) < T:
        s = int(rng.integers(0, S))
        pairs.add((s, int(rng.integers(0, caps[s]))))
    pairs = list(pairs)
    rng.shuffle(pairs)
    seqs = np.array([a for a, _ in pairs], np.int32)
    pos = np.array([b for _, b in pairs], np.int32)
    k, v, q = rand_bits(41, (T, 8, 64)), rand_bits(42, (T, 8, 64)), rand_bits(43, (T, 32, 64))
    want_pool, want_q, err = OP.append_rope(pool0, k, v, pos, seqs, bt, cos_o, sin_o, q)
    pool = to_dev_bf16(pool0, cuda_device)
    qd = to_dev_bf16(q, cuda_device)
    lib.kv_append_rope(to_dev_bf16(k, cuda_device), to_dev_bf16(v, cuda_device),
                       to_dev_i32(pos, cuda_device), to_dev_i32(bt, cuda_device), pool, cos_d, sin_d,
                       token_seq=to_dev_i32(seqs, cuda_device), q_in=qd, q_out=qd)
    torch.cuda.synchronize()
    assert np.array_equal(bits(pool), want_pool)
    assert np.array_equal(bits(qd), want_q)


def test_append_error_contract(lib, cuda_device, tables):
    cos_d, sin_d, cos_o, sin_o = tables
    pool0 = OP.new_pool(4, 0x1111)
    bt = np.array([[0, 1], [2, 9]], np.int32)     # page 9 is outside the pool
    k, v, q = rand_bits(51, (4, 8, 64)), rand_bits(52, (4, 8, 64)), rand_bits(53, (4, 32, 64))
    pos = np.array([3, 20, 0, 40], np.int32)      # token 3: position 40 is past 2 blocks
    seqs = np.array([0, 1, 5, 0], np.int32)       # token 2: row 5 does not exist
    want_pool, want_q, err = OP.append_rope(pool0, k, v, pos, seqs, bt, cos_o[:64], sin_o[:64], q)
    assert err
    pool = to_dev_bf16(pool0, cuda_device)
    qo = torch.full((4, 32, 64), 7.0, dtype=torch.bfloat16, device=cuda_device)
    errd = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    lib.kv_append_rope(to_dev_bf16(k, cuda_device), to_dev_bf16(v, cuda_device),
                       to_dev_i32(pos, cuda_device), to_dev_i32(bt, cuda_device), pool,
                       cos_d[:64].contiguous(), sin_d[:64].contiguous(),
                       token_seq=to_dev_i32(seqs, cuda_device), q_in=to_dev_bf16(q, cuda_device),
                       q_out=qo, d_err=errd)
    assert lib.pkv_read_device_error(errd) == lib.ERR_DEVICE_INDEX
    assert np.array_equal(bits(pool), want_pool)
    assert np.array_equal(bits(qo), want_q)


# ---------------------------------------------------------------- decode ----

def test_decode_single_sequence_prewritten(lib, cuda_device):
    case = W.case_single()
    pool = W.bf16_bits(W.fill_pool(case))
    q = W.bf16_bits(W.fill_queries(case))[0]
    out, code = run_decode(lib, cuda_device, q, pool, case.block_tables[0], case.seq_lens)
    ref, _ = OP.decode(q, pool, case.block_tables[0], case.seq_lens, case.scale)
    assert code == 0
    check_close(bf16_to_f64(out), ref, "single sequence, 37 tokens")


def make_case(lens, seed, extra_pages):
    """One-layer case with the given lengths on shuffled pages of a small pool."""
    lens = np.asarray(lens, np.int32)
    need = int(sum((int(n) + 15) // 16 for n in lens))
    rng = np.random.default_rng(seed)
    N = need + extra_pages
    perm = rng.permutation(N).astype(np.int32)
    bt = np.full((len(lens), 128), -1, np.int32)
    cur = 0
    for s, n in enumerate(lens):
        k = (int(n) + 15) // 16
        bt[s, :k] = perm[cur:cur + k]
        cur += k
    return W.DecodeCase(f"lens{len(lens)}", seed, 1, lens, N, bt[None])


def edge_case():
    case = make_case([1, 15, 16, 17, 31, 32, 2047, 2048, 0, 5, 1, 129], seed=21, extra_pages=7)
    pool_t = W.fill_pool(case)
    W.garbage_fill_unused(pool_t, case, 0)
    return case, W.bf16_bits(pool_t), W.bf16_bits(W.fill_queries(case))[0]


@pytest.mark.parametrize("compute", [0, 1])
def test_decode_edge_lengths_and_tail_garbage(lib, cuda_device, compute):
    case, pool, q = edge_case()
    bt = case.block_tables[0]
    out, code = run_decode(lib, cuda_device, q, pool, bt, case.seq_lens, compute=compute)
    ref, err = OP.decode(q, pool, bt, case.seq_lens, case.scale)
    assert code == 0 and not err
    got = bf16_to_f64(out)
    check_close(got, ref, f"edge lengths (compute={compute})")
    assert np.all(got[8] == 0)                      # seq_len 0 -> zeros
    for s in (0, 10):                               # one token -> V exactly
        for h in range(32):
            vb = pool[bt[s, 0], 1, h // 4, 0, :]
            assert np.array_equal(bits(out[s, h]), vb)


def test_decode_page_permutation_bit_invariant_and_deterministic(lib, cuda_device):
    case, pool, q = edge_case()
    bt = case.block_tables[0]
    out1, _ = run_decode(lib, cuda_device, q, pool, bt, case.seq_lens)
    out1b, _ = run_decode(lib, cuda_device, q, pool, bt, case.seq_lens)
    assert torch.equal(out1.view(torch.int16), out1b.view(torch.int16))
    perm = np.random.default_rng(5).permutation(case.num_pages)
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2, _ = run_decode(lib, cuda_device, q, pool2, bt2, case.seq_lens)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_decode_error_contract(lib, cuda_device):
    case, pool, q = edge_case()
    bt = case.block_tables[0].copy()
    good, code = run_decode(lib, cuda_device, q, pool, bt, case.seq_lens)
    assert code == 0
    bad_bt = bt.copy()
    bad_bt[6, 50] = case.num_pages + 3             # a needed page of seq 6 is out of range
    out, code = run_decode(lib, cuda_device, q, pool, bad_bt, case.seq_lens)
    assert code == lib.ERR_DEVICE_INDEX
    got = bits(out)
    assert np.all(got[6] == 0)
    keep = [s for s in range(len(case.seq_lens)) if s != 6]
    assert np.array_equal(got[keep], bits(good)[keep])
    lens = case.seq_lens.copy()
    lens[3] = -1
    lens[4] = 16 * 128 + 1
    out, code = run_decode(lib, cuda_device, q, pool, bt, lens)
    assert code == lib.ERR_DEVICE_INDEX
    got = bits(out)
    assert np.all(got[3] == 0) and np.all(got[4] == 0)
    ref, err = OP.decode(q, pool, bt, lens, case.scale)
    assert err
    check_close(bf16_to_f64(out), ref, "other sequences next to invalid lengths")


@pytest.mark.parametrize("compute", [0, 1])
def test_decode_mixed_batch8(lib, cuda_device, compute):
    case = W.case_mixed()
    pool = W.bf16_bits(W.fill_pool(case))
    q = W.bf16_bits(W.fill_queries(case))[0]
    bt = case.block_tables[0]
    out, code = run_decode(lib, cuda_device, q, pool, bt, case.seq_lens, compute=compute)
    ref, _ = OP.decode(q, pool, bt, case.seq_lens, case.scale)
    assert code == 0
    check_close(bf16_to_f64(out), ref, f"mixed batch 8 (compute={compute})")


@pytest.mark.parametrize("opts", [dict(min_units_per_warp=1), dict(min_units_per_warp=64),
                                  dict(ctas_per_sm=1), dict(max_seq_len=2048),
                                  dict(warps_per_cta=8, stages=2), dict(warps_per_cta=8, stages=4),
                                  dict(warps_per_cta=4, stages=2), dict(warps_per_cta=4, stages=4),
                                  dict(warps_per_cta=4, stages=2, min_units_per_warp=1),
                                  dict(warps_per_cta=16, stages=3), dict(combine=1),
                                  dict(combine=1, warps_per_cta=4, stages=2, min_units_per_warp=1),
                                  dict(combine=1, ctas_per_sm=1, min_units_per_warp=1),
                                  dict(schedule=1), dict(schedule=1, min_units_per_warp=1),
                                  dict(early_kv=1), dict(early_kv=1, max_seq_len=2048),
                                  dict(schedule=1, max_seq_len=2048)])
def test_decode_work_split_variants(lib, cuda_device, opts):
    """Different warp counts (including more warps than units) give the same answer."""
    case = make_case([3, 40, 17, 700, 1, 129, 2048, 16], seed=9, extra_pages=5)
    pool = W.bf16_bits(W.fill_pool(case))
    q = W.bf16_bits(W.fill_queries(case))[0]
    bt = case.block_tables[0]
    out, code = run_decode(lib, cuda_device, q, pool, bt, case.seq_lens, **opts)
    ref, _ = OP.decode(q, pool, bt, case.seq_lens, case.scale)
    assert code == 0
    check_close(bf16_to_f64(out), ref, f"split variant {opts}")


# ------------------------------------------------- full-size, sampled -------

def full_size_step_check(lib, dev, case, samples, tables, fused=True, schedule=0):
    """Run one bench-shaped step (append new token with q rotation, then decode,
    on every layer; fused into one call or as two calls) and compare sampled
    (layer, seq) outputs with the oracle."""
    cos_d, sin_d, cos_o, sin_o = tables
    pool = W.fill_pool(case, device=dev)
    q_raw = W.fill_queries(case, device=dev)
    k_new, v_new = W.fill_new_kv(case, device=dev)
    pos = W.new_positions(case)
    bt_all = to_dev_i32(case.block_tables, dev)
    lens = to_dev_i32(case.seq_lens, dev)
    posd = to_dev_i32(pos, dev)
    # inputs of the sampled sequences, copied before the step runs
    pre = {}
    for (l, s) in samples:
        ids = case.block_tables[l, s][case.block_tables[l, s] >= 0]
        pre[(l, s)] = (ids, bits(pool[torch.from_numpy(ids).to(dev).long()]))
    q_rot = torch.empty_like(q_raw)
    out = torch.empty_like(q_raw)
    ws = lib.alloc_workspace(case.num_seqs, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for l in range(case.num_layers):
        if fused:
            lib.paged_gqa_decode_append(q_raw[l], k_new[l], v_new[l], pool, bt_all[l], lens, out[l],
                                        cos_d, sin_d, case.scale, q_out=q_rot[l], workspace=ws,
                                        max_seq_len=case.max_seq_len, d_err=err, schedule=schedule)
        else:
            lib.kv_append_rope(k_new[l], v_new[l], posd, bt_all[l], pool, cos_d, sin_d,
                               q_in=q_raw[l], q_out=q_rot[l], d_err=err)
            lib.paged_gqa_decode(q_rot[l], pool, bt_all[l], lens, out[l], case.scale,
                                 workspace=ws, max_seq_len=case.max_seq_len, d_err=err,
                                 schedule=schedule)
    assert lib.pkv_read_device_error(err) == 0
    worst = 0.0
    for (l, s) in samples:
        ids, pages = pre[(l, s)]
        # the oracle's own view of these pages: renumber them 0..n-1
        bt_local = np.full((1, 128), -1, np.int32)
        bt_local[0, :len(ids)] = np.arange(len(ids))
        kb, vb = bits(k_new[l, s:s + 1]), bits(v_new[l, s:s + 1])
        qb = bits(q_raw[l, s:s + 1])
        want_pool, want_q, e = OP.append_rope(pages, kb, vb, pos[s:s + 1], None, bt_local,
                                              cos_o, sin_o, qb)
        assert not e
        got_pages = bits(pool[torch.from_numpy(ids).to(dev).long()])
        assert np.array_equal(got_pages, want_pool), f"pool pages of layer {l} seq {s}"
        assert np.array_equal(bits(q_rot[l, s:s + 1]), want_q)
        ref, _ = OP.decode(want_q, want_pool, bt_local, case.seq_lens[s:s + 1], case.scale)
        mx, _ = check_close(bf16_to_f64(out[l, s:s + 1]), ref, f"layer {l} seq {s}")
        worst = max(worst, mx)
    return worst


@pytest.mark.parametrize("fused,schedule", [(True, 0), (False, 0), (True, 1), (False, 1)])
def test_full_size_batch32_sampled(lib, cuda_device, tables, fused, schedule):
    case = W.case_batch32()
    samples = [(0, 0), (0, 31), (7, 13), (15, 5), (15, 31)]
    full_size_step_check(lib, cuda_device, case, samples, tables, fused=fused, schedule=schedule)


@pytest.mark.parametrize("schedule", [0, 1])
def test_full_size_stress256_sampled(lib, cuda_device, tables, schedule):
    case = W.case_stress()
    samples = [(0, 0), (3, 200), (9, 77), (15, 255)]
    full_size_step_check(lib, cuda_device, case, samples, tables, schedule=schedule)
    torch.cuda.empty_cache()


# ------------------------------------------------------- step graph, fused --

def test_workspace_counters_return_to_zero(lib, cuda_device):
    """Segments split across warps are merged by the last warp, which resets its counter."""
    case = make_case([700, 1, 1500, 33, 2048], seed=31, extra_pages=3)
    pool = W.bf16_bits(W.fill_pool(case))
    q = W.bf16_bits(W.fill_queries(case))[0]
    bt = case.block_tables[0]
    ws = lib.alloc_workspace(case.num_seqs, cuda_device)
    ref, _ = OP.decode(q, pool, bt, case.seq_lens, case.scale)
    for mu in (1, 3, 1000):          # many splits, some, none
        out, code = run_decode(lib, cuda_device, q, pool, bt, case.seq_lens, workspace=ws,
                               min_units_per_warp=mu)
        assert code == 0
        check_close(bf16_to_f64(out), ref, f"min_units_per_warp={mu}")
        cnt = ws[:8 * case.num_seqs * 4].view(torch.int32)
        assert int(cnt.abs().sum()) == 0


@pytest.mark.parametrize("fused", [True, False])
def test_decode_step_graph_matches_eager_and_oracle(lib, cuda_device, tables, fused):
    cos_d, sin_d, cos_o, sin_o = tables
    case = W.case_uniform(6, batch=4, layers=3, ctx=300, name="step_small")
    case.seq_lens[:] = [300, 17, 129, 256]
    dev = cuda_device
    pool0 = W.fill_pool(case, device=dev)
    q = W.fill_queries(case, device=dev)
    k, v = W.fill_new_kv(case, device=dev)
    pos = torch.from_numpy(W.new_positions(case)).to(dev)
    bt = torch.from_numpy(case.block_tables).to(dev)
    lens = torch.from_numpy(case.seq_lens).to(dev)
    outs = []
    for use_graph in (False, True):
        pool = pool0.clone()
        out = torch.empty_like(q)
        step = lib.DecodeStep(pool, bt, lens, pos, k, v, q, out, cos_d, sin_d, case.scale,
                              max_seq_len=300, use_graph=use_graph, fused=fused,
                              q_rot=torch.empty_like(q))
        step.run()
        assert step.error() == 0
        outs.append((bits(out), bits(pool), bits(step.q_rot)))
    assert all(np.array_equal(a, b) for a, b in zip(outs[0], outs[1]))
    # the decode-only graph of the step (layers >= 1 staging early) over the
    # step's pool and rotated q gives the step's output bit for bit
    if fused:
        out_step = out.clone()
        g = step.decode_only_graph()
        g.replay()
        assert step.error() == 0
        assert torch.equal(out.view(torch.int16), out_step.view(torch.int16))
    # without a q_rot buffer the fused step keeps no rotated queries; the rest is the same
    pool = pool0.clone()
    out = torch.empty_like(q)
    step = lib.DecodeStep(pool, bt, lens, pos, k, v, q, out, cos_d, sin_d, case.scale,
                          max_seq_len=300, fused=fused)
    assert (step.q_rot is None) == bool(fused)
    step.run()
    assert step.error() == 0
    assert np.array_equal(bits(out), outs[1][0]) and np.array_equal(bits(pool), outs[1][1])
    out_b, pool_b, qrot_b = outs[1]
    pool_in = bits(pool0)
    for l in range(case.num_layers):
        want_pool, want_q, e = OP.append_rope(pool_in, bits(k[l]), bits(v[l]), W.new_positions(case),
                                              None, case.block_tables[l], cos_o, sin_o, bits(q[l]))
        assert not e
        pool_in = want_pool
        assert np.array_equal(qrot_b[l], want_q)
        ref, _ = OP.decode(want_q, want_pool, case.block_tables[l], case.seq_lens, case.scale)
        check_close(OB.to_f64(out_b[l]), ref, f"step layer {l}")
    assert np.array_equal(pool_b, pool_in)


# ------------------------------------------------------- fused decode step --

def fused_case(lens, seed, layers=2):
    case = make_case(lens, seed=seed, extra_pages=6)
    # same lengths for every layer, separate pages per layer
    bt = case.block_tables[0]
    L = layers
    N = case.num_pages
    tables = np.full((L, len(lens), 128), -1, np.int32)
    for l in range(L):
        tables[l] = np.where(bt >= 0, bt + l * N, -1)
    return W.DecodeCase(case.name, seed, L, case.seq_lens, N * L, tables)


@pytest.mark.parametrize("warps,schedule", [(0, 0), (8, 0), (4, 0), (0, 1)])
def test_fused_append_decode_matches_oracle(lib, cuda_device, tables, warps, schedule):
    cos_d, sin_d, cos_o, sin_o = tables
    case = fused_case([1, 16, 17, 0, 2048, 333, 1500, 2], seed=41)
    dev = cuda_device
    pool0 = W.fill_pool(case)
    q = W.fill_queries(case)
    k, v = W.fill_new_kv(case)
    pool = pool0.to(dev)
    q_out = torch.full(q.shape, 3.0, dtype=torch.bfloat16, device=dev)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lens = torch.from_numpy(case.seq_lens).to(dev)
    for l in range(case.num_layers):
        lib.paged_gqa_decode_append(q[l].to(dev), k[l].to(dev), v[l].to(dev), pool,
                                    torch.from_numpy(case.block_tables[l]).to(dev), lens, out[l],
                                    cos_d, sin_d, case.scale, q_out=q_out[l], d_err=err,
                                    warps_per_cta=warps, max_seq_len=2048, schedule=schedule)
    assert lib.pkv_read_device_error(err) == 0
    want_pool = bits(pool0)
    for l in range(case.num_layers):
        want_pool, want_q, ref, e = OP.decode_step(want_pool, bits(q[l]), bits(k[l]), bits(v[l]),
                                                   case.block_tables[l], case.seq_lens, cos_o,
                                                   sin_o, case.scale)
        assert not e
        assert np.array_equal(bits(q_out[l]), want_q)
        check_close(bf16_to_f64(out[l]), ref, f"fused layer {l} warps {warps}")
    assert np.array_equal(bits(pool), want_pool)


@pytest.mark.parametrize("schedule", [0, 1])
@pytest.mark.parametrize("bad", ["last_page", "middle_page", "past_table"])
def test_fused_append_decode_error_contract(lib, cuda_device, tables, bad, schedule):
    cos_d, sin_d, cos_o, sin_o = tables
    case = fused_case([40, 70, 17], seed=43, layers=1)
    dev = cuda_device
    pool0 = W.fill_pool(case)
    q, (k, v) = W.fill_queries(case), W.fill_new_kv(case)
    bt = case.block_tables[0].copy()
    lens = case.seq_lens.copy()
    if bad == "last_page":
        bt[1, 4] = case.num_pages + 5      # the page that should receive seq 1's new token
    elif bad == "middle_page":
        bt[1, 1] = -1
    else:
        lens[1] = 65                       # position 64 is past the 64-entry rope table
        bt[1, 4] = bt[1, 3]
    pool = pool0.to(dev)
    out = torch.empty(q[0].shape, dtype=torch.bfloat16, device=dev)
    q_out = torch.full(q[0].shape, 3.0, dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.paged_gqa_decode_append(q[0].to(dev), k[0].to(dev), v[0].to(dev), pool,
                                torch.from_numpy(bt).to(dev), torch.from_numpy(lens).to(dev), out,
                                cos_d[:64].contiguous(), sin_d[:64].contiguous(), case.scale,
                                q_out=q_out, d_err=err, schedule=schedule)
    assert lib.pkv_read_device_error(err) == lib.ERR_DEVICE_INDEX
    want_pool, want_q, ref, e = OP.decode_step(bits(pool0), bits(q[0]), bits(k[0]), bits(v[0]),
                                               bt, lens, cos_o[:64], sin_o[:64], case.scale)
    assert e
    assert np.array_equal(bits(pool), want_pool)
    assert np.array_equal(bits(q_out), want_q)
    assert np.all(bits(out)[1] == 0)
    check_close(bf16_to_f64(out), ref, f"fused with a bad sequence ({bad})")


# ------------------------------------------------------- bounded waits ----

@pytest.mark.parametrize("schedule", [0, 1])
def test_bounded_wait_runs_out_and_reports_timeout(lib, cuda_device, schedule):
    """A wait that nothing completes (expire_first_wait) runs out after
    wait_limit_ns: the call reports PKV_ERR_TIMEOUT in the device error word,
    drains its copies and returns; after the workspace is zeroed again the
    same decode is exact (the context and the library stay usable)."""
    dev = cuda_device
    case = W.case_mixed(seed=95)
    pool = W.fill_pool(case, device=dev)
    q = W.fill_queries(case, device=dev)[0].contiguous()
    bt = torch.from_numpy(case.block_tables[0]).to(dev)
    lens = torch.from_numpy(case.seq_lens).to(dev)
    out = torch.empty_like(q)
    ws = lib.alloc_workspace(case.num_seqs, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.paged_gqa_decode(q, pool, bt, lens, out, case.scale, workspace=ws, d_err=err,
                         max_seq_len=case.max_seq_len, schedule=schedule,
                         wait_limit_ns=20000, expire_first_wait=1)
    assert lib.pkv_read_device_error(err) == lib.ERR_TIMEOUT
    ws.zero_()
    lib.paged_gqa_decode(q, pool, bt, lens, out, case.scale, workspace=ws, d_err=err,
                         max_seq_len=case.max_seq_len, schedule=schedule)
    assert lib.pkv_read_device_error(err) == 0
    want, _ = OP.decode(W.bf16_bits(q), W.bf16_bits(pool), case.block_tables[0], case.seq_lens,
                        case.scale)
    check_close(bf16_to_f64(out), want, "decode after a timeout")


def ragged24(seed):
    """24 lengths in [1, 2048] with the edges 1, 16, 17 and 2048 among them."""
    lens = np.random.default_rng(seed).integers(1, 2049, size=24).astype(np.int32)
    lens[:4] = [1, 16, 17, 2048]
    return lens


@pytest.mark.parametrize("seed", [61, 62])
def test_decode_one_segment_pairs_ragged(lib, cuda_device, seed):
    """24 sequences at a length bound of 2048: the default launch takes 8-warp
    CTAs, two per SM, one (sequence, KV head) segment each; ragged lengths put
    one-page, partial and full segments side by side."""
    case = make_case(ragged24(seed), seed, extra_pages=9)
    pool = W.bf16_bits(W.fill_pool(case))
    q = W.bf16_bits(W.fill_queries(case))[0]
    bt = case.block_tables[0]
    out, code = run_decode(lib, cuda_device, q, pool, bt, case.seq_lens, max_seq_len=2048)
    ref, _ = OP.decode(q, pool, bt, case.seq_lens, case.scale)
    assert code == 0
    check_close(bf16_to_f64(out), ref, "24 ragged sequences, one segment per CTA")


def test_fused_one_segment_pairs_ragged(lib, cuda_device, tables):
    """The fused step on the same grid, two layers: pool bit for bit, rotated
    q bit for bit, outputs against the oracle."""
    cos_d, sin_d, cos_o, sin_o = tables
    case = fused_case(ragged24(63), seed=63)
    dev = cuda_device
    pool0 = W.fill_pool(case)
    q = W.fill_queries(case)
    k, v = W.fill_new_kv(case)
    pool = pool0.to(dev)
    q_out = torch.full(q.shape, 3.0, dtype=torch.bfloat16, device=dev)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lens = torch.from_numpy(case.seq_lens).to(dev)
    for l in range(case.num_layers):
        lib.paged_gqa_decode_append(q[l].to(dev), k[l].to(dev), v[l].to(dev), pool,
                                    torch.from_numpy(case.block_tables[l]).to(dev), lens, out[l],
                                    cos_d, sin_d, case.scale, q_out=q_out[l], d_err=err,
                                    max_seq_len=2048, early_kv=int(l > 0))
    assert lib.pkv_read_device_error(err) == 0
    want_pool = bits(pool0)
    for l in range(case.num_layers):
        want_pool, want_q, ref, e = OP.decode_step(want_pool, bits(q[l]), bits(k[l]), bits(v[l]),
                                                   case.block_tables[l], case.seq_lens, cos_o,
                                                   sin_o, case.scale)
        assert not e
        assert np.array_equal(bits(q_out[l]), want_q)
        check_close(bf16_to_f64(out[l]), ref, f"fused, 24 ragged sequences, layer {l}")
    assert np.array_equal(bits(pool), want_pool)


# ------------------------------------------------ rounding of the rotations --

@pytest.mark.parametrize("warps,schedule", [(0, 0), (4, 0), (0, 1)])
def test_rotations_round_separately_on_cancelling_pairs(lib, cuda_device, tables, warps, schedule):
    """q and new K rows whose pairs nearly cancel under the rotation, where a
    fused multiply-add gives other bits: the fused step's rotated q and K (and,
    on the default grid, the append kernel's) are the oracle's, bit for bit.
    24 ragged sequences: by default the one-segment 8-warp grid; 4-warp CTAs
    and the dynamic schedule are the other grids."""
    cos_d, sin_d, cos_o, sin_o = tables
    dev = cuda_device
    case = fused_case(ragged24(66), seed=66, layers=1)
    S = len(case.seq_lens)
    pos = (case.seq_lens - 1).astype(np.int32)
    q = cancelling_rows(660, pos, 32, cos_o, sin_o)
    k = cancelling_rows(661, pos, 8, cos_o, sin_o)
    v = rand_bits(662, (S, 8, 64))
    pool0 = bits(W.fill_pool(case))
    bt = case.block_tables[0]
    want_pool, want_q, ref, e = OP.decode_step(pool0, q, k, v, bt, case.seq_lens, cos_o, sin_o,
                                               case.scale)
    assert not e
    pool = to_dev_bf16(pool0, dev)
    q_out = torch.full((S, 32, 64), 3.0, dtype=torch.bfloat16, device=dev)
    out = torch.empty((S, 32, 64), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.paged_gqa_decode_append(to_dev_bf16(q, dev), to_dev_bf16(k, dev), to_dev_bf16(v, dev), pool,
                                to_dev_i32(bt, dev), to_dev_i32(case.seq_lens, dev), out, cos_d,
                                sin_d, case.scale, q_out=q_out, d_err=err, warps_per_cta=warps,
                                max_seq_len=2048, schedule=schedule)
    assert lib.pkv_read_device_error(err) == 0
    assert np.array_equal(bits(q_out), want_q), "fused step: rotated q"
    assert np.array_equal(bits(pool), want_pool), "fused step: appended K/V"
    check_close(bf16_to_f64(out), ref, "fused step on cancelling pairs")
    if warps or schedule:
        return
    seqs = np.arange(S, dtype=np.int32)
    want_pool, want_q, e = OP.append_rope(pool0, k, v, pos, seqs, bt, cos_o, sin_o, q)
    assert not e
    pool = to_dev_bf16(pool0, dev)
    q_out = torch.empty((S, 32, 64), dtype=torch.bfloat16, device=dev)
    lib.kv_append_rope(to_dev_bf16(k, dev), to_dev_bf16(v, dev), to_dev_i32(pos, dev),
                       to_dev_i32(bt, dev), pool, cos_d, sin_d, token_seq=to_dev_i32(seqs, dev),
                       q_in=to_dev_bf16(q, dev), q_out=q_out, d_err=err)
    assert lib.pkv_read_device_error(err) == 0
    assert np.array_equal(bits(q_out), want_q), "append kernel: rotated q"
    assert np.array_equal(bits(pool), want_pool), "append kernel: appended K/V"
