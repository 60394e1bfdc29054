"""GPU parity of paged_gqa_prefill (causal attention of each sequence's newest
tokens over its own pages) against the FP64 oracle, through the C ABI.

Outputs (bf16) are compared with the oracle's FP64 rows within
max |err| <= 1.5e-2 and mean |err| <= 1e-3; inputs come from the seeded
generators in workloads.py.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import paged_kv as OP, rope as OR
from tests._util import bf16_to_f64, bits, check_close, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu
SCALE = 0.125
COMPUTE = [None, 2]   # tcgen05 (default) and the mma.sync comparison arm


@pytest.fixture(scope="module")
def lib(cuda_device):
    from paged_kv_gqa_append_gb300 import build
    build.build()
    import paged_kv_gqa_append_gb300 as m
    return m


def rand_bits(seed, shape):
    return W.bf16_bits(W.normal_bf16(shape, W.cpu_gen(seed)))


def make_case(seed, lens, q_lens, extra_pages=5, garbage=True):
    """A shuffled pool holding the sequences, tables, queries and row offsets."""
    rng = np.random.default_rng(seed)
    need = sum((n + 15) // 16 for n in lens)
    num_pages = need + extra_pages
    pool = rand_bits(seed + 1, (num_pages, 2, 8, 16, 64))
    if garbage:  # slots past each sequence's end hold NaN bits
        pool = pool.copy()
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((len(lens), 128), -1, np.int32)
    cur = 0
    for s, n in enumerate(lens):
        k = (n + 15) // 16
        bt[s, :k] = perm[cur:cur + k]
        cur += k
        if garbage and n % 16:
            pool[bt[s, k - 1], :, :, n % 16:, :] = 0x7FC0
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = rand_bits(seed + 2, (int(cu[-1]), 32, 64))
    return pool, bt, q, cu


def run_prefill(lib, dev, q, cu, pool, bt, lens, max_q_len=None, out_fill=None, compute=None):
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    if out_fill is not None:
        out.view(torch.int16).fill_(out_fill)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.paged_gqa_prefill(to_dev_bf16(q, dev), to_dev_i32(cu, dev), to_dev_bf16(pool, dev),
                          to_dev_i32(bt, dev), to_dev_i32(lens, dev), out, SCALE,
                          max_q_len=max_q_len, d_err=err, compute=compute)
    return out, lib.pkv_read_device_error(err)


@pytest.mark.parametrize("compute", COMPUTE)
def test_prefill_prompts_and_chunks_match_oracle(lib, cuda_device, compute):
    # whole prompts, chunks after a cached prefix, one-token chunks, ragged pages
    lens = [37, 16, 300, 1, 129, 64, 200, 45]
    q_lens = [37, 16, 64, 1, 129, 1, 33, 45]
    pool, bt, q, cu = make_case(100, lens, q_lens)
    out, code = run_prefill(lib, cuda_device, q, cu, pool, bt, lens, compute=compute)
    ref, err = OP.prefill(q, cu, pool, bt, np.array(lens), SCALE)
    assert code == 0 and not err
    check_close(bf16_to_f64(out), ref, "prefill mix")


@pytest.mark.parametrize("compute", COMPUTE)
def test_prefill_after_append_on_one_stream(lib, cuda_device, compute):
    """kv_append_rope of raw prompt K/V, then prefill over the rotated queries."""
    cos_d, sin_d = lib.rope_tables_device(cuda_device, 2048)
    cos_o, sin_o = OR.table(OR.inv_freq_llama3(), 2048)
    lens = [77, 150]
    pool0, bt, q_raw, cu = make_case(200, lens, lens, garbage=False)
    pool0 = OP.new_pool(pool0.shape[0], 0x7FC0)            # NaN until appended
    T = int(cu[-1])
    k, v = rand_bits(201, (T, 8, 64)), rand_bits(202, (T, 8, 64))
    seqs = np.concatenate([np.full(n, s, np.int32) for s, n in enumerate(lens)])
    pos = np.concatenate([np.arange(n, dtype=np.int32) for n in lens])
    want_pool, want_q, e = OP.append_rope(pool0, k, v, pos, seqs, bt, cos_o, sin_o, q_raw)
    assert not e
    ref, e2 = OP.prefill(want_q, cu, want_pool, bt, np.array(lens), SCALE)
    assert not e2
    dev = cuda_device
    pool = to_dev_bf16(pool0, dev)
    qr = torch.empty(T, 32, 64, dtype=torch.bfloat16, device=dev)
    btd = to_dev_i32(bt, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.kv_append_rope(to_dev_bf16(k, dev), to_dev_bf16(v, dev), to_dev_i32(pos, dev), btd, pool,
                       cos_d, sin_d, token_seq=to_dev_i32(seqs, dev), q_in=to_dev_bf16(q_raw, dev),
                       q_out=qr, d_err=err)
    out = torch.empty_like(qr)
    lib.paged_gqa_prefill(qr, to_dev_i32(cu, dev), pool, btd, to_dev_i32(lens, dev), out, SCALE,
                          d_err=err, compute=compute)
    assert lib.pkv_read_device_error(err) == 0
    assert np.array_equal(bits(pool), want_pool)
    check_close(bf16_to_f64(out), ref, "append then prefill")


@pytest.mark.parametrize("compute", COMPUTE)
@pytest.mark.parametrize("n", [2048, 1920])
def test_prefill_full_prompt_sampled(lib, cuda_device, n, compute):
    """A whole prompt of n tokens; sampled rows against the oracle's definition
    for that position (the row of position p is the one-query chunk of the
    first p + 1 tokens)."""
    lens, q_lens = [n, 333], [n, 100]
    pool, bt, q, cu = make_case(300 + n, lens, q_lens)
    out, code = run_prefill(lib, cuda_device, q, cu, pool, bt, lens, compute=compute)
    assert code == 0
    got = bf16_to_f64(out)
    rows = [0, 1, 15, 16, 17, 255, 1000, n // 2, n - 17, n - 1]
    for p in rows:
        ref, e = OP.prefill(q[p:p + 1], np.array([0, 1], np.int32), pool, bt[:1],
                            np.array([p + 1]), SCALE)
        assert not e
        check_close(got[p:p + 1], ref, f"prompt {n} position {p}")
    # the chunk of the second sequence: positions 233 .. 332
    ref2, _ = OP.prefill(q[n:], cu[1:] - n, pool, bt[1:], np.array([333]), SCALE)
    check_close(got[n:], ref2, "chunk after a prefix")


@pytest.mark.parametrize("compute", COMPUTE)
def test_prefill_error_contract(lib, cuda_device, compute):
    lens, q_lens = [40, 20, 30, 25], [40, 25, 10, 5]     # seq 1: q_len > n
    pool, bt, q, cu = make_case(400, lens, q_lens)
    bt[2, 1] = pool.shape[0] + 9                          # seq 2: a bad needed page
    out, code = run_prefill(lib, cuda_device, q, cu, pool, bt, lens, out_fill=0x1234, compute=compute)
    assert code == lib.ERR_DEVICE_INDEX
    ref, err = OP.prefill(q, cu, pool, bt, np.array(lens), SCALE)
    assert err
    got = bf16_to_f64(out)
    check_close(got[cu[0]:cu[1]], ref[cu[0]:cu[1]], "good sequence next to bad ones")
    check_close(got[cu[3]:cu[4]], ref[cu[3]:cu[4]], "good sequence after bad ones")
    assert np.all(got[cu[1]:cu[3]] == 0)
    # a grid bound below a q_len: that sequence's rows are zero, others unaffected
    out2, code2 = run_prefill(lib, cuda_device, q[:40], cu[:2], pool, bt[:1], lens[:1],
                              max_q_len=32, out_fill=0x1234, compute=compute)
    assert code2 == lib.ERR_DEVICE_INDEX and np.all(bf16_to_f64(out2) == 0)
    # row offsets outside [0, T): nothing is written
    bad_cu = np.array([0, 40, 90], np.int32)              # T is 70
    out3, code3 = run_prefill(lib, cuda_device, q[:70], bad_cu, pool, bt[:2], [40, 50],
                              out_fill=0x1234, compute=compute)
    assert code3 == lib.ERR_DEVICE_INDEX
    assert np.all(bits(out3)[40:] == 0x1234)


@pytest.mark.parametrize("compute", COMPUTE)
def test_prefill_deterministic(lib, cuda_device, compute):
    lens, q_lens = [500, 90], [500, 60]
    pool, bt, q, cu = make_case(500, lens, q_lens)
    a, _ = run_prefill(lib, cuda_device, q, cu, pool, bt, lens, compute=compute)
    b, _ = run_prefill(lib, cuda_device, q, cu, pool, bt, lens, compute=compute)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
