"""The allocation-free decode entry point, checked against the regular one.

paged_gqa_decode_noalloc serves callers that cannot allocate device memory
(for example a plug-in inside a host program that owns the device-memory
budget, or a serving loop that may not allocate after start-up): it takes no
workspace and uses a fixed array inside the library instead.  It runs the
same deterministic kernel as paged_gqa_decode, so its output must equal the
regular call's bit for bit; one case is also checked against the FP64
oracle.  This file is named so that pytest collects it last; it must pass on
its own in a fresh process as well as after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from oracle import paged_kv as OP
from tests._util import bf16_to_f64, check_close

pytestmark = pytest.mark.gpu

NOALLOC_BYTES = 4 * 1024 * 1024    # PKV_NOALLOC_WORKSPACE_BYTES in include/pkv.h
WORKSPACE_TOO_SMALL = 4


@pytest.fixture(scope="module")
def lib(cuda_device):
    from paged_kv_gqa_append_gb300 import build
    build.build()
    import paged_kv_gqa_append_gb300 as m
    return m


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _case(lens, seed):
    lens = np.asarray(lens, np.int32)
    rng = np.random.default_rng(seed)
    need = int(sum((int(n) + 15) // 16 for n in lens))
    N = need + 9
    perm = rng.permutation(N).astype(np.int32)
    bt = np.full((len(lens), 128), -1, np.int32)
    cur = 0
    for s, n in enumerate(lens):
        k = (int(n) + 15) // 16
        bt[s, :k] = perm[cur:cur + k]
        cur += k
    return W.DecodeCase("noalloc", seed, 1, lens, N, bt[None])


def _noalloc(lib, q, pool, bt, lens, out, num_seqs, max_seq_len, scale, err):
    return lib.lib.paged_gqa_decode_noalloc(
        _ptr(q), _ptr(pool), pool.shape[0], _ptr(bt), bt.shape[1], bt.shape[1], _ptr(lens),
        num_seqs, max_seq_len, _ptr(out), ctypes.c_float(scale), _ptr(err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _run_both(lib, dev, case, oracle=False):
    pool = W.fill_pool(case, device=dev)
    q = W.fill_queries(case, device=dev)[0].contiguous()
    bt = torch.from_numpy(case.block_tables[0]).to(dev)
    lens = torch.from_numpy(case.seq_lens).to(dev)
    ref = torch.empty_like(q)
    lib.paged_gqa_decode(q, pool, bt, lens, ref, case.scale, max_seq_len=case.max_seq_len)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = []
    for _ in range(2):                      # two calls in a row share the static workspace
        out = torch.full_like(q, float("nan"))
        st = _noalloc(lib, q, pool, bt, lens, out, case.num_seqs, case.max_seq_len, case.scale, err)
        assert st == 0, lib.lib.pkv_last_error()
        outs.append(out)
    assert lib.pkv_read_device_error(err) == 0
    for out in outs:                        # the same kernel on the same inputs: bit-identical
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    if oracle:
        want, _ = OP.decode(W.bf16_bits(q), W.bf16_bits(pool), case.block_tables[0],
                            case.seq_lens, case.scale)
        check_close(bf16_to_f64(outs[1]), want, "noalloc vs oracle")


def _largest_batch(lib):
    n = 1
    while lib.paged_gqa_decode_workspace_bytes(n + 1) <= NOALLOC_BYTES:
        n += 1
    return n


def test_noalloc_matches_regular_entry_point(lib, cuda_device):
    # lengths that split sequences across many CTAs and leave some empty
    _run_both(lib, cuda_device, _case([2048, 1, 0, 700, 17, 1500, 2047, 129], seed=71), oracle=True)
    # a second, larger batch reusing the same static array
    _run_both(lib, cuda_device, W.case_mixed(seed=72, batch=8))


def test_noalloc_largest_batch_that_fits(lib, cuda_device):
    n = _largest_batch(lib)
    assert lib.paged_gqa_decode_workspace_bytes(n) <= NOALLOC_BYTES
    lens = np.random.default_rng(73).integers(0, 49, size=n).astype(np.int32)
    _run_both(lib, cuda_device, _case(lens, seed=73))


def test_noalloc_rejects_batches_beyond_its_array(lib, cuda_device):
    dev = cuda_device
    n = _largest_batch(lib) + 1
    assert lib.paged_gqa_decode_workspace_bytes(n) > NOALLOC_BYTES
    # real buffers of the right sizes (zero lengths): nothing may be launched,
    # and nothing launched could read or write outside them
    q = torch.zeros(n, 32, 64, dtype=torch.bfloat16, device=dev)
    out = torch.full_like(q, float("nan"))
    pool = torch.zeros(8, 2, 8, 16, 64, dtype=torch.bfloat16, device=dev)
    bt = torch.full((n, 128), -1, dtype=torch.int32, device=dev)
    lens = torch.zeros(n, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    st = _noalloc(lib, q, pool, bt, lens, out, n, 16, 0.125, err)
    assert st == WORKSPACE_TOO_SMALL
    assert b"static workspace" in lib.lib.pkv_last_error()
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()   # untouched: the call launched nothing
