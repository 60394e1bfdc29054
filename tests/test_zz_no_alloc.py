"""The allocation-free decode entry point, checked against the regular one.

paged_gqa_decode_noalloc serves callers that cannot allocate device memory
(for example a plug-in inside a host program that owns the device-memory
budget, or a serving loop that may not allocate after start-up): it takes no
workspace and uses a fixed array inside the library instead.  This file is
named so that pytest collects it last; it must pass on its own in a fresh
process as well as after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from tests._util import MAX_ABS_TOL, MEAN_ABS_TOL

pytestmark = pytest.mark.gpu


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


def _run_both(lib, dev, case):
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
        st = lib.lib.paged_gqa_decode_noalloc(
            _ptr(q), _ptr(pool), pool.shape[0], _ptr(bt), bt.shape[1], bt.shape[1], _ptr(lens),
            case.num_seqs, case.max_seq_len, _ptr(out), ctypes.c_float(case.scale), _ptr(err),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, lib.lib.pkv_last_error()
        outs.append(out)
    assert lib.pkv_read_device_error(err) == 0
    a = ref.float()
    for out in outs:
        d = (out.float() - a).abs()
        assert torch.isfinite(out.float()).all()
        assert d.max().item() <= MAX_ABS_TOL and d.mean().item() <= MEAN_ABS_TOL


def test_noalloc_matches_regular_entry_point(lib, cuda_device):
    # lengths that split sequences across many CTAs and leave some empty
    _run_both(lib, cuda_device, _case([2048, 1, 0, 700, 17, 1500, 2047, 129], seed=71))
    # a second, larger batch reusing the same static array
    _run_both(lib, cuda_device, W.case_mixed(seed=72, batch=8))


def test_noalloc_rejects_batches_beyond_its_array(lib, cuda_device):
    n = 4096
    need = lib.paged_gqa_decode_workspace_bytes(n)
    assert need > 4 * 1024 * 1024
    fake = ctypes.c_void_p(0x1000)
    st = lib.lib.paged_gqa_decode_noalloc(fake, fake, 8, fake, 128, 128, fake, n, 2048, fake,
                                          ctypes.c_float(0.125), None,
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 4   # PKV_ERR_WORKSPACE_TOO_SMALL, nothing launched
    assert b"static workspace" in lib.lib.pkv_last_error()
