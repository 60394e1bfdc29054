"""Continuous-batching mix on the GPU, step for step against the oracle.

64 requests (prompts geometric, mean 300, clipped to [1, 1920]) run 128
decode steps each on 16 layers in a 128 MiB pool, admitted by the
admission-credit rule.  The C++ scheduler (driving the kernels) and the
oracle's scheduler must take identical decisions; every decode output of
layers 0 and 15 at every 16th step must match the FP64 oracle; the final pool
must equal the oracle's bit for bit.  The same run is made with the fused
decode step and with kv_append_rope followed by paged_gqa_decode, and on INT8
pages (the oracle's INT8 append and decode).
"""
import pytest

import workloads as W
from tests._mix import run_mix

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib(cuda_device):
    from paged_kv_gqa_append_gb300 import build
    build.build()
    import paged_kv_gqa_append_gb300 as m
    return m


@pytest.mark.parametrize("fused,static", [(True, False), (False, False), (True, True)])
def test_continuous_batching_mix_matches_oracle(lib, cuda_device, fused, static):
    # the full 64-request mix on the fused step; the two-call path and static
    # batching on its first 16 requests (same scheduler, same pool size)
    case = W.case_continuous() if fused and not static else W.case_continuous(requests=16)
    cos_d, sin_d = lib.rope_tables_device(cuda_device, W.MAX_CONTEXT)
    steps = run_mix(lib, cuda_device, case, fused, cos_d, sin_d, static)
    assert steps > case.decode_steps          # requests really overlapped in time


@pytest.mark.parametrize("fused", [True, False])
def test_continuous_batching_mix_int8_pages(lib, cuda_device, fused):
    # the first 16 requests of the mix on INT8 pages (same scheduler, same
    # page count): pages bit-exact at the end, outputs sampled as above
    case = W.case_continuous(requests=16)
    cos_d, sin_d = lib.rope_tables_device(cuda_device, W.MAX_CONTEXT)
    steps = run_mix(lib, cuda_device, case, fused, cos_d, sin_d, int8=True)
    assert steps > case.decode_steps


@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("staged", [False, True])
def test_native_layers_call_equals_per_layer_calls(lib, cuda_device, int8, staged):
    # paged_gqa_decode_append_layers (one C call, early staging on layers >= 1,
    # optionally after one copy of a packed step block) against L calls of the
    # per-layer entry point on copies of the same pool: pools, rotated q and
    # outputs bit for bit
    import numpy as np
    import torch
    dev = cuda_device
    L, S = 4, 6
    lens = np.array([1, 17, 300, 2048, 129, 64], np.int32)
    per = [(int(n) + 15) // 16 for n in lens]
    rng = np.random.default_rng(91)
    num_pages = L * sum(per) + 7
    perm = rng.permutation(num_pages).astype(np.int32)
    tab = np.full((L, S, 128), -1, np.int32)
    cur = 0
    for l in range(L):
        for s in range(S):
            tab[l, s, :per[s]] = perm[cur:cur + per[s]]
            cur += per[s]
    gen = W.cpu_gen(92)
    q = W.normal_bf16((L, S, 32, 64), gen).to(dev)
    k = W.normal_bf16((L, S, 8, 64), gen).to(dev)
    v = W.normal_bf16((L, S, 8, 64), gen).to(dev)
    if int8:
        pool0 = lib.new_int8_pool(num_pages, dev)
        pool0.copy_(torch.from_numpy(rng.integers(-127, 128, pool0.shape, dtype=np.int8).view(np.uint8)))
        blocks = pool0.view(num_pages, 8, W.I8_BLOCK_BYTES)
        scales = torch.from_numpy(rng.uniform(0.005, 0.03, (num_pages, 8, 32)).astype(np.float32))
        blocks[:, :, 2048:].copy_(scales.view(torch.uint8).view(num_pages, 8, 128).to(dev))
    else:
        pool0 = W.normal_bf16((num_pages, 2, 8, 16, 64), gen).to(dev)
    cos_d, sin_d = lib.rope_tables_device(dev, W.MAX_CONTEXT)
    ws = lib.alloc_workspace(S, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lens_d, tab_d = torch.from_numpy(lens).to(dev), torch.from_numpy(tab).to(dev)
    per_layer = lib.paged_gqa_decode_append_int8 if int8 else lib.paged_gqa_decode_append
    pool_a, out_a, qr_a = pool0.clone(), torch.empty_like(q), torch.empty_like(q)
    for l in range(L):
        per_layer(q[l], k[l], v[l], pool_a, tab_d[l], lens_d, out_a[l], cos_d, sin_d, 0.125,
                  q_out=qr_a[l], workspace=ws, max_seq_len=2048, d_err=err)
    pool_b, out_b, qr_b = pool0.clone(), torch.empty_like(q), torch.empty_like(q)
    kw = {}
    if staged:      # the tables and lengths reach the device with the call
        off = (4 * S + 15) // 16 * 16
        host = torch.zeros(off + tab.nbytes, dtype=torch.uint8).pin_memory()
        host[:4 * S].copy_(torch.from_numpy(lens.view(np.uint8)))
        host[off:].copy_(torch.from_numpy(tab.reshape(-1).view(np.uint8)))
        block = torch.zeros(host.numel(), dtype=torch.uint8, device=dev)
        lens_d = block[:4 * S].view(torch.int32)
        tab_d = block[off:].view(torch.int32).view(L, S, 128)
        kw = dict(host_stage=host, dev_stage=block)
    lib.paged_gqa_decode_append_layers(q, k, v, pool_b, tab_d, lens_d, out_b, cos_d, sin_d, 0.125,
                                       ws, max_seq_len=2048, d_err=err, q_out=qr_b, **kw)
    assert lib.pkv_read_device_error(err) == 0
    assert torch.equal(pool_a, pool_b)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(qr_a.view(torch.int16), qr_b.view(torch.int16))


@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("src_host", [False, True])
def test_layered_prompt_append_equals_per_layer_calls(lib, cuda_device, int8, src_host):
    # kv_append_rope_layers (one C call: per layer a copy of host rows into the
    # stage, then the append) with the batcher's one-row table view, against L
    # kv_append_rope(_int8) calls through the full table on a copy of the same
    # pool: the pools bit for bit, and no error
    import numpy as np
    import torch
    dev = cuda_device
    L, slots, P = 5, 6, 300
    npg = (P + 15) // 16
    rng = np.random.default_rng(93)
    num_pages = L * npg + 11
    perm = rng.permutation(num_pages).astype(np.int32)
    slot = 4
    tab = np.full((L, slots, 128), -1, np.int32)
    for l in range(L):
        tab[l, slot, :npg] = perm[l * npg:(l + 1) * npg]
    gen = W.cpu_gen(94)
    k = W.normal_bf16((L, P, 8, 64), gen)
    v = W.normal_bf16((L, P, 8, 64), gen)
    if int8:
        pool0 = lib.new_int8_pool(num_pages, dev)
    else:
        pool0 = W.normal_bf16((num_pages, 2, 8, 16, 64), gen).to(dev)
    cos_d, sin_d = lib.rope_tables_device(dev, W.MAX_CONTEXT)
    tab_d = torch.from_numpy(tab).to(dev)
    pos = torch.arange(P, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    per_layer = lib.kv_append_rope_int8 if int8 else lib.kv_append_rope
    pool_a = pool0.clone()
    rows = torch.full((P,), slot, dtype=torch.int32, device=dev)
    kd, vd = k.to(dev), v.to(dev)
    for l in range(L):
        per_layer(kd[l], vd[l], pos, tab_d[l], pool_a, cos_d, sin_d, token_seq=rows, d_err=err)
    pool_b = pool0.clone()
    if src_host:
        ks = [k[l].pin_memory() for l in range(L)]
        vs = [v[l].pin_memory() for l in range(L)]
        stage = torch.empty(2 * P * 1024, dtype=torch.uint8, device=dev)
    else:
        ks, vs, stage = [kd[l] for l in range(L)], [vd[l] for l in range(L)], None
    lib.kv_append_rope_layers(ks, vs, pos, tab_d[:, slot:slot + 1], pool_b, cos_d, sin_d,
                              token_seq=torch.zeros(P, dtype=torch.int32, device=dev), stage=stage,
                              d_err=err)
    torch.cuda.synchronize()
    assert lib.pkv_read_device_error(err) == 0
    assert torch.equal(pool_a.view(torch.uint8), pool_b.view(torch.uint8))
    assert not torch.equal(pool_a.view(torch.uint8), pool0.view(torch.uint8))
