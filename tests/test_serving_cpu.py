"""ContinuousBatcher's host logic on the CPU: admission by page credit, page
growth, block-table rows, the batch's table gather, token positions and
retirement.  The scheduler is the library's own C++ scheduler; the kernel
calls are replaced by oracle-backed stand-ins that also check the host-side
contract (int32 contiguous tables, max_seq_len bounding the lengths).  Each
run must take the oracle scheduler's decisions step for step, give the
oracle's outputs at every step and leave the pool equal to the oracle's bit
for bit, on bf16 and INT8 pages, fused and two-call steps, continuous and
static batching.
"""
import dataclasses

import pytest
import torch

from paged_kv_gqa_append_gb300 import build as B

B.build()  # no-op when libpkv.so is up to date
import paged_kv_gqa_append_gb300 as pkv  # noqa: E402
import workloads as W  # noqa: E402
from oracle import rope as OR  # noqa: E402
from tests import _fake_kernels as FK  # noqa: E402
from tests._mix import run_mix  # noqa: E402

DEV = torch.device("cpu")


@pytest.fixture
def serving_on_oracle(monkeypatch):
    FK.patch_serving(monkeypatch)
    from paged_kv_gqa_append_gb300.serving import ContinuousBatcher
    return ContinuousBatcher


def rope_tables():
    c, s = OR.table(OR.inv_freq_llama3(), W.MAX_CONTEXT)
    return torch.from_numpy(c), torch.from_numpy(s)


def small_mix(requests=6, pages=16):
    """Short prompts, 12 decode steps, 2 layers, and a pool that holds at most
    four short requests at a time, so requests queue (the longest waits for
    the whole pool), overlap and cross pages."""
    case = W.case_continuous(seed=11, requests=requests, mean_prompt=30.0, decode_steps=12,
                             num_layers=2)
    return dataclasses.replace(case, num_pages=pages)


@pytest.mark.parametrize("fused,static,int8", [
    (True, False, False), (False, False, False), (True, True, False),
    (True, False, True), (False, False, True)])
def test_batcher_matches_the_oracle_step_for_step(serving_on_oracle, fused, static, int8):
    case = small_mix()
    cos, sin = rope_tables()
    steps = run_mix(pkv, DEV, case, fused, cos, sin, static=static, int8=int8,
                    sample_every=1, sample_layers=(0, 1))
    assert steps > case.decode_steps                 # requests really queued
    assert steps < len(case.prompt_lens) * case.decode_steps or static


def test_prepare_and_launch_step_are_one_step(serving_on_oracle):
    # prepare_step advances the scheduler; launch_step takes [L, B, ...]
    # tensors and rejects any other shape before launching anything
    ContinuousBatcher = serving_on_oracle
    case = small_mix(requests=2, pages=32)
    cos, sin = rope_tables()
    pool = torch.zeros((case.num_pages, 2, 8, 16, 64), dtype=torch.bfloat16)
    cb = ContinuousBatcher(pool, case.num_layers, cos, sin, W.DEFAULT_SCALE, max_slots=4)
    for p in case.prompt_lens:
        assert cb.submit(int(p), case.allowed_new_tokens) >= 0
    src = lambda rid, l: W.request_kv(case.seed, rid, l, 0, cb.prompt[rid])
    assert cb.admit(src) == [0, 1]
    batch = cb.prepare_step()
    L, B = case.num_layers, 2
    assert batch.ids == [0, 1]
    assert list(batch.lens_h) == [int(p) + 1 for p in case.prompt_lens]
    # the packed host block: the lengths, then tables [L, B, P] padded with -1
    P = -(-int(batch.lens_h.max()) // W.PAGE_TOKENS)
    host = batch.host_block
    assert host.view(torch.int32)[:B].tolist() == list(batch.lens_h)
    off = (4 * B + 15) // 16 * 16
    tab = host[off:off + 4 * L * B * P].view(torch.int32).view(L, B, P)
    assert tuple(batch.tables.shape) == (L, B, P)
    for l in range(L):
        for b, rid in enumerate(batch.ids):
            row, _ = cb.sched.block_table(rid, l)
            assert tab[l, b].tolist() == list(row[:P])
    q = torch.zeros((L, 2, 32, 64), dtype=torch.bfloat16)
    kv = torch.zeros((L, 2, 8, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        cb.launch_step(batch, q[:, :1], kv, kv)
    with pytest.raises(ValueError):
        cb.launch_step(batch, q, kv[:1], kv)
    out = cb.launch_step(batch, q, kv, kv)
    assert tuple(out.shape) == (L, 2, 32, 64)
    assert cb.error() == 0
    # launch_step copied the block: the device views now hold it
    assert torch.equal(batch.tables.cpu(), tab) and batch.lens.tolist() == list(batch.lens_h)
    assert cb.uploaded_bytes > 0


def test_oversize_request_is_rejected(serving_on_oracle):
    ContinuousBatcher = serving_on_oracle
    cos, sin = rope_tables()
    pool = torch.zeros((8, 2, 8, 16, 64), dtype=torch.bfloat16)
    cb = ContinuousBatcher(pool, 2, cos, sin, W.DEFAULT_SCALE, max_slots=4)
    # 2 layers x ceil((64 + 33 - 1) / 16) = 12 pages > 8
    assert cb.submit(64, 33) == -1
    assert cb.rejected == [(64, 33)]
    assert cb.submit(16, 17) >= 0          # 2 x 2 pages fits
    with pytest.raises(pkv.PkvError):
        cb.submit(0, 5)                    # no prompt token
    assert list(cb.prompt) == [0]
