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
