"""GPU next-token argmax (pkv_argmax_f32) against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

from oracle import argmax as OA

pytestmark = pytest.mark.gpu
VOCAB = 128256  # Llama-3.2 vocabulary


@pytest.fixture(scope="module")
def lib(cuda_device):
    from paged_kv_gqa_append_gb300 import build
    build.build()
    import paged_kv_gqa_append_gb300 as m
    return m


def logits_with_specials(seed, rows, vocab):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, vocab)).astype(np.float32) * 4
    for r in range(rows):
        kind = r % 6
        if kind == 1:      # the maximum repeated at several positions
            m = x[r].max()
            x[r, rng.choice(vocab, size=min(3, vocab), replace=False)] = m
        elif kind == 2:    # NaNs sprinkled in, one of them at the front
            x[r, rng.choice(vocab, size=max(1, vocab // 7), replace=False)] = np.nan
            x[r, 0] = np.nan
        elif kind == 3:    # +inf twice
            x[r, rng.choice(vocab, size=min(2, vocab), replace=False)] = np.inf
        elif kind == 4:    # only -inf and NaN
            x[r] = -np.inf
            x[r, ::3] = np.nan
        elif kind == 5 and r % 12 == 5:
            x[r] = np.nan  # all NaN
    return x


@pytest.mark.parametrize("rows,vocab", [(1, VOCAB), (32, VOCAB), (257, 1000), (5, 3), (13, 7)])
def test_argmax_matches_oracle(lib, cuda_device, rows, vocab):
    x = logits_with_specials(rows * 7 + vocab, rows, vocab)
    got = lib.argmax_rows(torch.from_numpy(x).to(cuda_device)).cpu().numpy()
    assert np.array_equal(got, OA.argmax_rows(x))


def test_argmax_strided_unaligned_rows(lib, cuda_device):
    rows, vocab = 37, 1001
    buf = logits_with_specials(99, rows, vocab + 5)
    x = torch.from_numpy(buf).to(cuda_device)[:, :vocab]     # row stride 1006 floats
    got = lib.argmax_rows(x).cpu().numpy()
    assert np.array_equal(got, OA.argmax_rows(buf[:, :vocab]))
