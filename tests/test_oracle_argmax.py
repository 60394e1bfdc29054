"""Pins for the oracle's next-token argmax: a plain loop with the stated tie
and NaN rules on small rows, and hand-written special cases."""
import numpy as np

from oracle import argmax as A


def loop_argmax(row):
    """Scan left to right, keep the first strictly larger non-NaN value."""
    best_i, best_v = 0, None
    for i, v in enumerate(row):
        if np.isnan(v):
            continue
        if best_v is None or v > best_v:
            best_i, best_v = i, v
    return best_i


def test_matches_a_plain_scan_on_random_rows():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((50, 37)).astype(np.float32)
    x[:, ::5] = np.round(x[:, ::5])          # plenty of ties among rounded values
    x[3, :] = 1.0                             # a whole row of ties
    x[7, 10] = np.nan
    got = A.argmax_rows(x)
    assert got.dtype == np.int32
    assert list(got) == [loop_argmax(r) for r in x]


def test_hand_cases():
    nan, inf = np.float32(np.nan), np.float32(np.inf)
    rows = np.array([
        [0.0, 2.0, 2.0, 1.0],        # tie -> lowest index
        [nan, 1.0, nan, 0.5],        # NaN never wins
        [-inf, -inf, -inf, -inf],    # all -inf -> 0
        [nan, nan, nan, nan],        # all NaN -> 0
        [nan, -inf, nan, -inf],      # -inf beats NaN -> 1
        [1.0, inf, inf, 3.0],        # +inf wins, first one
    ], dtype=np.float32)
    assert list(A.argmax_rows(rows)) == [1, 1, 0, 0, 1, 1]
