"""Next-token selection: argmax over FP32 logits (oracle; test infrastructure only).

From the samir-vllm article, "Architecture et flux d'inference": the final
logits are produced in FP32 and a GPU argmax selects the next token.

Readings where the article is silent (the CUDA kernel follows the same rule):
  * the result is the smallest index of the row's largest value (ties go to
    the lowest token id);
  * a NaN never wins: it orders below every number, -inf included; the
    result is the first index holding the row's largest non-NaN value, and
    0 when every value of the row is NaN.
"""
from __future__ import annotations

import numpy as np


def argmax_rows(logits: np.ndarray) -> np.ndarray:
    """logits: float32 [rows][vocab] -> int32 [rows] token ids."""
    x = np.asarray(logits, dtype=np.float32)
    rows, vocab = x.shape
    out = np.zeros(rows, dtype=np.int32)
    for r in range(rows):
        finite = ~np.isnan(x[r])
        if not finite.any():
            continue
        best = x[r][finite].max()
        out[r] = int(np.flatnonzero(finite & (x[r] == best))[0])
    return out
