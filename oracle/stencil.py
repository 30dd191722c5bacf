"""Window sum (cooperative fetch + stencil) on the CPU.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

MLC course "Ep7: GPU and Hardware Acceleration", section "Window Sum
Example": B[i] = A[i] + A[i+1] + A[i+2] for float32 A of n + 2 elements and B
of n elements (the page's program uses n = 1024).  Generalised to a window of
w terms, B[i] = sum_{k < w} A[i + k].  Reading of the page: the terms are
added left to right in float32, ((A[i] + A[i+1]) + A[i+2]), exactly as the
expression is written; no reassociation, no wider accumulator.
"""
from __future__ import annotations

import numpy as np


def window_sum_f32(a: np.ndarray, n_out: int, window: int = 3) -> np.ndarray:
    """b[i] = a[i] + a[i+1] + ... + a[i+window-1], float32, left to right."""
    a = np.asarray(a, dtype=np.float32)
    if window < 1 or a.size < n_out + window - 1:
        raise ValueError("a holds %d elements, needs %d" % (a.size, n_out + window - 1))
    acc = a[0:n_out].copy()
    for k in range(1, window):
        acc = (acc + a[k:k + n_out]).astype(np.float32)  # one float32 addition per term
    return acc
