"""The SSMax scale g = RN32((1 + (pos+1)/2048)^0.1) in the Q/K kernel comes
from an FP32 estimate and a test of the lower midpoints of the 16 candidates
around it: the correctly rounded value is the largest candidate whose lower
midpoint's 10th power (four double products) is at most u = (2049 + pos)/2048.
This emulates that selection with IEEE double arithmetic in numpy, with the
estimate deliberately off by up to 4 ulps, and requires the oracle's
correctly rounded scale at every position below 2^20."""
from __future__ import annotations

import numpy as np
import pytest

import oracle


def _select(u: np.ndarray, est: np.ndarray) -> np.ndarray:
    bits = est.view(np.uint32).astype(np.int64)
    best = np.full(u.shape, -1)
    for k in range(16):
        f = (bits + (k - 8)).astype(np.uint32).view(np.float32).astype(np.float64)
        prev = (bits + (k - 9)).astype(np.uint32).view(np.float32).astype(np.float64)
        mid = 0.5 * (f + prev)
        m2 = mid * mid
        m4 = m2 * m2
        m8 = m4 * m4
        best = np.where(m8 * m2 <= u.astype(np.float64), k, best)
    assert (best >= 0).all() and (best < 15).all()
    return (bits + best - 8).astype(np.uint32).view(np.float32)


@pytest.fixture(scope="module")
def reference():
    p = np.arange(1 << 20, dtype=np.int64)
    return p, np.array([oracle.ssmax_scale(int(x)) for x in p], np.float32)


@pytest.mark.parametrize("offset", [-4, -1, 0, 3, 4])
def test_midpoint_selection_is_correctly_rounded_at_every_position(reference, offset):
    p, want = reference
    u = ((2049 + p).astype(np.float32) / np.float32(2048.0)).astype(np.float32)
    assert np.all(u.astype(np.float64) == (2049 + p) / 2048.0)  # u is exact in FP32
    est = np.exp2(np.float32(0.1) * np.log2(u)).astype(np.float32)
    est = (est.view(np.uint32).astype(np.int64) + offset).astype(np.uint32).view(np.float32)
    assert np.array_equal(_select(u, est), want)
