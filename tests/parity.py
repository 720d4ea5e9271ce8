"""Comparison helpers for the parity tests: BF16 bit patterns, ordered-integer
ULP distance, and the gate (every element within 1 BF16 ulp of the oracle and
at least 99.99% of elements bit-identical)."""
from __future__ import annotations

import numpy as np

MAX_ULP = 1
MIN_IDENTICAL = 0.9999


def bits(t) -> np.ndarray:
    """uint16 bit patterns of a bf16 torch tensor (any device) or a uint16 array."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    except ImportError:
        pass
    return np.asarray(t, dtype=np.uint16)


def _ordered(u: np.ndarray) -> np.ndarray:
    u = u.astype(np.int32)
    mag = u & 0x7FFF
    return np.where(u & 0x8000, -mag, mag)


def _is_nan(u: np.ndarray) -> np.ndarray:
    return ((u & 0x7F80) == 0x7F80) & ((u & 0x7F) != 0)


def ulp_distance(a, b) -> np.ndarray:
    a, b = bits(a), bits(b)
    d = np.abs(_ordered(a) - _ordered(b)).astype(np.int64)
    na, nb = _is_nan(a), _is_nan(b)
    d[na & nb] = 0
    d[na ^ nb] = 1 << 30
    return d


def compare(got, want) -> dict:
    d = ulp_distance(got, want)
    n = d.size
    same = int(np.count_nonzero(d == 0))
    return {"elements": n, "identical": same, "frac_identical": same / n if n else 1.0,
            "max_ulp": int(d.max()) if n else 0}


def assert_parity(got, want, label: str = "") -> dict:
    st = compare(got, want)
    assert st["max_ulp"] <= MAX_ULP, f"{label}: max ulp {st['max_ulp']} ({st})"
    assert st["frac_identical"] >= MIN_IDENTICAL, f"{label}: {st}"
    return st
