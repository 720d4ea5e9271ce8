"""The router kernel's correctly rounded sigmoid, restated step for step in C
(tests/router_sigmoid_method.c: a float-pair phase accepted by Ziv's rounding
test, a double-double phase for the rest), must give the oracle's correctly
rounded sigmoid bit for bit.

Every step of the kernel's method is a correctly rounded IEEE operation, so
the restatement reproduces the kernel's bits on the CPU. By default this
checks 1/64 of all 2^32 float inputs (every 64th block of 2^24 bit patterns),
every float with at most 8 significant bits, and the family z = m * 2^-23 near
0 whose sigmoid sits next to a rounding midpoint; with BEAM_EXHAUSTIVE=1 it
checks all 2^32 inputs (a few minutes on 8 cores). The GPU test
test_router_sigmoid_every_float_matches_the_oracle runs the kernel itself on
all of them."""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
CHUNK = 1 << 24
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def method(tmp_path_factory):
    so = tmp_path_factory.mktemp("sig") / "libsigmethod.so"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11",
                    os.path.join(HERE, "router_sigmoid_method.c"), "-o", str(so), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    lib.method_sigmoid_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int64]
    lib.method_sigmoid_range.argtypes = [ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int64]
    return lib


def _compare(z: np.ndarray, s: np.ndarray, o: np.ndarray) -> np.ndarray:
    """indices where the method and the oracle differ (NaN inputs: both NaN)"""
    nan = np.isnan(z)
    bad = (s.view(np.uint32) != o.view(np.uint32)) & ~nan
    bad |= nan & ~np.isnan(s)
    return np.nonzero(bad)[0]


def _check_chunk(method, olib, lo: int):
    s = np.empty(CHUNK, np.float32)
    ph = np.empty(CHUNK, np.uint8)
    method.method_sigmoid_range(lo, s.ctypes.data, ph.ctypes.data, CHUNK)
    z = (np.arange(CHUNK, dtype=np.uint64) + lo).astype(np.uint32).view(np.float32)
    o = np.empty(CHUNK, np.float32)
    olib.oracle_sigmoid_array(z.ctypes.data, o.ctypes.data, CHUNK)
    bad = _compare(z, s, o)
    return (bad[:5] + lo).tolist(), int((ph == 2).sum())


def _check_values(method, z: np.ndarray):
    z = np.ascontiguousarray(z, np.float32)
    s = np.empty_like(z)
    ph = np.empty(z.size, np.uint8)
    method.method_sigmoid_array(z.ctypes.data, s.ctypes.data, ph.ctypes.data, z.size)
    o = oracle.sigmoid_array(z, threads=THREADS)
    bad = _compare(z, s, o)
    return z[bad[:5]], int((ph == 2).sum())


def test_blocks_of_bit_patterns_match_the_oracle(method):
    olib = oracle._load()
    step = 1 if os.environ.get("BEAM_EXHAUSTIVE") == "1" else 64
    with ThreadPoolExecutor(THREADS) as ex:
        res = list(ex.map(lambda c: _check_chunk(method, olib, c * CHUNK), range(0, 256, step)))
    bad = [hex(b) for r in res for b in r[0]]
    assert not bad, f"method differs from the oracle at bit patterns {bad[:10]}"
    assert sum(r[1] for r in res) > 0  # the double-double phase was exercised
    assert oracle.sigmoid_undecided() == 0


def test_short_floats_and_the_near_midpoint_family_match_the_oracle(method):
    # every float with at most 8 significant bits, both signs, every exponent
    e = np.arange(256, dtype=np.uint32) << 23
    m = np.arange(256, dtype=np.uint32) << 15
    short = (e[:, None] | m[None, :]).ravel()
    short = np.concatenate([short, short | 0x80000000]).view(np.float32)
    # z = +-m 2^-23 (and 2^-24): 1/2 + z/4 is a float or a midpoint, and the
    # sigmoid lies within z^3/48 of it
    fam = np.arange(1, 1 << 18, dtype=np.float64)
    near = np.concatenate([fam * 2.0 ** -23, -fam * 2.0 ** -24, -fam * 2.0 ** -23,
                           fam * 2.0 ** -24]).astype(np.float32)
    z = np.concatenate([short, near])
    bad, phase2 = _check_values(method, z)
    assert bad.size == 0, f"method differs from the oracle at {[float(v).hex() for v in bad]}"
    assert phase2 > 1000  # these inputs lean on the double-double phase
    assert oracle.sigmoid_undecided() == 0
