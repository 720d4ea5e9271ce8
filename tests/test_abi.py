"""Host-only checks of the C ABI: the library builds, loads, exports every
function ``include/beam_boundary.h`` declares, and rejects bad arguments with
the documented status before touching CUDA (so these run without a GPU)."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

from sandwich_norm_residual_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "beam_boundary.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*BEAM_API\s+(?:const\s+)?\w+\s*\*?\s*(beam_\w+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for n in ("beam_boundary_fused", "beam_moe_combine_boundary", "beam_sync_status",
              "beam_status_string", "beam_version"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    # and nothing else of ours leaks out of the library
    ours = {n for n in exported if n.startswith("beam")}
    assert ours == set(declared_functions())
    assert set(_lib.SIGNATURES) == set(declared_functions())


def test_header_constants_match_binding():
    text = open(HEADER).read()
    enum = dict(re.findall(r"(BEAM_\w+)\s*=\s*(\d+)", text))
    for name, val in enum.items():
        assert getattr(_lib, name) == int(val), name
    assert _lib.BEAM_MAX_D == int(re.search(r"#define BEAM_MAX_D (\d+)", text).group(1))
    assert _lib.BEAM_MOE_TOPK == int(re.search(r"#define BEAM_MOE_TOPK (\d+)", text).group(1))
    assert ctypes.sizeof(_lib.LaunchOpts) == 32


def test_version_and_status_strings(lib):
    assert lib.beam_version() == 10000
    for s in range(0, 9):
        assert lib.beam_status_string(s)
    assert lib.beam_status_string(99) == b"unknown status"


# fake device addresses: never dereferenced, the calls fail validation first
A = 0x7F0000000000
D = 5120


def fused(lib, h=A, x=A + (1 << 32), pw=A + (2 << 32), qw=A + (3 << 32), n=2, eps=1e-6, T=4,
          d=D, y=A + (4 << 32)):
    return lib.beam_boundary_fused(None, h, x, pw, qw, n, eps, T, d, y)


def moe(lib, h=A, e=A + (1 << 32), w=A + (5 << 32), pw=A + (2 << 32), qw=A + (3 << 32), n=2,
        eps=1e-6, T=4, d=D, y=A + (4 << 32)):
    return lib.beam_moe_combine_boundary(None, h, e, w, pw, qw, n, eps, T, d, y)


@pytest.mark.parametrize("call", [fused, moe])
def test_shape_and_argument_errors(lib, call):
    assert call(lib, T=-1) == _lib.BEAM_ERR_SHAPE
    assert call(lib, d=0) == _lib.BEAM_ERR_SHAPE
    assert call(lib, d=12) == _lib.BEAM_ERR_SHAPE
    assert call(lib, d=_lib.BEAM_MAX_D + 8) == _lib.BEAM_ERR_SHAPE
    assert call(lib, n=0) == _lib.BEAM_ERR_ARG
    assert call(lib, eps=-1e-6) == _lib.BEAM_ERR_ARG
    assert call(lib, eps=float("nan")) == _lib.BEAM_ERR_ARG
    assert call(lib, eps=float("inf")) == _lib.BEAM_ERR_ARG
    # T = 0 is a no-op; pointers are not looked at
    assert call(lib, T=0, h=None, y=None) == _lib.BEAM_OK


def test_null_alignment_and_alias_errors_dense(lib):
    assert fused(lib, h=None) == _lib.BEAM_ERR_NULL
    assert fused(lib, x=None) == _lib.BEAM_ERR_NULL
    assert fused(lib, pw=None) == _lib.BEAM_ERR_NULL
    assert fused(lib, y=None) == _lib.BEAM_ERR_NULL
    assert fused(lib, h=A + 8) == _lib.BEAM_ERR_ALIGN
    assert fused(lib, qw=A + (3 << 32) + 2) == _lib.BEAM_ERR_ALIGN
    assert fused(lib, y=A) == _lib.BEAM_ERR_ALIAS                 # y over h
    assert fused(lib, y=A + (1 << 32) + 16) == _lib.BEAM_ERR_ALIAS  # y inside x
    assert fused(lib, x=A + 3 * D * 2) == _lib.BEAM_ERR_ALIAS       # x partly over h
    assert fused(lib, x=A + 4 * D * 2, y=A + (9 << 32)) != _lib.BEAM_ERR_ALIAS  # adjacent is fine
    assert fused(lib, pw=A + 64) == _lib.BEAM_ERR_ALIAS             # weight inside h


def test_null_alignment_and_alias_errors_moe(lib):
    assert moe(lib, e=None) == _lib.BEAM_ERR_NULL
    assert moe(lib, w=None) == _lib.BEAM_ERR_NULL
    assert moe(lib, w=A + (5 << 32) + 4) == _lib.BEAM_ERR_ALIGN
    assert moe(lib, y=A + (1 << 32) + 7 * D * 2 * 4) == _lib.BEAM_ERR_ALIAS  # y inside experts
    assert moe(lib, h=A + (1 << 32) + 16) == _lib.BEAM_ERR_ALIAS            # h inside experts
    assert moe(lib, y=A + (5 << 32)) == _lib.BEAM_ERR_ALIAS                 # y over weights


def test_bad_launch_options_are_rejected(lib):
    opts = _lib.LaunchOpts(flags=0x80)
    assert lib.beam_boundary_fused_ex(None, A, A + (1 << 32), A + (2 << 32), A + (3 << 32), 2,
                                      1e-6, 4, D, A + (4 << 32),
                                      ctypes.byref(opts)) == _lib.BEAM_ERR_ARG
    opts = _lib.LaunchOpts(vec_per_thread=9)
    assert lib.beam_boundary_fused_ex(None, A, A + (1 << 32), A + (2 << 32), A + (3 << 32), 2,
                                      1e-6, 4, D, A + (4 << 32),
                                      ctypes.byref(opts)) == _lib.BEAM_ERR_ARG
    # one vector per thread cannot cover D = 8192 with at most 512 threads
    opts = _lib.LaunchOpts(vec_per_thread=1)
    assert lib.beam_moe_combine_boundary_ex(None, A, A + (1 << 32), A + (5 << 32), A + (2 << 32),
                                            A + (3 << 32), 2, 1e-6, 4, 8192, A + (4 << 32),
                                            ctypes.byref(opts)) == _lib.BEAM_ERR_ARG


def _dense_ex(lib, **kw):
    opts = _lib.LaunchOpts(**kw)
    return lib.beam_boundary_fused_ex(None, A, A + (1 << 32), A + (2 << 32), A + (3 << 32), 2,
                                      1e-6, 4, D, A + (4 << 32), ctypes.byref(opts))


def test_bad_ring_options_are_rejected(lib):
    assert _dense_ex(lib, stages=1) == _lib.BEAM_ERR_ARG
    assert _dense_ex(lib, stages=9) == _lib.BEAM_ERR_ARG
    assert _dense_ex(lib, stages=-2) == _lib.BEAM_ERR_ARG
    assert _dense_ex(lib, prefetch_rows=9) == _lib.BEAM_ERR_ARG
    assert _dense_ex(lib, prefetch_rows=-2) == _lib.BEAM_ERR_ARG
    r = (ctypes.c_int32 * 3)(0, 1, 0)
    assert _dense_ex(lib, reserved=r) == _lib.BEAM_ERR_ARG
    # programmatic dependent launch is a valid option (the call then reaches CUDA)
    assert _dense_ex(lib, flags=_lib.BEAM_OPT_PDL) != _lib.BEAM_ERR_ARG
    # the wait test hook needs the ring kernel
    assert _dense_ex(lib, flags=_lib.BEAM_OPT_TEST_WAIT_TIMEOUT, stages=-1) == _lib.BEAM_ERR_ARG


def test_exact_count_rejects_null(lib):
    assert lib.beam_exact_sum_count(None, None, 0) == _lib.BEAM_ERR_NULL


def test_binding_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(ImportError, match="no CPU or PyTorch fallback"):
        _lib.load(str(tmp_path / "missing.so"))


def test_route_and_scaled_combine_argument_errors(lib):
    Z, Bi, I, W = A, A + (1 << 32), A + (2 << 32), A + (3 << 32)

    def route(T=4, E=256, ng=8, tg=4, k=8, sc=2.5, z=Z, b=Bi, i=I, w=W):
        return lib.beam_moe_route(None, z, b, T, E, ng, tg, k, sc, i, w)

    assert route(E=128) == _lib.BEAM_ERR_SHAPE
    assert route(T=-1) == _lib.BEAM_ERR_SHAPE
    assert route(ng=6) == _lib.BEAM_ERR_ARG          # not a power of two
    assert route(ng=64) == _lib.BEAM_ERR_ARG
    assert route(tg=9) == _lib.BEAM_ERR_ARG
    assert route(k=17) == _lib.BEAM_ERR_ARG
    assert route(ng=32, tg=1, k=9) == _lib.BEAM_ERR_ARG  # one group of 8 experts
    assert route(sc=float("inf")) == _lib.BEAM_ERR_ARG
    assert route(T=0, z=None) == _lib.BEAM_OK
    assert route(z=None) == _lib.BEAM_ERR_NULL
    assert route(z=Z + 4) == _lib.BEAM_ERR_ALIGN
    assert route(i=I + 2) == _lib.BEAM_ERR_ALIGN
    assert route(w=I + 16) == _lib.BEAM_ERR_ALIAS    # weights over the ids
    assert route(i=Z + 64) == _lib.BEAM_ERR_ALIAS    # ids inside the logits

    def route_ex(flags, T=4):
        return lib.beam_moe_route_ex(None, Z, Bi, T, 256, 8, 4, 8, 2.5, I, W, flags)

    assert route_ex(_lib.BEAM_OPT_FORCE_EXACT_SUM) == _lib.BEAM_ERR_ARG  # only BEAM_OPT_PDL
    assert route_ex(0x80) == _lib.BEAM_ERR_ARG
    assert route_ex(_lib.BEAM_OPT_PDL, T=0) == _lib.BEAM_OK

    def scaled(sc=2.5, **kw):
        args = dict(h=A, e=A + (1 << 32), w=A + (5 << 32), pw=A + (2 << 32), qw=A + (3 << 32),
                    y=A + (4 << 32))
        args.update(kw)
        return lib.beam_moe_combine_boundary_scaled(None, args["h"], args["e"], args["w"], sc,
                                                    args["pw"], args["qw"], 2, 1e-6, 4, D,
                                                    args["y"])

    assert scaled(sc=float("nan")) == _lib.BEAM_ERR_ARG
    assert scaled(e=None) == _lib.BEAM_ERR_NULL
    assert scaled(y=A) == _lib.BEAM_ERR_ALIAS


def test_qk_norm_argument_errors(lib):
    Q, K, QW, KW, P, TB = (A + (i << 32) for i in range(6))

    def qk(T=4, nq=48, nk=8, hd=128, eps=1e-6, mode=0, max_pos=100, q=Q, k=K, qw=QW, kw=KW, p=P,
           tb=TB):
        return lib.beam_qk_norm(None, q, k, qw, kw, p, tb, max_pos, T, nq, nk, hd, eps, mode)

    assert qk(hd=64) == _lib.BEAM_ERR_SHAPE
    assert qk(T=-1) == _lib.BEAM_ERR_SHAPE
    assert qk(mode=2) == _lib.BEAM_ERR_ARG
    assert qk(eps=-1.0) == _lib.BEAM_ERR_ARG
    assert qk(max_pos=0) == _lib.BEAM_ERR_ARG
    assert qk(T=0, q=None) == _lib.BEAM_OK
    assert qk(tb=None) == _lib.BEAM_ERR_NULL
    assert qk(p=None) == _lib.BEAM_ERR_NULL
    assert qk(q=Q + 8) == _lib.BEAM_ERR_ALIGN
    assert qk(k=Q + 4 * 48 * 128 * 2 - 256) == _lib.BEAM_ERR_ALIAS
    # SSMax needs no table
    assert qk(mode=1, tb=None, max_pos=0) != _lib.BEAM_ERR_NULL


def test_nvfp4_argument_errors(lib):
    H, X, PW, QW, Q, SF = (A + (i << 32) for i in range(6))
    E, W = A + (6 << 32), A + (7 << 32)

    def dense(T=4, d=D, gs=100.0, h=H, x=X, q=Q, sf=SF, opts=None):
        return lib.beam_boundary_fused_nvfp4(None, h, x, PW, QW, 2, 1e-6, T, d, gs, q, sf, opts)

    def moe(T=4, d=D, gs=100.0, h=H, q=Q, sf=SF, w=W, opts=None):
        return lib.beam_moe_combine_boundary_nvfp4(None, h, E, w, PW, QW, 2, 1e-6, T, d, gs, q, sf, opts)

    assert dense(d=520) == _lib.BEAM_ERR_SHAPE       # a multiple of 8, not of 16
    assert moe(d=520) == _lib.BEAM_ERR_SHAPE
    for gs in (0.0, -1.0, float("inf"), float("nan")):
        assert dense(gs=gs) == _lib.BEAM_ERR_ARG
        assert moe(gs=gs) == _lib.BEAM_ERR_ARG
    assert dense(T=0, h=None, q=None, sf=None) == _lib.BEAM_OK
    assert dense(q=None) == _lib.BEAM_ERR_NULL
    assert moe(sf=None) == _lib.BEAM_ERR_NULL
    assert dense(q=Q + 8) == _lib.BEAM_ERR_ALIGN
    assert dense(sf=Q + 4 * D // 2 - 1) == _lib.BEAM_ERR_ALIAS   # scales over the codes
    assert dense(q=X + 64) == _lib.BEAM_ERR_ALIAS                # codes inside x
    assert dense(sf=H + 2) == _lib.BEAM_ERR_ALIAS                # scales inside h
    assert moe(q=E + 4096) == _lib.BEAM_ERR_ALIAS                # codes inside the experts
    assert moe(sf=W + 8) == _lib.BEAM_ERR_ALIAS                  # scales inside the weights
    assert dense(x=H) != _lib.BEAM_ERR_ALIAS                     # x may be h itself
    ring = _lib.LaunchOpts(stages=2)
    hook = _lib.LaunchOpts(flags=_lib.BEAM_OPT_TEST_WAIT_TIMEOUT)
    assert dense(opts=ctypes.byref(ring)) == _lib.BEAM_ERR_ARG     # the ring writes no NVFP4
    assert dense(opts=ctypes.byref(hook)) == _lib.BEAM_ERR_ARG
    assert moe(opts=ctypes.byref(_lib.LaunchOpts(reserved=(0, 1, 0)))) == _lib.BEAM_ERR_ARG


def test_host_memory_calls_check_arguments_before_cuda(lib):
    H, X, PW, QW, Y, E, W = (A + (i << 32) for i in range(7))

    def dense(T=4, d=D, n=2, h=H, x=X, y=Y):
        return lib.beam_boundary_fused_host(None, h, x, PW, QW, n, 1e-6, T, d, y)

    def moe(T=4, d=D, h=H, e=E, w=W, y=Y):
        return lib.beam_moe_combine_boundary_host(None, h, e, w, PW, QW, 2, 1e-6, T, d, y)

    assert dense(d=12) == _lib.BEAM_ERR_SHAPE
    assert dense(n=0) == _lib.BEAM_ERR_ARG
    assert dense(T=0, h=None) == _lib.BEAM_OK
    assert dense(y=None) == _lib.BEAM_ERR_NULL
    assert moe(w=None) == _lib.BEAM_ERR_NULL
    assert dense(x=X + 8) == _lib.BEAM_ERR_ALIGN
    assert moe(e=E + 2) == _lib.BEAM_ERR_ALIGN
    assert dense(y=H + 64) == _lib.BEAM_ERR_ALIAS
    assert moe(h=E + 4096) == _lib.BEAM_ERR_ALIAS
    # valid arguments reach CUDA: without a GPU that is a CUDA or device error
    assert dense() in (_lib.BEAM_ERR_CUDA, _lib.BEAM_ERR_DEVICE)


def test_qk_norm_flags(lib):
    Q, K, QW, KW, P, TB = (A + (i << 32) for i in range(6))

    def qk(flags):
        return lib.beam_qk_norm_ex(None, Q, K, QW, KW, P, TB, 100, 4, 48, 8, 128, 1e-6, 0, flags)

    assert qk(0x8) == _lib.BEAM_ERR_ARG                          # not a Q/K flag
    assert qk(_lib.BEAM_OPT_TEST_WAIT_TIMEOUT) == _lib.BEAM_ERR_ARG
    for ok in (_lib.BEAM_OPT_PDL, _lib.BEAM_OPT_FORCE_EXACT_SUM | _lib.BEAM_OPT_PDL):
        assert qk(ok) in (_lib.BEAM_ERR_CUDA, _lib.BEAM_ERR_DEVICE)   # reaches CUDA
