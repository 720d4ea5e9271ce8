"""CPU oracle for the fused sublayer boundary -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The CUDA
library and its Python binding never touch it, and it shares no code with them.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, built with
``-ffp-contract=off``); this file compiles it with gcc and marshals numpy /
torch CPU buffers into it. Row ranges may be handed to several Python threads
(ctypes drops the GIL during the call); each call stays single-threaded C.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
# A test may point the loader at another build of oracle.c (a planted-mistake copy)
_SO_OVERRIDE = os.environ.get("BEAM_ORACLE_SO")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` beside its source with gcc."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = f"{_SO}.{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                    "-std=c11", _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if _SO_OVERRIDE:
                lib = ctypes.CDLL(_SO_OVERRIDE)
            else:
                build()
                lib = ctypes.CDLL(_SO)
            vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
            ld = ctypes.c_longdouble
            lib.oracle_bf16_rne.argtypes = [f32]
            lib.oracle_bf16_rne.restype = ctypes.c_uint16
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f32.restype = f32
            lib.oracle_sum_f32_exact.argtypes = [vp, i64]
            lib.oracle_sum_f32_exact.restype = f32
            lib.oracle_sum_squares.argtypes = [vp, i32]
            lib.oracle_sum_squares.restype = f32
            lib.oracle_rms_factor.argtypes = [f32, i32, f32]
            lib.oracle_rms_factor.restype = f32
            lib.oracle_rmsnorm.argtypes = [vp, vp, f32, i32, vp]
            lib.oracle_rmsnorm.restype = None
            lib.oracle_scales.argtypes = [i32, vp, vp]
            lib.oracle_scales.restype = None
            lib.oracle_moe_combine.argtypes = [vp, vp, i32, i32, vp]
            lib.oracle_moe_combine.restype = None
            lib.oracle_boundary.argtypes = [vp, vp, vp, vp, i32, f32, i64, i32, vp]
            lib.oracle_boundary.restype = i32
            lib.oracle_moe_boundary.argtypes = [vp, vp, vp, i32, vp, vp, i32, f32, i64, i32, vp]
            lib.oracle_moe_boundary.restype = i32
            lib.oracle_boundary_ld.argtypes = [vp, vp, vp, vp, i32, ld, i64, i32, vp]
            lib.oracle_boundary_ld.restype = i32
            lib.oracle_residual_ld.argtypes = [vp, vp, i32, i64]
            lib.oracle_residual_ld.restype = None
            lib.oracle_moe_combine_scaled.argtypes = [vp, vp, i32, i32, f32, vp]
            lib.oracle_moe_combine_scaled.restype = None
            lib.oracle_moe_boundary_scaled.argtypes = [vp, vp, vp, i32, f32, vp, vp, i32, f32, i64,
                                                       i32, vp]
            lib.oracle_moe_boundary_scaled.restype = i32
            lib.oracle_ssmax_scale.argtypes = [i64]
            lib.oracle_ssmax_scale.restype = f32
            lib.oracle_qk_norm.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, i32]
            lib.oracle_qk_norm.restype = i32
            u8 = ctypes.c_uint8
            for name, res, args in (("oracle_e4m3", u8, [f32]), ("oracle_e2m1", u8, [f32]),
                                    ("oracle_e4m3_to_f32", f32, [u8]),
                                    ("oracle_e2m1_to_f32", f32, [u8])):
                getattr(lib, name).argtypes = args
                getattr(lib, name).restype = res
            lib.oracle_nvfp4_row.argtypes = [vp, i32, f32, vp, vp]
            lib.oracle_nvfp4_row.restype = None
            lib.oracle_boundary_nvfp4.argtypes = [vp, vp, vp, vp, i32, f32, i64, i32, f32, vp, vp]
            lib.oracle_boundary_nvfp4.restype = i32
            lib.oracle_moe_boundary_nvfp4.argtypes = [vp, vp, vp, i32, vp, vp, i32, f32, i64, i32,
                                                      f32, vp, vp]
            lib.oracle_moe_boundary_nvfp4.restype = i32
            lib.oracle_route.argtypes = [vp, vp, i64, i32, i32, i32, i32, f32, vp, vp]
            lib.oracle_route.restype = i32
            lib.oracle_sigmoid.argtypes = [f32]
            lib.oracle_sigmoid.restype = f32
            lib.oracle_sigmoid_array.argtypes = [vp, vp, i64]
            lib.oracle_sigmoid_array.restype = None
            lib.oracle_sigmoid_undecided.argtypes = []
            lib.oracle_sigmoid_undecided.restype = ctypes.c_ulonglong
            _lib = lib
    return _lib


# ---------------------------------------------------------------- marshalling

def as_u16(a) -> np.ndarray:
    """BF16 bit patterns as a C-contiguous uint16 numpy array (torch bf16 or uint16 input)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            assert a.dtype == torch.bfloat16 and a.device.type == "cpu"
            return a.contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:
        pass
    a = np.asarray(a)
    assert a.dtype == np.uint16
    return np.ascontiguousarray(a)


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


def bf16_rne(f: float) -> int:
    return int(_load().oracle_bf16_rne(float(f)))


def bf16_to_f32(b: int) -> float:
    return float(_load().oracle_bf16_to_f32(int(b)))


def sum_f32_exact(t) -> float:
    t = np.ascontiguousarray(t, dtype=np.float32)
    return float(_load().oracle_sum_f32_exact(_p(t), t.size))


def sum_squares(v) -> float:
    v = as_u16(v)
    return float(_load().oracle_sum_squares(_p(v), v.size))


def rms_factor(S: float, D: int, eps: float) -> float:
    return float(_load().oracle_rms_factor(S, D, eps))


def rmsnorm(v, w, eps: float) -> np.ndarray:
    v, w = as_u16(v), as_u16(w)
    out = np.empty_like(v)
    _load().oracle_rmsnorm(_p(v), _p(w), eps, v.size, _p(out))
    return out


def scales(n: int) -> tuple[float, float]:
    c1, c2 = ctypes.c_float(), ctypes.c_float()
    _load().oracle_scales(n, ctypes.byref(c1), ctypes.byref(c2))
    return c1.value, c2.value


def moe_combine(e, w) -> np.ndarray:
    e = as_u16(e)
    w = np.ascontiguousarray(w, dtype=np.float32)
    K, D = e.shape
    out = np.empty(D, np.uint16)
    _load().oracle_moe_combine(_p(e), _p(w), K, D, _p(out))
    return out


def _row_split(T: int, threads: int):
    threads = max(1, min(threads, T))
    step = -(-T // threads) if T else 0
    return [(r, min(T, r + step)) for r in range(0, T, step)] if T else []


def boundary(h, x, post_w, pre_w, n: int, eps: float, threads: int = 1):
    """Dense boundary; returns (h', y) as uint16 arrays [T, D] (inputs are not modified)."""
    h = as_u16(h).copy()
    x, post_w, pre_w = as_u16(x), as_u16(post_w), as_u16(pre_w)
    T, D = h.shape
    y = np.empty_like(h)
    lib = _load()

    def run(lo_hi):
        lo, hi = lo_hi
        rc = lib.oracle_boundary(_p(h[lo:hi]), _p(x[lo:hi]), _p(post_w), _p(pre_w), n, eps,
                                 hi - lo, D, _p(y[lo:hi]))
        if rc != 0:
            raise ValueError("oracle_boundary: bad arguments")

    _run_rows(run, T, threads)
    return h, y


def moe_combine_scaled(e, w, scale: float) -> np.ndarray:
    e = as_u16(e)
    w = np.ascontiguousarray(w, dtype=np.float32)
    K, D = e.shape
    out = np.empty(D, np.uint16)
    _load().oracle_moe_combine_scaled(_p(e), _p(w), K, D, scale, _p(out))
    return out


def moe_boundary(h, expert_out, topk_w, post_w, pre_w, n: int, eps: float, threads: int = 1,
                 route_scale: float | None = None):
    """MoE combine + boundary; returns (h', y) as uint16 arrays [T, D]. With route_scale the
    scale is applied in the combine (x = bf16(scale * acc)) and topk_w are unscaled."""
    h = as_u16(h).copy()
    e = as_u16(expert_out)
    w = np.ascontiguousarray(topk_w.numpy() if hasattr(topk_w, "numpy") else topk_w,
                             dtype=np.float32)
    post_w, pre_w = as_u16(post_w), as_u16(pre_w)
    T, K, D = e.shape
    y = np.empty_like(h)
    lib = _load()

    def run(lo_hi):
        lo, hi = lo_hi
        if route_scale is None:
            rc = lib.oracle_moe_boundary(_p(h[lo:hi]), _p(e[lo:hi]), _p(w[lo:hi]), K, _p(post_w),
                                         _p(pre_w), n, eps, hi - lo, D, _p(y[lo:hi]))
        else:
            rc = lib.oracle_moe_boundary_scaled(_p(h[lo:hi]), _p(e[lo:hi]), _p(w[lo:hi]), K,
                                                route_scale, _p(post_w), _p(pre_w), n, eps,
                                                hi - lo, D, _p(y[lo:hi]))
        if rc != 0:
            raise ValueError("oracle_moe_boundary: bad arguments")

    _run_rows(run, T, threads)
    return h, y


def _run_rows(fn, T: int, threads: int):
    parts = _row_split(T, threads)
    if len(parts) <= 1:
        for p in parts:
            fn(p)
        return
    with ThreadPoolExecutor(len(parts)) as ex:
        list(ex.map(fn, parts))


def boundary_ld(h, x, post_w, pre_w, n: int, eps: float):
    """The boundary in long double with no rounding; numpy longdouble arrays in, (h', y) out."""
    h = np.array(h, dtype=np.longdouble, order="C")
    x = np.ascontiguousarray(x, dtype=np.longdouble)
    post_w = np.ascontiguousarray(post_w, dtype=np.longdouble)
    pre_w = np.ascontiguousarray(pre_w, dtype=np.longdouble)
    T, D = h.shape
    y = np.empty_like(h)
    rc = _load().oracle_boundary_ld(_p(h), _p(x), _p(post_w), _p(pre_w), n, eps, T, D, _p(y))
    if rc != 0:
        raise ValueError("oracle_boundary_ld: bad arguments")
    return h, y


def residual_ld(h, x, n: int) -> np.ndarray:
    h = np.array(h, dtype=np.longdouble, order="C")
    x = np.ascontiguousarray(x, dtype=np.longdouble)
    _load().oracle_residual_ld(_p(h), _p(x), n, h.size)
    return h


def sigmoid(z: float) -> float:
    return float(_load().oracle_sigmoid(z))


def sigmoid_array(z, threads: int = 1) -> np.ndarray:
    """The router sigmoid of every element of a float32 array (row-parallel over threads)."""
    z = np.ascontiguousarray(z, dtype=np.float32).ravel()
    s = np.empty_like(z)
    lib = _load()
    if threads <= 1 or z.size < 1 << 16:
        lib.oracle_sigmoid_array(_p(z), _p(s), z.size)
        return s
    step = -(-z.size // threads)
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda lo: lib.oracle_sigmoid_array(_p(z[lo:lo + step]), _p(s[lo:lo + step]),
                                                         min(step, z.size - lo)),
                    range(0, z.size, step)))
    return s


def sigmoid_undecided() -> int:
    """Sigmoid evaluations that neither precision level decided (expected: 0)."""
    return int(_load().oracle_sigmoid_undecided())


def route(logits, bias, n_group: int = 8, topk_group: int = 4, topk: int = 8,
          scale: float = 2.5, threads: int = 1):
    """Group-limited top-k routing; returns (idx int32 [T, topk], w float32 [T, topk])."""
    z = np.ascontiguousarray(logits.numpy() if hasattr(logits, "numpy") else logits,
                             dtype=np.float32)
    b = np.ascontiguousarray(bias.numpy() if hasattr(bias, "numpy") else bias, dtype=np.float32)
    T, E = z.shape
    idx = np.empty((T, topk), np.int32)
    w = np.empty((T, topk), np.float32)
    lib = _load()

    def run(lo_hi):
        lo, hi = lo_hi
        rc = lib.oracle_route(_p(z[lo:hi]), _p(b), hi - lo, E, n_group, topk_group, topk, scale,
                              _p(idx[lo:hi]), _p(w[lo:hi]))
        if rc != 0:
            raise ValueError("oracle_route: bad arguments")

    _run_rows(run, T, threads)
    return idx, w


def ssmax_scale(pos: int) -> float:
    return float(_load().oracle_ssmax_scale(int(pos)))


def qk_norm(q, k, q_w, k_w, pos, table, eps: float, mode: str = "rope", threads: int = 1):
    """Per-head Q/K RMSNorm then RoPE (mode "rope", FP32 cos/sin table [max_pos, 128]) or
    SSMax on the queries (mode "ssmax"); returns new (q, k) uint16 arrays."""
    q = as_u16(q).copy()
    k = as_u16(k).copy()
    q_w, k_w = as_u16(q_w), as_u16(k_w)
    pos = np.ascontiguousarray(pos.numpy() if hasattr(pos, "numpy") else pos, dtype=np.int32)
    T, nq, _ = q.shape
    nk = k.shape[1]
    if table is None:
        table = np.zeros((1, 128), np.float32)
    table = np.ascontiguousarray(table.numpy() if hasattr(table, "numpy") else table,
                                 dtype=np.float32)
    m = {"rope": 0, "ssmax": 1}[mode]
    lib = _load()

    def run(lo_hi):
        lo, hi = lo_hi
        rc = lib.oracle_qk_norm(_p(q[lo:hi]), _p(k[lo:hi]), _p(q_w), _p(k_w), _p(pos[lo:hi]),
                                _p(table), table.shape[0], hi - lo, nq, nk, eps, m)
        if rc != 0:
            raise ValueError("oracle_qk_norm: bad arguments")

    _run_rows(run, T, threads)
    return q, k


def e4m3(v: float) -> int:
    return int(_load().oracle_e4m3(float(v)))


def e2m1(v: float) -> int:
    return int(_load().oracle_e2m1(float(v)))


def e4m3_to_f32(b: int) -> float:
    return float(_load().oracle_e4m3_to_f32(int(b)))


def e2m1_to_f32(b: int) -> float:
    return float(_load().oracle_e2m1_to_f32(int(b)))


def nvfp4_row(y, gs: float):
    """Quantise one BF16 row (length a multiple of 16): (q [D/2] uint8, sf [D/16] uint8)."""
    y = as_u16(y)
    D = y.size
    q = np.empty(D // 2, np.uint8)
    sf = np.empty(D // 16, np.uint8)
    _load().oracle_nvfp4_row(_p(y), D, gs, _p(q), _p(sf))
    return q, sf


def boundary_nvfp4(h, x, post_w, pre_w, n: int, eps: float, gs: float, threads: int = 1):
    """Dense boundary with y as NVFP4; returns (h', q [T, D/2], sf [T, D/16])."""
    h = as_u16(h).copy()
    x, post_w, pre_w = as_u16(x), as_u16(post_w), as_u16(pre_w)
    T, D = h.shape
    q = np.empty((T, D // 2), np.uint8)
    sf = np.empty((T, D // 16), np.uint8)
    lib = _load()

    def run(lo_hi):
        lo, hi = lo_hi
        rc = lib.oracle_boundary_nvfp4(_p(h[lo:hi]), _p(x[lo:hi]), _p(post_w), _p(pre_w), n, eps,
                                       hi - lo, D, gs, _p(q[lo:hi]), _p(sf[lo:hi]))
        if rc != 0:
            raise ValueError("oracle_boundary_nvfp4: bad arguments")

    _run_rows(run, T, threads)
    return h, q, sf


def moe_boundary_nvfp4(h, expert_out, topk_w, post_w, pre_w, n: int, eps: float, gs: float,
                       threads: int = 1):
    """MoE boundary with y as NVFP4; returns (h', q [T, D/2], sf [T, D/16])."""
    h = as_u16(h).copy()
    e = as_u16(expert_out)
    w = np.ascontiguousarray(topk_w.numpy() if hasattr(topk_w, "numpy") else topk_w,
                             dtype=np.float32)
    post_w, pre_w = as_u16(post_w), as_u16(pre_w)
    T, K, D = e.shape
    q = np.empty((T, D // 2), np.uint8)
    sf = np.empty((T, D // 16), np.uint8)
    lib = _load()

    def run(lo_hi):
        lo, hi = lo_hi
        rc = lib.oracle_moe_boundary_nvfp4(_p(h[lo:hi]), _p(e[lo:hi]), _p(w[lo:hi]), K,
                                           _p(post_w), _p(pre_w), n, eps, hi - lo, D, gs,
                                           _p(q[lo:hi]), _p(sf[lo:hi]))
        if rc != 0:
            raise ValueError("oracle_moe_boundary_nvfp4: bad arguments")

    _run_rows(run, T, threads)
    return h, q, sf
