"""Seeded synthetic inputs for the sublayer-boundary workloads.

This module only draws random numbers (see ``synth.c`` for the exact
generator definition) and converts them to BF16 storage with torch's own
round-to-nearest-even cast. It holds none of the boundary's arithmetic, and it
is the one piece of code that both the CUDA path's harness and the CPU oracle's
harness use: the same bytes reach both sides.

Shapes and distributions follow the decoder the boundary sits in: hidden size
5120, 104 boundaries per forward (52 layers x 2 sublayers), an 8 x 2048-token
prefill chunk, and top-8 routing with FP32 routing weights that already carry
the routing scale of 2.5 (Beam blog pages: "Model architecture",
"MoE and residual stream"; "Agent-driven optimization", change 1).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .configs import (DECODE_CHAIN_T64, DENSE_DECODE_T4, DENSE_PREFILL_T16384,  # noqa: F401
                      MOE_STRESS_T131072, MOE_T16384, STREAMS, WORKLOADS, Config)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` next to its source (plain gcc, no GPU needed)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = f"{_SO}.{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                    _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            u64, i32, f64 = ctypes.c_uint64, ctypes.c_int, ctypes.c_double
            vp = ctypes.c_void_p
            lib.synth_normal.argtypes = [u64, u64, u64, u64, f64, f64, vp, i32]
            lib.synth_normal.restype = None
            lib.synth_student_t3_unit.argtypes = [u64, u64, u64, u64, vp, i32]
            lib.synth_student_t3_unit.restype = None
            lib.synth_bernoulli.argtypes = [u64, u64, u64, u64, f64, vp, i32]
            lib.synth_bernoulli.restype = None
            lib.synth_topk_weights.argtypes = [u64, u64, u64, u64, i32, f64, vp, i32]
            lib.synth_topk_weights.restype = i32
            lib.synth_words.argtypes = [u64, u64, u64, u64, vp]
            lib.synth_words.restype = None
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def normal(seed: int, stream: int, count: int, start: int = 0,
           scale: float = 1.0, offset: float = 0.0, out: np.ndarray | None = None) -> np.ndarray:
    """FP32 values ``offset + scale * N(0,1)`` for indices ``start .. start+count-1``."""
    a = np.empty(count, np.float32) if out is None else out
    assert a.dtype == np.float32 and a.size == count and a.flags.c_contiguous
    _load().synth_normal(seed, stream, start, count, scale, offset, _ptr(a), _threads())
    return a


def student_t3_unit(seed: int, stream: int, count: int, start: int = 0,
                    out: np.ndarray | None = None) -> np.ndarray:
    """FP32 Student-t(3) values divided by sqrt(3), i.e. unit variance."""
    a = np.empty(count, np.float32) if out is None else out
    assert a.dtype == np.float32 and a.size == count and a.flags.c_contiguous
    _load().synth_student_t3_unit(seed, stream, start, count, _ptr(a), _threads())
    return a


def bernoulli(seed: int, stream: int, count: int, p: float, start: int = 0) -> np.ndarray:
    a = np.empty(count, np.uint8)
    _load().synth_bernoulli(seed, stream, start, count, p, _ptr(a), _threads())
    return a.astype(bool)


def topk_weights(seed: int, stream: int, rows: int, k: int = 8, scale: float = 2.5,
                 row_start: int = 0) -> np.ndarray:
    """[rows, k] FP32 routing weights: logistic of N(0,1) draws, renormalised, times ``scale``."""
    a = np.empty((rows, k), np.float32)
    rc = _load().synth_topk_weights(seed, stream, row_start, rows, k, scale, _ptr(a), _threads())
    if rc != 0:
        raise ValueError("k must be in 1..64")
    return a


def words(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    a = np.empty(count, np.uint64)
    _load().synth_words(seed, stream, start, count, _ptr(a))
    return a


def to_bf16(a: np.ndarray):
    """BF16 storage of FP32 values via torch's round-to-nearest-even cast (a CPU tensor)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)


# --------------------------------------------------------------------------- workloads

def dense_inputs(cfg: Config, row_start: int = 0, rows: int | None = None, step: int = 0) -> dict:
    """h, x [rows, D] and post_w, pre_w [D] for a dense boundary (BF16 CPU tensors).

    For the decode chain, ``step`` selects the boundary (0-based) and x and the
    norm weights are drawn fresh per step; h is the chain's initial stream."""
    D = cfg.D
    rows = cfg.T - row_start if rows is None else rows
    n0 = row_start * D
    cnt = rows * D
    h = to_bf16(normal(cfg.seed, STREAMS["h"], cnt, n0).reshape(rows, D))
    x = to_bf16(normal(cfg.seed, STREAMS["x"] + 16 * step, cnt, n0).reshape(rows, D))
    post_w = to_bf16(normal(cfg.seed, STREAMS["post_w"] + 16 * step, D, 0, 0.1, 1.0))
    pre_w = to_bf16(normal(cfg.seed, STREAMS["pre_w"] + 16 * step, D, 0, 0.1, 1.0))
    return dict(h=h, x=x, post_w=post_w, pre_w=pre_w)


def expert_rows_f32(cfg: Config, row_start: int, rows: int) -> np.ndarray:
    """FP32 expert outputs [rows, K, D] for tokens ``row_start ..`` (before BF16 storage)."""
    K, D = cfg.K, cfg.D
    n0 = row_start * K * D
    cnt = rows * K * D
    if cfg.expert_dist == "normal":
        e = normal(cfg.seed, STREAMS["e"], cnt, n0)
    elif cfg.expert_dist == "t3_outliers":
        e = student_t3_unit(cfg.seed, STREAMS["e"], cnt, n0)
        sel = bernoulli(cfg.seed, STREAMS["outlier"], rows * K, cfg.outlier_p, row_start * K)
        e = e.reshape(rows * K, D)
        e[sel] *= np.float32(cfg.outlier_scale)
    else:
        raise ValueError(cfg.expert_dist)
    return e.reshape(rows, K, D)


def expert_rows(cfg: Config, row_start: int, rows: int, out=None, chunk_rows: int = 2048):
    """BF16 expert outputs [rows, K, D] (CPU tensor; filled in chunks to bound FP32 scratch)."""
    import torch
    if out is None:
        out = torch.empty((rows, cfg.K, cfg.D), dtype=torch.bfloat16)
    for r in range(0, rows, chunk_rows):
        m = min(chunk_rows, rows - r)
        out[r:r + m].copy_(to_bf16(expert_rows_f32(cfg, row_start + r, m)))
    return out


def moe_inputs(cfg: Config, row_start: int = 0, rows: int | None = None, pin: bool = False) -> dict:
    """h [rows, D], expert_out [rows, K, D], topk_w [rows, K] FP32, post_w, pre_w [D]."""
    import torch
    D = cfg.D
    rows = cfg.T - row_start if rows is None else rows
    h = to_bf16(normal(cfg.seed, STREAMS["h"], rows * D, row_start * D).reshape(rows, D))
    e_out = torch.empty((rows, cfg.K, D), dtype=torch.bfloat16, pin_memory=pin)
    expert_rows(cfg, row_start, rows, out=e_out)
    w = torch.from_numpy(topk_weights(cfg.seed, STREAMS["topk"], rows, cfg.K, cfg.route_scale,
                                      row_start))
    post_w = to_bf16(normal(cfg.seed, STREAMS["post_w"], D, 0, 0.1, 1.0))
    pre_w = to_bf16(normal(cfg.seed, STREAMS["pre_w"], D, 0, 0.1, 1.0))
    return dict(h=h, expert_out=e_out, topk_w=w, post_w=post_w, pre_w=pre_w)


def layer_chain_inputs(chain: Config, moe: Config) -> tuple:
    """The decode chain as a decoder runs it: boundary s (0-based, n = chain.n + s)
    follows an attention sublayer when s is even (dense: x [T, D]) and an MoE
    sublayer when s is odd (expert rows [T, K, D] and routing weights [T, K]:
    tokens s*T .. s*T + T - 1 of the MoE workload's generator). Norm weights and
    the initial stream come from dense_inputs(chain, step=s). Returns (h0, steps)."""
    import torch
    T = chain.T
    h0 = dense_inputs(chain)["h"]
    steps = []
    for s in range(chain.steps):
        d = dense_inputs(chain, step=s)
        if s % 2 == 0:
            steps.append(dict(kind="dense", x=d["x"], post_w=d["post_w"], pre_w=d["pre_w"]))
        else:
            r0 = s * T
            w = topk_weights(moe.seed, STREAMS["topk"], T, moe.K, moe.route_scale, r0)
            steps.append(dict(kind="moe", expert_out=expert_rows(moe, r0, T),
                              topk_w=torch.from_numpy(w), post_w=d["post_w"], pre_w=d["pre_w"]))
    return h0, steps
