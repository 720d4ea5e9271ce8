"""Fused sublayer boundary of the Beam decoder on GB300 (sm_103a).

Python binding of ``libbeamboundary`` (C ABI: ``include/beam_boundary.h``).
This module only marshals torch CUDA tensors into the C calls; every step of
the boundary runs in the library's CUDA kernels. There is no CPU or PyTorch
fallback: without the built library, calls raise ``ImportError``.

    y = boundary_fused(h, x, post_w, pre_w, n, eps)          # h updated in place
    y = moe_combine_boundary(h, expert_out, topk_w, post_w, pre_w, n, eps)
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import LaunchOpts  # noqa: F401

__all__ = ["boundary_fused", "moe_combine_boundary", "boundary_fused_host",
           "moe_combine_boundary_host", "boundary_fused_nvfp4",
           "moe_combine_boundary_nvfp4", "moe_route", "router_sigmoid", "qk_norm", "sync_status",
           "exact_sum_count",
           "version", "BeamError", "LaunchOpts", "library"]


class BeamError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.load().beam_status_string(status).decode()
        super().__init__(f"{where}: status {status} ({msg})")


def library() -> ctypes.CDLL:
    """The loaded ``libbeamboundary.so`` (raises ImportError when it is not built)."""
    return _lib.load()


def _stream_ptr(stream) -> int | None:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream or None


def _check(t, name: str, dtype, ndim: int):
    """Type, dtype, rank and layout of one operand (devices: ``_on_current_device``)."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")


def _shape(t, name: str, shape: tuple):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)} (got {tuple(t.shape)})")


def _on_current_device(**tensors):
    """Every operand on one CUDA device, the current one: the library launches on the
    current device and takes the pointers as they are, so a tensor elsewhere would
    reach the kernel as a foreign address. Checked after the shapes, before any launch."""
    import torch
    devs = {name: t.device for name, t in tensors.items()}
    if len(set(devs.values())) != 1:
        raise ValueError("operands must all be on one device: "
                         + ", ".join(f"{n} on {d}" for n, d in devs.items()))
    dev = next(iter(devs.values()))
    if dev.type != "cuda":
        raise ValueError(f"operands must be CUDA tensors (got {dev})")
    cur = torch.cuda.current_device()
    if dev.index != cur:
        raise ValueError(f"operands are on {dev} but the current device is cuda:{cur}: "
                         f"call under `with torch.cuda.device({dev.index}):`")


def _opts(opts):
    if opts is None:
        return None
    if isinstance(opts, dict):
        opts = LaunchOpts(**opts)
    return ctypes.byref(opts)


def boundary_fused(h, x, post_w, pre_w, n: int, eps: float = 1e-6, y=None, stream=None, opts=None):
    """Dense boundary on torch CUDA tensors; updates ``h`` in place and returns ``y``.

    h, x: [T, D] bfloat16; post_w, pre_w: [D] bfloat16; n >= 1 (index of the residual add).
    """
    import torch
    _check(h, "h", torch.bfloat16, 2)
    _check(x, "x", torch.bfloat16, 2)
    _check(post_w, "post_w", torch.bfloat16, 1)
    _check(pre_w, "pre_w", torch.bfloat16, 1)
    T, D = h.shape
    if x.shape != h.shape or post_w.shape[0] != D or pre_w.shape[0] != D:
        raise ValueError("shape mismatch: h, x [T, D]; post_w, pre_w [D]")
    if y is None:
        y = torch.empty_like(h)
    _check(y, "y", torch.bfloat16, 2)
    _shape(y, "y", (T, D))
    _on_current_device(h=h, x=x, post_w=post_w, pre_w=pre_w, y=y)
    lib = _lib.load()
    args = (_stream_ptr(stream), h.data_ptr(), x.data_ptr(), post_w.data_ptr(), pre_w.data_ptr(),
            int(n), float(eps), T, D, y.data_ptr())
    st = lib.beam_boundary_fused(*args) if opts is None else lib.beam_boundary_fused_ex(
        *args, _opts(opts))
    if st != 0:
        raise BeamError(st, "beam_boundary_fused")
    return y


def moe_combine_boundary(h, expert_out, topk_w, post_w, pre_w, n: int, eps: float = 1e-6, y=None,
                         stream=None, opts=None, route_scale: float | None = None):
    """MoE boundary: combine the top-8 expert outputs with FP32 weights, then the dense boundary.

    h: [T, D] bf16; expert_out: [T, 8, D] bf16; topk_w: [T, 8] float32 with the routing
    scale included, or, when ``route_scale`` is given, without it (the kernel then applies
    it to the combined sum).
    """
    import torch
    _check(h, "h", torch.bfloat16, 2)
    _check(expert_out, "expert_out", torch.bfloat16, 3)
    _check(topk_w, "topk_w", torch.float32, 2)
    _check(post_w, "post_w", torch.bfloat16, 1)
    _check(pre_w, "pre_w", torch.bfloat16, 1)
    T, D = h.shape
    K = _lib.BEAM_MOE_TOPK
    if expert_out.shape != (T, K, D) or topk_w.shape != (T, K):
        raise ValueError(f"shape mismatch: expert_out [T, {K}, D], topk_w [T, {K}]")
    if post_w.shape[0] != D or pre_w.shape[0] != D:
        raise ValueError("shape mismatch: post_w, pre_w [D]")
    if y is None:
        y = torch.empty_like(h)
    _check(y, "y", torch.bfloat16, 2)
    _shape(y, "y", (T, D))
    _on_current_device(h=h, expert_out=expert_out, topk_w=topk_w, post_w=post_w, pre_w=pre_w, y=y)
    lib = _lib.load()
    if route_scale is not None:
        if opts is not None:
            raise ValueError("route_scale and opts cannot be combined")
        st = lib.beam_moe_combine_boundary_scaled(
            _stream_ptr(stream), h.data_ptr(), expert_out.data_ptr(), topk_w.data_ptr(),
            float(route_scale), post_w.data_ptr(), pre_w.data_ptr(), int(n), float(eps), T, D,
            y.data_ptr())
        if st != 0:
            raise BeamError(st, "beam_moe_combine_boundary_scaled")
        return y
    args = (_stream_ptr(stream), h.data_ptr(), expert_out.data_ptr(), topk_w.data_ptr(),
            post_w.data_ptr(), pre_w.data_ptr(), int(n), float(eps), T, D, y.data_ptr())
    st = lib.beam_moe_combine_boundary(*args) if opts is None else \
        lib.beam_moe_combine_boundary_ex(*args, _opts(opts))
    if st != 0:
        raise BeamError(st, "beam_moe_combine_boundary")
    return y


def _check_any(t, name: str, dtype, ndim: int):
    """A CUDA tensor or a CPU tensor (page-locked, or pageable where the device
    reads pageable memory: the library decides)."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type not in ("cuda", "cpu"):
        raise ValueError(f"{name} must be a CUDA or CPU tensor (got {t.device})")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")


def _like_host(h):
    import torch
    if h.device.type == "cuda":
        return torch.empty_like(h)
    return torch.empty(h.shape, dtype=h.dtype, pin_memory=True)


def boundary_fused_host(h, x, post_w, pre_w, n: int, eps: float = 1e-6, y=None, stream=None):
    """Dense boundary on a batch in host memory: h, x, y (and the weights) may be
    page-locked CPU tensors (``tensor.pin_memory()``), read and written by the kernels
    over the CPU-GPU link. Asynchronous on ``stream`` (default: the current CUDA
    stream): synchronise before touching the host tensors. Returns y (page-locked
    CPU when h is on the CPU)."""
    import torch
    _check_any(h, "h", torch.bfloat16, 2)
    _check_any(x, "x", torch.bfloat16, 2)
    _check_any(post_w, "post_w", torch.bfloat16, 1)
    _check_any(pre_w, "pre_w", torch.bfloat16, 1)
    T, D = h.shape
    if x.shape != h.shape or post_w.shape[0] != D or pre_w.shape[0] != D:
        raise ValueError("shape mismatch: h, x [T, D]; post_w, pre_w [D]")
    if y is None:
        y = _like_host(h)
    _check_any(y, "y", torch.bfloat16, 2)
    _shape(y, "y", (T, D))
    st = _lib.load().beam_boundary_fused_host(_stream_ptr(stream), h.data_ptr(), x.data_ptr(),
                                              post_w.data_ptr(), pre_w.data_ptr(), int(n),
                                              float(eps), T, D, y.data_ptr())
    if st != 0:
        raise BeamError(st, "beam_boundary_fused_host")
    return y


def moe_combine_boundary_host(h, expert_out, topk_w, post_w, pre_w, n: int, eps: float = 1e-6,
                              y=None, stream=None):
    """MoE boundary on a batch in host memory (see ``boundary_fused_host``)."""
    import torch
    _check_any(h, "h", torch.bfloat16, 2)
    _check_any(expert_out, "expert_out", torch.bfloat16, 3)
    _check_any(topk_w, "topk_w", torch.float32, 2)
    _check_any(post_w, "post_w", torch.bfloat16, 1)
    _check_any(pre_w, "pre_w", torch.bfloat16, 1)
    T, D = h.shape
    K = _lib.BEAM_MOE_TOPK
    if (expert_out.shape != (T, K, D) or topk_w.shape != (T, K) or post_w.shape[0] != D
            or pre_w.shape[0] != D):
        raise ValueError(f"shape mismatch: h [T, D]; expert_out [T, {K}, D]; topk_w [T, {K}]")
    if y is None:
        y = _like_host(h)
    _check_any(y, "y", torch.bfloat16, 2)
    _shape(y, "y", (T, D))
    st = _lib.load().beam_moe_combine_boundary_host(
        _stream_ptr(stream), h.data_ptr(), expert_out.data_ptr(), topk_w.data_ptr(),
        post_w.data_ptr(), pre_w.data_ptr(), int(n), float(eps), T, D, y.data_ptr())
    if st != 0:
        raise BeamError(st, "beam_moe_combine_boundary_host")
    return y


def _nvfp4_out(h, q, sf):
    import torch
    T, D = h.shape
    if D % 16:
        raise ValueError("NVFP4 output needs D to be a multiple of 16")
    if q is None:
        q = torch.empty((T, D // 2), dtype=torch.uint8, device=h.device)
    if sf is None:
        sf = torch.empty((T, D // 16), dtype=torch.uint8, device=h.device)
    _check(q, "y_fp4", torch.uint8, 2)
    _check(sf, "y_scale", torch.uint8, 2)
    if tuple(q.shape) != (T, D // 2) or tuple(sf.shape) != (T, D // 16):
        raise ValueError("shape mismatch: y_fp4 [T, D/2]; y_scale [T, D/16]")
    return q, sf


def boundary_fused_nvfp4(h, x, post_w, pre_w, n: int, eps: float, y_global_scale: float,
                         y_fp4=None, y_scale=None, stream=None, opts=None):
    """Dense boundary with y as NVFP4; updates h in place, returns (y_fp4 [T, D/2] uint8,
    y_scale [T, D/16] uint8)."""
    import torch
    for t, name in ((h, "h"), (x, "x")):
        _check(t, name, torch.bfloat16, 2)
    _check(post_w, "post_w", torch.bfloat16, 1)
    _check(pre_w, "pre_w", torch.bfloat16, 1)
    T, D = h.shape
    if x.shape != h.shape or post_w.shape[0] != D or pre_w.shape[0] != D:
        raise ValueError("shape mismatch: h, x [T, D]; post_w, pre_w [D]")
    q, sf = _nvfp4_out(h, y_fp4, y_scale)
    _on_current_device(h=h, x=x, post_w=post_w, pre_w=pre_w, y_fp4=q, y_scale=sf)
    st = _lib.load().beam_boundary_fused_nvfp4(_stream_ptr(stream), h.data_ptr(), x.data_ptr(),
                                               post_w.data_ptr(), pre_w.data_ptr(), int(n),
                                               float(eps), T, D, float(y_global_scale),
                                               q.data_ptr(), sf.data_ptr(), _opts(opts))
    if st != 0:
        raise BeamError(st, "beam_boundary_fused_nvfp4")
    return q, sf


def moe_combine_boundary_nvfp4(h, expert_out, topk_w, post_w, pre_w, n: int, eps: float,
                               y_global_scale: float, y_fp4=None, y_scale=None, stream=None,
                               opts=None):
    """MoE boundary with y as NVFP4; updates h in place, returns (y_fp4, y_scale)."""
    import torch
    _check(h, "h", torch.bfloat16, 2)
    _check(expert_out, "expert_out", torch.bfloat16, 3)
    _check(topk_w, "topk_w", torch.float32, 2)
    _check(post_w, "post_w", torch.bfloat16, 1)
    _check(pre_w, "pre_w", torch.bfloat16, 1)
    T, D = h.shape
    if (expert_out.shape != (T, _lib.BEAM_MOE_TOPK, D) or topk_w.shape != (T, _lib.BEAM_MOE_TOPK)
            or post_w.shape[0] != D or pre_w.shape[0] != D):
        raise ValueError("shape mismatch: h [T, D]; expert_out [T, 8, D]; topk_w [T, 8]")
    q, sf = _nvfp4_out(h, y_fp4, y_scale)
    _on_current_device(h=h, expert_out=expert_out, topk_w=topk_w, post_w=post_w, pre_w=pre_w,
                       y_fp4=q, y_scale=sf)
    st = _lib.load().beam_moe_combine_boundary_nvfp4(
        _stream_ptr(stream), h.data_ptr(), expert_out.data_ptr(), topk_w.data_ptr(),
        post_w.data_ptr(), pre_w.data_ptr(), int(n), float(eps), T, D, float(y_global_scale),
        q.data_ptr(), sf.data_ptr(), _opts(opts))
    if st != 0:
        raise BeamError(st, "beam_moe_combine_boundary_nvfp4")
    return q, sf


def moe_route(logits, bias, n_group: int = 8, topk_group: int = 4, topk: int = 8,
              route_scale: float = 2.5, idx=None, w=None, stream=None, pdl: bool = False):
    """Group-limited top-k routing on torch CUDA tensors.

    logits: [T, 256] float32 router logits; bias: [256] float32 correction bias.
    pdl: launch with programmatic dependent launch (BEAM_OPT_PDL).
    Returns (idx int32 [T, topk], w float32 [T, topk]).
    """
    import torch
    _check(logits, "logits", torch.float32, 2)
    _check(bias, "bias", torch.float32, 1)
    T, E = logits.shape
    if bias.shape[0] != E:
        raise ValueError("bias must have one entry per expert")
    if idx is None:
        idx = torch.empty((T, topk), dtype=torch.int32, device=logits.device)
    if w is None:
        w = torch.empty((T, topk), dtype=torch.float32, device=logits.device)
    _check(idx, "idx", torch.int32, 2)
    _check(w, "w", torch.float32, 2)
    _shape(idx, "idx", (T, topk))
    _shape(w, "w", (T, topk))
    _on_current_device(logits=logits, bias=bias, idx=idx, w=w)
    st = _lib.load().beam_moe_route_ex(_stream_ptr(stream), logits.data_ptr(), bias.data_ptr(), T, E,
                                       int(n_group), int(topk_group), int(topk), float(route_scale),
                                       idx.data_ptr(), w.data_ptr(), _lib.BEAM_OPT_PDL if pdl else 0)
    if st != 0:
        raise BeamError(st, "beam_moe_route_ex")
    return idx, w


def router_sigmoid(z, out=None, stream=None, fast: bool = False):
    """The router's correctly rounded FP32 sigmoid of every element of ``z`` (float32 CUDA
    tensor, any shape, contiguous); ``out`` may be ``z`` (in place). With ``fast``, the
    routing first pass's approximation instead (within 2^-19 of the exact sigmoid)."""
    import torch
    if not isinstance(z, torch.Tensor) or z.dtype != torch.float32 or not z.is_contiguous():
        raise TypeError("z must be a contiguous float32 tensor")
    if out is None:
        out = torch.empty_like(z)
    if not isinstance(out, torch.Tensor) or out.dtype != torch.float32 or not out.is_contiguous():
        raise TypeError("out must be a contiguous float32 tensor")
    _shape(out, "out", tuple(z.shape))
    _on_current_device(z=z, out=out)
    fn = _lib.load().beam_router_sigmoid_fast if fast else _lib.load().beam_router_sigmoid
    st = fn(_stream_ptr(stream), z.data_ptr(), out.data_ptr(), z.numel())
    if st != 0:
        raise BeamError(st, "beam_router_sigmoid_fast" if fast else "beam_router_sigmoid")
    return out


def qk_norm(q, k, q_w, k_w, pos, eps: float = 1e-6, mode: str = "rope", rope_table=None,
            stream=None, force_exact: bool = False, pdl: bool = False):
    """Per-head Q/K RMSNorm then RoPE (mode "rope") or SSMax (mode "ssmax"), in place.

    q: [T, n_q, 128] bf16; k: [T, n_kv, 128] bf16; q_w, k_w: [128] bf16; pos: [T] int32;
    rope_table: [max_pos, 128] float32 (cos | sin), needed for mode "rope".
    """
    import torch
    _check(q, "q", torch.bfloat16, 3)
    _check(k, "k", torch.bfloat16, 3)
    _check(q_w, "q_w", torch.bfloat16, 1)
    _check(k_w, "k_w", torch.bfloat16, 1)
    _check(pos, "pos", torch.int32, 1)
    T = q.shape[0]
    if k.shape[0] != T or pos.shape[0] != T or q.shape[2] != k.shape[2]:
        raise ValueError("shape mismatch: q [T, nq, 128], k [T, nk, 128], pos [T]")
    hd = q.shape[2]
    _shape(q_w, "q_w", (hd,))
    _shape(k_w, "k_w", (hd,))
    m = {"rope": _lib.BEAM_QK_ROPE, "ssmax": _lib.BEAM_QK_SSMAX}[mode]
    tab, max_pos = 0, 0
    ops = dict(q=q, k=k, q_w=q_w, k_w=k_w, pos=pos)
    if mode == "rope":
        _check(rope_table, "rope_table", torch.float32, 2)
        if rope_table.shape[1] != hd:
            raise ValueError(f"rope_table must be [max_pos, {hd}] (cos | sin)")
        tab, max_pos = rope_table.data_ptr(), rope_table.shape[0]
        ops["rope_table"] = rope_table
    _on_current_device(**ops)
    st = _lib.load().beam_qk_norm_ex(_stream_ptr(stream), q.data_ptr(), k.data_ptr(), q_w.data_ptr(),
                                     k_w.data_ptr(), pos.data_ptr(), tab or None, max_pos, T,
                                     q.shape[1], k.shape[1], q.shape[2], float(eps), m,
                                     (_lib.BEAM_OPT_FORCE_EXACT_SUM if force_exact else 0)
                                     | (_lib.BEAM_OPT_PDL if pdl else 0))
    if st != 0:
        raise BeamError(st, "beam_qk_norm")
    return q, k


def sync_status(stream=None) -> None:
    """Synchronise the stream and raise BeamError if a kernel reported a device-side error."""
    st = _lib.load().beam_sync_status(_stream_ptr(stream))
    if st != 0:
        raise BeamError(st, "beam_sync_status")


def exact_sum_count(reset: bool = False, stream=None) -> int:
    """Row sums that took the exact integer path on this device (diagnostics)."""
    v = ctypes.c_uint64(0)
    st = _lib.load().beam_exact_sum_count(_stream_ptr(stream), ctypes.byref(v), int(reset))
    if st != 0:
        raise BeamError(st, "beam_exact_sum_count")
    return int(v.value)


def version() -> int:
    return int(_lib.load().beam_version())
