"""The Python binding refuses wrong shapes and devices before any launch.

The C calls trust T * D and take device addresses as they are, so a caller-given
output that is too small, or an operand on another device, must be caught in
the binding. These run on the CPU: every check fires before the library is
loaded or a CUDA call is made (meta tensors stand in for a second device)."""
from __future__ import annotations

import pytest
import torch

import sandwich_norm_residual_gb300 as snr

T, D = 4, 64


def bf(*shape, device="cpu"):
    return torch.zeros(shape, dtype=torch.bfloat16, device=device)


def dense_args(device="cpu"):
    return bf(T, D, device=device), bf(T, D, device=device), bf(D), bf(D)


def test_dense_refuses_a_y_of_the_wrong_shape():
    h, x, pw, qw = dense_args()
    for bad in (bf(T - 1, D), bf(T, D - 8), bf(2 * T, D // 2)):
        with pytest.raises(ValueError, match="y must have shape"):
            snr.boundary_fused(h, x, pw, qw, 2, y=bad)


def test_moe_refuses_a_y_of_the_wrong_shape():
    h = bf(T, D)
    e = bf(T, 8, D)
    w = torch.zeros((T, 8), dtype=torch.float32)
    with pytest.raises(ValueError, match="y must have shape"):
        snr.moe_combine_boundary(h, e, w, bf(D), bf(D), 2, y=bf(T, D // 2))


def test_host_variants_refuse_a_y_of_the_wrong_shape():
    h, x, pw, qw = dense_args()
    with pytest.raises(ValueError, match="y must have shape"):
        snr.boundary_fused_host(h, x, pw, qw, 2, y=bf(T + 1, D))
    e = bf(T, 8, D)
    w = torch.zeros((T, 8), dtype=torch.float32)
    with pytest.raises(ValueError, match="y must have shape"):
        snr.moe_combine_boundary_host(h, e, w, pw, qw, 2, y=bf(T, 2 * D))


def test_mixed_devices_are_refused():
    h, x, pw, qw = dense_args()
    with pytest.raises(ValueError, match="one device"):
        snr.boundary_fused(h, x.to("meta"), pw, qw, 2)
    with pytest.raises(ValueError, match="one device"):
        snr.boundary_fused(h, x, pw, qw, 2, y=bf(T, D, device="meta"))
    e = bf(T, 8, D)
    w = torch.zeros((T, 8), dtype=torch.float32, device="meta")
    with pytest.raises(ValueError, match="one device"):
        snr.moe_combine_boundary(h, e, w, pw, qw, 2)


def test_cpu_operands_are_refused_by_the_device_calls():
    h, x, pw, qw = dense_args()
    with pytest.raises(ValueError, match="CUDA tensors"):
        snr.boundary_fused(h, x, pw, qw, 2)
    with pytest.raises(ValueError, match="CUDA tensors"):
        snr.boundary_fused_nvfp4(h, x, pw, qw, 2, 1e-6, 1.0)


def test_routing_and_qk_norm_check_their_outputs_and_weights():
    z = torch.zeros((T, 256), dtype=torch.float32)
    b = torch.zeros(256, dtype=torch.float32)
    with pytest.raises(ValueError, match="idx must have shape"):
        snr.moe_route(z, b, idx=torch.zeros((T, 4), dtype=torch.int32))
    with pytest.raises(ValueError, match="w must have shape"):
        snr.moe_route(z, b, w=torch.zeros((T + 1, 8), dtype=torch.float32))
    q, k = bf(T, 2, 128), bf(T, 1, 128)
    pos = torch.zeros(T, dtype=torch.int32)
    with pytest.raises(ValueError, match="q_w must have shape"):
        snr.qk_norm(q, k, bf(64), bf(128), pos, mode="ssmax")
    with pytest.raises(ValueError, match="rope_table"):
        snr.qk_norm(q, k, bf(128), bf(128), pos, mode="rope",
                    rope_table=torch.zeros((16, 64), dtype=torch.float32))
