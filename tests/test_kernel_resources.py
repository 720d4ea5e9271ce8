"""Register budgets that set how many CTAs of the default launch shapes fit on
an SM (65,536 registers, allocated per warp in steps of 8 per thread). Past
these budgets residency drops silently: the MoE boundary, built for 2 CTAs of
320 threads per SM, ran 38% slower when a code change left room for only 1.
Read from ptxas's resource summary (-Xptxas -v) of an sm_103a build; no GPU
needed."""
from __future__ import annotations

import re
import subprocess

import pytest

from sandwich_norm_residual_gb300 import build

REGFILE = 65536


@pytest.fixture(scope="module")
def registers(tmp_path_factory) -> dict[str, int]:
    out = tmp_path_factory.mktemp("res") / "lib.so"
    r = subprocess.run([build.nvcc()] + build.flags(True) + build.SOURCES + ["-o", str(out)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    regs, cur = {}, None
    for line in r.stderr.splitlines():
        m = re.search(r"Compiling entry function '(\w+)'", line)
        if m:
            cur = subprocess.run(["c++filt", m.group(1)], capture_output=True,
                                 text=True).stdout.strip()
        m = re.search(r"Used (\d+) registers", line)
        if m and cur:
            regs[cur] = int(m.group(1))
    return regs


def ctas_per_sm(regs: int, threads: int) -> int:
    per_thread = -(-regs // 8) * 8
    return REGFILE // (per_thread * threads)


def find(registers, pattern: str) -> int:
    hits = [v for k, v in registers.items() if pattern in k]
    assert len(hits) == 1, (pattern, [k for k in registers if pattern in k])
    return hits[0]


@pytest.mark.parametrize("quant", ["false", "true"])
def test_moe_boundary_keeps_two_ctas_of_320_threads(registers, quant):
    # D = 5120: 2 vectors per thread, 320 threads; the L2 rule asks for 2 CTAs/SM
    regs = find(registers, f"boundary_kernel<2, true, true, {quant}>")
    assert ctas_per_sm(regs, 320) >= 2, regs


@pytest.mark.parametrize("quant", ["false", "true"])
def test_dense_boundary_keeps_four_ctas_of_128_threads(registers, quant):
    regs = find(registers, f"boundary_kernel<5, false, true, {quant}>")
    assert ctas_per_sm(regs, 128) >= 4, regs


@pytest.mark.parametrize("mode", [0, 1])
def test_qk_norm_keeps_two_blocks_of_256_threads(registers, mode):
    # two 8-head batches in flight per warp, RoPE (mode 0) and SSMax alike
    assert ctas_per_sm(find(registers, f"qk_norm_kernel<{mode}>("), 256) >= 2


@pytest.mark.parametrize("params", ["8, 4, 8", "0, 0, 0"])
def test_routing_keeps_five_blocks_of_256_threads(registers, params):
    assert ctas_per_sm(find(registers, f"route_kernel<{params}>("), 256) >= 5
