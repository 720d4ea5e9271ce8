"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded input bytes.

Gate for every output (h' and y): each BF16 element within 1 ulp of the
oracle (ordered-integer distance) and >= 99.99% bit-identical. The kernels'
row sums are exact (certified compensated sum, exact integer fallback), so
these tests expect and report 100%.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
import sandwich_norm_residual_gb300 as snr
import synth
from parity import assert_parity, bits, compare
from sandwich_norm_residual_gb300 import build
from synth import (DECODE_CHAIN_T64, DENSE_DECODE_T4, DENSE_PREFILL_T16384, MOE_STRESS_T131072,
                   MOE_T16384)

pytestmark = pytest.mark.gpu
THREADS = max(1, min(32, os.cpu_count() or 1))
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    snr.library()
    torch.cuda.init()


def to_dev(inp: dict) -> dict:
    return {k: v.to(DEV) for k, v in inp.items()}


def gpu_dense(inp, n, eps, opts=None, stream=None):
    d = to_dev(inp)
    y = snr.boundary_fused(d["h"], d["x"], d["post_w"], d["pre_w"], n, eps, opts=opts,
                           stream=stream)
    snr.sync_status(stream)
    return bits(d["h"]), bits(y)


def gpu_moe(inp, n, eps, opts=None):
    d = to_dev(inp)
    y = snr.moe_combine_boundary(d["h"], d["expert_out"], d["topk_w"], d["post_w"], d["pre_w"],
                                 n, eps, opts=opts)
    snr.sync_status()
    return bits(d["h"]), bits(y)


def oracle_dense(inp, n, eps):
    return oracle.boundary(inp["h"], inp["x"], inp["post_w"], inp["pre_w"], n, eps,
                           threads=THREADS)


def oracle_moe(inp, n, eps):
    return oracle.moe_boundary(inp["h"], inp["expert_out"], inp["topk_w"], inp["post_w"],
                               inp["pre_w"], n, eps, threads=THREADS)


def check(got, want, label):
    st_h = assert_parity(got[0], want[0], f"{label} h'")
    st_y = assert_parity(got[1], want[1], f"{label} y")
    print(f"{label}: h' {st_h}  y {st_y}")
    return st_h, st_y


def bf16(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def random_dense(T, D, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return dict(h=bf16(rng.standard_normal((T, D))), x=bf16(rng.standard_normal((T, D)) * scale),
                post_w=bf16(1 + 0.1 * rng.standard_normal(D)),
                pre_w=bf16(1 + 0.1 * rng.standard_normal(D)))


# --------------------------------------------------------------- the five workloads

def test_dense_decode_T4():
    cfg = DENSE_DECODE_T4
    inp = synth.dense_inputs(cfg)
    check(gpu_dense(inp, cfg.n, cfg.eps), oracle_dense(inp, cfg.n, cfg.eps), cfg.name)


def test_decode_chain_T64_every_step_and_unit_variance():
    cfg = DECODE_CHAIN_T64
    h0 = synth.dense_inputs(cfg)["h"]
    h_gpu = h0.to(DEV)
    h_ref = oracle.as_u16(h0).copy()
    xn_sq = 0.0
    for s in range(cfg.steps):
        n = cfg.n + s
        inp = synth.dense_inputs(cfg, step=s)
        d = to_dev(inp)
        y = snr.boundary_fused(h_gpu, d["x"], d["post_w"], d["pre_w"], n, cfg.eps)
        h_ref, y_ref = oracle.boundary(h_ref, inp["x"], inp["post_w"], inp["pre_w"], n, cfg.eps,
                                       threads=THREADS)
        snr.sync_status()
        assert_parity(bits(h_gpu), h_ref, f"chain step {s} h'")
        assert_parity(bits(y), y_ref, f"chain step {s} y")
        xn = np.stack([oracle.rmsnorm(inp["x"][t], inp["post_w"], cfg.eps) for t in range(cfg.T)])
        xnf = (xn.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        xn_sq += float(np.mean(xnf * xnf))
    # depth scaling keeps the stream at (var(h_1) + sum_n mean(xn_n^2)) / N
    h1 = h0.float().numpy().astype(np.float64)
    pred = (np.mean(h1 * h1) + xn_sq) / (cfg.steps + 1)
    got = float(np.mean(h_gpu.float().cpu().numpy().astype(np.float64) ** 2))
    sigma = np.sqrt(2.0 / h1.size)
    assert abs(got - pred) < 5 * sigma, (got, pred)


def test_dense_prefill_T16384_full():
    cfg = DENSE_PREFILL_T16384
    inp = synth.dense_inputs(cfg)
    check(gpu_dense(inp, cfg.n, cfg.eps), oracle_dense(inp, cfg.n, cfg.eps), cfg.name)


def test_moe_T16384_full():
    cfg = MOE_T16384
    inp = synth.moe_inputs(cfg)
    check(gpu_moe(inp, cfg.n, cfg.eps), oracle_moe(inp, cfg.n, cfg.eps), cfg.name)


@pytest.mark.slow
def test_moe_stress_T131072_every_row():
    """T = 131072 on the GPU in one launch, then every row of h' and y against the
    oracle, row-parallel on the host cores. The 1024 sampled rows (half of them tokens
    with a x100 expert row) are compared first, as a quick sub-check."""
    cfg = MOE_STRESS_T131072
    T, D, K = cfg.T, cfg.D, cfg.K
    e_host = torch.empty((T, K, D), dtype=torch.bfloat16)
    chunk = 2048
    for r in range(0, T, chunk):
        synth.expert_rows(cfg, r, min(chunk, T - r), out=e_host[r:r + chunk])
    e = e_host.to(DEV)
    h_host = synth.to_bf16(synth.normal(cfg.seed, synth.STREAMS["h"], T * D).reshape(T, D))
    w_host = torch.from_numpy(synth.topk_weights(cfg.seed, synth.STREAMS["topk"], T, K,
                                                 cfg.route_scale))
    pw = synth.to_bf16(synth.normal(cfg.seed, synth.STREAMS["post_w"], D, 0, 0.1, 1.0))
    qw = synth.to_bf16(synth.normal(cfg.seed, synth.STREAMS["pre_w"], D, 0, 0.1, 1.0))
    h = h_host.to(DEV)
    y = snr.moe_combine_boundary(h, e, w_host.to(DEV), pw.to(DEV), qw.to(DEV), cfg.n, cfg.eps)
    snr.sync_status()
    del e
    h_out, y_out = bits(h), bits(y)
    del h, y

    def rows_input(idx):
        return dict(h=h_host[idx], expert_out=e_host[idx], topk_w=w_host[idx], post_w=pw, pre_w=qw)

    outl = synth.bernoulli(cfg.seed, synth.STREAMS["outlier"], T * K, cfg.outlier_p)
    outl_tok = np.unique(np.nonzero(outl)[0] // K)
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([rng.choice(outl_tok, min(512, outl_tok.size), replace=False),
                                     rng.choice(T, 512, replace=False)]))
    idx = torch.from_numpy(rows)
    check((h_out[rows], y_out[rows]), oracle_moe(rows_input(idx), cfg.n, cfg.eps),
          f"{cfg.name} ({rows.size} sampled rows)")

    same_h = same_y = 0
    for r in range(0, T, 8192):
        sl = slice(r, min(T, r + 8192))
        want_h, want_y = oracle_moe(rows_input(sl), cfg.n, cfg.eps)
        st_h = assert_parity(h_out[sl], want_h, f"{cfg.name} rows {r}.. h'")
        st_y = assert_parity(y_out[sl], want_y, f"{cfg.name} rows {r}.. y")
        same_h += st_h["identical"]
        same_y += st_y["identical"]
    n = T * D
    print(f"{cfg.name}: all {T} rows, h' {same_h / n:.6f} and y {same_y / n:.6f} bit-identical")
    assert same_h == n and same_y == n


# --------------------------------------------------------------- shapes and edge cases

@pytest.mark.parametrize("T,D,n", [(1, 5120, 2), (3, 5120, 104), (7, 5120, 105), (1000, 5120, 7),
                                   (5, 8, 2), (9, 128, 3), (33, 8192, 20), (2, 16, 1),
                                   (300, 4096, 52), (4, 32768, 9), (17, 1000, 5)])
def test_dense_shapes(T, D, n):
    inp = random_dense(T, D, seed=T * 7 + D)
    check(gpu_dense(inp, n, 1e-6), oracle_dense(inp, n, 1e-6), f"dense T={T} D={D} n={n}")


@pytest.mark.parametrize("T,D,n", [(1, 5120, 20), (3, 5120, 2), (257, 5120, 104), (6, 8, 3),
                                   (11, 2048, 1), (2, 32768, 50), (13, 1000, 4)])
def test_moe_shapes(T, D, n):
    rng = np.random.default_rng(T + D)
    z = rng.standard_normal((T, 8))
    s = 1 / (1 + np.exp(-z))
    inp = dict(h=bf16(rng.standard_normal((T, D))),
               expert_out=bf16(rng.standard_normal((T, 8, D))),
               topk_w=torch.from_numpy((2.5 * s / s.sum(1, keepdims=True)).astype(np.float32)),
               post_w=bf16(1 + 0.1 * rng.standard_normal(D)),
               pre_w=bf16(1 + 0.1 * rng.standard_normal(D)))
    check(gpu_moe(inp, n, 1e-6), oracle_moe(inp, n, 1e-6), f"moe T={T} D={D} n={n}")


def test_zero_rows_eps_zero_and_outlier_rows():
    T, D = 12, 5120
    inp = random_dense(T, D, seed=5)
    x = inp["x"].float()
    x[0] = 0.0                      # zero branch: r1 = 1/sqrt(eps)
    x[1] *= 100.0                   # outlier row
    x[2] *= 1e-25                   # tiny: squares underflow or turn subnormal
    x[3, ::7] *= 3e4                # a few huge elements
    x[4] = 1e19                     # squares near the FP32 range; the sum overflows
    inp["x"] = x.to(torch.bfloat16)
    h = inp["h"].float()
    h[5] = 0.0
    inp["h"] = h.to(torch.bfloat16)
    for eps in (1e-6, 0.0):
        if eps == 0.0:
            inp["x"][0] = inp["x"][6]  # eps = 0 only on rows that are not all zero
            inp["h"][5] = inp["h"][7]
        check(gpu_dense(inp, 3, eps), oracle_dense(inp, 3, eps), f"edge rows eps={eps}")


def test_non_finite_inputs_propagate_like_the_oracle():
    T, D = 4, 512
    inp = random_dense(T, D, seed=6)
    inp["x"][0, 5] = float("inf")
    inp["x"][1, 9] = float("nan")
    inp["h"][2, 3] = float("-inf")
    check(gpu_dense(inp, 2, 1e-6), oracle_dense(inp, 2, 1e-6), "non-finite")


def test_rows_at_rounding_ties_take_the_exact_path():
    """Rows whose exact sum of squares sits on (or within 2^-40 of) an FP32
    midpoint cannot be certified; the exact path must decide, bit for bit."""
    T, D = 8, 5120
    rng = np.random.default_rng(8)
    x = np.zeros((T, D), np.float32)
    for t in range(T):
        x[t, 0] = 1.0
        x[t, 1] = 2.0 ** -12            # square 2^-24: 1 + 2^-24 is an FP32 tie
        if t % 2:
            x[t, 2] = 2.0 ** -20        # square 2^-40 breaks the tie upwards
        x[t, 3:3 + 64] = rng.choice([2.0 ** -30, 0.0], 64).astype(np.float32)
    inp = dict(h=bf16(rng.standard_normal((T, D))), x=bf16(x),
               post_w=bf16(np.ones(D)), pre_w=bf16(np.ones(D)))
    snr.exact_sum_count(reset=True)
    check(gpu_dense(inp, 2, 0.0), oracle_dense(inp, 2, 0.0), "tie rows")
    assert snr.exact_sum_count() >= T


def test_launch_shape_does_not_change_a_bit():
    T, D = 200, 5120
    inp = random_dense(T, D, seed=10)
    ref = None
    shapes = [dict(vec_per_thread=v, ctas_per_sm=c, stages=st)
              for v in (2, 3, 4, 5, 6, 7, 8)  # one vector per thread would need 640 threads
              for c in (0, 1) for st in (-1, 0)]
    shapes += [dict(vec_per_thread=5, stages=st, ctas_per_sm=c) for st in (2, 3, 5, 8)
               for c in (0, 1, 3)]
    shapes += [dict(stages=-1, prefetch_rows=pf) for pf in (-1, 1, 4)]
    for opts in shapes:
        got = gpu_dense(inp, 11, 1e-6, opts=opts)
        if ref is None:
            ref = got
            check(got, oracle_dense(inp, 11, 1e-6), "launch-shape sweep reference")
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), opts


def test_moe_launch_shape_does_not_change_a_bit():
    cfg = MOE_T16384
    m = synth.moe_inputs(cfg, rows=96)
    ref = gpu_moe(m, cfg.n, cfg.eps)
    check(ref, oracle_moe(m, cfg.n, cfg.eps), "moe launch-shape reference")
    for v in (2, 3, 4, 5, 8):
        for pf in (-1, 1, 3):
            got = gpu_moe(m, cfg.n, cfg.eps, opts=dict(vec_per_thread=v, prefetch_rows=pf))
            assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), (v, pf)


def test_ring_kernel_at_a_hidden_size_where_fewer_slots_fit():
    # 4 * D bytes per slot: D = 16384 leaves room for three slots, D = 32768 for none
    for T, D in ((40, 16384), (5, 32768)):
        inp = random_dense(T, D, seed=D)
        check(gpu_dense(inp, 3, 1e-6), oracle_dense(inp, 3, 1e-6), f"ring D={D}")


def test_bounded_wait_runs_out_reports_timeout_and_leaves_later_rows_untouched():
    """The test hook withholds the bulk copy of each CTA's second row. That slot wait gives
    up after 1 ms; the CTA stores nothing for that row or any later one (h and y keep
    their bytes), drains its copies in flight and returns; the status word reports the
    timeout. Each CTA's first row (rows 0 .. grid-1) is computed exactly. The context
    stays usable."""
    T, D = 2048, 5120
    inp = random_dense(T, D, seed=16)
    d = to_dev(inp)
    sentinel = 0x40E0  # BF16 7.0
    y = torch.full((T, D), 7.0, dtype=torch.bfloat16, device=DEV)
    opts = dict(flags=snr._lib.BEAM_OPT_TEST_WAIT_TIMEOUT)
    snr.boundary_fused(d["h"], d["x"], d["post_w"], d["pre_w"], 5, 1e-6, y=y, opts=opts)
    with pytest.raises(snr.BeamError) as ei:
        snr.sync_status()
    assert ei.value.status == snr._lib.BEAM_ERR_TIMEOUT
    h_out, y_out = bits(d["h"]), bits(y)
    h_in = oracle.as_u16(inp["h"])
    written = (y_out != sentinel).any(1)
    G = int(written.sum())
    assert 1 <= G < T and written[:G].all(), G  # exactly the first row of every CTA
    want_h, want_y = oracle_dense(inp, 5, 1e-6)
    assert np.array_equal(h_out[:G], want_h[:G]) and np.array_equal(y_out[:G], want_y[:G])
    assert np.array_equal(h_out[G:], h_in[G:]) and (y_out[G:] == sentinel).all()
    print(f"timed-out launch: {G} first rows computed, {T - G} rows untouched")
    # the status was cleared and the context still works
    snr.sync_status()
    check(gpu_dense(inp, 5, 1e-6), oracle_dense(inp, 5, 1e-6), "next call")


def test_forced_exact_path_is_bit_identical_and_counted():
    T, D = 300, 5120
    inp = random_dense(T, D, seed=12)
    fast = gpu_dense(inp, 4, 1e-6)
    snr.exact_sum_count(reset=True)
    exact = gpu_dense(inp, 4, 1e-6, opts=dict(flags=snr._lib.BEAM_OPT_FORCE_EXACT_SUM))
    assert snr.exact_sum_count() == 2 * T
    assert np.array_equal(fast[0], exact[0]) and np.array_equal(fast[1], exact[1])
    cfg = MOE_T16384
    m = synth.moe_inputs(cfg, rows=64)
    a = gpu_moe(m, cfg.n, cfg.eps)
    b = gpu_moe(m, cfg.n, cfg.eps, opts=dict(flags=snr._lib.BEAM_OPT_FORCE_EXACT_SUM))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    check(b, oracle_moe(m, cfg.n, cfg.eps), "moe forced exact")


def test_certification_is_rare_on_the_prefill_workload():
    cfg = DENSE_PREFILL_T16384
    inp = synth.dense_inputs(cfg)
    snr.exact_sum_count(reset=True)
    gpu_dense(inp, cfg.n, cfg.eps)
    n_exact = snr.exact_sum_count()
    print(f"exact-path row sums: {n_exact} of {2 * cfg.T}")
    assert n_exact <= 2 * cfg.T * 1e-3


def test_branch_may_be_the_stream_itself():
    T, D = 16, 5120
    inp = random_dense(T, D, seed=13)
    d = to_dev(inp)
    y = snr.boundary_fused(d["h"], d["h"], d["post_w"], d["pre_w"], 6, 1e-6)
    snr.sync_status()
    want = oracle.boundary(inp["h"], inp["h"], inp["post_w"], inp["pre_w"], 6, 1e-6)
    check((bits(d["h"]), bits(y)), want, "x is h")


def test_guard_bands_and_untouched_neighbours():
    """Operands sit inside larger buffers filled with a canary; nothing outside
    the operands may change (a bounds check without compute-sanitizer)."""
    T, D, pad = 37, 5120, 4096
    inp = random_dense(T, D, seed=14)
    canary = torch.tensor(0x7E5A, dtype=torch.int16)

    def padded(t):
        flat = torch.full((t.numel() + 2 * pad,), 0x7E5A, dtype=torch.int16, device=DEV)
        flat[pad:pad + t.numel()].copy_(t.reshape(-1).view(torch.int16))
        return flat

    bufs = {k: padded(v) for k, v in inp.items()}
    ybuf = torch.full((T * D + 2 * pad,), 0x7E5A, dtype=torch.int16, device=DEV)
    view = {k: b[pad:pad + inp[k].numel()].view(torch.bfloat16).reshape(inp[k].shape)
            for k, b in bufs.items()}
    y = ybuf[pad:pad + T * D].view(torch.bfloat16).reshape(T, D)
    snr.boundary_fused(view["h"], view["x"], view["post_w"], view["pre_w"], 2, 1e-6, y=y)
    snr.sync_status()
    for b in list(bufs.values()) + [ybuf]:
        assert (b[:pad] == canary).all() and (b[-pad:] == canary).all()
    assert torch.equal(bufs["x"][pad:-pad].cpu(), inp["x"].reshape(-1).view(torch.int16))
    check((bits(view["h"]), bits(y)), oracle_dense(inp, 2, 1e-6), "guard bands")


def test_zero_tokens_is_a_no_op_and_streams_are_honoured():
    h = torch.zeros((0, 5120), dtype=torch.bfloat16, device=DEV)
    w = torch.ones(5120, dtype=torch.bfloat16, device=DEV)
    y = snr.boundary_fused(h, h, w, w, 2, 1e-6)
    assert y.shape == (0, 5120)
    inp = random_dense(64, 5120, seed=15)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got = gpu_dense(inp, 9, 1e-6, stream=s)
    check(got, oracle_dense(inp, 9, 1e-6), "side stream")


# --------------------------------------------------------------- decode chain: graphs and PDL

def _chain_inputs(cfg):
    steps = [synth.dense_inputs(cfg, step=s) for s in range(cfg.steps)]
    return synth.dense_inputs(cfg)["h"], steps


@pytest.mark.parametrize("pdl", [False, True])
@pytest.mark.parametrize("graph", [False, True])
def test_decode_chain_with_cuda_graph_and_pdl_matches_the_oracle(pdl, graph):
    """All 104 boundaries of the T = 64 decode chain back to back on one stream
    (optionally captured in one CUDA graph, optionally with programmatic
    dependent launches); every step's y and the final stream are exact."""
    cfg = DECODE_CHAIN_T64
    h0, steps = _chain_inputs(cfg)
    dev_steps = [to_dev(s) for s in steps]
    h = h0.to(DEV)
    ys = [torch.empty_like(h) for _ in steps]
    opts = dict(flags=snr._lib.BEAM_OPT_PDL) if pdl else None
    stream = torch.cuda.Stream()

    def run_chain():
        for s, d in enumerate(dev_steps):
            snr.boundary_fused(h, d["x"], d["post_w"], d["pre_w"], cfg.n + s, cfg.eps, y=ys[s],
                               opts=opts, stream=stream)

    with torch.cuda.stream(stream):
        run_chain()  # first call on the device sets up the launch shapes (before any capture)
    torch.cuda.synchronize()
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run_chain()
        h.copy_(h0.to(DEV))
        for y in ys:
            y.zero_()
        torch.cuda.synchronize()
        g.replay()
    else:
        h.copy_(h0.to(DEV))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            run_chain()
    torch.cuda.synchronize()
    snr.sync_status()

    h_ref = oracle.as_u16(h0).copy()
    for s, inp in enumerate(steps):
        h_ref, y_ref = oracle.boundary(h_ref, inp["x"], inp["post_w"], inp["pre_w"], cfg.n + s,
                                       cfg.eps, threads=THREADS)
        assert_parity(bits(ys[s]), y_ref, f"chain step {s} y (graph={graph}, pdl={pdl})")
    check((bits(h), bits(ys[-1])), (h_ref, y_ref), f"chain graph={graph} pdl={pdl}")


def test_pdl_on_the_prefill_and_moe_workloads():
    cfg = DENSE_PREFILL_T16384
    inp = synth.dense_inputs(cfg, rows=2048)
    opts = dict(flags=snr._lib.BEAM_OPT_PDL)
    check(gpu_dense(inp, cfg.n, cfg.eps, opts=opts), oracle_dense(inp, cfg.n, cfg.eps), "dense pdl")
    m = synth.moe_inputs(MOE_T16384, rows=512)
    check(gpu_moe(m, 20, 1e-6, opts=opts), oracle_moe(m, 20, 1e-6), "moe pdl")
    check(gpu_dense(inp, cfg.n, cfg.eps, opts=dict(flags=snr._lib.BEAM_OPT_PDL, stages=2)),
          oracle_dense(inp, cfg.n, cfg.eps), "dense ring pdl")


# --------------------------------------------------------------- routing and the scaled combine

def _router_inputs(T, seed):
    z = (synth.normal(seed, 8, T * 256) * 2.0).reshape(T, 256).astype(np.float32)
    b = (synth.normal(seed, 9, 256) * 0.05).astype(np.float32)
    return z, b


def _check_routing(idx_g, w_g, idx_o, w_o, label):
    """Expert ids are index work and the weights are FP32 results of exact steps (the
    sigmoid is correctly rounded on both sides): both must be identical, bit for bit
    (NaN weights: NaN on both sides)."""
    same = (idx_g == idx_o).all(1)
    assert same.all(), (label, np.nonzero(~same)[0][:5], idx_g[~same][:2], idx_o[~same][:2])
    nan = np.isnan(w_o)
    assert np.array_equal(np.isnan(w_g), nan), label
    assert np.array_equal(w_g.view(np.uint32)[~nan], w_o.view(np.uint32)[~nan]), label
    print(f"{label}: {idx_g.shape[0]} tokens, identical experts and weights")


@pytest.mark.parametrize("ng,tg,k,scale", [(8, 4, 8, 2.5), (1, 1, 8, 1.0), (32, 4, 6, 1.0),
                                           (4, 2, 16, 2.5)])
def test_routing_matches_the_oracle(ng, tg, k, scale):
    T = 16384 if (ng, tg, k) == (8, 4, 8) else 1024
    z, b = _router_inputs(T, 3)
    idx_g, w_g = snr.moe_route(torch.from_numpy(z).to(DEV), torch.from_numpy(b).to(DEV), ng, tg, k,
                               scale)
    snr.sync_status()
    idx_o, w_o = oracle.route(z, b, ng, tg, k, scale, threads=THREADS)
    _check_routing(idx_g.cpu().numpy(), w_g.cpu().numpy(), idx_o, w_o,
                   f"route ng={ng} tg={tg} k={k}")


@pytest.mark.parametrize("ng,tg,k", [(8, 4, 8), (4, 2, 16)])
def test_routing_chain_with_pdl_in_a_cuda_graph(ng, tg, k):
    """Eight routings back to back as programmatic dependent launches in one CUDA
    graph, each writing its weights over the first logits of the next one: every
    layer's ids and weights equal the oracle run in sequence, so no launch read
    its logits before the launch in front of it had written them. (8, 4, 8) runs
    the compiled Beam router, (4, 2, 16) the kernel with run-time parameters."""
    T, L = 64, 8
    rng = np.random.default_rng(77 + k)
    z = [(rng.standard_normal((T, 256)) * 2).astype(np.float32) for _ in range(L + 1)]
    b = (rng.standard_normal(256) * 0.05).astype(np.float32)
    dz = [torch.from_numpy(t).to(DEV) for t in z]
    db = torch.from_numpy(b).to(DEV)
    idx = [torch.empty((T, k), dtype=torch.int32, device=DEV) for _ in range(L)]
    w = [dz[i + 1].view(-1)[:T * k].view(T, k) for i in range(L)]  # layer i's weights: layer i+1's logits
    stream = torch.cuda.Stream()

    def run():
        for i in range(L):
            snr.moe_route(dz[i], db, ng, tg, k, idx=idx[i], w=w[i], stream=stream, pdl=True)

    with torch.cuda.stream(stream):
        run()
    torch.cuda.synchronize()
    for t, d in zip(z, dz):
        d.copy_(torch.from_numpy(t).to(DEV))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    g.replay()
    torch.cuda.synchronize()
    snr.sync_status()
    zc = [t.copy() for t in z]
    for i in range(L):
        idx_o, w_o = oracle.route(zc[i], b, ng, tg, k)
        zc[i + 1].reshape(-1)[:T * k] = w_o.reshape(-1)
        _check_routing(idx[i].cpu().numpy(), w[i].cpu().numpy(), idx_o, w_o, f"route pdl layer {i}")


def test_routing_with_infinite_and_extreme_logits():
    """Logits of +-inf, +-100, -95 (a subnormal sigmoid) and +-50 beside ordinary ones:
    the sigmoid saturates to exactly 1, underflows to 0 or is a subnormal, on both sides
    alike."""
    T = 2048
    z, b = _router_inputs(T, 13)
    rng = np.random.default_rng(13)
    extremes = np.array([np.inf, -np.inf, 100.0, -100.0, -95.0, 50.0, -50.0], np.float32)
    pick = rng.random((T, 256)) < 0.05
    z[pick] = extremes[rng.integers(0, extremes.size, int(pick.sum()))]
    idx_g, w_g = snr.moe_route(torch.from_numpy(z).to(DEV), torch.from_numpy(b).to(DEV))
    snr.sync_status()
    idx_o, w_o = oracle.route(z, b, threads=THREADS)
    assert np.isfinite(w_g.cpu().numpy()).all()
    _check_routing(idx_g.cpu().numpy(), w_g.cpu().numpy(), idx_o, w_o, "route extreme logits")


@pytest.mark.parametrize("ng,tg,k", [(8, 4, 8), (4, 2, 16), (32, 4, 6), (1, 1, 8)])
def test_routing_with_nan_logits_and_non_finite_bias(ng, tg, k):
    """NaN logits (2% of them, and whole NaN groups on some tokens), a NaN, a +inf and a
    -inf correction bias: NaN scores rank below every number on both sides, so the same
    experts are chosen; weights that involve a NaN score are NaN on both sides."""
    T = 2048
    z, b = _router_inputs(T, 14)
    rng = np.random.default_rng(14)
    z[rng.random((T, 256)) < 0.02] = np.nan
    for t in range(16):
        g = t % 8
        z[t, 32 * g:32 * g + 32] = np.nan
    b[7], b[100], b[200] = np.nan, np.inf, -np.inf
    idx_g, w_g = snr.moe_route(torch.from_numpy(z).to(DEV), torch.from_numpy(b).to(DEV), ng, tg, k,
                               2.5)
    snr.sync_status()
    idx_o, w_o = oracle.route(z, b, ng, tg, k, 2.5, threads=THREADS)
    _check_routing(idx_g.cpu().numpy(), w_g.cpu().numpy(), idx_o, w_o,
                   f"route NaN ng={ng} tg={tg} k={k}")


@pytest.mark.slow
def test_router_sigmoid_every_float_matches_the_oracle():
    """All 2^32 float inputs through the kernel's sigmoid (beam_router_sigmoid, the
    function the router scores with) against the oracle's correctly rounded sigmoid:
    identical bits (NaN inputs: NaN outputs). The routing first pass's fast sigmoid
    (beam_router_sigmoid_fast) must stay within 2^-19 of the exact sigmoid on every
    input: within 2^-19 - 2^-25 of the oracle's value, itself within half an ulp
    (at most 2^-25) of the exact one."""
    chunk = 1 << 28
    bad = bad_fast = 0
    worst = 0.0
    for c in range((1 << 32) // chunk):
        lo = c * chunk
        start = lo if lo < (1 << 31) else lo - (1 << 32)
        zg = torch.arange(start, start + chunk, dtype=torch.int32, device=DEV).view(torch.float32)
        sg = snr.router_sigmoid(zg)
        fg = snr.router_sigmoid(zg, fast=True)
        snr.sync_status()
        got = sg.cpu().numpy().view(np.uint32)
        fast = fg.cpu().numpy()
        del zg, sg, fg
        z = np.arange(lo, lo + chunk, dtype=np.uint32).view(np.float32)
        want = oracle.sigmoid_array(z, threads=THREADS)
        nan = np.isnan(z)
        diff = (got != want.view(np.uint32)) & ~nan
        diff |= nan & ~np.isnan(got.view(np.float32))
        n = int(diff.sum())
        if n:
            print("first differences:", [hex(lo + int(i)) for i in np.nonzero(diff)[0][:5]])
        bad += n
        with np.errstate(invalid="ignore"):
            err = np.abs(fast.astype(np.float64) - want.astype(np.float64))
        err[nan] = 0.0
        nf = int((err > 2.0 ** -19 - 2.0 ** -25).sum()) + int((nan & ~np.isnan(fast)).sum())
        if nf:
            print("fast sigmoid beyond its bound at", [hex(lo + int(i)) for i in np.nonzero(err > 2.0 ** -19 - 2.0 ** -25)[0][:5]])
        bad_fast += nf
        worst = max(worst, float(err.max()))
    print(f"fast sigmoid: largest distance to the correctly rounded value {worst:.3g} (2^{np.log2(worst):.2f})")
    assert bad == 0 and bad_fast == 0
    assert oracle.sigmoid_undecided() == 0


@pytest.mark.parametrize("ng,tg,k", [(8, 4, 8), (4, 2, 16), (32, 4, 6)])
def test_routing_exact_ties_go_to_the_lower_index(ng, tg, k):
    """Logits drawn from five values with no bias: experts, and often whole groups, tie
    exactly. Equal logits give equal scores on each side, and no two different pairs of
    the five scores sum to nearly the same group score, so both sides see the same ties
    and must break every one towards the lower index: identical selections on every
    token."""
    vals = np.array([0.3, 0.7, 1.1, 1.9, 2.6], np.float32)
    sig = 1.0 / (1.0 + np.exp(-vals.astype(np.float64)))
    pair_sums = np.sort([sig[i] + sig[j] for i in range(5) for j in range(i, 5)])
    assert np.diff(pair_sums).min() > 1e-3
    rng = np.random.default_rng(71)
    T = 4096
    hi = rng.integers(1, 6, (T, 8))  # group g of token t draws from the first hi values
    z = np.empty((T, 256), np.float32)
    for g in range(8):
        z[:, 32 * g:32 * (g + 1)] = vals[(rng.random((T, 32)) * hi[:, g:g + 1]).astype(int)]
    b = np.zeros(256, np.float32)
    idx_g, w_g = snr.moe_route(torch.from_numpy(z).to(DEV), torch.from_numpy(b).to(DEV), ng, tg, k,
                               2.5)
    snr.sync_status()
    idx_o, w_o = oracle.route(z, b, ng, tg, k, 2.5, threads=THREADS)
    _check_routing(idx_g.cpu().numpy(), w_g.cpu().numpy(), idx_o, w_o, f"route ties ng={ng}")


def test_routing_then_the_scaled_combine_boundary():
    """route (weights without the scale) -> boundary with the scale applied in the combine;
    and scale 1 reproduces the plain combine bit for bit."""
    cfg = MOE_T16384
    T = 512
    z, b = _router_inputs(T, 5)
    _, w = snr.moe_route(torch.from_numpy(z).to(DEV), torch.from_numpy(b).to(DEV), route_scale=1.0)
    m = synth.moe_inputs(cfg, rows=T)
    m["topk_w"] = w.cpu()
    d = to_dev(m)
    y = snr.moe_combine_boundary(d["h"], d["expert_out"], d["topk_w"], d["post_w"], d["pre_w"],
                                 cfg.n, cfg.eps, route_scale=2.5)
    snr.sync_status()
    want = oracle.moe_boundary(m["h"], m["expert_out"], m["topk_w"], m["post_w"], m["pre_w"],
                               cfg.n, cfg.eps, threads=THREADS, route_scale=2.5)
    check((bits(d["h"]), bits(y)), want, "route + scaled combine")
    d1 = to_dev(m)
    y1 = snr.moe_combine_boundary(d1["h"], d1["expert_out"], d1["topk_w"], d1["post_w"],
                                  d1["pre_w"], cfg.n, cfg.eps, route_scale=1.0)
    plain = gpu_moe(m, cfg.n, cfg.eps)
    assert np.array_equal(bits(d1["h"]), plain[0]) and np.array_equal(bits(y1), plain[1])


# --------------------------------------------------------------- per-head Q/K norm with RoPE / SSMax

def _qk_case(T, nq, nk, seed, max_pos):
    rng = np.random.default_rng(seed)
    q = bf16(rng.standard_normal((T, nq, 128)) * 2)
    k = bf16(rng.standard_normal((T, nk, 128)) * 2)
    qw = bf16(1 + 0.1 * rng.standard_normal(128))
    kw = bf16(1 + 0.1 * rng.standard_normal(128))
    pos = torch.from_numpy(rng.integers(0, max_pos, T).astype(np.int32))
    inv = 10000.0 ** (-np.arange(0, 128, 2) / 128.0)
    ang = np.arange(max_pos)[:, None] * inv[None, :]
    table = torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], 1).astype(np.float32))
    return q, k, qw, kw, pos, table


@pytest.mark.parametrize("mode", ["rope", "ssmax"])
# T = 16384: one warp walks all 7 batches of its token; T = 700 and 1000: a
# token's batches split over several warps of 2 or 3 batches each (ragged last
# batch at 45 + 7 heads), which runs the two-batch pipeline on short runs
@pytest.mark.parametrize("T,nq,nk", [(16384, 48, 8), (5, 3, 1), (33, 48, 8), (7, 0, 8), (2, 48, 0),
                                     (700, 48, 8), (1000, 45, 7)])
def test_qk_norm_matches_the_oracle(mode, T, nq, nk):
    max_pos = 4096 if mode == "rope" else 1 << 20
    q, k, qw, kw, pos, table = _qk_case(T, nq, nk, T + nq, max_pos if mode == "rope" else 64)
    if mode == "ssmax":
        pos = torch.from_numpy(np.random.default_rng(T).integers(0, max_pos, T).astype(np.int32))
    dq, dk = q.to(DEV), k.to(DEV)
    snr.qk_norm(dq, dk, qw.to(DEV), kw.to(DEV), pos.to(DEV), 1e-6, mode,
                rope_table=table.to(DEV) if mode == "rope" else None)
    snr.sync_status()
    wq, wk = oracle.qk_norm(q, k, qw, kw, pos, table if mode == "rope" else None, 1e-6, mode,
                            threads=THREADS)
    st_q = assert_parity(bits(dq), wq, f"qk {mode} q") if nq else None
    st_k = assert_parity(bits(dk), wk, f"qk {mode} k") if nk else None
    print(f"qk_norm {mode} T={T} nq={nq} nk={nk}: q {st_q} k {st_k}")


@pytest.mark.parametrize("mode", ["rope", "ssmax"])
def test_qk_norm_non_finite_and_zero_heads_match_the_oracle(mode):
    """Beside finite heads: a NaN element (its head goes NaN), +-inf elements (the
    head's factor is 0, so NaN at the element, and under RoPE at its rotation
    partner, zeros elsewhere) and an all-zero head; every output identical."""
    q, k, qw, kw, pos, table = _qk_case(9, 48, 8, 91, 512)
    q[0, 1, 7] = float("nan")
    q[1, 0, 70] = float("inf")
    k[2, 1, 3] = float("-inf")
    q[3, 2, :] = 0.0
    k[4, 0, 64] = float("nan")
    dq, dk = q.to(DEV), k.to(DEV)
    snr.qk_norm(dq, dk, qw.to(DEV), kw.to(DEV), pos.to(DEV), 1e-6, mode,
                rope_table=table.to(DEV) if mode == "rope" else None)
    snr.sync_status()
    wq, wk = oracle.qk_norm(q, k, qw, kw, pos, table if mode == "rope" else None, 1e-6, mode)
    for got, want, name in ((bits(dq), wq, "q"), (bits(dk), wk, "k")):
        st = compare(got, want)
        assert st["frac_identical"] == 1.0, (mode, name, st)


def test_ssmax_scale_at_every_position_below_a_million():
    """End to end at all 2^20 positions: a query head of ones, norm weight 1 and eps 0
    give out = bf16(g), which must equal the BF16 rounding of the oracle's scale (the
    FP32 midpoint selection itself is checked exhaustively on the CPU in
    test_ssmax_method.py; BF16 output shows only the top 8 bits of g)."""
    T = 1 << 20
    q = torch.ones((T, 1, 128), dtype=torch.bfloat16)
    k = torch.ones((T, 0, 128), dtype=torch.bfloat16)
    w = torch.ones(128, dtype=torch.bfloat16)
    pos = torch.arange(T, dtype=torch.int32)
    dq = q.to(DEV)
    snr.qk_norm(dq, k.to(DEV), w.to(DEV), w.to(DEV), pos.to(DEV), 0.0, "ssmax")
    snr.sync_status()
    want = np.array([oracle.ssmax_scale(p) for p in range(T)], np.float32)
    got = bits(dq[:, 0, 0]).astype(np.uint32) << 16
    assert np.array_equal(got, bits(torch.from_numpy(want).to(torch.bfloat16)).astype(np.uint32) << 16)


def test_qk_norm_forced_exact_path_and_bad_positions():
    q, k, qw, kw, pos, table = _qk_case(64, 48, 8, 90, 512)
    a = (q.to(DEV), k.to(DEV))
    snr.qk_norm(*a, qw.to(DEV), kw.to(DEV), pos.to(DEV), 1e-6, "rope", rope_table=table.to(DEV))
    snr.exact_sum_count(reset=True)
    b = (q.to(DEV), k.to(DEV))
    snr.qk_norm(*b, qw.to(DEV), kw.to(DEV), pos.to(DEV), 1e-6, "rope", rope_table=table.to(DEV),
                force_exact=True)
    assert snr.exact_sum_count() == 64 * 56
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    # a token with a position outside the table is left as it was and reported
    bad = pos.clone()
    bad[3] = 512
    c = (q.to(DEV), k.to(DEV))
    snr.qk_norm(*c, qw.to(DEV), kw.to(DEV), bad.to(DEV), 1e-6, "rope", rope_table=table.to(DEV))
    with pytest.raises(snr.BeamError) as ei:
        snr.sync_status()
    assert ei.value.status == snr._lib.BEAM_ERR_ARG
    assert torch.equal(c[0][3].cpu(), q[3]) and torch.equal(c[1][3].cpu(), k[3])
    keep = torch.arange(64) != 3
    assert torch.equal(c[0][keep], a[0][keep])
    snr.sync_status()  # cleared


# --------------------------------------------------------------- y as NVFP4

def gpu_dense_nvfp4(inp, n, eps, gs, opts=None, stream=None):
    d = to_dev(inp)
    q, sf = snr.boundary_fused_nvfp4(d["h"], d["x"], d["post_w"], d["pre_w"], n, eps, gs,
                                     opts=opts, stream=stream)
    snr.sync_status(stream)
    return bits(d["h"]), q.cpu().numpy(), sf.cpu().numpy()


def gpu_moe_nvfp4(inp, n, eps, gs, opts=None):
    d = to_dev(inp)
    q, sf = snr.moe_combine_boundary_nvfp4(d["h"], d["expert_out"], d["topk_w"], d["post_w"],
                                           d["pre_w"], n, eps, gs, opts=opts)
    snr.sync_status()
    return bits(d["h"]), q.cpu().numpy(), sf.cpu().numpy()


def check_nvfp4(got, want, label):
    """h' bit for bit; every E2M1 code byte and E4M3 scale byte identical."""
    assert_parity(got[0], want[0], f"{label} h'")
    for g, w, name in ((got[1], want[1], "codes"), (got[2], want[2], "scales")):
        assert g.shape == w.shape, (label, name, g.shape, w.shape)
        bad = np.argwhere(g != w)
        assert bad.size == 0, (f"{label} {name}: {len(bad)} of {g.size} bytes differ, first at "
                               f"{bad[:4].tolist()}: got {g[tuple(bad[0])]:#04x} "
                               f"want {w[tuple(bad[0])]:#04x}")
    print(f"{label}: h' identical, {got[1].size} code bytes and {got[2].size} scales identical")


# 448 * 6 / amax(y) with amax(y) near 8 is the usual per-tensor scale; the
# others drive the E4M3 scales subnormal, to zero, and into saturation
GLOBAL_SCALES = (336.0, 1.0, 1e-3, 1e5)


def test_nvfp4_dense_prefill_full():
    cfg = DENSE_PREFILL_T16384
    inp = synth.dense_inputs(cfg)
    want = oracle.boundary_nvfp4(inp["h"], inp["x"], inp["post_w"], inp["pre_w"], cfg.n, cfg.eps,
                                 336.0, threads=THREADS)
    check_nvfp4(gpu_dense_nvfp4(inp, cfg.n, cfg.eps, 336.0), want, f"{cfg.name} nvfp4")


def test_nvfp4_moe_full():
    cfg = MOE_T16384
    inp = synth.moe_inputs(cfg)
    want = oracle.moe_boundary_nvfp4(inp["h"], inp["expert_out"], inp["topk_w"], inp["post_w"],
                                     inp["pre_w"], cfg.n, cfg.eps, 336.0, threads=THREADS)
    check_nvfp4(gpu_moe_nvfp4(inp, cfg.n, cfg.eps, 336.0), want, f"{cfg.name} nvfp4")


@pytest.mark.parametrize("gs", GLOBAL_SCALES)
def test_nvfp4_global_scales_and_zero_and_outlier_rows(gs):
    T, D = 40, 5120
    inp = random_dense(T, D, seed=21)
    x = inp["x"].float()
    x[0] = 0.0          # y is pre_w-scaled h' alone
    x[1] *= 100.0       # outlier branch
    x[2, ::16] *= 3e4   # one huge element in every block
    inp["x"] = x.to(torch.bfloat16)
    h = inp["h"].float()
    h[3] = 0.0
    h[3, 17] = 1.0      # one non-zero block in a row
    h[4, :32] = 0.0     # whole blocks of zeros: sf = 0
    inp["h"] = h.to(torch.bfloat16)
    want = oracle.boundary_nvfp4(inp["h"], inp["x"], inp["post_w"], inp["pre_w"], 3, 1e-6, gs)
    check_nvfp4(gpu_dense_nvfp4(inp, 3, 1e-6, gs), want, f"nvfp4 gs={gs}")


@pytest.mark.parametrize("T,D,n", [(1, 16, 2), (5, 48, 3), (257, 528, 7), (3, 5136, 104),
                                   (17, 16384, 11), (2, 32768, 5)])
def test_nvfp4_shapes(T, D, n):
    inp = random_dense(T, D, seed=T * 31 + D)
    want = oracle.boundary_nvfp4(inp["h"], inp["x"], inp["post_w"], inp["pre_w"], n, 1e-6, 336.0)
    check_nvfp4(gpu_dense_nvfp4(inp, n, 1e-6, 336.0), want, f"nvfp4 T={T} D={D}")
    rng = np.random.default_rng(D)
    m = dict(h=inp["h"], expert_out=bf16(rng.standard_normal((T, 8, D))),
             topk_w=torch.from_numpy(rng.uniform(0, 0.4, (T, 8)).astype(np.float32)),
             post_w=inp["post_w"], pre_w=inp["pre_w"])
    want = oracle.moe_boundary_nvfp4(m["h"], m["expert_out"], m["topk_w"], m["post_w"], m["pre_w"],
                                     n, 1e-6, 336.0)
    check_nvfp4(gpu_moe_nvfp4(m, n, 1e-6, 336.0), want, f"moe nvfp4 T={T} D={D}")


def test_nvfp4_launch_shapes_forced_exact_and_pdl():
    """Every vectors-per-thread choice, the exact row-sum path (for MoE it parks
    the combined x in the h row), and PDL give the same bytes."""
    T, D = 96, 5120
    inp = random_dense(T, D, seed=22)
    want = oracle.boundary_nvfp4(inp["h"], inp["x"], inp["post_w"], inp["pre_w"], 9, 1e-6, 336.0)
    force, pdl = snr._lib.BEAM_OPT_FORCE_EXACT_SUM, snr._lib.BEAM_OPT_PDL
    for v in (2, 3, 4, 5, 6, 7, 8):
        for flags in (0, force, pdl):
            got = gpu_dense_nvfp4(inp, 9, 1e-6, 336.0, opts=dict(vec_per_thread=v, flags=flags))
            check_nvfp4(got, want, f"dense nvfp4 vpt={v} flags={flags}")
    cfg = MOE_T16384
    m = synth.moe_inputs(cfg, rows=64)
    want = oracle.moe_boundary_nvfp4(m["h"], m["expert_out"], m["topk_w"], m["post_w"],
                                     m["pre_w"], cfg.n, cfg.eps, 336.0)
    for v in (2, 3, 4, 5, 8):
        for flags in (0, force, pdl):
            snr.exact_sum_count(reset=True)
            got = gpu_moe_nvfp4(m, cfg.n, cfg.eps, 336.0, opts=dict(vec_per_thread=v, flags=flags))
            if flags == force:
                assert snr.exact_sum_count() == 2 * 64
            check_nvfp4(got, want, f"moe nvfp4 vpt={v} flags={flags}")


def test_nvfp4_non_finite_values_match_the_oracle():
    """Rows whose y is all NaN (NaN or -inf in x), a row with an infinite h, and
    pre-norm weights holding a NaN and +-inf, which put NaN and infinite values
    in blocks of every other row: the block amax skips NaN, an infinite amax
    saturates the scale, infinite values saturate their codes and a NaN value's
    code is +6 (0x7)."""
    rng = np.random.default_rng(81)
    T, D = 6, 256
    inp = random_dense(T, D, seed=81)
    inp["x"][0, 7] = float("nan")
    inp["h"][1, 9] = float("inf")
    inp["x"][2, 3] = float("-inf")
    inp["pre_w"][5] = float("nan")
    inp["pre_w"][40] = float("inf")
    inp["pre_w"][41] = float("-inf")
    want = oracle.boundary_nvfp4(inp["h"], inp["x"], inp["post_w"], inp["pre_w"], 3, 1e-6, 336.0)
    assert (want[2] == 0x7E).any() and (want[1] == 0x77).any()  # the cases are present
    check_nvfp4(gpu_dense_nvfp4(inp, 3, 1e-6, 336.0), want, "dense nvfp4 non-finite")
    m = dict(h=inp["h"], expert_out=bf16(rng.standard_normal((T, 8, D))),
             topk_w=torch.from_numpy(rng.uniform(0, 0.4, (T, 8)).astype(np.float32)),
             post_w=inp["post_w"], pre_w=inp["pre_w"])
    m["expert_out"][0, 3, 11] = float("nan")
    want = oracle.moe_boundary_nvfp4(m["h"], m["expert_out"], m["topk_w"], m["post_w"], m["pre_w"],
                                     3, 1e-6, 336.0)
    check_nvfp4(gpu_moe_nvfp4(m, 3, 1e-6, 336.0), want, "moe nvfp4 non-finite")


def test_nvfp4_agrees_with_quantising_the_bf16_output():
    """The quantised call equals the BF16 call followed by the oracle's NVFP4
    quantiser on its y, row by row."""
    cfg = MOE_T16384
    m = synth.moe_inputs(cfg, rows=128)
    h_bf, y_bf = gpu_moe(m, cfg.n, cfg.eps)
    h_q, q, sf = gpu_moe_nvfp4(m, cfg.n, cfg.eps, 336.0)
    assert np.array_equal(h_bf, h_q)
    for t in range(y_bf.shape[0]):
        qr, sr = oracle.nvfp4_row(y_bf[t], 336.0)
        assert np.array_equal(q[t], qr) and np.array_equal(sf[t], sr), t


def test_nvfp4_branch_is_the_stream_guard_bands_and_zero_tokens():
    T, D = 21, 5120
    inp = random_dense(T, D, seed=23)
    d = to_dev(inp)
    qbuf = torch.full((T + 2, D // 2), 0xA5, dtype=torch.uint8, device=DEV)
    sbuf = torch.full((T + 2, D // 16), 0xA5, dtype=torch.uint8, device=DEV)
    q, sf = snr.boundary_fused_nvfp4(d["h"], d["h"], d["post_w"], d["pre_w"], 6, 1e-6, 336.0,
                                     y_fp4=qbuf[1:T + 1], y_scale=sbuf[1:T + 1])
    snr.sync_status()
    for b in (qbuf, sbuf):
        assert (b[0] == 0xA5).all() and (b[-1] == 0xA5).all()
    want = oracle.boundary_nvfp4(inp["h"], inp["h"], inp["post_w"], inp["pre_w"], 6, 1e-6, 336.0)
    check_nvfp4((bits(d["h"]), q.cpu().numpy(), sf.cpu().numpy()), want, "nvfp4 x is h")
    h0 = torch.zeros((0, D), dtype=torch.bfloat16, device=DEV)
    q0, s0 = snr.boundary_fused_nvfp4(h0, h0, d["post_w"], d["pre_w"], 2, 1e-6, 336.0)
    assert q0.shape == (0, D // 2) and s0.shape == (0, D // 16)


# --------------------------------------------------------------- batch in host memory

def pinned(inp: dict) -> dict:
    return {k: v.pin_memory() for k, v in inp.items()}


def test_host_memory_dense_and_moe_full_match_the_oracle():
    """Every operand page-locked in host memory: the kernels read and write it over
    the CPU-GPU link; results equal the oracle and the device path bit for bit."""
    cfg = DENSE_PREFILL_T16384
    inp = synth.dense_inputs(cfg)
    hp = pinned(inp)
    y = snr.boundary_fused_host(hp["h"], hp["x"], hp["post_w"], hp["pre_w"], cfg.n, cfg.eps)
    snr.sync_status()
    assert y.device.type == "cpu" and y.is_pinned()
    want = oracle_dense(inp, cfg.n, cfg.eps)
    check((bits(hp["h"]), bits(y)), want, f"{cfg.name} host memory")
    cfg = MOE_T16384
    m = synth.moe_inputs(cfg)
    mp = pinned(m)
    y = snr.moe_combine_boundary_host(mp["h"], mp["expert_out"], mp["topk_w"], mp["post_w"],
                                      mp["pre_w"], cfg.n, cfg.eps)
    snr.sync_status()
    check((bits(mp["h"]), bits(y)), oracle_moe(m, cfg.n, cfg.eps), f"{cfg.name} host memory")


def test_host_memory_mixed_with_device_operands_and_a_side_stream():
    T, D = 300, 5120
    inp = random_dense(T, D, seed=31)
    want = oracle_dense(inp, 5, 1e-6)
    hp = pinned(inp)
    pw, qw = inp["post_w"].to(DEV), inp["pre_w"].to(DEV)
    y_dev = torch.empty((T, D), dtype=torch.bfloat16, device=DEV)   # h on the host, y on the device
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        snr.boundary_fused_host(hp["h"], hp["x"], pw, qw, 5, 1e-6, y=y_dev, stream=s)
    snr.sync_status(s)
    check((bits(hp["h"]), bits(y_dev)), want, "host h and x, device weights and y")
    cfg = MOE_T16384
    m = synth.moe_inputs(cfg, rows=200)
    wantm = oracle_moe(m, cfg.n, cfg.eps)
    e_dev = m["expert_out"].to(DEV)                                  # expert rows already on the GPU
    mp = pinned({k: v for k, v in m.items() if k != "expert_out"})
    y = snr.moe_combine_boundary_host(mp["h"], e_dev, mp["topk_w"], mp["post_w"], mp["pre_w"],
                                      cfg.n, cfg.eps)
    snr.sync_status()
    check((bits(mp["h"]), bits(y)), wantm, "host h, device expert rows")


def test_host_memory_pageable_is_read_or_refused():
    """Pageable memory works only where the device reads the host's page tables;
    elsewhere the call refuses it with BEAM_ERR_ARG before launching."""
    T, D = 8, 5120
    inp = random_dense(T, D, seed=32)
    want = oracle_dense(inp, 3, 1e-6)
    h = inp["h"].clone()
    y = torch.empty((T, D), dtype=torch.bfloat16)
    try:
        snr.boundary_fused_host(h, inp["x"], inp["post_w"], inp["pre_w"], 3, 1e-6, y=y)
        snr.sync_status()
    except snr.BeamError as e:
        assert e.status == snr._lib.BEAM_ERR_ARG
        assert torch.equal(h, inp["h"])      # nothing ran
        print("pageable host memory refused (no pageable access on this device)")
        return
    check((bits(h), bits(y)), want, "pageable host memory")


@pytest.mark.parametrize("pdl", [False, True])
@pytest.mark.parametrize("graph", [False, True])
def test_decoder_layer_chain_alternating_dense_and_moe_matches_the_oracle(pdl, graph):
    """104 boundaries as the decoder runs them at T = 64: attention (dense) and MoE
    boundaries in turn, n = 2..105, back to back on one stream (optionally one CUDA
    graph, optionally programmatic dependent launches); every step exact."""
    cfg = DECODE_CHAIN_T64
    h0, steps = synth.layer_chain_inputs(cfg, MOE_T16384)
    dev_steps = [{k: (v.to(DEV) if k != "kind" else v) for k, v in s.items()} for s in steps]
    h = h0.to(DEV)
    ys = [torch.empty_like(h) for _ in steps]
    opts = dict(flags=snr._lib.BEAM_OPT_PDL) if pdl else None
    stream = torch.cuda.Stream()

    def run_chain():
        for s, d in enumerate(dev_steps):
            if d["kind"] == "dense":
                snr.boundary_fused(h, d["x"], d["post_w"], d["pre_w"], cfg.n + s, cfg.eps, y=ys[s],
                                   opts=opts, stream=stream)
            else:
                snr.moe_combine_boundary(h, d["expert_out"], d["topk_w"], d["post_w"], d["pre_w"],
                                         cfg.n + s, cfg.eps, y=ys[s], opts=opts, stream=stream)

    with torch.cuda.stream(stream):
        run_chain()  # sets up the launch shapes before any capture
    torch.cuda.synchronize()
    h.copy_(h0.to(DEV))
    torch.cuda.synchronize()
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run_chain()
        h.copy_(h0.to(DEV))
        for y in ys:
            y.zero_()
        torch.cuda.synchronize()
        g.replay()
    else:
        with torch.cuda.stream(stream):
            run_chain()
    torch.cuda.synchronize()
    snr.sync_status()

    h_ref = oracle.as_u16(h0).copy()
    for s, inp in enumerate(steps):
        if inp["kind"] == "dense":
            h_ref, y_ref = oracle.boundary(h_ref, inp["x"], inp["post_w"], inp["pre_w"], cfg.n + s,
                                           cfg.eps, threads=THREADS)
        else:
            h_ref, y_ref = oracle.moe_boundary(h_ref, inp["expert_out"], inp["topk_w"],
                                               inp["post_w"], inp["pre_w"], cfg.n + s, cfg.eps,
                                               threads=THREADS)
        assert_parity(bits(ys[s]), y_ref, f"layer chain step {s} ({inp['kind']}) y")
    check((bits(h), bits(ys[-1])), (h_ref, y_ref), f"layer chain graph={graph} pdl={pdl}")


# --------------------------------------------------------------- seeded random shapes

def _fuzz_cases(seed: int, count: int):
    rng = np.random.default_rng(seed)
    for _ in range(count):
        T = int(rng.integers(1, 300))
        D = 8 * int(rng.integers(1, 1025))            # 8 .. 8192, any multiple of 8
        n = int(rng.integers(1, 200))
        eps = float(rng.choice([0.0, 1e-6, 1e-5, 1e-3]))
        scale = float(10.0 ** rng.uniform(-3, 3))
        yield rng, T, D, n, eps, scale


def test_random_shapes_dense_and_moe_match_the_oracle():
    for i, (rng, T, D, n, eps, scale) in enumerate(_fuzz_cases(101, 12)):
        inp = dict(h=bf16(rng.standard_normal((T, D))),
                   x=bf16(rng.standard_normal((T, D)) * scale),
                   post_w=bf16(1 + 0.3 * rng.standard_normal(D)),
                   pre_w=bf16(1 + 0.3 * rng.standard_normal(D)))
        if eps == 0.0:
            inp["x"][0] = bf16(np.ones(D))  # eps = 0 only on rows that are not all zero
        check(gpu_dense(inp, n, eps), oracle_dense(inp, n, eps), f"fuzz {i} dense T={T} D={D} n={n}")
        m = dict(h=inp["h"], expert_out=bf16(rng.standard_normal((T, 8, D)) * scale),
                 topk_w=torch.from_numpy(rng.uniform(0, 0.5, (T, 8)).astype(np.float32)),
                 post_w=inp["post_w"], pre_w=inp["pre_w"])
        check(gpu_moe(m, n, max(eps, 1e-6)), oracle_moe(m, n, max(eps, 1e-6)),
              f"fuzz {i} moe T={T} D={D} n={n}")


def test_random_shapes_nvfp4_match_the_oracle():
    for i, (rng, T, D, n, eps, scale) in enumerate(_fuzz_cases(202, 10)):
        D = 16 * max(1, D // 16)
        gs = float(10.0 ** rng.uniform(-2, 4))
        inp = random_dense(T, D, seed=1000 + i, scale=scale)
        want = oracle.boundary_nvfp4(inp["h"], inp["x"], inp["post_w"], inp["pre_w"], n, 1e-6, gs)
        check_nvfp4(gpu_dense_nvfp4(inp, n, 1e-6, gs), want, f"fuzz {i} nvfp4 T={T} D={D} gs={gs:.3g}")


def test_random_head_counts_qk_norm_match_the_oracle():
    rng = np.random.default_rng(303)
    for i in range(8):
        T, nq, nk = int(rng.integers(1, 100)), int(rng.integers(0, 64)), int(rng.integers(0, 16))
        if nq + nk == 0:
            nk = 1
        q, k, qw, kw, pos, table = _qk_case(T, nq, nk, 400 + i, 3000)
        for mode in ("rope", "ssmax"):
            dq, dk = q.to(DEV), k.to(DEV)
            snr.qk_norm(dq, dk, qw.to(DEV), kw.to(DEV), pos.to(DEV), 1e-6, mode,
                        rope_table=table.to(DEV) if mode == "rope" else None)
            snr.sync_status()
            wq, wk = oracle.qk_norm(q, k, qw, kw, pos, table if mode == "rope" else None, 1e-6, mode)
            assert_parity(bits(dq), wq, f"fuzz {i} qk {mode} q T={T} nq={nq}")
            assert_parity(bits(dk), wk, f"fuzz {i} qk {mode} k T={T} nk={nk}")


@pytest.mark.parametrize("mode", ["rope", "ssmax"])
def test_qk_norm_chain_with_pdl_in_a_cuda_graph(mode):
    """Eight Q/K norms (one per layer) back to back as programmatic dependent
    launches captured in one CUDA graph; each layer's q and k exact."""
    layers = [_qk_case(64, 48, 8, 700 + i, 4096) for i in range(8)]
    dev_layers = [tuple(t.to(DEV) for t in case) for case in layers]
    stream = torch.cuda.Stream()

    def run():
        for q, k, qw, kw, pos, table in dev_layers:
            snr.qk_norm(q, k, qw, kw, pos, 1e-6, mode, rope_table=table if mode == "rope" else None,
                        stream=stream, pdl=True)

    with torch.cuda.stream(stream):
        run()
    torch.cuda.synchronize()
    for (q, k, *_), (dq, dk, *_) in zip(layers, dev_layers):
        dq.copy_(q.to(DEV))
        dk.copy_(k.to(DEV))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    g.replay()
    torch.cuda.synchronize()
    snr.sync_status()
    for i, ((q, k, qw, kw, pos, table), (dq, dk, *_)) in enumerate(zip(layers, dev_layers)):
        wq, wk = oracle.qk_norm(q, k, qw, kw, pos, table if mode == "rope" else None, 1e-6, mode)
        assert_parity(bits(dq), wq, f"qk pdl layer {i} q")
        assert_parity(bits(dk), wk, f"qk pdl layer {i} k")
