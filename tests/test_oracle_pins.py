"""Pins for the CPU oracle, checked against things other than the oracle itself.

Each test ties one part of the oracle to a library routine (torch's BF16 cast,
IEEE float32 arithmetic in numpy), to exact rational arithmetic, to a closed
form of the depth-scaled residual, to an invariant the pages state, or to the
hand-worked examples in ``tests/golden/hand_examples.txt``.
"""
from __future__ import annotations

import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.txt")
f32 = np.float32


# ----------------------------------------------------------------- helpers

def bf16_bits(vals) -> np.ndarray:
    """BF16 bit patterns of FP32 values via torch's cast (a library routine)."""
    t = torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def nearest_f32(q: Fraction) -> np.float32:
    """The FP32 value nearest to the rational q, ties to even (brute force on neighbours)."""
    if q == 0:
        return f32(0.0)
    c = f32(float(q)) if abs(q) < Fraction(2) ** 128 else f32(np.inf)
    best = None
    cands = {c, np.nextafter(c, f32(np.inf)), np.nextafter(c, f32(-np.inf))}
    for v in cands:
        if not np.isfinite(v):
            continue
        d = abs(Fraction(float(v)) - q)
        key = (d, int(np.array(v).view(np.uint32)) & 1)  # ties: even significand first
        if best is None or key < best[0]:
            best = (key, v)
    # beyond the largest finite float by at least half an ulp -> infinity
    fmax = Fraction(float(np.finfo(np.float32).max))
    half_ulp = Fraction(2) ** (127 - 24)
    if q >= fmax + half_ulp:
        return f32(np.inf)
    return best[1]


def exact_sum(vals) -> Fraction:
    return sum((Fraction(float(v)) for v in vals), Fraction(0))


def load_golden():
    ex = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, val = line.split(":", 1)
        name, field = key.split(".")
        vals = [float(v) for v in val.split()]
        ex.setdefault(name, {})[field] = vals if field in (
            "h", "x", "post_w", "pre_w", "h_out", "y") else vals[0]
    return ex


# ------------------------------------------------------------- BF16 rounding

def test_bf16_rne_matches_torch_cast_on_random_bit_patterns():
    rng = np.random.default_rng(123)
    u = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    vals = u.view(np.float32)
    want = bf16_bits(vals)
    got = np.array([oracle.bf16_rne(float(v)) for v in vals], dtype=np.uint16)
    nan = np.isnan(vals)
    assert np.array_equal(got[~nan], want[~nan])
    assert all(((g & 0x7F80) == 0x7F80) and (g & 0x7F) for g in got[nan])


def test_bf16_rne_ties_subnormals_and_overflow():
    cases = []
    for hi in (0x3F80, 0x3F81, 0x0001, 0x0002, 0x807F, 0x7F7F, 0xFF7F, 0x0080):
        for lo in (0x7FFF, 0x8000, 0x8001, 0x0000, 0xFFFF):
            cases.append(np.uint32((hi << 16) | lo))
    vals = np.array(cases, dtype=np.uint32).view(np.float32)
    want = bf16_bits(vals)
    got = np.array([oracle.bf16_rne(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)
    assert oracle.bf16_rne(float("inf")) == 0x7F80
    assert oracle.bf16_rne(float("-inf")) == 0xFF80


# -------------------------------------------------- exact sum, rounded once

@pytest.mark.parametrize("seed", range(6))
def test_exact_sum_is_nearest_float_of_rational_sum(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 400))
    # spread exponents widely, include subnormals and zeros
    mant = rng.random(n).astype(np.float32)
    expo = rng.integers(-150, 40, size=n)
    t = np.ldexp(mant, expo).astype(np.float32)
    t[rng.random(n) < 0.05] = 0.0
    got = oracle.sum_f32_exact(t)
    assert f32(got) == nearest_f32(exact_sum(t))


def test_exact_sum_ties_go_to_even():
    one, e24, e40 = 1.0, 2.0 ** -24, 2.0 ** -40
    # 1 + 2^-24 is the midpoint of 1 and 1 + 2^-23: ties to the even one, 1
    assert oracle.sum_f32_exact([one, e24]) == 1.0
    # a tiny extra term breaks the tie upwards
    assert oracle.sum_f32_exact([one, e24, e40]) == 1.0 + 2.0 ** -23
    # (1 + 2^-23) + 2^-24 is a midpoint with an odd lower neighbour: rounds up
    assert oracle.sum_f32_exact([1.0 + 2.0 ** -23, e24]) == 1.0 + 2.0 ** -22
    # many tiny terms that together pass the midpoint
    assert oracle.sum_f32_exact([one] + [2.0 ** -30] * 65) == 1.0 + 2.0 ** -23


def test_exact_sum_subnormal_exact_and_overflow():
    tiny = float(np.array(1, np.uint32).view(np.float32))  # 2^-149
    assert oracle.sum_f32_exact([tiny] * 7) == 7 * tiny
    assert oracle.sum_f32_exact([2.0 ** -126 - tiny, tiny]) == 2.0 ** -126
    big = float(f32(1.5 * 2.0 ** 127))
    assert math.isinf(oracle.sum_f32_exact([big, big]))
    assert math.isnan(oracle.sum_f32_exact([1.0, float("nan")]))
    assert math.isinf(oracle.sum_f32_exact([1.0, float("inf")]))
    assert oracle.sum_f32_exact([]) == 0.0


@pytest.mark.parametrize("seed", range(4))
def test_sum_squares_uses_fp32_products_and_one_rounding(seed):
    rng = np.random.default_rng(100 + seed)
    D = 257
    v = rng.standard_normal(D).astype(np.float32) * np.float32(2.0) ** rng.integers(-70, 10, D)
    b = bf16_bits(v)
    xf = bits_to_f32(b)
    sq = xf * xf  # numpy float32 products: IEEE RN, subnormals kept
    assert f32(oracle.sum_squares(b)) == nearest_f32(exact_sum(sq))


def test_rms_factor_matches_ieee_float32_steps():
    rng = np.random.default_rng(7)
    for _ in range(2000):
        S = f32(rng.random() * 10.0 ** int(rng.integers(-3, 6)))
        D = int(rng.integers(1, 9000))
        eps = f32([0.0, 1e-6, 1e-5][rng.integers(0, 3)])
        want = f32(1.0) / np.sqrt(S / f32(D) + eps)
        assert f32(oracle.rms_factor(float(S), D, float(eps))) == want


# -------------------------------------------------------------------- RMSNorm

def test_rmsnorm_single_element_closed_form():
    rng = np.random.default_rng(11)
    for _ in range(500):
        x = f32(rng.standard_normal() * 4)
        w = f32(1 + 0.1 * rng.standard_normal())
        xb, wb = bf16_bits([x])[0], bf16_bits([w])[0]
        xf, wf = bits_to_f32([xb])[0], bits_to_f32([wb])[0]
        r = f32(1.0) / np.sqrt(xf * xf + f32(1e-6))
        want = bf16_bits([(xf * r) * wf])[0]
        got = oracle.rmsnorm(np.array([xb], np.uint16), np.array([wb], np.uint16), 1e-6)[0]
        assert got == want


@pytest.mark.parametrize("k", [-20, -3, 1, 9])
def test_rmsnorm_is_invariant_to_power_of_two_scaling_with_zero_eps(k):
    rng = np.random.default_rng(5)
    D = 640
    x = bf16_bits(rng.standard_normal(D))
    w = bf16_bits(1 + 0.1 * rng.standard_normal(D))
    xs = bf16_bits(bits_to_f32(x) * f32(2.0 ** k))  # exact scaling
    assert np.array_equal(oracle.rmsnorm(x, w, 0.0), oracle.rmsnorm(xs, w, 0.0))


def test_rmsnorm_unit_weights_give_unit_rms_and_weights_multiply():
    rng = np.random.default_rng(6)
    D = 5120
    x = bf16_bits(rng.standard_normal(D) * 3.7)
    ones = bf16_bits(np.ones(D))
    y = bits_to_f32(oracle.rmsnorm(x, ones, 1e-6)).astype(np.float64)
    assert abs(np.mean(y * y) - 1.0) < 2.0 ** -9
    twos = bf16_bits(np.full(D, 2.0))
    y2 = bits_to_f32(oracle.rmsnorm(x, twos, 1e-6))
    assert np.array_equal(y2, (2 * y).astype(np.float32))


@pytest.mark.parametrize("seed", range(3))
def test_rmsnorm_matches_torch_cpu_composition(seed):
    """Independent restatement: exact rational sum, then torch float32 ops and torch's BF16 cast."""
    rng = np.random.default_rng(40 + seed)
    D = 1024
    x = bf16_bits(rng.standard_normal(D))
    w = bf16_bits(1 + 0.1 * rng.standard_normal(D))
    xt = torch.from_numpy(bits_to_f32(x).copy())
    wt = torch.from_numpy(bits_to_f32(w).copy())
    S = nearest_f32(exact_sum((xt * xt).numpy()))
    # numpy's float32 sqrt is IEEE correctly rounded; torch's CPU sqrt is not always
    r = torch.tensor(f32(1.0) / np.sqrt(S / f32(D) + f32(1e-6)))
    want = ((xt * r) * wt).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.rmsnorm(x, w, 1e-6), want)


def _nearest_f32_of_fsum(vals: np.ndarray) -> np.float32:
    """RN32 of the exact sum: fsum gives the correctly rounded double; if that double
    is exactly halfway between two floats the exact rational decides."""
    d = math.fsum(vals.astype(np.float64).tolist())
    c = f32(d)
    lo, hi = np.nextafter(c, f32(-np.inf)), np.nextafter(c, f32(np.inf))
    if d in ((float(c) + float(lo)) / 2, (float(c) + float(hi)) / 2):
        return nearest_f32(exact_sum(vals))
    return c


def test_rmsnorm_matches_torch_cpu_composition_on_a_million_elements():
    """Order of the two FP32 products, (v r) w, shows in about one element per
    million, so this cross-check runs on 256 rows of 5120."""
    rng = np.random.default_rng(44)
    T, D = 256, 5120
    x = bf16_bits(rng.standard_normal((T, D)))
    w = bf16_bits(1 + 0.1 * rng.standard_normal(D))
    xt = torch.from_numpy(bits_to_f32(x).copy())
    wt = torch.from_numpy(bits_to_f32(w).copy())
    sq = (xt * xt).numpy()
    S = np.array([_nearest_f32_of_fsum(sq[t]) for t in range(T)], np.float32).reshape(T, 1)
    r = torch.from_numpy(f32(1.0) / np.sqrt(S / f32(D) + f32(1e-6)))
    want = ((xt * r) * wt).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.stack([oracle.rmsnorm(x[t], w, 1e-6) for t in range(T)])
    assert np.array_equal(got, want)


# ------------------------------------------------------ depth-scaled residual

@pytest.mark.parametrize("n", [1, 2, 3, 7, 20, 104, 105, 1000])
def test_scales_are_rounded_sqrt_and_keep_unit_variance(n):
    c1, c2 = oracle.scales(n)
    getcontext().prec = 50
    t1 = (Decimal(n - 1) / Decimal(n)).sqrt()
    t2 = 1 / Decimal(n).sqrt()
    for c, t in ((c1, t1), (c2, t2)):
        c = f32(c)
        ulp = float(np.spacing(c)) if c != 0 else 2.0 ** -149
        assert abs(Decimal(float(c)) - t) <= Decimal(ulp)
    # (sqrt((n-1)/n))^2 + (1/sqrt(n))^2 = 1 up to the FP32 rounding of c1, c2
    assert abs(float(c1) ** 2 + float(c2) ** 2 - 1.0) < 2.0 ** -22


def test_n1_makes_the_stream_the_normalised_branch():
    rng = np.random.default_rng(9)
    T, D = 3, 520
    h = bf16_bits(rng.standard_normal((T, D)))
    x = bf16_bits(rng.standard_normal((T, D)))
    pw = bf16_bits(1 + 0.1 * rng.standard_normal(D))
    qw = bf16_bits(1 + 0.1 * rng.standard_normal(D))
    h2, y = oracle.boundary(h, x, pw, qw, 1, 1e-6)
    for t in range(T):
        xn = oracle.rmsnorm(x[t], pw, 1e-6)
        assert np.array_equal(np.abs(bits_to_f32(h2[t])), np.abs(bits_to_f32(xn)))
        assert np.array_equal(h2[t] & 0x7FFF, xn & 0x7FFF)
        assert np.array_equal(y[t], oracle.rmsnorm(h2[t], qw, 1e-6))


def test_post_and_pre_weights_are_not_swapped():
    # D = 1, n = 1 (c1 = 0, c2 = 1): h' = bf16(x r1 w_post), y = bf16(h' r2 w_pre)
    one = bf16_bits([1.0])
    h2, y = oracle.boundary(bf16_bits([[0.0]]), bf16_bits([[1.0]]), bf16_bits([2.0]),
                            bf16_bits([0.5]), 1, 1e-6)
    assert bits_to_f32(h2)[0, 0] == 2.0 and bits_to_f32(y)[0, 0] == 0.5
    h2s, ys = oracle.boundary(bf16_bits([[0.0]]), bf16_bits([[1.0]]), bf16_bits([0.5]),
                              bf16_bits([2.0]), 1, 1e-6)
    assert bits_to_f32(h2s)[0, 0] == 0.5 and bits_to_f32(ys)[0, 0] == 2.0
    assert one[0] == 0x3F80


@pytest.mark.parametrize("name", ["A", "B", "C"])
def test_hand_worked_examples(name):
    ex = load_golden()[name]
    D = int(ex["D"])
    h = bf16_bits([ex["h"]])
    x = bf16_bits([ex["x"]])
    h2, y = oracle.boundary(h, x, bf16_bits(ex["post_w"]), bf16_bits(ex["pre_w"]), int(ex["n"]),
                            float(ex["eps"]))
    assert h2.shape == (1, D)
    assert np.array_equal(bits_to_f32(h2)[0], np.array(ex["h_out"], np.float32))
    if "y" in ex:
        assert np.array_equal(bits_to_f32(y)[0], np.array(ex["y"], np.float32))


def test_long_double_residual_chain_closed_form():
    """Applying n = 2..N to h1 gives (h1 + sum_n x_n) / sqrt(N): the products of
    sqrt((j-1)/j) telescope to sqrt(k/N)."""
    rng = np.random.default_rng(21)
    N, M = 105, 64
    h1 = rng.standard_normal(M)
    xs = rng.standard_normal((N - 1, M))
    h = np.array(h1, dtype=np.longdouble)
    for n in range(2, N + 1):
        h = oracle.residual_ld(h, xs[n - 2], n)
    closed = (h1.astype(np.longdouble) + xs.astype(np.longdouble).sum(0)) / np.sqrt(
        np.longdouble(N))
    assert np.max(np.abs(h - closed)) < 1e-14


def test_long_double_boundary_matches_bf16_oracle_within_rounding():
    rng = np.random.default_rng(22)
    T, D = 4, 512
    hb = bf16_bits(rng.standard_normal((T, D)))
    xb = bf16_bits(rng.standard_normal((T, D)))
    pw = bf16_bits(1 + 0.1 * rng.standard_normal(D))
    qw = bf16_bits(1 + 0.1 * rng.standard_normal(D))
    n = 9
    h2, y = oracle.boundary(hb, xb, pw, qw, n, 1e-6)
    hl, yl = oracle.boundary_ld(bits_to_f32(hb), bits_to_f32(xb), bits_to_f32(pw),
                                bits_to_f32(qw), n, 1e-6)
    hl, yl = hl.astype(np.float64), yl.astype(np.float64)
    h0 = bits_to_f32(hb).astype(np.float64)
    xf = bits_to_f32(xb).astype(np.float64)
    xn_ld = xf / np.sqrt(np.mean(xf * xf, 1, keepdims=True) + 1e-6) * bits_to_f32(pw)
    c1, c2 = math.sqrt((n - 1) / n), 1 / math.sqrt(n)
    # BF16 keeps 8 significant bits (unit roundoff 2^-8): each of xn, a, b, h' is off by
    # at most 2^-8 relative, so h' is off by at most 2^-8 (|c1 h| + 2 |c2 xn| + |h'|)
    # (cancellation in a + b makes this absolute, not relative to h')
    dh = np.abs(bits_to_f32(h2) - hl)
    bound_h = 2.0 ** -8 * (np.abs(c1 * h0) + 2 * np.abs(c2 * xn_ld) + np.abs(hl)) * 1.01 + 1e-7
    assert (dh <= bound_h).all()
    # y = h' r2 w: carries h''s error, r2's relative error and its own rounding
    qwf = bits_to_f32(qw).astype(np.float64)
    r2 = 1 / np.sqrt(np.mean(hl * hl, 1, keepdims=True) + 1e-6)
    dy = np.abs(bits_to_f32(y) - yl)
    bound_y = bound_h * r2 * np.abs(qwf) + 2.0 ** -7 * np.abs(yl) + 1e-7
    assert np.mean(dh) < 0.25 * np.mean(bound_h)  # typical error well inside the bound
    assert (dy <= bound_y).all()


def _chain(T, D, steps, seed, weights_fixed=False):
    rng = np.random.default_rng(seed)
    h1 = bf16_bits(rng.standard_normal((T, D)))
    h = h1.copy()
    xn_sum = np.zeros((T, D), np.longdouble)
    xn_sq = 0.0
    for s in range(steps):
        n = s + 2
        x = bf16_bits(rng.standard_normal((T, D)))
        pw = bf16_bits(np.ones(D) if weights_fixed else 1 + 0.1 * rng.standard_normal(D))
        qw = bf16_bits(1 + 0.1 * rng.standard_normal(D))
        xn = np.stack([oracle.rmsnorm(x[t], pw, 1e-6) for t in range(T)])
        xnf = bits_to_f32(xn).astype(np.float64)
        xn_sum += xnf
        xn_sq += np.mean(xnf * xnf)
        h, _ = oracle.boundary(h, x, pw, qw, n, 1e-6)
    return h1, h, xn_sum, xn_sq


def test_bf16_chain_follows_closed_form_of_depth_scaling():
    T, D, steps = 2, 512, 104
    h1, h, xn_sum, _ = _chain(T, D, steps, 31)
    closed = (bits_to_f32(h1).astype(np.longdouble) + xn_sum) / np.sqrt(np.longdouble(steps + 1))
    got = bits_to_f32(h).astype(np.float64)
    rel_rms = np.sqrt(np.mean((got - closed.astype(np.float64)) ** 2) /
                      np.mean(closed.astype(np.float64) ** 2))
    # 104 steps of three BF16 roundings each, damped by the depth scaling
    assert rel_rms < 0.03


def test_chain_keeps_unit_variance_statistically():
    """sqrt((n-1)/n)^2 + (1/sqrt(n))^2 = 1: with unit-variance h and branches the
    stream keeps unit variance; here the prediction uses the data's own branch
    second moments: var(h_N) = (var(h_1) + sum_n mean(xn_n^2)) / N."""
    T, D, steps = 8, 5120, 104
    h1, h, _, xn_sq = _chain(T, D, steps, 32)
    h1f = bits_to_f32(h1).astype(np.float64)
    pred = (np.mean(h1f * h1f) + xn_sq) / (steps + 1)
    got = np.mean(bits_to_f32(h).astype(np.float64) ** 2)
    sigma = math.sqrt(2.0 / (T * D))
    assert abs(got - pred) < 5 * sigma
    assert abs(pred - 1.0099) < 0.02  # E[w^2] = 1.01 for weights 1 + 0.1 N(0,1)


# --------------------------------------------------------------- MoE combine

def test_moe_one_hot_weights_reduce_to_a_single_scaled_expert():
    rng = np.random.default_rng(50)
    K, D = 8, 256
    e = bf16_bits(rng.standard_normal((K, D)))
    for k in range(K):
        w = np.zeros(K, np.float32)
        w[k] = f32(rng.random() * 2.5)
        want = bf16_bits(w[k] * bits_to_f32(e[k]))
        assert np.array_equal(oracle.moe_combine(e, w), want)


def test_moe_equal_experts_power_of_two_values_sum_exactly():
    K, D = 8, 64
    vals = np.float32(2.0) ** np.arange(-10, 54, dtype=np.float32)[:D] * np.where(
        np.arange(D) % 2, 1, -1).astype(np.float32)
    vals = np.clip(vals, -2.0 ** 100, 2.0 ** 100).astype(np.float32)
    e = np.tile(bf16_bits(vals), (K, 1))
    w = np.full(K, 2.5 / 8, np.float32)
    got = bits_to_f32(oracle.moe_combine(e, w))
    assert np.array_equal(got, (2.5 * bits_to_f32(e[0])).astype(np.float32))


def test_moe_boundary_with_one_unit_expert_is_the_dense_boundary():
    rng = np.random.default_rng(51)
    T, D = 3, 384
    h = bf16_bits(rng.standard_normal((T, D)))
    x = bf16_bits(rng.standard_normal((T, D)))
    pw = bf16_bits(1 + 0.1 * rng.standard_normal(D))
    qw = bf16_bits(1 + 0.1 * rng.standard_normal(D))
    hd, yd = oracle.boundary(h, x, pw, qw, 5, 1e-6)
    hm, ym = oracle.moe_boundary(h, x.reshape(T, 1, D), np.ones((T, 1), np.float32), pw, qw, 5,
                                 1e-6)
    assert np.array_equal(hd, hm) and np.array_equal(yd, ym)


def _fma_chain_exact(e_bits: np.ndarray, w: np.ndarray) -> np.ndarray:
    """acc <- RN32(w_k e_k + acc) for k ascending, each step from the exact rational."""
    ef = bits_to_f32(e_bits)
    K, D = ef.shape
    acc = [Fraction(0)] * D
    for k in range(K):
        wk = Fraction(float(w[k]))
        acc = [Fraction(float(nearest_f32(wk * Fraction(float(ef[k, j])) + acc[j])))
               for j in range(D)]
    return bf16_bits([float(a) for a in acc])


def test_moe_combine_is_an_fma_chain_in_expert_order():
    """Each step is one rounding of w_k e_k + acc (exact rational, then RN32), k ascending."""
    rng = np.random.default_rng(52)
    K, D = 8, 512
    e = bf16_bits(rng.standard_normal((K, D)))
    w = (rng.random(K) * 0.6).astype(np.float32)
    assert np.array_equal(oracle.moe_combine(e, w), _fma_chain_exact(e, w))


def test_moe_combine_fused_multiply_add_decides_a_bf16_tie():
    # w1 e1 = (1 + 2^-23)(1 + 2^-7) = 1 + 2^-7 + 2^-23 + 2^-30. Fused with acc = 1 the sum
    # 2 + 2^-7 + 2^-23 + 2^-30 rounds up to 2 + 2^-7 + 2^-22, past the BF16 midpoint
    # 2 + 2^-7, so x = 2 + 2^-6. Rounding the product first gives 2 + 2^-7 + 2^-23,
    # an FP32 tie that goes to the even 2 + 2^-7, a BF16 tie that goes to 2.
    e = bf16_bits([[1.0], [1.0078125]])
    w = np.array([1.0, 1.0 + 2.0 ** -23], np.float32)
    got = oracle.moe_combine(e, w)
    assert bits_to_f32(got)[0] == 2.015625
    assert np.array_equal(got, _fma_chain_exact(e, w))


def test_moe_combine_order_decides_a_bf16_tie():
    # 1, 2^-8, 2^-24, 2^-24 in this order: 1 + 2^-8, then two FP32 ties that stay at the
    # even 1 + 2^-8, a BF16 tie -> 1. Summed from the last expert: 2^-23 + 2^-8 + 1 is
    # exact and passes the BF16 midpoint -> 1 + 2^-7.
    e = bf16_bits([[1.0], [2.0 ** -8], [2.0 ** -24], [2.0 ** -24]])
    w = np.ones(4, np.float32)
    got = oracle.moe_combine(e, w)
    assert bits_to_f32(got)[0] == 1.0
    assert np.array_equal(got, _fma_chain_exact(e, w))


def test_moe_combine_rounds_once_after_the_fp32_sum():
    # experts 1, 2^-8, 2^-8 with unit weights: the FP32 sum 1 + 2^-7 is a BF16 value.
    # Rounding the running sum to BF16 after each expert would give 1 + 2^-8 -> 1
    # (a tie, to even) and stay at 1.
    e = bf16_bits([[1.0], [2.0 ** -8], [2.0 ** -8]])
    got = bits_to_f32(oracle.moe_combine(e, np.array([1.0, 1.0, 1.0], np.float32)))
    assert got[0] == 1.0078125


# ------------------------------------------------------------ input generator

def test_generator_is_counter_based_and_seeded():
    a = synth.normal(3, 2, 1000)
    b = synth.normal(3, 2, 400, start=600)
    assert np.array_equal(a[600:], b)
    assert not np.array_equal(a, synth.normal(4, 2, 1000))
    assert not np.array_equal(a, synth.normal(3, 5, 1000))


def test_generator_distributions():
    z = synth.normal(0, 1, 400000).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.var() - 1) < 0.01
    t = synth.student_t3_unit(0, 9, 400000).astype(np.float64)
    assert abs(np.median(t)) < 0.01
    # t3 / sqrt(3): P(|t| > 1) = P(|T3| > sqrt(3)) = 0.18165 (closed form of the t3 CDF)
    p = np.mean(np.abs(t) > 1.0)
    assert abs(p - 0.18165) < 0.004
    w = synth.topk_weights(3, 6, 1000)
    assert np.allclose(w.sum(1), 2.5, atol=1e-5) and (w > 0).all()
    m = synth.bernoulli(4, 7, 200000, 1e-3)
    assert 120 < m.sum() < 290


# ------------------------------------------------------------------- routing

def _sigmoid_exact_f32(z: float) -> np.float32:
    getcontext().prec = 60
    v = Decimal(1) / (Decimal(1) + (-Decimal(float(z))).exp())
    return nearest_f32(Fraction(v))


def test_router_sigmoid_is_the_correctly_rounded_fp32_value():
    rng = np.random.default_rng(60)
    zs = np.concatenate([rng.standard_normal(1500) * 3, rng.uniform(-30, 30, 500),
                         [0.0, 1e-8, -1e-8, 17.0, -17.0, 88.0, -88.0]]).astype(np.float32)
    for z in zs:
        assert f32(oracle.sigmoid(float(z))) == _sigmoid_exact_f32(float(z)), z


def test_router_sigmoid_next_to_rounding_midpoints_and_at_the_ends():
    # z = m 2^-23 (and -m 2^-24): 1/2 + z/4 is a float or a rounding midpoint and
    # the sigmoid lies only about z^3/48 below (above) it, far inside a double's
    # rounding error; subnormal results below z = -87.3; 0 and 1 at the ends
    zs = [m * 2.0 ** -23 for m in range(1, 65)] + [-m * 2.0 ** -24 for m in range(1, 65)]
    zs += [-m * 2.0 ** -23 for m in range(1, 33)] + [m * 2.0 ** -22 for m in range(1, 33)]
    zs += [-87.5, -90.0, -95.25, -100.0, -103.5, -103.96, -103.98, 16.5, 17.0, 17.33, 17.5, 50.0]
    for z in zs:
        z = float(f32(z))
        assert f32(oracle.sigmoid(z)) == _sigmoid_exact_f32(z), z.hex()
    assert oracle.sigmoid(0.0) == 0.5 and oracle.sigmoid(-0.0) == 0.5
    assert oracle.sigmoid(math.inf) == 1.0 and oracle.sigmoid(-math.inf) == 0.0
    assert oracle.sigmoid(104.0) == 1.0 and oracle.sigmoid(-104.0) == 0.0
    assert math.isnan(oracle.sigmoid(math.nan))
    # 3 2^-23: 1/2 + z/4 = 1/2 + 1.5 2^-24 is the midpoint of 1/2 + 2^-24 and
    # 1/2 + 2^-23 (a tie would go to the latter, the even one); the sigmoid is
    # about 2^-71 below it, so it rounds down
    assert oracle.sigmoid(3 * 2.0 ** -23) == 0.5 + 2.0 ** -24
    assert oracle.sigmoid_undecided() == 0


def _route_inputs(T, E, seed, bias_scale=0.1):
    rng = np.random.default_rng(seed)
    z = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    b = (rng.standard_normal(E) * bias_scale).astype(np.float32)
    return z, b


def _biased(z, b):
    s = np.array([[oracle.sigmoid(float(v)) for v in row] for row in z], np.float32)
    return s, (s + b).astype(np.float32)


def _order(v, eligible):
    """indices of the eligible entries by descending value, ties by lower index (numpy lexsort)"""
    idx = np.nonzero(eligible)[0]
    return idx[np.lexsort((idx, -v[idx].astype(np.float64)))]


def test_routing_without_groups_is_a_plain_top_k_of_biased_scores():
    z, b = _route_inputs(16, 64, 61)
    idx, w = oracle.route(z, b, n_group=1, topk_group=1, topk=6, scale=1.0)
    s, bb = _biased(z, b)
    for t in range(z.shape[0]):
        assert np.array_equal(idx[t], _order(bb[t], np.ones(64, bool))[:6])


def test_group_limited_routing_matches_a_numpy_restatement():
    z, b = _route_inputs(24, 256, 62)
    idx, w = oracle.route(z, b)  # 8 groups of 32, keep 4, top 8, scale 2.5
    s, bb = _biased(z, b)
    for t in range(z.shape[0]):
        g = bb[t].reshape(8, 32)
        top2 = -np.sort(-g, axis=1)[:, :2]
        gscore = (top2[:, 0] + top2[:, 1]).astype(np.float32)
        kept = _order(gscore, np.ones(8, bool))[:4]
        elig = np.zeros(256, bool)
        for k in kept:
            elig[32 * k:32 * k + 32] = True
        want = _order(bb[t], elig)[:8]
        assert np.array_equal(idx[t], want)
        assert all(e // 32 in kept for e in idx[t])
        # weights: unbiased scores, running FP32 sum in output order, (s / sum) * 2.5
        sel = s[t, idx[t]]
        tot = sel[0]
        for v in sel[1:]:
            tot = f32(tot + v)
        assert np.array_equal(w[t], ((sel / tot).astype(np.float32) * f32(2.5)).astype(np.float32))
        assert abs(float(w[t].astype(np.float64).sum()) - 2.5) < 1e-5


def test_routing_hand_example_with_a_group_tie():
    # E = 8, two groups of 4, z = 0 so every sigmoid is exactly 0.5
    z = np.zeros((1, 8), np.float32)
    b = np.array([0.125, 0.375, 0, 0, 0.25, 0.25, 0.25, 0], np.float32)
    # biased 0.625 0.875 0.5 0.5 | 0.75 0.75 0.75 0.5: both group scores are 1.5 -> group 0
    idx, w = oracle.route(z, b, n_group=2, topk_group=1, topk=2, scale=2.5)
    assert idx.tolist() == [[1, 0]] and w.tolist() == [[1.25, 1.25]]
    # both groups kept: 0.875 first, then the first of the three 0.75 (expert 4)
    idx, w = oracle.route(z, b, n_group=2, topk_group=2, topk=2, scale=2.5)
    assert idx.tolist() == [[1, 4]] and w.tolist() == [[1.25, 1.25]]
    # the weights come from the unbiased scores: a larger bias does not raise them
    idx, w = oracle.route(np.array([[0, 2, 0, 0, 0, 0, 0, 0]], np.float32),
                          np.array([1, 0, 0, 0, 0, 0, 0, 0], np.float32), 1, 1, 2, 1.0)
    s1 = oracle.sigmoid(2.0)
    assert idx.tolist() == [[0, 1]]
    assert w[0, 0] == f32(f32(0.5) / f32(0.5 + s1)) and w[0, 0] < w[0, 1]


def test_routing_ranks_nan_scores_below_every_number():
    # E = 8 in two groups of 4, z = 0 (every sigmoid 1/2) unless NaN; a NaN
    # logit gives a NaN score, which ranks after every number (NaNs among
    # themselves by index)
    b = np.array([0, 0.5, 0, 0, 0.25, 0.5, 0.25, 0], np.float32)
    # group 0 biased 0.5 NaN 0.5 0.5 -> 1.0; group 1: 0.75 1.0 0.75 0.5 -> 1.75
    z = np.zeros((1, 8), np.float32)
    z[0, 1] = np.nan
    idx, w = oracle.route(z, b, n_group=2, topk_group=1, topk=2, scale=1.0)
    assert idx.tolist() == [[5, 4]] and w.tolist() == [[0.5, 0.5]]
    # group 0: 0.5 1.0 0.5 0.5 -> 1.5; group 1: NaN 1.0 0.75 0.5 -> 1.75
    z = np.zeros((1, 8), np.float32)
    z[0, 4] = np.nan
    idx, w = oracle.route(z, b, n_group=2, topk_group=1, topk=2, scale=1.0)
    assert idx.tolist() == [[5, 6]]
    # group 1 all NaN: its score is NaN and group 0 is kept; with both groups
    # kept, the NaN experts come after every number, lowest index first
    z = np.zeros((1, 8), np.float32)
    z[0, 4:] = np.nan
    idx, w = oracle.route(z, b, n_group=2, topk_group=1, topk=3, scale=1.0)
    assert idx.tolist() == [[1, 0, 2]]
    idx, w = oracle.route(z, b, n_group=2, topk_group=2, topk=6, scale=1.0)
    assert idx.tolist() == [[1, 0, 2, 3, 4, 5]] and np.isnan(w).all()


def test_scaled_combine_by_a_power_of_two_equals_prescaled_weights():
    rng = np.random.default_rng(70)
    e = bf16_bits(rng.standard_normal((8, 512)))
    w = (rng.random(8) * 0.3).astype(np.float32)
    for k in (-3, 1, 2):
        sc = f32(2.0 ** k)
        assert np.array_equal(oracle.moe_combine_scaled(e, w, float(sc)),
                              oracle.moe_combine(e, (w * sc).astype(np.float32)))
    assert np.array_equal(oracle.moe_combine_scaled(e, w, 1.0), oracle.moe_combine(e, w))


def test_scaled_combine_rounds_the_scaled_fp32_sum_once():
    rng = np.random.default_rng(71)
    e = bf16_bits(rng.standard_normal((8, 96)))
    w = (rng.random(8) * 0.3).astype(np.float32)
    ef = bits_to_f32(e)
    acc = [Fraction(0)] * 96
    for k in range(8):
        acc = [Fraction(float(nearest_f32(Fraction(float(w[k])) * Fraction(float(ef[k, j])) + acc[j])))
               for j in range(96)]
    want = bf16_bits([float(nearest_f32(Fraction(5, 2) * a)) for a in acc])
    assert np.array_equal(oracle.moe_combine_scaled(e, w, 2.5), want)


# ------------------------------------------------------------ Q/K norm, RoPE, SSMax

def _qk_inputs(T, nq, nk, seed):
    rng = np.random.default_rng(seed)
    q = bf16_bits(rng.standard_normal((T, nq, 128)) * 3)
    k = bf16_bits(rng.standard_normal((T, nk, 128)) * 3)
    qw = bf16_bits(1 + 0.1 * rng.standard_normal(128))
    kw = bf16_bits(1 + 0.1 * rng.standard_normal(128))
    return q, k, qw, kw


def _table(rows, c, s):
    t = np.zeros((rows, 128), np.float32)
    t[:, :64] = c
    t[:, 64:] = s
    return t


def test_rope_identity_quarter_and_half_turn_rotations():
    q, k, qw, kw = _qk_inputs(3, 4, 2, 80)
    pos = np.array([0, 1, 2], np.int32)
    tab = np.stack([_table(1, 1, 0)[0], _table(1, 0, 1)[0], _table(1, -1, 0)[0]])
    qo, ko = oracle.qk_norm(q, k, qw, kw, pos, tab, 1e-6)
    for t in range(3):
        for h in range(4):
            vn = oracle.rmsnorm(q[t, h], qw, 1e-6)
            f = bits_to_f32(vn)
            want = {0: f, 1: np.concatenate([-f[64:], f[:64]]), 2: -f}[t]
            assert np.array_equal(bits_to_f32(qo[t, h]), want.astype(np.float32))
        vk = bits_to_f32(oracle.rmsnorm(k[t, 1], kw, 1e-6))
        assert np.array_equal(bits_to_f32(ko[t, 1]), {0: vk, 1: np.concatenate([-vk[64:], vk[:64]]),
                                                      2: -vk}[t].astype(np.float32))


def test_rope_matches_float32_rotation_steps_and_keeps_pair_norms():
    q, k, qw, kw = _qk_inputs(4, 6, 2, 81)
    rng = np.random.default_rng(82)
    ang = rng.uniform(-np.pi, np.pi, (16, 64))
    tab = np.concatenate([np.cos(ang), np.sin(ang)], 1).astype(np.float32)
    pos = np.array([3, 9, 0, 15], np.int32)
    qo, _ = oracle.qk_norm(q, k, qw, kw, pos, tab, 1e-6)
    for t in range(4):
        c, s = tab[pos[t], :64], tab[pos[t], 64:]
        for h in range(6):
            f = bits_to_f32(oracle.rmsnorm(q[t, h], qw, 1e-6))
            a, b = f[:64], f[64:]
            lo = bf16_bits((a * c) - (b * s))
            hi = bf16_bits((b * c) + (a * s))
            assert np.array_equal(qo[t, h], np.concatenate([lo, hi]))
            o = bits_to_f32(qo[t, h]).astype(np.float64)
            n_in = a.astype(np.float64) ** 2 + b.astype(np.float64) ** 2
            n_out = o[:64] ** 2 + o[64:] ** 2
            assert np.all(np.abs(n_out - n_in) <= 2.0 ** -6 * n_in + 1e-12)


def test_rope_uses_the_row_of_each_tokens_position():
    q, k, qw, kw = _qk_inputs(3, 2, 1, 83)
    tab = _table(8, 1, 0)
    tab[5] = _table(1, 0, 1)[0]          # a quarter turn only at position 5
    qo, _ = oracle.qk_norm(q, k, qw, kw, np.array([4, 5, 6], np.int32), tab, 1e-6)
    for t, turned in ((0, False), (1, True), (2, False)):
        f = bits_to_f32(oracle.rmsnorm(q[t, 0], qw, 1e-6))
        want = np.concatenate([-f[64:], f[:64]]) if turned else f
        assert np.array_equal(bits_to_f32(qo[t, 0]), want.astype(np.float32))


@pytest.mark.parametrize("p", [0, 1, 2047, 6143, 100000, 1048575])
def test_ssmax_scale_is_the_rounded_power(p):
    getcontext().prec = 60
    x = Decimal(1) + Decimal(p + 1) / Decimal(2048)
    exact = (Decimal("0.1") * x.ln()).exp()
    assert f32(oracle.ssmax_scale(p)) == nearest_f32(Fraction(exact))
    if p == 2047:
        assert abs(oracle.ssmax_scale(p) - 2.0 ** 0.1) < 1e-7


def test_ssmax_scales_queries_only_and_keys_keep_their_norm():
    q, k, qw, kw = _qk_inputs(2, 3, 2, 84)
    pos = np.array([10, 70000], np.int32)
    qo, ko = oracle.qk_norm(q, k, qw, kw, pos, None, 1e-6, mode="ssmax")
    for t in range(2):
        g = f32(oracle.ssmax_scale(int(pos[t])))
        for h in range(3):
            f = bits_to_f32(oracle.rmsnorm(q[t, h], qw, 1e-6))
            assert np.array_equal(qo[t, h], bf16_bits(f * g))
        for h in range(2):
            assert np.array_equal(ko[t, h], oracle.rmsnorm(k[t, h], kw, 1e-6))
    # queries and keys use their own norm weights
    qo2, ko2 = oracle.qk_norm(q, k, kw, qw, pos, None, 1e-6, mode="ssmax")
    assert not np.array_equal(ko2, ko)


# -------------------------------------------------------------------- NVFP4 output

def test_e4m3_matches_torch_float8_cast_in_range():
    rng = np.random.default_rng(90)
    v = np.concatenate([rng.uniform(-448, 448, 4000), rng.standard_normal(4000) * 0.01,
                        np.ldexp(rng.integers(1, 16, 500) * 0.5 + 0.25, rng.integers(-9, 8, 500))])
    v = v.astype(np.float32)
    v = v[np.abs(v) <= 448]  # torch's cast turns larger values into NaN; these saturate
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3(float(x)) for x in v], np.uint8)
    assert np.array_equal(got, want)
    assert oracle.e4m3_to_f32(oracle.e4m3(1e6)) == 448.0        # saturates
    assert oracle.e4m3_to_f32(oracle.e4m3(-470.0)) == -448.0


def test_e4m3_decoder_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle.e4m3_to_f32(int(c)) for c in codes], np.float32)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(got[~np.isnan(got)], want[~np.isnan(want)])


def test_e2m1_rounding_table():
    # the eight magnitudes 0 0.5 1 1.5 2 3 4 6; halfway cases go to the even code
    cases = {0.25: 0.0, 0.26: 0.5, 0.75: 1.0, 1.25: 1.0, 1.3: 1.5, 1.75: 2.0, 2.5: 2.0,
             2.6: 3.0, 3.5: 4.0, 5.0: 4.0, 5.1: 6.0, 6.0: 6.0, 7.0: 6.0, 1e9: 6.0, -1.75: -2.0,
             -5.0: -4.0, 0.0: 0.0}
    for v, want in cases.items():
        assert oracle.e2m1_to_f32(oracle.e2m1(v)) == want, v
    assert oracle.e2m1(-0.1) == 0x8   # the sign is kept (-0)


def test_e4m3_and_e2m1_saturate_all_the_way_to_infinity():
    """Saturation holds for every magnitude beyond the largest value, infinity
    included (a nearest-distance search would tie once the distances round alike)."""
    for v in (448.0, 449.0, 1e6, 1e17, 1e20, 3.4e38, math.inf):
        assert oracle.e4m3(v) == 0x7E and oracle.e4m3(-v) == 0xFE, v
    for v in (6.0, 6.5, 1e9, 1e17, 1e20, 3.4e38, math.inf):
        assert oracle.e2m1(v) == 0x7 and oracle.e2m1(-v) == 0xF, v


def test_nan_codes_follow_the_reading():
    # E4M3FN keeps NaN as 0x7F; E2M1 has no NaN, and a NaN converts to +6 (0x7),
    # as the hardware's saturating conversion does
    assert oracle.e4m3(math.nan) == 0x7F
    assert oracle.e2m1(math.nan) == 0x7
    # E4M3FN has no infinity: S.1111.111 is NaN, and 0x7E = 448 is the largest value
    assert math.isnan(oracle.e4m3_to_f32(0x7F)) and math.isnan(oracle.e4m3_to_f32(0xFF))
    assert oracle.e4m3_to_f32(0x7E) == 448.0 and oracle.e4m3_to_f32(0xFE) == -448.0


def test_nvfp4_block_amax_skips_nan_and_an_infinite_amax_saturates_the_scale():
    y = np.zeros(32, np.float32)
    y[:4] = [math.inf, 1.0, -2.0, math.nan]  # amax inf: scale 448; codes +6, 0, -0, +6
    y[16:18] = [math.nan, 3.0]               # amax 3 (NaN skipped): scale 0.5; +6, 6
    q, sf = oracle.nvfp4_row(bf16_bits(y), 1.0)
    assert sf[0] == 0x7E and oracle.e4m3_to_f32(int(sf[1])) == 0.5
    nib = [int(q[i // 2]) >> (4 * (i % 2)) & 0xF for i in range(32)]
    assert nib[:4] == [0x7, 0x0, 0x8, 0x7] and nib[4:16] == [0] * 12
    assert nib[16:18] == [0x7, 0x7] and nib[18:] == [0] * 14


def test_nvfp4_hand_block():
    # gs = 1, amax = 3: sf = e4m3(3/6) = 0.5, q = e2m1(2 y)
    y = np.array([1, 2, 3, -1, 0.25, 0, -3, 0.5, 1.5, -2, 0.125, 0, 0, 0, 0, 0.75], np.float32)
    q, sf = oracle.nvfp4_row(bf16_bits(y), 1.0)
    assert oracle.e4m3_to_f32(int(sf[0])) == 0.5
    nib = [int(q[i // 2]) >> (4 * (i % 2)) & 0xF for i in range(16)]
    vals = [oracle.e2m1_to_f32(c) for c in nib]
    assert vals == [2, 4, 6, -2, 0.5, 0, -6, 1, 3, -4, 0, 0, 0, 0, 0, 1.5]
    # an all-zero block has scale 0 and zero codes
    q, sf = oracle.nvfp4_row(np.zeros(16, np.uint16), 448.0)
    assert sf[0] == 0 and not q.any()


def _load_nvfp4_golden():
    vals = {}
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "nvfp4_reciprocal_scale.txt")):
        if line.startswith("#") or ":" not in line:
            continue
        k, v = line.split(":", 1)
        vals[k.strip()] = v.split()
    return vals


def test_nvfp4_block_scale_is_one_reciprocal_factor_per_block():
    # hand-worked block (tests/golden/nvfp4_reciprocal_scale.txt): every value is
    # multiplied by inv = RN32(gs / sf); dividing each RN32(y * gs) by sf instead
    # gives other codes on six of the sixteen values
    g = _load_nvfp4_golden()
    gs = float(np.array([int(g["gs_bits"][0], 16)], np.uint32).view(np.float32)[0])
    y = np.array([float(v) for v in g["y"]], np.float32)
    q, sf = oracle.nvfp4_row(bf16_bits(y), gs)
    assert int(sf[0]) == int(g["sf_code"][0], 16)
    nib = [int(q[i // 2]) >> (4 * (i % 2)) & 0xF for i in range(16)]
    assert nib == [int(c) for c in g["codes"]]
    assert nib != [int(c) for c in g["per_element_codes"]]


def test_nvfp4_dequantises_within_half_a_step():
    rng = np.random.default_rng(91)
    y = bf16_bits(rng.standard_normal(5120) * 2)
    yf = bits_to_f32(y).astype(np.float64)
    gs = 448.0 * 6.0 / float(np.abs(yf).max())
    q, sf = oracle.nvfp4_row(y, gs)
    for blk in range(5120 // 16):
        s = oracle.e4m3_to_f32(int(sf[blk]))
        seg = yf[blk * 16:(blk + 1) * 16]
        codes = [int(q[(blk * 16 + i) // 2]) >> (4 * (i % 2)) & 0xF for i in range(16)]
        deq = np.array([oracle.e2m1_to_f32(c) for c in codes]) * s / gs
        amax = np.abs(seg).max()
        # scale rounding (E4M3, 4 significant bits) may clip the top value a little; the
        # grid step near amax is 2 (in scaled units) -> half a step is amax/6, plus clipping
        assert np.all(np.abs(deq - seg) <= amax / 6 + 2 ** -4 * amax + 1e-12)


def test_nvfp4_boundaries_are_the_bf16_boundaries_then_the_row_quantiser():
    rng = np.random.default_rng(92)
    T, D, n, eps, gs = 6, 512, 5, 1e-6, 336.0
    h = bf16_bits(rng.standard_normal((T, D)))
    x = bf16_bits(rng.standard_normal((T, D)))
    pw, qw = bf16_bits(1 + 0.1 * rng.standard_normal(D)), bf16_bits(1 + 0.1 * rng.standard_normal(D))
    h1, y = oracle.boundary(h, x, pw, qw, n, eps)
    h2, q, sf = oracle.boundary_nvfp4(h, x, pw, qw, n, eps, gs)
    assert np.array_equal(h1, h2)
    for t in range(T):
        qr, sr = oracle.nvfp4_row(y[t], gs)
        assert np.array_equal(q[t], qr) and np.array_equal(sf[t], sr)
    e = bf16_bits(rng.standard_normal((T, 8, D)))
    w = rng.uniform(0, 0.4, (T, 8)).astype(np.float32)
    h1, y = oracle.moe_boundary(h, e, w, pw, qw, n, eps)
    h2, q, sf = oracle.moe_boundary_nvfp4(h, e, w, pw, qw, n, eps, gs)
    assert np.array_equal(h1, h2)
    for t in range(T):
        qr, sr = oracle.nvfp4_row(y[t], gs)
        assert np.array_equal(q[t], qr) and np.array_equal(sf[t], sr)
