"""The oracle's pins must catch plausible mistakes.

Each case below plants one mistake in a copy of ``oracle/oracle.c`` (on the
CPU, in a temporary directory), builds it, and runs the pin suite
``test_oracle_pins.py`` against that build. Every planted mistake must make at
least one pin fail.
"""
from __future__ import annotations

import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("residual coefficients swapped",
     "oracle_bf16_rne(c1 * oracle_bf16_to_f32(h[j]))", "oracle_bf16_rne(c2 * oracle_bf16_to_f32(h[j]))"),
    ("scaled stream not rounded to BF16",
     "float a = oracle_bf16_to_f32(oracle_bf16_rne(c1 * oracle_bf16_to_f32(h[j])));",
     "float a = c1 * oracle_bf16_to_f32(h[j]);"),
    ("scaled branch not rounded to BF16",
     "float b = oracle_bf16_to_f32(oracle_bf16_rne(c2 * oracle_bf16_to_f32(xn[j])));",
     "float b = c2 * oracle_bf16_to_f32(xn[j]);"),
    ("post-norm uses the pre-norm weight",
     "oracle_rmsnorm(x, post_w, eps, D, xn);", "oracle_rmsnorm(x, pre_w, eps, D, xn);"),
    ("next pre-norm reads the branch instead of the new stream",
     "oracle_rmsnorm(h, pre_w, eps, D, y);", "oracle_rmsnorm(x, pre_w, eps, D, y);"),
    ("mean over D - 1", "float ms = S / (float)D;", "float ms = S / (float)(D - 1);"),
    ("eps dropped", "float v = ms + eps;", "float v = ms;"),
    ("c1 without the square root",
     "*c1 = (float)sqrt((double)(n - 1) / (double)n);", "*c1 = (float)((double)(n - 1) / (double)n);"),
    ("c2 = 1/n", "*c2 = (float)(1.0 / sqrt((double)n));", "*c2 = (float)(1.0 / (double)n);"),
    ("BF16 ties rounded away from zero",
     "(rest == 0x8000u && (keep & 1u))", "(rest == 0x8000u)"),
    ("BF16 rounding truncates", "if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1;",
     "if (0) keep += 1;"),
    ("sum rounding ignores ties-to-even", "if (half && (sticky || (m & 1u))) m += 1;",
     "if (half) m += 1;"),
    ("sum rounding drops the sticky bits", "if (half && (sticky || (m & 1u))) m += 1;",
     "if (half && (m & 1u)) m += 1;"),
    ("weight applied before the rms factor",
     "float p = oracle_bf16_to_f32(v[j]) * r;\n        float q = p * oracle_bf16_to_f32(w[j]);",
     "float p = oracle_bf16_to_f32(v[j]) * oracle_bf16_to_f32(w[j]);\n        float q = p * r;"),
    ("MoE running sum rounded to BF16 per expert",
     "acc = fmaf(w[k], oracle_bf16_to_f32(e[(int64_t)k * D + j]), acc);",
     "acc = oracle_bf16_to_f32(oracle_bf16_rne(fmaf(w[k], oracle_bf16_to_f32(e[(int64_t)k * D + j]), acc)));"),
    ("MoE product and add rounded separately",
     "acc = fmaf(w[k], oracle_bf16_to_f32(e[(int64_t)k * D + j]), acc);",
     "acc = acc + w[k] * oracle_bf16_to_f32(e[(int64_t)k * D + j]);"),
    ("MoE experts combined in reverse order",
     "for (int k = 0; k < K; ++k) acc = fmaf(", "for (int k = K - 1; k >= 0; --k) acc = fmaf("),
    ("MoE uses the first routing weight for every expert", "fmaf(w[k],", "fmaf(w[0],"),
    ("MoE expert row index dropped", "e[(int64_t)k * D + j]", "e[(int64_t)k + j]"),
    ("routing group score from the best expert only", "                top = top + b[g * gs + i2];",
     "                top = top + 0.0f * b[g * gs + i2];"),
    ("routing chooses by the unbiased score", "            b[e] = s[e] + bias[e];", "            b[e] = s[e];"),
    ("routing weights from the biased score", "        for (int k = 0; k < topk; ++k) {\n            float q = s[id[k]] / sum;",
     "        for (int k = 0; k < topk; ++k) {\n            float q = b[id[k]] / sum;"),
    ("routing ties to the higher index", "    return isnan(b) || a > b;", "    return isnan(b) || a >= b;"),
    ("routing weights not renormalised", "            float q = s[id[k]] / sum;", "            float q = s[id[k]];"),
    ("routing scale not applied", "            w_out[t * topk + k] = q * scale;", "            w_out[t * topk + k] = q;"),
    ("routing sigmoid of the wrong sign", "hi = z >= 0.0f ? 1.0 / (1.0 + e) : e / (1.0 + e);",
     "hi = z >= 0.0f ? e / (1.0 + e) : 1.0 / (1.0 + e);"),
    ("RoPE pairs neighbours instead of halves",
     "float a = oracle_bf16_to_f32(vn[j]), b = oracle_bf16_to_f32(vn[j + 64]);",
     "float a = oracle_bf16_to_f32(vn[j]), b = oracle_bf16_to_f32(vn[(j + 1) % 128]);"),
    ("RoPE sine sign flipped", "out[j] = oracle_bf16_rne(ac - bs);", "out[j] = oracle_bf16_rne(ac + bs);"),
    ("RoPE table row of the token index", "rope_row(vn, table + p * 128, row);",
     "rope_row(vn, table + t * 128, row);"),
    ("SSMax with the 0-based position", "return (float)pow(1.0 + (double)(pos + 1) / 2048.0, 0.1);",
     "return (float)pow(1.0 + (double)pos / 2048.0, 0.1);"),
    ("SSMax also scales keys", "            } else if (is_q) {", "            } else if (1) {"),
    ("keys normalised with the query weight", "oracle_rmsnorm(row, is_q ? qw : kw, eps, 128, vn);",
     "oracle_rmsnorm(row, qw, eps, 128, vn);"),
    ("NVFP4 block max without the absolute value",
     "float a = fabsf(oracle_bf16_to_f32(y[blk * 16 + j]));", "float a = oracle_bf16_to_f32(y[blk * 16 + j]);"),
    ("NVFP4 scale without the E2M1 maximum", "float t = amax / 6.0f;", "float t = amax;"),
    ("NVFP4 nibbles swapped", "q[(blk * 16 + j) / 2] = (uint8_t)(lo | (hi << 4));",
     "q[(blk * 16 + j) / 2] = (uint8_t)(hi | (lo << 4));"),
    ("FP8/FP4 ties away from zero", "if (d < bd || (d == bd && (c & 1u) == 0 && (best & 1u))) { best = c; bd = d; }",
     "if (d < bd || (d == bd && c > best)) { best = c; bd = d; }"),
    ("NVFP4 quantises with the global scale inverted", "const float inv = sv != 0.0f ? gs / sv : 0.0f;",
     "const float inv = sv != 0.0f ? 1.0f / (gs * sv) : 0.0f;"),
    ("FP8/FP4 saturation left to the distance search",
     "    if (mag >= value(n_codes - 1)) return n_codes - 1;\n", ""),
    ("NVFP4 block max takes NaN", "if (a > amax) amax = a;", "if (!(a <= amax)) amax = a;"),
    ("NVFP4 per-element division instead of one reciprocal factor per block",
     "float a = oracle_bf16_to_f32(y[blk * 16 + j]) * inv;\n                float b = oracle_bf16_to_f32(y[blk * 16 + j + 1]) * inv;",
     "float a = (oracle_bf16_to_f32(y[blk * 16 + j]) * gs) / sv;\n                float b = (oracle_bf16_to_f32(y[blk * 16 + j + 1]) * gs) / sv;"),
    ("E2M1 NaN encoded as zero", "    if (isnan(v)) return 0x7;\n", "    if (isnan(v)) return 0x0;\n"),
    ("routing keeps one group too many", "for (int k = 0; k < topk_group; ++k) {",
     "for (int k = 0; k <= topk_group && k < n_group; ++k) {"),
    ("router sigmoid without the split form near 0",
     "const int small = fabsf(z) < 0x1p-4f;", "const int small = 0;"),
    ("router sigmoid rounding test without the neighbouring candidates",
     "for (int i = 0; i < 3; ++i) {", "for (int i = 0; i < 1; ++i) {"),
    ("routing ranks a NaN score first",
     "    if (isnan(a)) return 0;\n    return isnan(b) || a > b;",
     "    if (isnan(a)) return 1;\n    return isnan(b) || a > b;"),
    ("RoPE cross term with the cosine", "bc = b * c, as = a * s;", "bc = b * c, as = a * c;"),
    ("SSMax exponent 0.2", "(double)(pos + 1) / 2048.0, 0.1);", "(double)(pos + 1) / 2048.0, 0.2);"),
    ("E4M3 subnormals one binade low", "ldexpf((float)m / 8.0f, -6)", "ldexpf((float)m / 8.0f, -7)"),
    ("E2M1 smallest step 0.25", "(m ? 0.5f : 0.0f)", "(m ? 0.25f : 0.0f)"),
    ("long-double residual coefficient squared",
     "long double c1 = sqrtl((long double)(n - 1) / (long double)n);\n    long double c2 = 1.0L / sqrtl((long double)n);\n    for (int64_t i",
     "long double c1 = (long double)(n - 1) / (long double)n;\n    long double c2 = 1.0L / sqrtl((long double)n);\n    for (int64_t i"),
]


def _run_mutant(case, tmp):
    name, old, new = case
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site not found: {name}"
    mutated = src.replace(old, new)
    tag = "".join(c if c.isalnum() else "_" for c in name)
    c_path = os.path.join(tmp, f"{tag}.c")
    so_path = os.path.join(tmp, f"{tag}.so")
    with open(c_path, "w") as f:
        f.write(mutated)
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11", c_path,
                    "-o", so_path, "-lm"], check=True)
    env = dict(os.environ, BEAM_ORACLE_SO=so_path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    return name, r.returncode


@pytest.mark.slow
def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
            results = list(ex.map(lambda c: _run_mutant(c, tmp), MUTANTS))
    survivors = [name for name, rc in results if rc == 0]
    assert not survivors, f"mistakes no pin caught: {survivors}"
