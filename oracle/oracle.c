/*
 * CPU oracle for the fused sublayer boundary of the Beam decoder.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the package's smoke check and the
 * bench's CPU-baseline leg are the only callers. The CUDA library never links,
 * loads or calls this file, and this file shares no code with it.
 *
 * What it computes (one token row at a time, plain loops, one thread):
 *
 *   Sandwich norm and depth-scaled residual (Beam blog, SGLang page,
 *   "Sandwich normalization and depth-scaled residual"; vLLM page, "MoE and
 *   residual stream"): every branch has an input and an output RMSNorm, and
 *   the n-th residual add is  h <- sqrt((n-1)/n) * h + x / sqrt(n).
 *   Both scaled operands are rounded to the activation dtype (BF16) before the
 *   add (SGLang page, same section). The fused boundary keeps FP32 math and
 *   the BF16 rounding points of the unfused code (vLLM page, "Agent-driven
 *   optimization", change 1), and the unfused code writes the normalised
 *   branch (SGLang page, same section), so that branch is a BF16 tensor.
 *
 *   RMSNorm, FP32 math (the pages give no formula; the standard RMS norm):
 *     S   = RN32( sum_j RN32(v_j * v_j) )   exact sum, rounded once
 *     ms  = RN32(S / D)
 *     r   = RN32(1 / RN32(sqrt(RN32(ms + eps))))
 *     out = bf16( RN32( RN32(v_j * r) * w_j ) )
 *   The pages leave the order of the FP32 sum open and accept FP32
 *   reduction-order differences as noise (SGLang page, "BF16 MoE kernel
 *   optimization" and "Reinforcement learning in Miles"); the oracle takes the
 *   one order-free FP32 value, the exact sum rounded once to nearest-even.
 *
 *   Boundary, per row:
 *     xn_j = rmsnorm(x, post_w)_j                      (BF16)
 *     c1   = RN32(sqrt((n-1)/n)), c2 = RN32(1/sqrt(n))  (evaluated in double)
 *     a_j  = bf16(RN32(c1 * h_j)),  b_j = bf16(RN32(c2 * xn_j))
 *     h'_j = bf16(RN32(a_j + b_j))                     (stored over h)
 *     y_j  = rmsnorm(h', pre_w)_j                      (BF16)
 *
 *   MoE combine in front of the boundary (vLLM page, change 3: after the MoE
 *   the norm kernel also combines the top-8 expert outputs; SGLang page,
 *   "Fusion optimizations": the BF16 MoE path folds the local expert sum,
 *   the routing scale and the BF16 rounding together; "Dense layers and
 *   grouped MoE routing": FP32 routing coefficients):
 *     acc_j = 0; for k = 0..K-1: acc_j = fma(w_k, e_kj, acc_j)   (FP32)
 *     x_j   = bf16(acc_j)
 *   The routing scale of 2.5 is already inside w.
 *
 * bf16(v) is IEEE-754 round-to-nearest-even from FP32 to the 8-bit
 * significand; any NaN becomes the quiet NaN 0x7FFF; overflow gives +-inf;
 * subnormals are kept. Build with -ffp-contract=off so that no mul+add pair is
 * fused behind the source's back.
 *
 * The *_ld functions repeat the boundary in long double with no rounding at
 * all; they exist for the hand-worked and closed-form checks.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef uint16_t bf16_t;

static float f32_of_bits(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t bits_of_f32(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

float oracle_bf16_to_f32(bf16_t b) { return f32_of_bits((uint32_t)b << 16); }

bf16_t oracle_bf16_rne(float f) {
    uint32_t u = bits_of_f32(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) return 0x7FFF;
    uint32_t keep = u >> 16;      /* sign, exponent and the top 7 fraction bits */
    uint32_t rest = u & 0xFFFFu;  /* the 16 dropped bits */
    /* above the halfway point, or exactly halfway with an odd kept part: round the
     * magnitude up; a carry out of the fraction correctly bumps the exponent,
     * up to infinity */
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1;
    return (bf16_t)keep;
}

/* ------------------------------------------------------------------------
 * Exact sum of non-negative floats, rounded once to FP32.
 *
 * A finite float t >= 0 with biased exponent field E and fraction f is
 * m * 2^(q - 149) with m = (E ? 2^23 + f : f) < 2^24 and q = (E ? E - 1 : 0).
 * The sum is held exactly as the integer N = sum m * 2^q in a little-endian
 * array of single bits; the value is N * 2^-149. 320 bits hold 2^43 terms.
 * ---------------------------------------------------------------------- */
#define ACC_BITS 320

typedef struct {
    uint8_t bit[ACC_BITS];
    int any_nan, any_inf, any_negative;
} exact_acc;

static void acc_init(exact_acc* a) { memset(a, 0, sizeof *a); }

static void acc_add(exact_acc* a, float t) {
    uint32_t u = bits_of_f32(t);
    uint32_t E = (u >> 23) & 0xFFu, f = u & 0x7FFFFFu;
    if (E == 0xFFu) {
        if (f) a->any_nan = 1;
        else if (u >> 31) a->any_negative = 1;
        else a->any_inf = 1;
        return;
    }
    if ((u >> 31) && (u & 0x7FFFFFFFu)) { a->any_negative = 1; return; }
    uint32_t m = E ? (f | 0x800000u) : f;
    int q = E ? (int)E - 1 : 0;
    for (int i = 0; i < 24; ++i) {
        if (!((m >> i) & 1u)) continue;
        int p = q + i; /* add 2^p with carry */
        while (a->bit[p]) a->bit[p++] = 0;
        a->bit[p] = 1;
    }
}

static float acc_round(const exact_acc* a) {
    if (a->any_nan || a->any_negative) return NAN;
    if (a->any_inf) return INFINITY;
    int top = -1;
    for (int p = ACC_BITS - 1; p >= 0; --p)
        if (a->bit[p]) { top = p; break; }
    if (top < 0) return 0.0f;
    if (top <= 23) {
        /* N < 2^24: N * 2^-149 is a subnormal or lies in the first normal
         * binade; either way it is exact and its bit pattern is N itself */
        uint32_t v = 0;
        for (int p = top; p >= 0; --p) v = (v << 1) | a->bit[p];
        return f32_of_bits(v);
    }
    int lo = top - 23; /* keep bits lo..top (24 bits) */
    uint32_t m = 0;
    for (int p = top; p >= lo; --p) m = (m << 1) | a->bit[p];
    int half = a->bit[lo - 1], sticky = 0;
    for (int p = lo - 2; p >= 0; --p) sticky |= a->bit[p];
    if (half && (sticky || (m & 1u))) m += 1;
    if (m == (1u << 24)) { m >>= 1; lo += 1; }
    /* value = m * 2^(lo - 149) with m in [2^23, 2^24): biased exponent lo + 1 */
    uint32_t Eb = (uint32_t)lo + 1u;
    if (Eb >= 255u) return INFINITY;
    return f32_of_bits((Eb << 23) | (m & 0x7FFFFFu));
}

/* RN32 of the exact sum of t[0..n-1]; every t must be >= 0 (else NaN) */
float oracle_sum_f32_exact(const float* t, int64_t n) {
    exact_acc* a = (exact_acc*)malloc(sizeof(exact_acc));
    if (!a) return NAN;
    acc_init(a);
    for (int64_t i = 0; i < n; ++i) acc_add(a, t[i]);
    float s = acc_round(a);
    free(a);
    return s;
}

/* S = RN32(sum_j RN32(v_j * v_j)) over a BF16 row */
float oracle_sum_squares(const bf16_t* v, int D) {
    exact_acc a;
    acc_init(&a);
    for (int j = 0; j < D; ++j) {
        float vj = oracle_bf16_to_f32(v[j]);
        float sq = vj * vj;
        acc_add(&a, sq);
    }
    return acc_round(&a);
}

/* r = 1 / sqrt(S / D + eps), each operation in FP32 */
float oracle_rms_factor(float S, int D, float eps) {
    float ms = S / (float)D;
    float v = ms + eps;
    float root = sqrtf(v);
    return 1.0f / root;
}

/* out_j = bf16((v_j * r) * w_j), r from the row's mean square */
void oracle_rmsnorm(const bf16_t* v, const bf16_t* w, float eps, int D, bf16_t* out) {
    float r = oracle_rms_factor(oracle_sum_squares(v, D), D, eps);
    for (int j = 0; j < D; ++j) {
        float p = oracle_bf16_to_f32(v[j]) * r;
        float q = p * oracle_bf16_to_f32(w[j]);
        out[j] = oracle_bf16_rne(q);
    }
}

/* depth-scaled residual coefficients for the n-th add (n >= 1) */
void oracle_scales(int n, float* c1, float* c2) {
    *c1 = (float)sqrt((double)(n - 1) / (double)n);
    *c2 = (float)(1.0 / sqrt((double)n));
}

/* x_j = bf16(RN32(scale * fma chain over k of w_k * e_kj)), e is [K, D], w is [K].
 * With the routing scale carried in w, scale is 1 and the product is exact. */
static void moe_combine_scaled(const bf16_t* e, const float* w, int K, int D, float scale, bf16_t* x_out) {
    for (int j = 0; j < D; ++j) {
        float acc = 0.0f;
        for (int k = 0; k < K; ++k) acc = fmaf(w[k], oracle_bf16_to_f32(e[(int64_t)k * D + j]), acc);
        x_out[j] = oracle_bf16_rne(scale * acc);
    }
}

void oracle_moe_combine(const bf16_t* e, const float* w, int K, int D, bf16_t* x_out) {
    moe_combine_scaled(e, w, K, D, 1.0f, x_out);
}

void oracle_moe_combine_scaled(const bf16_t* e, const float* w, int K, int D, float scale, bf16_t* x_out) {
    moe_combine_scaled(e, w, K, D, scale, x_out);
}

/* one row of the boundary given its (BF16) branch output x */
static void boundary_row(bf16_t* h, const bf16_t* x, const bf16_t* post_w, const bf16_t* pre_w,
                         float c1, float c2, float eps, int D, bf16_t* y, bf16_t* xn) {
    oracle_rmsnorm(x, post_w, eps, D, xn);
    for (int j = 0; j < D; ++j) {
        float a = oracle_bf16_to_f32(oracle_bf16_rne(c1 * oracle_bf16_to_f32(h[j])));
        float b = oracle_bf16_to_f32(oracle_bf16_rne(c2 * oracle_bf16_to_f32(xn[j])));
        h[j] = oracle_bf16_rne(a + b);
    }
    oracle_rmsnorm(h, pre_w, eps, D, y);
}

/* Dense boundary. h [T,D] in/out; x, y [T,D]; post_w, pre_w [D]. Returns 0, or -1 on bad sizes. */
int oracle_boundary(bf16_t* h, const bf16_t* x, const bf16_t* post_w, const bf16_t* pre_w, int n,
                    float eps, int64_t T, int D, bf16_t* y) {
    if (n < 1 || D < 1 || T < 0) return -1;
    float c1, c2;
    oracle_scales(n, &c1, &c2);
    bf16_t* xn = (bf16_t*)malloc(sizeof(bf16_t) * (size_t)D);
    if (!xn) return -1;
    for (int64_t t = 0; t < T; ++t)
        boundary_row(h + t * D, x + t * D, post_w, pre_w, c1, c2, eps, D, y + t * D, xn);
    free(xn);
    return 0;
}

/* MoE boundary with the routing scale applied in the combine */
int oracle_moe_boundary_scaled(bf16_t* h, const bf16_t* e, const float* topk_w, int K, float scale,
                               const bf16_t* post_w, const bf16_t* pre_w, int n, float eps, int64_t T,
                               int D, bf16_t* y) {
    if (n < 1 || D < 1 || T < 0 || K < 1) return -1;
    float c1, c2;
    oracle_scales(n, &c1, &c2);
    bf16_t* x = (bf16_t*)malloc(sizeof(bf16_t) * (size_t)D * 2);
    if (!x) return -1;
    for (int64_t t = 0; t < T; ++t) {
        moe_combine_scaled(e + t * (int64_t)K * D, topk_w + t * K, K, D, scale, x);
        boundary_row(h + t * D, x, post_w, pre_w, c1, c2, eps, D, y + t * D, x + D);
    }
    free(x);
    return 0;
}

/* MoE boundary. e [T,K,D]; topk_w [T,K] FP32; other operands as the dense boundary. */
int oracle_moe_boundary(bf16_t* h, const bf16_t* e, const float* topk_w, int K,
                        const bf16_t* post_w, const bf16_t* pre_w, int n, float eps, int64_t T,
                        int D, bf16_t* y) {
    if (n < 1 || D < 1 || T < 0 || K < 1) return -1;
    float c1, c2;
    oracle_scales(n, &c1, &c2);
    bf16_t* x = (bf16_t*)malloc(sizeof(bf16_t) * (size_t)D * 2);
    if (!x) return -1;
    for (int64_t t = 0; t < T; ++t) {
        oracle_moe_combine(e + t * (int64_t)K * D, topk_w + t * K, K, D, x);
        boundary_row(h + t * D, x, post_w, pre_w, c1, c2, eps, D, y + t * D, x + D);
    }
    free(x);
    return 0;
}

/* ---- long double, no rounding anywhere ----------------------------------- */

static void rmsnorm_ld(const long double* v, const long double* w, long double eps, int D,
                       long double* out) {
    long double s = 0.0L;
    for (int j = 0; j < D; ++j) s += v[j] * v[j];
    long double r = 1.0L / sqrtl(s / (long double)D + eps);
    for (int j = 0; j < D; ++j) out[j] = v[j] * r * w[j];
}

int oracle_boundary_ld(long double* h, const long double* x, const long double* post_w,
                       const long double* pre_w, int n, long double eps, int64_t T, int D,
                       long double* y) {
    if (n < 1 || D < 1 || T < 0) return -1;
    long double c1 = sqrtl((long double)(n - 1) / (long double)n);
    long double c2 = 1.0L / sqrtl((long double)n);
    long double* xn = (long double*)malloc(sizeof(long double) * (size_t)D);
    if (!xn) return -1;
    for (int64_t t = 0; t < T; ++t) {
        rmsnorm_ld(x + t * D, post_w, eps, D, xn);
        for (int j = 0; j < D; ++j) h[t * D + j] = c1 * h[t * D + j] + c2 * xn[j];
        rmsnorm_ld(h + t * D, pre_w, eps, D, y + t * D);
    }
    free(xn);
    return 0;
}

/* residual update alone, long double: h <- sqrt((n-1)/n) h + x / sqrt(n) */
void oracle_residual_ld(long double* h, const long double* x, int n, int64_t count) {
    long double c1 = sqrtl((long double)(n - 1) / (long double)n);
    long double c2 = 1.0L / sqrtl((long double)n);
    for (int64_t i = 0; i < count; ++i) h[i] = c1 * h[i] + c2 * x[i];
}

/* ------------------------------------------------------------------------
 * Group-limited top-k routing in front of the MoE combine (vLLM page, "MoE
 * and residual stream": sigmoid scores plus a correction bias pick the best
 * 4 of 8 expert groups, then the top 8 experts, and the renormalised weights
 * are scaled by 2.5; SGLang page, "Dense layers and grouped MoE routing":
 * FP32 logits and routing coefficients; HF page: 8 groups of 32 experts).
 *
 * Per token, FP32 throughout:
 *   s_e = RN32(1 / (1 + exp(-z_e)))       the sigmoid, correctly rounded
 *   b_e = RN32(s_e + bias_e)              biased score, used only to choose
 *   group score = RN32(top1 + top2) of the b_e in the group (the pages say the
 *                 routing matches DeepSeek-V3, whose group score is the sum of
 *                 the group's two best biased scores)
 *   keep the topk_group best groups; among their experts take the topk best
 *   b_e. Ties go to the lower index; the output is in descending b_e. A NaN
 *   score (the pages do not speak of one) ranks below every number, NaNs
 *   among themselves by index: one total order, so exactly topk_group groups
 *   and topk experts are kept whatever the inputs hold.
 *   sum = RN32 running sum of the chosen s_e in output order
 *   w_k = RN32(RN32(s_k / sum) * scale)
 *
 * The sigmoid is the FP32 value nearest to 1 / (1 + e^-z), found by Ziv's
 * strategy (A. Ziv, "Fast evaluation of elementary mathematical functions
 * with correctly rounded last bit", ACM TOMS 17(3), 1991): evaluate with a
 * known error bound and accept the rounding when every value within the bound
 * rounds alike; otherwise evaluate again with more precision. Each level
 * forms the value as hi + lo:
 *   |z| >= 2^-4: hi = 1/(1+e) for z >= 0, e/(1+e) for z < 0, e = e^-|z|
 *                (lo = 0); exp within 1 ulp, then one add and one division:
 *                within 3 ulps of the exact value, relative.
 *   |z| <  2^-4: hi = 1/2, lo = tanh(z/2)/2 (sigma(z) = (1 + tanh(z/2))/2),
 *                tanh within a few ulps of lo. Near 0 the value sits within
 *                z^3/48 of 1/2 + z/4, which is a rounding midpoint for every
 *                z that is an odd multiple of 2^-23 (2^-24 below zero); a
 *                bound relative to lo, not to the value, decides those.
 *   level 1: double, accepted with the bound 2^-49 relative to hi or lo;
 *   level 2: long double (64 or 113 significant bits), bound 2^-(p-4).
 * For z != 0 the exact value is transcendental (Lindemann-Weierstrass), so
 * it never sits on a rounding midpoint and some precision always decides; a
 * value that level 2 still leaves open is counted (oracle_sigmoid_undecided)
 * and the tests require that count to stay 0.
 * ---------------------------------------------------------------------- */

static unsigned long long g_sigmoid_undecided;

/* 1 when every value of [hi + lo - eb, hi + lo + eb] rounds to the same
 * binary32 value *out. The candidates are RN32(hi + lo) and its two
 * neighbours (hi + lo rounded first may fall on a midpoint that the exact
 * sum does not reach). The midpoints between neighbouring floats are exact in
 * double; hi - midpoint is exact (Sterbenz) and adding lo and eb keeps its
 * sign, so each comparison is decided correctly. */
static int rn32_certain(double hi, double lo, double eb, float* out) {
    const float f0 = (float)(hi + lo);
    const float cand[3] = {f0, nextafterf(f0, -INFINITY), nextafterf(f0, INFINITY)};
    *out = f0;
    for (int i = 0; i < 3; ++i) {
        const float f = cand[i];
        const double m_lo = 0.5 * ((double)f + (double)nextafterf(f, -INFINITY));
        const double m_hi = 0.5 * ((double)f + (double)nextafterf(f, INFINITY));
        if (((hi - m_lo) + lo) - eb > 0.0 && ((hi - m_hi) + lo) + eb < 0.0) {
            *out = f;
            return 1;
        }
    }
    return 0;
}

static int rn32_certain_l(long double hi, long double lo, long double eb, float* out) {
    const float f0 = (float)(hi + lo);
    const float cand[3] = {f0, nextafterf(f0, -INFINITY), nextafterf(f0, INFINITY)};
    *out = f0;
    for (int i = 0; i < 3; ++i) {
        const float f = cand[i];
        const long double m_lo = 0.5L * ((long double)f + (long double)nextafterf(f, -INFINITY));
        const long double m_hi = 0.5L * ((long double)f + (long double)nextafterf(f, INFINITY));
        if (((hi - m_lo) + lo) - eb > 0.0L && ((hi - m_hi) + lo) + eb < 0.0L) {
            *out = f;
            return 1;
        }
    }
    return 0;
}

static float sigmoid_rn32(float z) {
    if (isnan(z)) return z;
    float r;
    const int small = fabsf(z) < 0x1p-4f;
    {
        double hi = 0.5, lo = 0.0;
        if (small) {
            lo = 0.5 * tanh(0.5 * (double)z);
        } else {
            const double e = exp(-fabs((double)z));
            hi = z >= 0.0f ? 1.0 / (1.0 + e) : e / (1.0 + e);
        }
        if (rn32_certain(hi, lo, ldexp(small ? fabs(lo) : hi, -49) + 0x1p-1070, &r)) return r;
    }
    {
        long double hi = 0.5L, lo = 0.0L;
        if (small) {
            lo = 0.5L * tanhl(0.5L * (long double)z);
        } else {
            const long double e = expl(-fabsl((long double)z));
            hi = z >= 0.0f ? 1.0L / (1.0L + e) : e / (1.0L + e);
        }
        if (rn32_certain_l(hi, lo, ldexpl(small ? fabsl(lo) : hi, 4 - LDBL_MANT_DIG) + 0x1p-1070L, &r))
            return r;
    }
    __atomic_fetch_add(&g_sigmoid_undecided, 1ull, __ATOMIC_RELAXED);
    return r;
}

/* a ranks before b: a larger number, or a number against a NaN; equal values
 * (and two NaNs) are left to the index */
static int score_before(float a, float b) {
    if (isnan(a)) return 0;
    return isnan(b) || a > b;
}

/* index of the best of the first n values of v whose taken[] flag is 0
 * (ties: the lower index); -1 if none */
static int best_free(const float* v, const unsigned char* taken, int n) {
    int best = -1;
    for (int i = 0; i < n; ++i) {
        if (taken[i]) continue;
        if (best < 0 || score_before(v[i], v[best])) best = i;
    }
    return best;
}

int oracle_route(const float* logits, const float* bias, int64_t T, int E, int n_group,
                 int topk_group, int topk, float scale, int32_t* idx_out, float* w_out) {
    if (E < 1 || n_group < 1 || E % n_group || topk_group < 1 || topk_group > n_group || topk < 1 ||
        topk > (E / n_group) * topk_group || E > 4096 || topk > 64)
        return -1;
    const int gs = E / n_group;
    float s[4096], b[4096], gscore[4096];
    unsigned char taken[4096], gtaken[4096];
    for (int64_t t = 0; t < T; ++t) {
        const float* z = logits + t * E;
        for (int e = 0; e < E; ++e) {
            s[e] = sigmoid_rn32(z[e]);
            b[e] = s[e] + bias[e];
        }
        /* group scores: sum of the group's two best biased scores */
        for (int g = 0; g < n_group; ++g) {
            memset(taken, 0, (size_t)gs);
            int i1 = best_free(b + g * gs, taken, gs);
            float top = b[g * gs + i1];
            if (gs > 1) {
                taken[i1] = 1;
                int i2 = best_free(b + g * gs, taken, gs);
                top = top + b[g * gs + i2];
            }
            gscore[g] = top;
        }
        /* keep the topk_group best groups; experts outside them are not eligible */
        memset(gtaken, 0, (size_t)n_group);
        memset(taken, 1, (size_t)E);
        for (int k = 0; k < topk_group; ++k) {
            int g = best_free(gscore, gtaken, n_group);
            gtaken[g] = 1;
            memset(taken + g * gs, 0, (size_t)gs);
        }
        /* topk best biased scores among the eligible experts, in descending order */
        float sum = 0.0f;
        int32_t* id = idx_out + t * topk;
        for (int k = 0; k < topk; ++k) {
            int e = best_free(b, taken, E);
            taken[e] = 1;
            id[k] = e;
            sum = (k == 0) ? s[e] : sum + s[e];
        }
        for (int k = 0; k < topk; ++k) {
            float q = s[id[k]] / sum;
            w_out[t * topk + k] = q * scale;
        }
    }
    return 0;
}

/* the FP32 sigmoid the router uses, exposed for the pins */
float oracle_sigmoid(float z) { return sigmoid_rn32(z); }

/* the same over an array (tests compare whole ranges of inputs) */
void oracle_sigmoid_array(const float* z, float* s, int64_t n) {
    for (int64_t i = 0; i < n; ++i) s[i] = sigmoid_rn32(z[i]);
}

/* sigmoid values that the two precision levels left undecided (none are expected) */
unsigned long long oracle_sigmoid_undecided(void) { return __atomic_load_n(&g_sigmoid_undecided, __ATOMIC_RELAXED); }

/* ------------------------------------------------------------------------
 * Per-head Q/K RMSNorm with RoPE or SSMax (vLLM page, "Beam model
 * architecture": Q and K are RMS-normalised per head before RoPE or SSMax;
 * 48 query heads, 8 KV heads, head dimension 128; sliding-window layers use
 * RoPE, full-attention layers use no positional encoding and scale each query
 * by (1 + p/2048)^0.1 with p the 1-based position; HF page: the same scale
 * written with the 0-based position, (1 + (pos+1)/2048)^0.1; FP32 at the norm,
 * RoPE and query-scaling positions).
 *
 * Per head row v[0..127] (BF16), weight w:
 *   vn_j = bf16((v_j * r) * w_j)  as oracle_rmsnorm (exact FP32 sum, one rounding)
 * RoPE (rotate-half pairs j and j + 64, cos/sin from the caller's FP32 table
 * row of the token's position: c_j = table[pos][j], s_j = table[pos][64 + j]):
 *   out_j      = bf16(RN32(RN32(vn_j * c_j)      - RN32(vn_{j+64} * s_j)))
 *   out_{j+64} = bf16(RN32(RN32(vn_{j+64} * c_j) + RN32(vn_j * s_j)))
 * SSMax (queries only; keys keep vn):
 *   g = RN32((1 + (pos + 1) / 2048)^0.1)   (evaluated in double, rounded once)
 *   out_j = bf16(RN32(vn_j * g))
 * ---------------------------------------------------------------------- */

float oracle_ssmax_scale(int64_t pos) {
    return (float)pow(1.0 + (double)(pos + 1) / 2048.0, 0.1);
}

static void rope_row(const bf16_t* vn, const float* cs, bf16_t* out) {
    for (int j = 0; j < 64; ++j) {
        float a = oracle_bf16_to_f32(vn[j]), b = oracle_bf16_to_f32(vn[j + 64]);
        float c = cs[j], s = cs[64 + j];
        float ac = a * c, bs = b * s, bc = b * c, as = a * s;
        out[j] = oracle_bf16_rne(ac - bs);
        out[j + 64] = oracle_bf16_rne(bc + as);
    }
}

/* mode 0: RoPE on q and k; mode 1: SSMax on q, norm only on k.
 * q [T, nq, 128] and k [T, nk, 128] are overwritten. Returns 0, or -1 on bad arguments. */
int oracle_qk_norm(bf16_t* q, bf16_t* k, const bf16_t* qw, const bf16_t* kw, const int32_t* pos,
                   const float* table, int64_t max_pos, int64_t T, int nq, int nk, float eps,
                   int mode) {
    if (T < 0 || nq < 0 || nk < 0 || (mode != 0 && mode != 1)) return -1;
    bf16_t vn[128];
    for (int64_t t = 0; t < T; ++t) {
        const int64_t p = pos[t];
        if (p < 0 || (mode == 0 && p >= max_pos)) return -1;
        const float g = oracle_ssmax_scale(p);
        for (int hh = 0; hh < nq + nk; ++hh) {
            const int is_q = hh < nq;
            bf16_t* row = is_q ? q + (t * nq + hh) * 128 : k + (t * nk + (hh - nq)) * 128;
            oracle_rmsnorm(row, is_q ? qw : kw, eps, 128, vn);
            if (mode == 0) {
                rope_row(vn, table + p * 128, row);
            } else if (is_q) {
                for (int j = 0; j < 128; ++j) row[j] = oracle_bf16_rne(oracle_bf16_to_f32(vn[j]) * g);
            } else {
                memcpy(row, vn, sizeof vn);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * NVFP4 output of the next pre-norm (SGLang page, "Fusion optimizations": the
 * fusable boundary is extended to NVFP4). The pages give no format; this
 * follows NVIDIA's published NVFP4 layout:
 *   elements FP4 E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit:
 *   0, 0.5, 1, 1.5, 2, 3, 4, 6), two per byte, element 2i in the low nibble;
 *   one FP8 E4M3 (OCP E4M3FN, bias 7, largest 448) scale per 16 consecutive
 *   elements; an FP32 global scale gs from the caller.
 * The steps of a block are those of TensorRT-LLM's open-source FP4 quantiser
 * (which vLLM and SGLang reuse for NVFP4 activations): the block scale is
 * gs * (amax / 6) rounded to E4M3, and every value is multiplied by one
 * per-block FP32 factor, the reciprocal of (E4M3 scale / gs), before its
 * saturating nearest-even E2M1 conversion. That code forms the factor from
 * hardware reciprocal approximations; this reading takes each step as one
 * correctly rounded FP32 operation. Per block of the BF16 row y:
 *   amax = max |y_j|
 *   sf   = E4M3(RN32(RN32(amax / 6) * gs))           nearest, ties to even, saturating
 *   inv  = RN32(gs / sf)                              one factor per block
 *   q_j  = sf == 0 ? +0 : E2M1(RN32(y_j * inv))
 * Both conversions are written out as a nearest search over the format's
 * finite values (ties to the even code, magnitudes above the largest value,
 * infinities included, saturate; the sign is kept). A NaN converts to E4M3's
 * NaN code 0x7F. E2M1 has no NaN and neither the pages nor the recipe say
 * what a NaN becomes; the reading sends it to the largest code, +6 (0x7), as
 * saturation does with every value beyond the finite range. The block amax
 * skips NaN values (a maximum ignores them).
 * ---------------------------------------------------------------------- */

static float e4m3_value(unsigned code) { /* finite codes 0..0x7E of the magnitude */
    unsigned e = (code >> 3) & 0xF, m = code & 7;
    return e ? ldexpf(1.0f + (float)m / 8.0f, (int)e - 7) : ldexpf((float)m / 8.0f, -6);
}

static float e2m1_value(unsigned code) {
    unsigned e = (code >> 1) & 3, m = code & 1;
    return e ? ldexpf(1.0f + (float)m / 2.0f, (int)e - 1) : (m ? 0.5f : 0.0f);
}

/* nearest code (magnitude) among n_codes values, ties to the even code; saturates */
static unsigned nearest_code(float mag, float (*value)(unsigned), unsigned n_codes) {
    /* saturating: the largest value and anything beyond it, infinity included
     * (a distance search would tie once the distances round alike) */
    if (mag >= value(n_codes - 1)) return n_codes - 1;
    unsigned best = 0;
    double bd = fabs((double)mag - (double)value(0));
    for (unsigned c = 1; c < n_codes; ++c) {
        double d = fabs((double)mag - (double)value(c));
        if (d < bd || (d == bd && (c & 1u) == 0 && (best & 1u))) { best = c; bd = d; }
    }
    return best;
}

uint8_t oracle_e4m3(float v) {
    if (isnan(v)) return 0x7F;
    unsigned s = signbit(v) ? 0x80u : 0u;
    return (uint8_t)(s | nearest_code(fabsf(v), e4m3_value, 0x7F));
}

uint8_t oracle_e2m1(float v) {
    if (isnan(v)) return 0x7;
    unsigned s = signbit(v) ? 0x8u : 0u;
    return (uint8_t)(s | nearest_code(fabsf(v), e2m1_value, 8));
}

float oracle_e4m3_to_f32(uint8_t b) {
    if ((b & 0x7Fu) == 0x7Fu) return NAN; /* E4M3FN: S.1111.111 is NaN (there is no infinity) */
    float m = e4m3_value(b & 0x7Fu);
    return (b & 0x80u) ? -m : m;
}

float oracle_e2m1_to_f32(uint8_t b) {
    float m = e2m1_value(b & 7u);
    return (b & 8u) ? -m : m;
}

/* quantise a BF16 row of D (a multiple of 16) values: q [D/2] bytes, sf [D/16] bytes */
void oracle_nvfp4_row(const bf16_t* y, int D, float gs, uint8_t* q, uint8_t* sf) {
    for (int blk = 0; blk < D / 16; ++blk) {
        float amax = 0.0f;
        for (int j = 0; j < 16; ++j) {
            float a = fabsf(oracle_bf16_to_f32(y[blk * 16 + j]));
            if (a > amax) amax = a;
        }
        float t = amax / 6.0f;
        uint8_t s = oracle_e4m3(t * gs);
        float sv = oracle_e4m3_to_f32(s);
        sf[blk] = s;
        const float inv = sv != 0.0f ? gs / sv : 0.0f;
        for (int j = 0; j < 16; j += 2) {
            uint8_t lo = 0, hi = 0;
            if (sv != 0.0f) {
                float a = oracle_bf16_to_f32(y[blk * 16 + j]) * inv;
                float b = oracle_bf16_to_f32(y[blk * 16 + j + 1]) * inv;
                lo = oracle_e2m1(a);
                hi = oracle_e2m1(b);
            }
            q[(blk * 16 + j) / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* dense boundary whose y leaves as NVFP4 */
int oracle_boundary_nvfp4(bf16_t* h, const bf16_t* x, const bf16_t* post_w, const bf16_t* pre_w,
                          int n, float eps, int64_t T, int D, float gs, uint8_t* q, uint8_t* sf) {
    if (D % 16) return -1;
    bf16_t* y = (bf16_t*)malloc(sizeof(bf16_t) * (size_t)D);
    if (!y) return -1;
    for (int64_t t = 0; t < T; ++t) {
        if (oracle_boundary(h + t * D, x + t * D, post_w, pre_w, n, eps, 1, D, y) != 0) { free(y); return -1; }
        oracle_nvfp4_row(y, D, gs, q + t * (D / 2), sf + t * (D / 16));
    }
    free(y);
    return 0;
}

/* MoE boundary whose y leaves as NVFP4 */
int oracle_moe_boundary_nvfp4(bf16_t* h, const bf16_t* e, const float* topk_w, int K,
                              const bf16_t* post_w, const bf16_t* pre_w, int n, float eps, int64_t T,
                              int D, float gs, uint8_t* q, uint8_t* sf) {
    if (D % 16) return -1;
    bf16_t* y = (bf16_t*)malloc(sizeof(bf16_t) * (size_t)D);
    if (!y) return -1;
    for (int64_t t = 0; t < T; ++t) {
        if (oracle_moe_boundary(h + t * D, e + t * (int64_t)K * D, topk_w + t * K, K, post_w, pre_w, n, eps, 1,
                                D, y) != 0) {
            free(y);
            return -1;
        }
        oracle_nvfp4_row(y, D, gs, q + t * (D / 2), sf + t * (D / 16));
    }
    free(y);
    return 0;
}
