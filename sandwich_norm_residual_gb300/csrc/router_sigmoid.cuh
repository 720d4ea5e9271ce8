// Correctly rounded FP32 sigmoid of the MoE router, sm_103a.
//
// The routing rule scores each expert with the FP32 sigmoid of its logit
// (vLLM page, "MoE and residual stream"; SGLang page, "Dense layers and
// grouped MoE routing": FP32 routing). Its exact FP32 value is
// s = RN32(1 / (1 + e^-z)), the float nearest the real sigmoid. It is found by
// Ziv's strategy (A. Ziv, "Fast evaluation of elementary mathematical
// functions with correctly rounded last bit", ACM TOMS 17(3), 1991): an
// evaluation with a known error bound is accepted when every value within the
// bound rounds to the same float; otherwise the value is evaluated again with
// more precision.
//
// Phase 1 (FP32 pipes, every value), float-float arithmetic. With a = |z| and
// k = rint(a * 32/ln2) = 32 K + j (0 <= j < 32):
//   e^-a = 2^-K * 2^(-j/32) * e^s,   s = k ln2/32 - a,   |s| <= ln2/64 (+ rounding of k)
//   - s: Cody-Waite reduction, ln2/32 = L1 + L2 + L3 in floats with L1 of 11
//     significant bits (k < 2^13, so k L1 and a - k L1 are exact), k L2 split
//     exactly with an FMA; s is a float pair sh + sl.
//   - e^s: Taylor series to s^5 (the rest is below 2^-48.6); 1 + sh + sh^2/2
//     as an error-free pair, the small terms (sh^2's rounding, s^3..s^5,
//     sl e^sh) in plain floats.
//   - 2^(-j/32): 32 float pairs, one table entry per lane, fetched by shuffle.
//   - M = 2^(-j/32) e^s, t = 2^-K M; sigma = 1/(1+t) for z >= 0 and
//     2^-K M/(1+t) for z < 0, with 1/(1+t) refined from the FP32 reciprocal
//     by one Newton step in float-pair arithmetic.
//   Error budget, relative: reduction 2^-50, series truncation 2^-48.6,
//   rounding of the small terms and of the pair products <= 2^-44 each,
//   Newton step 2^-45; accepted with the bound 2^-42. About one value in
//   10^5 falls inside its bound and goes to phase 2.
// Phase 2 (rare): the same steps in double-double arithmetic (Taylor series to
// s^12, table of 2^(-j/32) as double pairs, one Newton step on the double
// reciprocal), within 2^-100 of the exact value, then rounded to the nearest
// float by comparing the pair with the exact midpoints.
//
// Every operation of both phases is a correctly rounded IEEE operation (no
// approximate hardware functions), so a CPU running the same steps reproduces
// every bit. Every one of the 2^32 float inputs has been compared with the CPU
// oracle's correctly rounded sigmoid, both through a CPU restatement of these
// steps and through this code on the GPU.
#pragma once

#include <cstdint>

namespace beam {

// 2^(-j/32), j = 0..31, as float pairs (hi = RN32, lo = RN32 of the rest)
__device__ const float2 kExp2NegF[32] = {
    {0x1p+0f, 0x0p+0f},                    {0x1.f50766p-1f, -0x1.246ebp-27f},
    {0x1.ea4afap-1f, 0x1.52486cp-28f},     {0x1.dfc974p-1f, -0x1.908c94p-26f},
    {0x1.d5818ep-1f, -0x1.822dbcp-28f},    {0x1.cb720ep-1f, -0x1.8837ccp-28f},
    {0x1.c199bep-1f, -0x1.3d56b2p-28f},    {0x1.b7f77p-1f, -0x1.a09438p-26f},
    {0x1.ae89fap-1f, -0x1.a94b14p-27f},    {0x1.a5503cp-1f, -0x1.b83b54p-26f},
    {0x1.9c4918p-1f, 0x1.51f848p-28f},     {0x1.93737cp-1f, -0x1.e64744p-26f},
    {0x1.8ace54p-1f, 0x1.15506ep-28f},     {0x1.82589ap-1f, -0x1.accc7cp-27f},
    {0x1.7a1148p-1f, -0x1.829fdp-26f},     {0x1.71f75ep-1f, 0x1.1d8beep-26f},
    {0x1.6a09e6p-1f, 0x1.9fcef4p-27f},     {0x1.6247ecp-1f, -0x1.f8b55p-26f},
    {0x1.5ab07ep-1f, -0x1.5bd5ecp-28f},    {0x1.5342b6p-1f, -0x1.2c561p-26f},
    {0x1.4bfdaep-1f, -0x1.593abcp-26f},    {0x1.44e086p-1f, 0x1.8624b4p-31f},
    {0x1.3dea64p-1f, 0x1.824684p-26f},     {0x1.371a74p-1f, -0x1.18aac6p-26f},
    {0x1.306fep-1f, 0x1.4636e2p-26f},      {0x1.29e9ep-1f, -0x1.5c0424p-26f},
    {0x1.2387a6p-1f, 0x1.ceac48p-26f},     {0x1.1d4874p-1f, -0x1.d2e8cap-26f},
    {0x1.172b84p-1f, -0x1.c15742p-28f},    {0x1.11301ep-1f, -0x1.fdb496p-26f},
    {0x1.0b5586p-1f, 0x1.9f3122p-26f},     {0x1.059b0ep-1f, -0x1.9d4f52p-26f},
};

// 2^(-j/32) as double pairs
__device__ const double2 kExp2NegD[32] = {
    {0x1p+0, 0x0p+0},
    {0x1.f50765b6e454p-1, 0x1.9d3e12dd8a18bp-55},
    {0x1.ea4afa2a490dap-1, -0x1.e9c23179c2893p-55},
    {0x1.dfc97337b9b5fp-1, -0x1.1a5cd4f184b5cp-55},
    {0x1.d5818dcfba487p-1, 0x1.2ed02d75b3707p-56},
    {0x1.cb720dcef9069p-1, 0x1.503cbd1e949dbp-57},
    {0x1.c199bdd85529cp-1, 0x1.11065895048ddp-56},
    {0x1.b7f76f2fb5e47p-1, -0x1.5584f7e54ac3bp-57},
    {0x1.ae89f995ad3adp-1, 0x1.7a1cd345dcc81p-55},
    {0x1.a5503b23e255dp-1, -0x1.d2f6edb8d41e1p-55},
    {0x1.9c49182a3f09p-1, 0x1.c7c46b071f2bep-57},
    {0x1.93737b0cdc5e5p-1, -0x1.75fc781b57ebcp-58},
    {0x1.8ace5422aa0dbp-1, 0x1.6e9f156864b27p-55},
    {0x1.82589994cce13p-1, -0x1.d4c1dd41532d8p-55},
    {0x1.7a11473eb0187p-1, -0x1.41577ee04992fp-56},
    {0x1.71f75e8ec5f74p-1, -0x1.16e4786887a99p-56},
    {0x1.6a09e667f3bcdp-1, -0x1.bdd3413b26456p-55},
    {0x1.6247eb03a5585p-1, -0x1.383c17e40b497p-55},
    {0x1.5ab07dd485429p-1, 0x1.6324c054647adp-55},
    {0x1.5342b569d4f82p-1, -0x1.07abe1db13cadp-56},
    {0x1.4bfdad5362a27p-1, 0x1.d4397afec42e2p-57},
    {0x1.44e086061892dp-1, 0x1.89b7a04ef80dp-60},
    {0x1.3dea64c123422p-1, 0x1.ada0911f09ebcp-56},
    {0x1.371a7373aa9cbp-1, -0x1.63aeabf42eae2p-55},
    {0x1.306fe0a31b715p-1, 0x1.6f46ad23182e4p-56},
    {0x1.29e9df51fdee1p-1, 0x1.612e8afad1255p-56},
    {0x1.2387a6e756238p-1, 0x1.9b07eb6c70573p-55},
    {0x1.1d4873168b9aap-1, 0x1.e016e00a2643cp-55},
    {0x1.172b83c7d517bp-1, -0x1.19041b9d78a76p-56},
    {0x1.11301d0125b51p-1, -0x1.6c51039449b3ap-55},
    {0x1.0b5586cf9890fp-1, 0x1.8a62e4adc610bp-55},
    {0x1.059b0d3158574p-1, 0x1.d73e2a475b465p-56},
};

// 1/n! as double pairs, n = 0..5 (the Taylor coefficients of e^s kept exact
// to 2^-106); n = 6..12 as doubles
__device__ const double2 kInvFactD[6] = {
    {0x1p+0, 0x0p+0},
    {0x1p+0, 0x0p+0},
    {0x1p-1, 0x0p+0},
    {0x1.5555555555555p-3, 0x1.5555555555555p-57},
    {0x1.5555555555555p-5, 0x1.5555555555555p-59},
    {0x1.1111111111111p-7, 0x1.1111111111111p-63},
};

struct SigmoidLane {  // this lane's entry of the 2^(-j/32) table (lane l holds j = l)
    float hi, lo;
};

__device__ __forceinline__ SigmoidLane sigmoid_lane_table() {
    const float2 t = __ldg(&kExp2NegF[threadIdx.x & 31]);
    return SigmoidLane{t.x, t.y};
}

// ---------------------------------------------------------------- float pairs

// a + b = s + e exactly, any a, b (Knuth)
__device__ __forceinline__ void two_sum_f(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    const float ap = __fsub_rn(s, bp);
    e = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

// a + b = s + e exactly when exponent(a) >= exponent(b) (Dekker)
__device__ __forceinline__ void fast_two_sum_f(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    e = __fsub_rn(b, __fsub_rn(s, a));
}

// ---------------------------------------------------------------- double pairs

struct DD {
    double h, l;
};

__device__ __forceinline__ DD dd_fast(double a, double b) {
    const double s = __dadd_rn(a, b);
    return DD{s, __dsub_rn(b, __dsub_rn(s, a))};
}

__device__ __forceinline__ DD dd_two_sum(double a, double b) {
    const double s = __dadd_rn(a, b);
    const double bp = __dsub_rn(s, a);
    const double ap = __dsub_rn(s, bp);
    return DD{s, __dadd_rn(__dsub_rn(a, ap), __dsub_rn(b, bp))};
}

__device__ __forceinline__ DD dd_mul(DD a, DD b) {
    const double p = __dmul_rn(a.h, b.h);
    double e = __fma_rn(a.h, b.h, -p);
    e = __fma_rn(a.h, b.l, e);
    e = __fma_rn(a.l, b.h, e);
    return dd_fast(p, e);
}

__device__ __forceinline__ DD dd_add(DD a, DD b) {
    DD s = dd_two_sum(a.h, b.h);
    return dd_fast(s.h, __dadd_rn(s.l, __dadd_rn(a.l, b.l)));
}

// Phase 2: the sigmoid of z in double-double, rounded to the nearest float.
// Only for |z| < 104 and z not NaN (phase 1 settles the rest).
__device__ __noinline__ float router_sigmoid_dd(float z) {
    const double a = fabs((double)z);
    const bool neg = z < 0.0f;
    // k = rint(a 32/ln2) by the 1.5 * 2^52 shifter (k < 2^13)
    const double kk = __fma_rn(a, 0x1.71547652b82fep+5, 0x1.8p52);
    const long long k = __double_as_longlong(kk) - __double_as_longlong(0x1.8p52);
    const double kd = __dsub_rn(kk, 0x1.8p52);
    const int j = (int)(k & 31), K = (int)(k >> 5);
    // s = k ln2/32 - a, with ln2/32 = L1 (40 bits) + L2 + L3
    const double r1 = __fma_rn(-kd, 0x1.62e42fefa2p-6, a);  // a - k L1, exact
    const double p2 = __dmul_rn(kd, 0x1.9ef35793c7673p-46);
    const double p2e = __fma_rn(kd, 0x1.9ef35793c7673p-46, -p2);
    DD s = dd_two_sum(p2, -r1);
    s.l = __dadd_rn(s.l, __fma_rn(kd, 0x1.f97b57a079a19p-108, p2e));
    // e^s: Taylor series, terms s^6..s^12 in double, s^0..s^5 in pairs
    double tail = 0x1.1eed8eff8d898p-29;                     // 1/12!
    tail = __fma_rn(tail, s.h, 0x1.ae64567f544e4p-26);        // 1/11!
    tail = __fma_rn(tail, s.h, 0x1.27e4fb7789f5cp-22);        // 1/10!
    tail = __fma_rn(tail, s.h, 0x1.71de3a556c734p-19);        // 1/9!
    tail = __fma_rn(tail, s.h, 0x1.a01a01a01a01ap-16);        // 1/8!
    tail = __fma_rn(tail, s.h, 0x1.a01a01a01a01ap-13);        // 1/7!
    tail = __fma_rn(tail, s.h, 0x1.6c16c16c16c17p-10);        // 1/6!
    DD e = DD{tail, 0.0};
    for (int n = 5; n >= 0; --n) {
        const double2 c = kInvFactD[n];
        e = dd_add(dd_mul(e, s), DD{c.x, c.y});
    }
    const double2 tj = kExp2NegD[j];
    const DD m = dd_mul(DD{tj.x, tj.y}, e);                    // 2^(-j/32) e^s
    const double sc = __hiloint2double((int)((uint32_t)(1023 - K) << 20), 0);  // 2^-K, K <= 150
    const DD t = DD{__dmul_rn(m.h, sc), __dmul_rn(m.l, sc)};
    const DD d = dd_add(DD{1.0, 0.0}, t);
    // q = 1/d: the double reciprocal and one Newton step
    const double q1 = __drcp_rn(d.h);
    double er = __fma_rn(-d.h, q1, 1.0);
    er = __fma_rn(-d.l, q1, er);
    const DD q = dd_fast(q1, __dmul_rn(q1, er));
    DD v = neg ? dd_mul(m, q) : q;
    if (neg) v = DD{__dmul_rn(v.h, sc), __dmul_rn(v.l, sc)};  // exact scaling
    // nearest float to v.h + v.l: RN32(v.h) or a neighbour, decided against
    // the exact midpoints
    const float f0 = __double2float_rn(v.h);
    const uint32_t b0 = __float_as_uint(f0);
    float best = f0;
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        const uint32_t bc = c == 0 ? b0 : c == 1 ? (b0 ? b0 - 1u : 0x80000001u) : b0 + 1u;
        const float f = __uint_as_float(bc);
        const float fd = __uint_as_float(bc ? (bc == 0x80000001u ? 0x80000002u : bc - 1u) : 0x80000001u);
        const float fu = __uint_as_float(bc == 0x80000001u ? 0u : bc + 1u);
        const double mlo = 0.5 * ((double)f + (double)fd), mhi = 0.5 * ((double)f + (double)fu);
        if (__dadd_rn(__dsub_rn(v.h, mlo), v.l) > 0.0 && __dadd_rn(__dsub_rn(v.h, mhi), v.l) < 0.0) {
            best = f;
            break;
        }
    }
    return best;
}

// Phase 1; returns the float and whether the rounding is certain. Settles
// NaN (returned as the canonical NaN), |z| >= 104 (1 or +0) outright.
__device__ __forceinline__ float router_sigmoid_ff(float z, SigmoidLane lt, bool& ok) {
    const float a = fabsf(z);
    const bool neg = z < 0.0f;
    const float big = 0x1.8p23f;
    const float kk = __fmaf_rn(a, 0x1.715476p+5f, big);       // 1.5 * 2^23 + rint(a 32/ln2)
    const int k = __float_as_int(kk) - __float_as_int(big);
    const float kf = __fsub_rn(kk, big);
    const int j = k & 31, K = k >> 5;
    // s = k ln2/32 - a = sh + sl
    const float r1 = __fmaf_rn(-kf, 0x1.62cp-6f, a);           // a - k L1, exact
    const float p2 = __fmul_rn(kf, 0x1.217f7ep-17f);
    const float p2e = __fmaf_rn(kf, 0x1.217f7ep-17f, -p2);
    float sh, sl;
    two_sum_f(p2, -r1, sh, sl);
    sl = __fadd_rn(sl, __fmaf_rn(kf, -0x1.c610cap-42f, p2e));
    // e^s = (1 + sh + sh^2/2) + small terms
    const float qh = __fmul_rn(sh, sh);
    const float ql = __fmaf_rn(sh, sh, -qh);
    float c = __fmaf_rn(sh, 0x1.111112p-7f, 0x1.555556p-5f);   // 1/120, 1/24
    c = __fmaf_rn(sh, c, 0x1.555556p-3f);                      // 1/6
    const float p3 = __fmul_rn(__fmul_rn(qh, sh), c);
    float e1h, e1l, e2h, e2l;
    fast_two_sum_f(1.0f, sh, e1h, e1l);
    fast_two_sum_f(e1h, __fmul_rn(0.5f, qh), e2h, e2l);
    float lo = __fmaf_rn(sl, e2h, p3);
    lo = __fmaf_rn(0.5f, ql, lo);
    lo = __fadd_rn(lo, e1l);
    lo = __fadd_rn(lo, e2l);
    float eh, el;
    fast_two_sum_f(e2h, lo, eh, el);
    // M = 2^(-j/32) e^s
    const float th = __shfl_sync(0xFFFFFFFFu, lt.hi, j);
    const float tl = __shfl_sync(0xFFFFFFFFu, lt.lo, j);
    const float mh = __fmul_rn(th, eh);
    float ml = __fmaf_rn(th, eh, -mh);
    ml = __fmaf_rn(th, el, ml);
    ml = __fmaf_rn(tl, eh, ml);
    // d = 1 + 2^-K M (2^-K clamped at 2^-64: below it t no longer matters)
    const int kc = K < 64 ? K : 64;
    const float sc = __uint_as_float((uint32_t)(127 - kc) << 23);
    const float tph = __fmul_rn(mh, sc), tpl = __fmul_rn(ml, sc);
    const float dh = __fadd_rn(1.0f, tph);
    const float dl = __fadd_rn(__fsub_rn(tph, __fsub_rn(dh, 1.0f)), tpl);
    // q = 1/d: the FP32 reciprocal and one Newton step
    const float y0 = __frcp_rn(dh);
    float er = __fmaf_rn(-dh, y0, 1.0f);
    er = __fmaf_rn(-dl, y0, er);
    const float qqh = y0, qql = __fmul_rn(y0, er);
    // v = num q, num = M (z < 0) or 1 (z >= 0); the result is 2^-Ks v
    const float nh = neg ? mh : 1.0f, nl = neg ? ml : 0.0f;
    float vh = __fmul_rn(nh, qqh);
    float vl = __fmaf_rn(nh, qqh, -vh);
    vl = __fmaf_rn(nh, qql, vl);
    vl = __fmaf_rn(nl, qqh, vl);
    fast_two_sum_f(vh, vl, vh, vl);
    const int ks = neg ? K : 0;
    // rounding of 2^-ks v, done in the v domain: the result's grid there is
    // G = 2^gexp, the larger of v's ulp and the subnormal spacing 2^(ks-149)
    const int ev = (__float_as_int(vh) >> 23) & 0xFF;          // vh in [0.2, 1.1]: normal
    const int gexp = max(ev - 150, ks - 149);
    const bool sub = ks - 149 > ev - 150;
    const float G = __uint_as_float((uint32_t)(gexp + 127) << 23);
    float cnd, gdn;
    float n = 0.0f;
    if (!sub) {
        cnd = vh;
        const bool pow2 = (__float_as_int(vh) & 0x7FFFFF) == 0;
        gdn = (pow2 && ks - 149 <= ev - 151) ? __fmul_rn(0.5f, G) : G;
    } else {
        n = rintf(__fmul_rn(vh, __uint_as_float((uint32_t)(127 - gexp) << 23)));
        cnd = __fmul_rn(n, G);
        gdn = G;
    }
    const float dv = __fadd_rn(__fsub_rn(vh, cnd), vl);
    const float mg = __fmaf_rn(0x1p-42f, vh, __fmul_rn(0x1p-22f, G));
    ok = __fadd_rn(dv, mg) < __fmul_rn(0.5f, G) && __fsub_rn(dv, mg) > -__fmul_rn(0.5f, gdn);
    float res = sub ? __uint_as_float((uint32_t)n) : __fmul_rn(cnd, __uint_as_float((uint32_t)(127 - ks) << 23));
    if (!(a < 104.0f)) {  // saturated, or NaN
        ok = true;
        res = (a != a) ? __int_as_float(0x7FFFFFFF) : (neg ? 0.0f : 1.0f);
    }
    return res;
}

// A fast FP32 sigmoid for the router's first pass, 1 / (1 + 2^(-z log2 e))
// from the hardware's approximate base-2 exponential and reciprocal (ftz).
// Not correctly rounded: its distance to the exact sigmoid stays below
// kFastSigmoidSlack on every float input (NaN gives NaN), which a test checks
// on all 2^32 of them against the correctly rounded oracle.
constexpr float kFastSigmoidSlack = 0x1p-19f;

__device__ __forceinline__ float router_sigmoid_fast(float z) {
    float e, s;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(__fmul_rn(z, -1.44269504088896340736f)));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(s) : "f"(__fadd_rn(1.0f, e)));
    return s;
}

// The correctly rounded sigmoid. Call with all 32 lanes of the warp (phase 1
// reads the table by shuffle); phase 2 runs only in the lanes that need it.
__device__ __forceinline__ float router_sigmoid(float z, SigmoidLane lt) {
    bool ok;
    float s = router_sigmoid_ff(z, lt, ok);
    if (!ok) s = router_sigmoid_dd(z);
    return s;
}

}  // namespace beam
