/*
 * CPU restatement of the router's correctly rounded sigmoid
 * (sandwich_norm_residual_gb300/csrc/router_sigmoid.cuh), step for step, for
 * the exhaustive check in test_router_sigmoid_method.py.
 *
 * Every step of the kernel's two phases is a correctly rounded IEEE operation
 * (add, subtract, multiply, fused multiply-add, reciprocal, round to integer,
 * conversions), so the same steps on the CPU give the same bits. The lane
 * table the kernel reads by shuffle is a plain array here. Built with
 * -ffp-contract=off so that no multiply and add are fused behind our back.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static const float kTabF[32][2] = {
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

static const double kTabD[32][2] = {
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

static const double kInvFact[6][2] = {
    {0x1p+0, 0x0p+0}, {0x1p+0, 0x0p+0}, {0x1p-1, 0x0p+0},
    {0x1.5555555555555p-3, 0x1.5555555555555p-57},
    {0x1.5555555555555p-5, 0x1.5555555555555p-59},
    {0x1.1111111111111p-7, 0x1.1111111111111p-63},
};

static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static double u2d(uint64_t u) { double d; memcpy(&d, &u, 8); return d; }
static int64_t d2i(double d) { int64_t u; memcpy(&u, &d, 8); return u; }

static void two_sum_f(float a, float b, float* s, float* e) {
    *s = a + b;
    float bp = *s - a, ap = *s - bp;
    *e = (a - ap) + (b - bp);
}
static void fast_two_sum_f(float a, float b, float* s, float* e) {
    float t = a + b;
    *e = b - (t - a);
    *s = t;
}

typedef struct { double h, l; } dd;
static dd dd_fast(double a, double b) { double s = a + b; dd r = {s, b - (s - a)}; return r; }
static dd dd_two_sum(double a, double b) {
    double s = a + b, bp = s - a, ap = s - bp;
    dd r = {s, (a - ap) + (b - bp)};
    return r;
}
static dd dd_mul(dd a, dd b) {
    double p = a.h * b.h, e = fma(a.h, b.h, -p);
    e = fma(a.h, b.l, e);
    e = fma(a.l, b.h, e);
    return dd_fast(p, e);
}
static dd dd_add(dd a, dd b) {
    dd s = dd_two_sum(a.h, b.h);
    return dd_fast(s.h, s.l + (a.l + b.l));
}

static float sigmoid_dd(float z) {
    const double a = fabs((double)z);
    const int neg = z < 0.0f;
    const double kk = fma(a, 0x1.71547652b82fep+5, 0x1.8p52);
    const int64_t k = d2i(kk) - d2i(0x1.8p52);
    const double kd = kk - 0x1.8p52;
    const int j = (int)(k & 31), K = (int)(k >> 5);
    const double r1 = fma(-kd, 0x1.62e42fefa2p-6, a);
    const double p2 = kd * 0x1.9ef35793c7673p-46;
    const double p2e = fma(kd, 0x1.9ef35793c7673p-46, -p2);
    dd s = dd_two_sum(p2, -r1);
    s.l = s.l + fma(kd, 0x1.f97b57a079a19p-108, p2e);
    double tail = 0x1.1eed8eff8d898p-29;
    tail = fma(tail, s.h, 0x1.ae64567f544e4p-26);
    tail = fma(tail, s.h, 0x1.27e4fb7789f5cp-22);
    tail = fma(tail, s.h, 0x1.71de3a556c734p-19);
    tail = fma(tail, s.h, 0x1.a01a01a01a01ap-16);
    tail = fma(tail, s.h, 0x1.a01a01a01a01ap-13);
    tail = fma(tail, s.h, 0x1.6c16c16c16c17p-10);
    dd e = {tail, 0.0};
    for (int n = 5; n >= 0; --n) {
        dd c = {kInvFact[n][0], kInvFact[n][1]};
        e = dd_add(dd_mul(e, s), c);
    }
    const dd tj = {kTabD[j][0], kTabD[j][1]};
    const dd m = dd_mul(tj, e);
    const double sc = u2d((uint64_t)(uint32_t)(1023 - K) << 52);
    const dd t = {m.h * sc, m.l * sc};
    const dd one = {1.0, 0.0};
    const dd d = dd_add(one, t);
    const double q1 = 1.0 / d.h;
    double er = fma(-d.h, q1, 1.0);
    er = fma(-d.l, q1, er);
    const dd q = dd_fast(q1, q1 * er);
    dd v = neg ? dd_mul(m, q) : q;
    if (neg) { v.h = v.h * sc; v.l = v.l * sc; }
    const float f0 = (float)v.h;
    const uint32_t b0 = f2u(f0);
    float best = f0;
    for (int c = 0; c < 3; ++c) {
        const uint32_t bc = c == 0 ? b0 : c == 1 ? (b0 ? b0 - 1u : 0x80000001u) : b0 + 1u;
        const float f = u2f(bc);
        const float fd = u2f(bc ? (bc == 0x80000001u ? 0x80000002u : bc - 1u) : 0x80000001u);
        const float fu = u2f(bc == 0x80000001u ? 0u : bc + 1u);
        const double mlo = 0.5 * ((double)f + (double)fd), mhi = 0.5 * ((double)f + (double)fu);
        if ((v.h - mlo) + v.l > 0.0 && (v.h - mhi) + v.l < 0.0) { best = f; break; }
    }
    return best;
}

static float sigmoid_ff(float z, int* ok) {
    const float a = fabsf(z);
    const int neg = z < 0.0f;
    const float big = 0x1.8p23f;
    const float kk = fmaf(a, 0x1.715476p+5f, big);
    const int k = (int)(f2u(kk) - f2u(big));
    const float kf = kk - big;
    const int j = k & 31, K = k >> 5;
    const float r1 = fmaf(-kf, 0x1.62cp-6f, a);
    const float p2 = kf * 0x1.217f7ep-17f;
    const float p2e = fmaf(kf, 0x1.217f7ep-17f, -p2);
    float sh, sl;
    two_sum_f(p2, -r1, &sh, &sl);
    sl = sl + fmaf(kf, -0x1.c610cap-42f, p2e);
    const float qh = sh * sh;
    const float ql = fmaf(sh, sh, -qh);
    float c = fmaf(sh, 0x1.111112p-7f, 0x1.555556p-5f);
    c = fmaf(sh, c, 0x1.555556p-3f);
    const float p3 = (qh * sh) * c;
    float e1h, e1l, e2h, e2l;
    fast_two_sum_f(1.0f, sh, &e1h, &e1l);
    fast_two_sum_f(e1h, 0.5f * qh, &e2h, &e2l);
    float lo = fmaf(sl, e2h, p3);
    lo = fmaf(0.5f, ql, lo);
    lo = lo + e1l;
    lo = lo + e2l;
    float eh, el;
    fast_two_sum_f(e2h, lo, &eh, &el);
    const float th = kTabF[j & 31][0], tl = kTabF[j & 31][1];
    const float mh = th * eh;
    float ml = fmaf(th, eh, -mh);
    ml = fmaf(th, el, ml);
    ml = fmaf(tl, eh, ml);
    const int kc = K < 64 ? K : 64;
    const float sc = u2f((uint32_t)(127 - kc) << 23);
    const float tph = mh * sc, tpl = ml * sc;
    const float dh = 1.0f + tph;
    const float dl = (tph - (dh - 1.0f)) + tpl;
    const float y0 = 1.0f / dh;
    float er = fmaf(-dh, y0, 1.0f);
    er = fmaf(-dl, y0, er);
    const float qqh = y0, qql = y0 * er;
    const float nh = neg ? mh : 1.0f, nl = neg ? ml : 0.0f;
    float vh = nh * qqh;
    float vl = fmaf(nh, qqh, -vh);
    vl = fmaf(nh, qql, vl);
    vl = fmaf(nl, qqh, vl);
    fast_two_sum_f(vh, vl, &vh, &vl);
    const int ks = neg ? K : 0;
    const int ev = (int)((f2u(vh) >> 23) & 0xFF);
    const int gexp = (ev - 150) > (ks - 149) ? (ev - 150) : (ks - 149);
    const int sub = ks - 149 > ev - 150;
    const float G = u2f((uint32_t)(gexp + 127) << 23);
    float cnd, gdn, n = 0.0f;
    if (!sub) {
        cnd = vh;
        const int pow2 = (f2u(vh) & 0x7FFFFF) == 0;
        gdn = (pow2 && ks - 149 <= ev - 151) ? 0.5f * G : G;
    } else {
        n = rintf(vh * u2f((uint32_t)(127 - gexp) << 23));
        cnd = n * G;
        gdn = G;
    }
    const float dv = (vh - cnd) + vl;
    const float mg = fmaf(0x1p-42f, vh, 0x1p-22f * G);
    *ok = (dv + mg) < 0.5f * G && (dv - mg) > -(0.5f * gdn);
    float res = sub ? u2f((uint32_t)n) : cnd * u2f((uint32_t)(127 - ks) << 23);
    if (!(a < 104.0f)) {
        *ok = 1;
        res = (a != a) ? u2f(0x7FFFFFFFu) : (neg ? 0.0f : 1.0f);
    }
    return res;
}

/* s[i] = the kernel's sigmoid of z[i]; phase[i] = 1 or 2 (which phase decided) */
void method_sigmoid_array(const float* z, float* s, uint8_t* phase, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        int ok;
        float v = sigmoid_ff(z[i], &ok);
        if (!ok) v = sigmoid_dd(z[i]);
        s[i] = v;
        phase[i] = ok ? 1 : 2;
    }
}

/* the same over the bit patterns lo .. lo + n - 1 */
void method_sigmoid_range(uint32_t lo, float* s, uint8_t* phase, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        const float z = u2f(lo + (uint32_t)i);
        int ok;
        float v = sigmoid_ff(z, &ok);
        if (!ok) v = sigmoid_dd(z);
        s[i] = v;
        phase[i] = ok ? 1 : 2;
    }
}
