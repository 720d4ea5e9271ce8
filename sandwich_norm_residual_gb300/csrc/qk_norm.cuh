// Per-head Q/K RMSNorm with RoPE or SSMax, sm_103a (vLLM page, "Beam model
// architecture": Q and K are RMS-normalised per head before RoPE or SSMax;
// 48 query heads, 8 KV heads, head dimension 128; SSMax scales each query by
// (1 + (pos+1)/2048)^0.1 with pos 0-based).
//
// Per head row v (128 BF16), FP32 math:
//   vn_j = bf16((v_j r) w_j), r = 1/sqrt(RN32(sum v^2)/128 + eps)  (exact row sum)
//   RoPE:  out_j      = bf16(RN32(vn_j c_j)      - RN32(vn_{j+64} s_j))
//          out_{j+64} = bf16(RN32(vn_{j+64} c_j) + RN32(vn_j s_j)),
//          c_j = table[pos][j], s_j = table[pos][64 + j]   (rotate-half pairs)
//   SSMax: out_j = bf16(RN32(vn_j g)), g = RN32((1 + (pos+1)/2048)^0.1) for
//          queries (evaluated in double); keys keep vn.
//
// One warp per token walks its heads, 8 rows at a time. Lane l holds
// elements 4l .. 4l+3 of a row, so the RoPE partner of lane l is lane l ^ 16.
#pragma once

#include "row_sum.cuh"
#include "tma.cuh"

namespace beam {

constexpr int kQKHeadDim = 128;
constexpr int kQKBatch = 8;

struct QKParams {
    uint16_t* q;          // [T, nq, 128] in/out
    uint16_t* k;          // [T, nk, 128] in/out
    const uint16_t* qw;   // [128]
    const uint16_t* kw;   // [128]
    const int32_t* pos;   // [T]
    const float* table;   // [max_pos, 128] FP32 cos | sin (RoPE)
    long long max_pos;
    long long T;
    int nq, nk;
    float eps;
    float errk;
    int mode;             // 0 RoPE, 1 SSMax
    unsigned flags;       // kFlagForceExact
};

// Exact RN32 sum of the squares of a 128-element row held as 4 values per
// lane, for one warp (no shared memory): 32-bit chunk sums of each FP32 term
// m * 2^q * 2^-149 in nine 64-bit registers, added across the warp, carried
// and rounded to nearest even.
__device__ __noinline__ float exact_warp_sum_squares(float v0, float v1, float v2, float v3) {
    unsigned long long acc[9];
#pragma unroll
    for (int L = 0; L < 9; ++L) acc[L] = 0ull;
    int nan = 0, inf = 0;
    const float v[4] = {v0, v1, v2, v3};
    for (int i = 0; i < 4; ++i) {
        const float t = __fmul_rn(v[i], v[i]);
        const uint32_t u = __float_as_uint(t);
        const uint32_t E = (u >> 23) & 0xFFu, f = u & 0x7FFFFFu;
        if (E == 0xFFu) {
            if (f) nan = 1; else inf = 1;
            continue;
        }
        const uint32_t M = E ? (f | 0x800000u) : f;
        const uint32_t q = E ? E - 1u : 0u;
        const unsigned long long w = (unsigned long long)M << (q & 31u);
        const uint32_t k = q >> 5, lo = (uint32_t)w, hi = (uint32_t)(w >> 32);
#pragma unroll
        for (uint32_t L = 0; L < 9; ++L) {
            acc[L] += (L == k) ? lo : 0u;
            acc[L] += (L == k + 1u) ? hi : 0u;
        }
    }
#pragma unroll
    for (int L = 0; L < 9; ++L)
        for (int off = 16; off; off >>= 1) acc[L] += __shfl_xor_sync(0xFFFFFFFFu, acc[L], off);
    const int any_nan = __any_sync(0xFFFFFFFFu, nan), any_inf = __any_sync(0xFFFFFFFFu, inf);
    if ((threadIdx.x & 31) == 0) atomicAdd(&g_exact_sum_count, 1ull);
    if (any_nan) return __uint_as_float(0x7FFFFFFFu);
    if (any_inf) return __uint_as_float(0x7F800000u);
    uint32_t Lw[10];
    unsigned long long carry = 0ull;
    for (int L = 0; L < 10; ++L) {
        const unsigned long long s = carry + (L < 9 ? acc[L] : 0ull);
        Lw[L] = (uint32_t)s;
        carry = s >> 32;
    }
    return limbs_to_f32(Lw);
}

__global__ void __launch_bounds__(256) qk_norm_kernel(const QKParams p) {
    const int lane = threadIdx.x & 31;
    const long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= p.T) return;  // whole warps leave together
    const unsigned full = 0xFFFFFFFFu;
    const bool force_exact = (p.flags & kFlagForceExact) != 0;

    const long long pos = p.pos[t];
    if (pos < 0 || (p.mode == 0 && pos >= p.max_pos)) {
        if (lane == 0) atomicOr(&g_status_word, 2u);  // reported as a bad argument
        return;
    }
    // per-lane constants: weights, and cos/sin (RoPE) or the query scale (SSMax)
    const uint2 qwv = __ldg(reinterpret_cast<const uint2*>(p.qw) + lane);
    const uint2 kwv = __ldg(reinterpret_cast<const uint2*>(p.kw) + lane);
    float c[4] = {0.f, 0.f, 0.f, 0.f}, s[4] = {0.f, 0.f, 0.f, 0.f}, g = 1.0f;
    if (p.mode == 0) {
        const float* row = p.table + pos * kQKHeadDim + 4 * (lane & 15);
        const float4 cc = __ldg(reinterpret_cast<const float4*>(row));
        const float4 ss = __ldg(reinterpret_cast<const float4*>(row + 64));
        c[0] = cc.x; c[1] = cc.y; c[2] = cc.z; c[3] = cc.w;
        s[0] = ss.x; s[1] = ss.y; s[2] = ss.z; s[3] = ss.w;
    } else {
        double gd = 0.0;
        if (lane == 0) gd = pow(1.0 + (double)(pos + 1) / 2048.0, 0.1);
        g = (float)__shfl_sync(full, gd, 0);
    }
    const bool upper = lane >= 16;  // holds elements j + 64 of the rotate-half pairs
    const int nh = p.nq + p.nk;

    for (int h0 = 0; h0 < nh; h0 += kQKBatch) {
        uint2 v[kQKBatch];
        uint16_t* rowp[kQKBatch];
#pragma unroll
        for (int b = 0; b < kQKBatch; ++b) {
            const int hh = h0 + b;
            rowp[b] = hh < p.nq ? p.q + ((size_t)t * p.nq + hh) * kQKHeadDim
                                : p.k + ((size_t)t * p.nk + (hh - p.nq)) * kQKHeadDim;
            v[b] = hh < nh ? *reinterpret_cast<const uint2*>(rowp[b] + 4 * lane) : make_uint2(0, 0);
        }
#pragma unroll
        for (int b = 0; b < kQKBatch; ++b) {
            const int hh = h0 + b;
            if (hh >= nh) break;
            const bool is_q = hh < p.nq;
            const float2 x01 = bf2_to_f2(v[b].x), x23 = bf2_to_f2(v[b].y);
            // compensated sum of squares, both FP32 lanes, then the warp
            float2 sa = make_float2(0.f, 0.f), ca = make_float2(0.f, 0.f);
            two_sum_acc2(sa, ca, mul2_rn(x01, x01));
            two_sum_acc2(sa, ca, mul2_rn(x23, x23));
            float S = sa.x, C = ca.x;
            ff_merge(S, C, sa.y, ca.y);
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                const float s2 = __shfl_xor_sync(full, S, off), c2 = __shfl_xor_sync(full, C, off);
                ff_merge(S, C, s2, c2);
            }
            float Sr;
            if (!certify_round(S, C, p.errk, &Sr) || force_exact)  // warp-uniform
                Sr = exact_warp_sum_squares(x01.x, x01.y, x23.x, x23.y);
            const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(Sr, 128.0f), p.eps)));
            const float2 rv = make_float2(r, r);
            const uint2 wv = is_q ? qwv : kwv;
            const uint32_t n01 = f2_to_bf2(mul2_rn(mul2_rn(x01, rv), bf2_to_f2(wv.x)));
            const uint32_t n23 = f2_to_bf2(mul2_rn(mul2_rn(x23, rv), bf2_to_f2(wv.y)));
            uint2 out;
            if (p.mode == 0) {
                const uint32_t m01 = __shfl_xor_sync(full, n01, 16), m23 = __shfl_xor_sync(full, n23, 16);
                const float2 a01 = bf2_to_f2(n01), a23 = bf2_to_f2(n23);
                const float2 b01 = bf2_to_f2(m01), b23 = bf2_to_f2(m23);
                const float2 c01 = make_float2(c[0], c[1]), c23 = make_float2(c[2], c[3]);
                const float2 s01 = make_float2(s[0], s[1]), s23 = make_float2(s[2], s[3]);
                const float2 p01 = mul2_rn(a01, c01), p23 = mul2_rn(a23, c23);
                const float2 q01 = mul2_rn(b01, s01), q23 = mul2_rn(b23, s23);
                out.x = f2_to_bf2(upper ? add2_rn(p01, q01) : sub2_rn(p01, q01));
                out.y = f2_to_bf2(upper ? add2_rn(p23, q23) : sub2_rn(p23, q23));
            } else if (is_q) {
                const float2 gv = make_float2(g, g);
                out.x = f2_to_bf2(mul2_rn(bf2_to_f2(n01), gv));
                out.y = f2_to_bf2(mul2_rn(bf2_to_f2(n23), gv));
            } else {
                out = make_uint2(n01, n23);
            }
            *reinterpret_cast<uint2*>(rowp[b] + 4 * lane) = out;
        }
    }
}

}  // namespace beam
