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
//          queries (correctly rounded, see ssmax_scale); keys keep vn.
//
// One warp per token walks its heads: each pass takes 4 heads, one per group
// of 8 lanes, and lane i of a group holds elements 8i .. 8i+7 and 64+8i ..
// 64+8i+7 of its head: both halves of every rotate-half pair are in the same
// lane, which keeps the 8 cos and 8 sin values it needs in registers for the
// whole token. The row sums merge over 3 shuffle levels. Two batches of 8 heads
// are in flight at a time.
#pragma once

#include "row_sum.cuh"
#include "tma.cuh"

namespace beam {

constexpr int kQKHeadDim = 128;
constexpr int kQKBatch = 8;           // heads per batch (two passes of 4)

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

// Exact RN32 sum of the squares of a 128-element row held by a group of 8
// lanes (16 BF16 values per lane in a, b), without shared memory: 32-bit
// chunk sums of each FP32 term m * 2^q * 2^-149 in nine 64-bit registers,
// added over the group (xor 1, 2, 4), carried and rounded to nearest even.
// Every lane of the warp must call it; each group gets its own row's sum.
__device__ __noinline__ float exact_group_sum_squares(uint4 a, uint4 b) {
    unsigned long long acc[9];
#pragma unroll
    for (int L = 0; L < 9; ++L) acc[L] = 0ull;
    int nan = 0, inf = 0;
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    for (int i = 0; i < 16; ++i) {
        const uint32_t bits = (i & 1) ? (w[i >> 1] & 0xFFFF0000u) : (w[i >> 1] << 16);
        const float x = __uint_as_float(bits);
        const float t = __fmul_rn(x, x);
        const uint32_t u = __float_as_uint(t);
        const uint32_t E = (u >> 23) & 0xFFu, f = u & 0x7FFFFFu;
        if (E == 0xFFu) {
            if (f) nan = 1; else inf = 1;
            continue;
        }
        const uint32_t M = E ? (f | 0x800000u) : f;
        const uint32_t q = E ? E - 1u : 0u;
        const unsigned long long v = (unsigned long long)M << (q & 31u);
        const uint32_t k = q >> 5, lo = (uint32_t)v, hi = (uint32_t)(v >> 32);
#pragma unroll
        for (uint32_t L = 0; L < 9; ++L) {
            acc[L] += (L == k) ? lo : 0u;
            acc[L] += (L == k + 1u) ? hi : 0u;
        }
    }
#pragma unroll
    for (int L = 0; L < 9; ++L)
        for (int off = 4; off; off >>= 1) acc[L] += __shfl_xor_sync(0xFFFFFFFFu, acc[L], off);
    for (int off = 4; off; off >>= 1) {
        nan |= __shfl_xor_sync(0xFFFFFFFFu, nan, off);
        inf |= __shfl_xor_sync(0xFFFFFFFFu, inf, off);
    }
    if (nan) return __uint_as_float(0x7FFFFFFFu);
    if (inf) return __uint_as_float(0x7F800000u);
    uint32_t Lw[10];
    unsigned long long carry = 0ull;
    for (int L = 0; L < 10; ++L) {
        const unsigned long long s = carry + (L < 9 ? acc[L] : 0ull);
        Lw[L] = (uint32_t)s;
        carry = s >> 32;
    }
    return limbs_to_f32(Lw);
}

// Largest SSMax position: u = (2049 + pos) / 2048 is then exact in FP32.
constexpr long long kSSMaxMaxPos = (1ll << 24) - 2050;

// g = RN32(u^0.1), u = (2049 + pos)/2048, without a double pow (the FP64 pipe
// is narrow). An FP32 estimate 2^(0.1 log2 u) is within a few ulps; lanes
// 0..15 each take the candidate est + (lane - 8) ulps and test whether the
// 10th power of its lower midpoint (exact in double, four double products,
// relative error ~4e-16) is <= u. The 10th power is increasing, so the
// correctly rounded g is the largest candidate that passes (no midpoint's
// 10th power equals u for these positions: u^0.1 is irrational).
// Called by the whole warp.
__device__ __forceinline__ float ssmax_scale(long long pos, int lane) {
    const float u = __fdiv_rn((float)(2049 + pos), 2048.0f);
    const float est = exp2f(__fmul_rn(0.1f, log2f(u)));
    bool below = false;
    if (lane < 16) {
        const uint32_t b = __float_as_uint(est) + (uint32_t)(lane - 8);
        const double mid = 0.5 * ((double)__uint_as_float(b) + (double)__uint_as_float(b - 1u));
        const double m2 = __dmul_rn(mid, mid), m4 = __dmul_rn(m2, m2), m8 = __dmul_rn(m4, m4);
        below = __dmul_rn(m8, m2) <= (double)u;
    }
    const unsigned mask = __ballot_sync(0xFFFFFFFFu, below) & 0xFFFFu;
    return __uint_as_float(__float_as_uint(est) + (uint32_t)((31 - __clz(mask)) - 8));
}

__global__ void __launch_bounds__(256, 2) qk_norm_kernel(const QKParams p) {
    const int lane = threadIdx.x & 31, grp = lane >> 3, li = lane & 7;
    const long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= p.T) return;  // whole warps leave together
    const unsigned full = 0xFFFFFFFFu;
    const bool force_exact = (p.flags & kFlagForceExact) != 0;

    const long long pos = p.pos[t];
    if (pos < 0 || (p.mode == 0 && pos >= p.max_pos) || (p.mode != 0 && pos > kSSMaxMaxPos)) {
        if (lane == 0) atomicOr(&g_status_word, 2u);  // reported as a bad argument
        return;
    }
    const int nh = p.nq + p.nk;
    // ask L2 for the token's whole q and k rows now, so that DRAM streams all
    // its heads while the batches below are loaded and processed
    if (lane == 0) {
        if (p.nq) prefetch_l2(p.q + (size_t)t * p.nq * kQKHeadDim, (uint32_t)p.nq * kQKHeadDim * 2u);
        if (p.nk) prefetch_l2(p.k + (size_t)t * p.nk * kQKHeadDim, (uint32_t)p.nk * kQKHeadDim * 2u);
    }

    // ---- loads of one batch: pass b takes head h0 + 4b + grp
    auto row_of = [&](int hh) -> uint16_t* {
        return hh < p.nq ? p.q + ((size_t)t * p.nq + hh) * kQKHeadDim
                         : p.k + ((size_t)t * p.nk + (hh - p.nq)) * kQKHeadDim;
    };
    auto load = [&](uint4 (&v)[2][2], int h0) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int hh = h0 + 4 * b + grp;
            if (hh < nh) {
                const uint4* r = reinterpret_cast<const uint4*>(row_of(hh) + 8 * li);
                v[b][0] = r[0];  // elements 8 li ..
                v[b][1] = r[8];  // elements 64 + 8 li ..
            } else {
                v[b][0] = v[b][1] = make_uint4(0, 0, 0, 0);
            }
        }
    };
    uint4 va[2][2], vb[2][2];
    load(va, 0);

    // ---- per-lane constants: weights and cos/sin (RoPE) or the query scale (SSMax)
    const uint4* qwp = reinterpret_cast<const uint4*>(p.qw + 8 * li);
    const uint4* kwp = reinterpret_cast<const uint4*>(p.kw + 8 * li);
    const uint4 qw0 = __ldg(qwp), qw1 = __ldg(qwp + 8), kw0 = __ldg(kwp), kw1 = __ldg(kwp + 8);
    // cos and sin of this lane's 8 pairs (RoPE), for every head of the token
    float2 cv[4], sv[4];
    if (p.mode == 0) {
        const float4* cs = reinterpret_cast<const float4*>(p.table + pos * kQKHeadDim + 8 * li);
        const float4 c0 = __ldg(cs), c1 = __ldg(cs + 1), s0 = __ldg(cs + 16), s1 = __ldg(cs + 17);
        cv[0] = make_float2(c0.x, c0.y); cv[1] = make_float2(c0.z, c0.w);
        cv[2] = make_float2(c1.x, c1.y); cv[3] = make_float2(c1.z, c1.w);
        sv[0] = make_float2(s0.x, s0.y); sv[1] = make_float2(s0.z, s0.w);
        sv[2] = make_float2(s1.x, s1.y); sv[3] = make_float2(s1.z, s1.w);
    }
    const float g = p.mode != 0 ? ssmax_scale(pos, lane) : 1.0f;

    auto process = [&](const uint4 (&v)[2][2], int h0) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int hh = h0 + 4 * b + grp;
            const bool live = hh < nh, is_q = hh < p.nq;
            const uint32_t w[8] = {v[b][0].x, v[b][0].y, v[b][0].z, v[b][0].w,
                                   v[b][1].x, v[b][1].y, v[b][1].z, v[b][1].w};
            // compensated sum of squares over the group's 128 values
            float2 sa = make_float2(0.f, 0.f), ca = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 x = bf2_to_f2(w[i]);
                two_sum_acc2(sa, ca, mul2_rn(x, x));
            }
            float S = sa.x, C = ca.x;
            ff_merge(S, C, sa.y, ca.y);
#pragma unroll
            for (int off = 4; off; off >>= 1) {
                const float so = __shfl_xor_sync(full, S, off), co = __shfl_xor_sync(full, C, off);
                ff_merge(S, C, so, co);
            }
            float Sr;
            const bool need = !certify_round(S, C, p.errk, &Sr) || force_exact;  // group-uniform
            if (__any_sync(full, need)) {
                const float Sx = exact_group_sum_squares(v[b][0], v[b][1]);
                if (need) {
                    Sr = Sx;
                    if (li == 0 && live) atomicAdd(&g_exact_sum_count, 1ull);
                }
            }
            // Sr / 128 as an exact scaling by 2^-7 (the same rounding of the same value)
            const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(Sr, 0x1p-7f), p.eps)));
            const float2 rv = make_float2(r, r);
            const uint4 w0 = is_q ? qw0 : kw0, w1 = is_q ? qw1 : kw1;
            const uint32_t ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            uint32_t n[8], o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) n[i] = f2_to_bf2(mul2_rn(mul2_rn(bf2_to_f2(w[i]), rv), bf2_to_f2(ww[i])));
            if (p.mode == 0) {
                // words i (elements j) and i + 4 (elements j + 64) form the pairs.
                // The products are packed; the sums are scalar __fadd_rn /
                // __fsub_rn, which never merge into an FMA (a packed add whose
                // only operand is a packed product was measured to fuse into an
                // FMA despite its explicit rounding modifier).
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 a = bf2_to_f2(n[i]), b = bf2_to_f2(n[i + 4]);
                    const float2 ac = mul2_rn(a, cv[i]), bs = mul2_rn(b, sv[i]);
                    const float2 bc = mul2_rn(b, cv[i]), as = mul2_rn(a, sv[i]);
                    o[i] = f2_to_bf2(make_float2(__fsub_rn(ac.x, bs.x), __fsub_rn(ac.y, bs.y)));
                    o[i + 4] = f2_to_bf2(make_float2(__fadd_rn(bc.x, as.x), __fadd_rn(bc.y, as.y)));
                }
            } else if (is_q) {
                const float2 gv = make_float2(g, g);
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = f2_to_bf2(mul2_rn(bf2_to_f2(n[i]), gv));
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = n[i];
            }
            if (live) {
                uint4* dst = reinterpret_cast<uint4*>(row_of(hh) + 8 * li);
                dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                dst[8] = make_uint4(o[4], o[5], o[6], o[7]);
            }
        }
    };

    for (int h0 = 0; h0 < nh; h0 += 2 * kQKBatch) {
        if (h0 + kQKBatch < nh) load(vb, h0 + kQKBatch);
        process(va, h0);
        if (h0 + kQKBatch >= nh) break;
        if (h0 + 2 * kQKBatch < nh) load(va, h0 + 2 * kQKBatch);
        process(vb, h0 + kQKBatch);
    }
}

}  // namespace beam
