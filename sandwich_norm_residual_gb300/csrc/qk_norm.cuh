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
// One warp per token walks its heads, 8 heads per pass (4 lanes each), after
// asking L2 for all of the token's rows. Lane i of a head's group holds elements 16i .. 16i+15
// and 64+16i .. 64+16i+15: both halves of every rotate-half pair are in the
// same lane, which reads its 16 cos and 16 sin values from the token's table
// row, staged once per warp in shared memory. Each lane folds its 32 squares into two compensated sums; the
// row sum merges them in the lane, then over 2 shuffle levels (4 merge levels
// in all). Against 8 lanes per head, 4 lanes halve the per-head work that
// every lane of a group repeats (merges, certification, 1/sqrt): measured
// 7-8% faster.
#pragma once

#include "row_sum.cuh"
#include "tma.cuh"

namespace beam {

constexpr int kQKHeadDim = 128;
constexpr int kQKBatch = 8;           // heads per pass (one per group of 4 lanes)

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
    unsigned flags;       // kFlagForceExact
    int warps_per_token;  // warps sharing a token's heads (few tokens: more warps per token)
    int batches_per_warp; // 8-head batches each of them takes
};

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

// Exact RN32 sum of the squares of a 128-element row held by a group of 4
// lanes (32 BF16 values per lane in a..d), without shared memory: 32-bit
// chunk sums of each FP32 term m * 2^q * 2^-149 in nine 64-bit registers,
// added over the group (xor 2, 1), carried and rounded to nearest even.
// Every lane of the warp must call it; each group gets its own row's sum.
__device__ __noinline__ float exact_group_sum_squares(uint4 a, uint4 b, uint4 c, uint4 d) {
    unsigned long long acc[9];
#pragma unroll
    for (int L = 0; L < 9; ++L) acc[L] = 0ull;
    int nan = 0, inf = 0;
    const uint32_t w[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
    for (int i = 0; i < 32; ++i) {
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
        for (int off = 2; off; off >>= 1) acc[L] += __shfl_xor_sync(0xFFFFFFFFu, acc[L], off);
    for (int off = 2; off; off >>= 1) {
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

// MODE 0: RoPE, 1: SSMax. Each warp keeps two batches in registers: the next
// batch is loaded before the current one is processed, while the token's rows
// are already on their way to L2; 2 blocks of 8 warps per SM (at most 128
// registers). Measured at T = 16384 against one batch in flight at 3 blocks per
// SM: RoPE 112.9 -> 109.0 us, SSMax 96.1 -> 85.5 us at 3 blocks and 83.9 us at
// 2 (three batches in flight were slower); RoPE's cos and sin read per batch
// from shared memory instead of held in 32 registers for the whole token:
// 109.2 -> 101.2 us; the norm weights from a per-warp shared-memory copy
// instead of L1: RoPE 101.0 -> 100.1 us, SSMax 83.9 -> 81.9 us.
template <int MODE>
__global__ void __launch_bounds__(256, 2) qk_norm_kernel(const QKParams p) {
    const int lane = threadIdx.x & 31, grp = lane >> 2, li = lane & 3;
    // warp gw takes heads [hbeg, hend) of token gw / warps_per_token
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const bool split = p.warps_per_token > 1;  // launch-uniform: no 64-bit division otherwise
    const long long t = split ? gw / p.warps_per_token : gw;
    const int nh = p.nq + p.nk;
    const int hbeg = split ? (int)(gw % p.warps_per_token) * p.batches_per_warp * kQKBatch : 0;
    const int hend = min(nh, hbeg + p.batches_per_warp * kQKBatch);
    if (t >= p.T || hbeg >= nh) return;  // whole warps leave together
    const unsigned full = 0xFFFFFFFFu;
    const bool force_exact = (p.flags & kFlagForceExact) != 0;

    // with a programmatic launch this part overlaps the previous kernel on the
    // stream: ask L2 for this warp's q and k rows (a hint that returns no data),
    // so that DRAM streams all of them while the batches below are loaded and
    // processed; then wait for that kernel before reading anything
    pdl_trigger();
    if (lane == 0) {
        const int qe = min(hend, p.nq), kb = max(hbeg, p.nq) - p.nq, ke = hend - p.nq;
        if (qe > hbeg)
            prefetch_l2(p.q + ((size_t)t * p.nq + hbeg) * kQKHeadDim, (uint32_t)(qe - hbeg) * kQKHeadDim * 2u);
        if (ke > kb)
            prefetch_l2(p.k + ((size_t)t * p.nk + kb) * kQKHeadDim, (uint32_t)(ke - kb) * kQKHeadDim * 2u);
    }
    pdl_wait();

    const long long pos = p.pos[t];
    if (pos < 0 || (MODE == 0 && pos >= p.max_pos) || (MODE != 0 && pos > kSSMaxMaxPos)) {
        if (lane == 0) atomicOr(&g_status_word, 2u);  // reported as a bad argument
        return;
    }
    auto row_of = [&](int hh) -> uint16_t* {
        return hh < p.nq ? p.q + ((size_t)t * p.nq + hh) * kQKHeadDim
                         : p.k + ((size_t)t * p.nk + (hh - p.nq)) * kQKHeadDim;
    };
    auto load = [&](uint4 (&v)[4], int h0) {
        const int hh = h0 + grp;
        if (hh < nh) {
            const uint4* r = reinterpret_cast<const uint4*>(row_of(hh) + 16 * li);
            v[0] = r[0];
            v[1] = r[1];
            v[2] = r[8];
            v[3] = r[9];
        } else {
            v[0] = v[1] = v[2] = v[3] = make_uint4(0, 0, 0, 0);
        }
    };
    uint4 v[4];
    load(v, hbeg);

    // the q and k norm weights widened to FP32, one copy per warp, laid out like
    // the table below (q at 0, k at 160): 16-byte reads in distinct banks, and
    // no unpacking per batch (SSMax 81.7 -> 80.6 us at T = 16384)
    __shared__ __align__(16) float wsf[8][320];
    {
        const uint4 wv = __ldg(reinterpret_cast<const uint4*>(lane < 16 ? p.qw : p.kw) + (lane & 15));
        const int e = 8 * (lane & 15);
        float* d = &wsf[threadIdx.x >> 5][(lane < 16 ? 0 : 160) + 80 * (e >> 6) + 20 * ((e >> 4) & 3) + (e & 15)];
        const float2 w01 = bf2_to_f2(wv.x), w23 = bf2_to_f2(wv.y), w45 = bf2_to_f2(wv.z), w67 = bf2_to_f2(wv.w);
        reinterpret_cast<float4*>(d)[0] = make_float4(w01.x, w01.y, w23.x, w23.y);
        reinterpret_cast<float4*>(d)[1] = make_float4(w45.x, w45.y, w67.x, w67.y);
    }
    __syncwarp();
    // RoPE: the token's table row, one per warp: lane chunk li's 16 cos at
    // 20 li, its 16 sin at 80 + 20 li (the padding puts the 16-byte reads of a
    // head's 4 lanes in distinct banks: 100.0 -> 98.4 us at T = 16384)
    __shared__ __align__(16) float tab[8][160];
    const float4* cs = reinterpret_cast<const float4*>(&tab[threadIdx.x >> 5][20 * li]);
    if (MODE == 0) {
        const int e = 4 * lane;  // elements e .. e+3 of the row: cos or sin, chunk, offset in the chunk
        *reinterpret_cast<float4*>(&tab[threadIdx.x >> 5][80 * (e >> 6) + 20 * ((e >> 4) & 3) + (e & 15)]) =
            __ldg(reinterpret_cast<const float4*>(p.table + pos * kQKHeadDim) + lane);
        __syncwarp();
    }
    const float g = MODE != 0 ? ssmax_scale(pos, lane) : 1.0f;

    auto process = [&](const uint4 (&v)[4], int h0) {
        const int hh = h0 + grp;
        const bool live = hh < nh, is_q = hh < p.nq;
        const uint32_t w[16] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w,
                                v[2].x, v[2].y, v[2].z, v[2].w, v[3].x, v[3].y, v[3].z, v[3].w};
        // compensated sums of squares of the lower and upper halves, merged
        // in the lane, then over the group's 4 lanes
        float2 sa = make_float2(0.f, 0.f), ca = sa, sb = sa, cb = sa;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 xa = bf2_to_f2(w[i]), xb = bf2_to_f2(w[i + 8]);
            two_sum_acc2(sa, ca, mul2_rn(xa, xa));
            two_sum_acc2(sb, cb, mul2_rn(xb, xb));
        }
        float S = sa.x, C = ca.x, S2 = sb.x, C2 = cb.x;
        ff_merge(S, C, sa.y, ca.y);
        ff_merge(S2, C2, sb.y, cb.y);
        ff_merge(S, C, S2, C2);
#pragma unroll
        for (int off = 2; off; off >>= 1) {
            const float so = __shfl_xor_sync(full, S, off), co = __shfl_xor_sync(full, C, off);
            ff_merge(S, C, so, co);
        }
        float Sr;
        const bool need = !certify_round(S, C, p.errk, &Sr) || force_exact;  // group-uniform
        if (__any_sync(full, need)) {
            const float Sx = exact_group_sum_squares(v[0], v[1], v[2], v[3]);
            if (need) {
                Sr = Sx;
                if (li == 0 && live) atomicAdd(&g_exact_sum_count, 1ull);
            }
        }
        const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(Sr, 0x1p-7f), p.eps)));
        const float2 rv = make_float2(r, r);
        const float4* wf = reinterpret_cast<const float4*>(&wsf[threadIdx.x >> 5][(is_q ? 0 : 160) + 20 * li]);
        uint32_t n[16], o[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 wq = wf[j < 4 ? j : j + 16];
            const int i = 2 * j;
            n[i] = f2_to_bf2(mul2_rn(mul2_rn(bf2_to_f2(w[i]), rv), make_float2(wq.x, wq.y)));
            n[i + 1] = f2_to_bf2(mul2_rn(mul2_rn(bf2_to_f2(w[i + 1]), rv), make_float2(wq.z, wq.w)));
        }
        if (MODE == 0) {
            float2 cv[8], sv[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 c = cs[i], sn = cs[20 + i];
                cv[2 * i] = make_float2(c.x, c.y);
                cv[2 * i + 1] = make_float2(c.z, c.w);
                sv[2 * i] = make_float2(sn.x, sn.y);
                sv[2 * i + 1] = make_float2(sn.z, sn.w);
            }
            // words i (elements j) and i + 8 (elements j + 64) form the pairs.
            // The products are packed; the sums are scalar __fadd_rn /
            // __fsub_rn, which never merge into an FMA (a packed add whose only
            // operand is a packed product was measured to fuse into an FMA
            // despite its explicit rounding modifier).
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 a = bf2_to_f2(n[i]), b = bf2_to_f2(n[i + 8]);
                const float2 ac = mul2_rn(a, cv[i]), bs = mul2_rn(b, sv[i]);
                const float2 bc = mul2_rn(b, cv[i]), as = mul2_rn(a, sv[i]);
                o[i] = f2_to_bf2(make_float2(__fsub_rn(ac.x, bs.x), __fsub_rn(ac.y, bs.y)));
                o[i + 8] = f2_to_bf2(make_float2(__fadd_rn(bc.x, as.x), __fadd_rn(bc.y, as.y)));
            }
        } else if (is_q) {
            const float2 gv = make_float2(g, g);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = f2_to_bf2(mul2_rn(bf2_to_f2(n[i]), gv));
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = n[i];
        }
        if (live) {
            uint4* dst = reinterpret_cast<uint4*>(row_of(hh) + 16 * li);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            dst[8] = make_uint4(o[8], o[9], o[10], o[11]);
            dst[9] = make_uint4(o[12], o[13], o[14], o[15]);
        }
    };

    for (int h0 = hbeg; h0 < hend; h0 += kQKBatch) {
        uint4 vn[4];
        const bool more = h0 + kQKBatch < hend;
        if (more) load(vn, h0 + kQKBatch);
        process(v, h0);
        if (more) {
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = vn[i];
        }
    }
}

}  // namespace beam
