// Fused sublayer-boundary kernels for sm_103a (dense and MoE-combine).
//
// One CTA owns one token row at a time (persistent grid: rows blockIdx.x,
// blockIdx.x + gridDim.x, ...). Thread t holds the 16-byte vectors
// t, t + NT, ..., t + (VPT-1) NT of the row (8 BF16 each), so every load and
// store of a warp covers 512 contiguous bytes. A row never leaves registers
// between its loads and its two stores: HBM sees read h, read x (or the 8
// expert rows and 8 routing weights), write h', write y.
//
// Per row (FP32 math, BF16 rounding points of the unfused code):
//   [MoE] acc = fma chain over k of w_k * e_k (k ascending), x = bf16(acc)
//   S1 = RN32(sum x^2), r1 = 1/sqrt(S1/D + eps)
//   xn = bf16((x r1) post_w)
//   h' = bf16(bf16(c1 h) + bf16(c2 xn))                 (stored over h)
//   S2 = RN32(sum h'^2), r2 = 1/sqrt(S2/D + eps)
//   y  = bf16((h' r2) pre_w)
// Elementwise work runs on packed f32x2 arithmetic; BF16 <-> FP32 is a shift
// or mask one way and cvt.rn.bf16x2.f32 the other.
#pragma once

#include "row_sum.cuh"

namespace beam {

struct BoundaryParams {
    uint16_t* h;            // [T, D] in/out
    const uint16_t* x;      // [T, D] (dense)
    const uint16_t* e;      // [T, K, D] (MoE)
    const float* w;         // [T, K] (MoE)
    const uint16_t* post_w; // [D]
    const uint16_t* pre_w;  // [D]
    uint16_t* y;            // [T, D]
    long long T;
    int D;
    int nvec;               // D / 8
    float c1, c2, eps;
    float errk;             // certified-rounding error factor for this launch shape
    unsigned flags;
};

constexpr unsigned kFlagForceExact = 1u;
constexpr int kMaxThreads = 512;
constexpr int kTopK = 8;

// streaming loads: read-only operands bypass L1 allocation
__device__ __forceinline__ uint4 ld_stream_ro(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// h is read here and overwritten later by the same thread: no .nc
__device__ __forceinline__ uint4 ld_stream_rw(const void* p) {
    uint4 r;
    asm("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// the "memory" clobber keeps the stores ahead of the barrier that precedes
// the exact path's re-reads
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ uint32_t word(const uint4& v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}
__device__ __forceinline__ void set_word(uint4& v, int q, uint32_t w) {
    if (q == 0) v.x = w; else if (q == 1) v.y = w; else if (q == 2) v.z = w; else v.w = w;
}

// Block-wide compensated sum of the squares of the row held in v[] (zeros in
// unused slots). Returns true with *out = RN32(exact sum) when the rounding
// is certified; false when the exact path must decide. The barrier inside
// also orders every store this block issued before the call ahead of any
// load after it (the exact path re-reads rows through L2).
template <int VPT>
__device__ __forceinline__ bool block_sum_squares(const uint4 (&v)[VPT], float errk,
                                                  float2 (*red)[32], int& buf, float* out) {
    float2 s = make_float2(0.f, 0.f), c = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float2 f = bf2_to_f2(word(v[i], q));
            two_sum_acc2(s, c, __fmul2_rn(f, f));
        }
    float S = s.x, C = c.x;
    ff_merge(S, C, s.y, c.y);
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        float s2 = __shfl_xor_sync(0xFFFFFFFFu, S, off);
        float c2 = __shfl_xor_sync(0xFFFFFFFFu, C, off);
        ff_merge(S, C, s2, c2);
    }
    const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if ((threadIdx.x & 31) == 0) red[buf][warp] = make_float2(S, C);
    __syncthreads();
    float2 t0 = red[buf][0];
    S = t0.x;
    C = t0.y;
    for (int w = 1; w < nw; ++w) {
        float2 tw = red[buf][w];
        ff_merge(S, C, tw.x, tw.y);
    }
    buf ^= 1;  // the next reduction writes the other buffer: one barrier per reduction
    return certify_round(S, C, errk, out);
}

__device__ __forceinline__ float rms_factor(float S, int D, float eps) {
    float ms = __fdiv_rn(S, (float)D);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
}

template <int VPT, bool MOE>
__global__ void __launch_bounds__(kMaxThreads) boundary_kernel(const BoundaryParams p) {
    __shared__ float2 red[2][32];
    __shared__ ExactScratch sc;
    const int tid = threadIdx.x, nt = blockDim.x;
    const bool force_exact = (p.flags & kFlagForceExact) != 0;
    const float2 c1 = make_float2(p.c1, p.c1), c2 = make_float2(p.c2, p.c2);
    int buf = 0;

    for (long long row = blockIdx.x; row < p.T; row += gridDim.x) {
        const size_t base = (size_t)row * (size_t)p.D;
        uint4 xv[VPT], hv[VPT];

        // ---- branch output x (dense: load; MoE: FP32 fma chain over the 8 experts)
        if (MOE) {
            const float4 wa = __ldg(reinterpret_cast<const float4*>(p.w + row * kTopK));
            const float4 wb = __ldg(reinterpret_cast<const float4*>(p.w + row * kTopK + 4));
            const float wk[kTopK] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
            float2 acc[VPT][4];
#pragma unroll
            for (int i = 0; i < VPT; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[i][q] = make_float2(0.f, 0.f);
            const uint16_t* erow = p.e + (size_t)row * kTopK * (size_t)p.D;
#pragma unroll
            for (int k = 0; k < kTopK; ++k) {
                const float2 w2 = make_float2(wk[k], wk[k]);
#pragma unroll
                for (int i = 0; i < VPT; ++i) {
                    const int vi = tid + i * nt;
                    if (vi < p.nvec) {
                        uint4 ev = ld_stream_ro(erow + (size_t)k * p.D + (size_t)vi * 8);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            acc[i][q] = __ffma2_rn(w2, bf2_to_f2(word(ev, q)), acc[i][q]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < VPT; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) set_word(xv[i], q, f2_to_bf2(acc[i][q]));
        } else {
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int vi = tid + i * nt;
                xv[i] = vi < p.nvec ? ld_stream_ro(p.x + base + (size_t)vi * 8) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int vi = tid + i * nt;
            hv[i] = vi < p.nvec ? ld_stream_rw(p.h + base + (size_t)vi * 8) : make_uint4(0, 0, 0, 0);
        }

        // ---- post-norm sum; the exact path reads x from global memory: the
        // input row (dense) or, for MoE, the combined x parked in this y row
        float S1;
        if (!block_sum_squares<VPT>(xv, p.errk, red, buf, &S1) || force_exact) {
            const uint16_t* srow = p.x + base;
            if (MOE) {
#pragma unroll
                for (int i = 0; i < VPT; ++i) {
                    const int vi = tid + i * nt;
                    if (vi < p.nvec) st_stream(p.y + base + (size_t)vi * 8, xv[i]);
                }
                __syncthreads();
                srow = p.y + base;
            }
            S1 = exact_row_sum_squares(srow, p.D, &sc);
        }
        const float r1 = rms_factor(S1, p.D, p.eps);
        const float2 r1v = make_float2(r1, r1);

        // ---- xn, depth-scaled residual, store h' over h
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int vi = tid + i * nt;
            if (vi < p.nvec) {
                const uint4 pw = __ldg(reinterpret_cast<const uint4*>(p.post_w) + vi);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float2 xf = bf2_to_f2(word(xv[i], q));
                    float2 xn = bf2_to_f2(f2_to_bf2(__fmul2_rn(__fmul2_rn(xf, r1v), bf2_to_f2(word(pw, q)))));
                    float2 a = bf2_to_f2(f2_to_bf2(__fmul2_rn(c1, bf2_to_f2(word(hv[i], q)))));
                    float2 b = bf2_to_f2(f2_to_bf2(__fmul2_rn(c2, xn)));
                    set_word(hv[i], q, f2_to_bf2(__fadd2_rn(a, b)));
                }
                st_stream(p.h + base + (size_t)vi * 8, hv[i]);
            }
        }

        // ---- pre-norm sum of h' (the exact path re-reads the h row just stored)
        float S2;
        if (!block_sum_squares<VPT>(hv, p.errk, red, buf, &S2) || force_exact)
            S2 = exact_row_sum_squares(p.h + base, p.D, &sc);
        const float r2 = rms_factor(S2, p.D, p.eps);
        const float2 r2v = make_float2(r2, r2);

        // ---- y = bf16((h' r2) pre_w)
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int vi = tid + i * nt;
            if (vi < p.nvec) {
                const uint4 qw = __ldg(reinterpret_cast<const uint4*>(p.pre_w) + vi);
                uint4 yv;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    set_word(yv, q, f2_to_bf2(__fmul2_rn(__fmul2_rn(bf2_to_f2(word(hv[i], q)), r2v),
                                                         bf2_to_f2(word(qw, q)))));
                st_stream(p.y + base + (size_t)vi * 8, yv);
            }
        }
    }
}

}  // namespace beam
