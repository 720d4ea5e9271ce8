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
#include "tma.cuh"

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
    int prefetch_rows;      // rows of this CTA's sequence to prefetch into L2 ahead of use
    int stages;             // ring slots per CTA (ring kernel)
    unsigned long long wait_ns;       // bound of every mbarrier wait
    unsigned long long test_wait_ns;  // bound of the test hook's wait
    float route_scale;      // MoE: x = bf16(route_scale * acc); 1 when the weights carry it
    uint8_t* yq;            // NVFP4 y: [T, D/2] E2M1 codes, element 2i in the low nibble
    uint8_t* ysf;           // NVFP4 y: [T, D/16] E4M3 block scales
    float y_gs;             // NVFP4 y: global scale
};

constexpr unsigned kFlagForceExact = 1u;
constexpr unsigned kFlagTestWaitTimeout = 2u;
constexpr int kMaxStages = 8;
constexpr int kMaxThreads = 512;
constexpr int kTopK = 8;

// Streaming accesses. Every row is read once and written once, so loads and
// stores bypass L1 and mark their L2 lines evict_first: the written rows leave
// L2 first, ahead of the next rows that the L2 prefetch brought in (evict_last)
// and that these loads then consume (measured on GB300 at T = 16384: the MoE
// boundary 281 -> 272 us, the dense boundary 114.5 -> 113.5 us).

// read-only operands (expert rows; never h)
__device__ __forceinline__ uint4 ld_stream_ro(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p), "l"(l2_evict_first()));
    return r;
}

// h (read here and overwritten later by the same thread) and x (which may be
// h itself): no .nc
__device__ __forceinline__ uint4 ld_stream_rw(const void* p) {
    uint4 r;
    asm("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p), "l"(l2_evict_first()));
    return r;
}

// the "memory" clobber keeps the stores ahead of the barrier that precedes
// the exact path's re-reads
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(l2_evict_first()) : "memory");
}
__device__ __forceinline__ void st_stream_u32(void* p, uint32_t v) {
    asm volatile("st.global.L2::cache_hint.u32 [%0], %1, %2;" :: "l"(p), "r"(v), "l"(l2_evict_first()) : "memory");
}
__device__ __forceinline__ void st_stream_u8(void* p, uint32_t v) {
    asm volatile("st.global.L2::cache_hint.u8 [%0], %1, %2;" :: "l"(p), "r"(v), "l"(l2_evict_first()) : "memory");
}



// One thread asks L2 for the inputs of row r (branch rows and h)
template <bool MOE>
__device__ __forceinline__ void prefetch_row(const BoundaryParams& p, long long r) {
    if (r >= p.T) return;
    const uint32_t row_bytes = (uint32_t)p.D * 2u;
    if (MOE) prefetch_l2_keep(p.e + (size_t)r * kTopK * (size_t)p.D, row_bytes * kTopK);
    else prefetch_l2_keep(p.x + (size_t)r * (size_t)p.D, row_bytes);
    prefetch_l2_keep(p.h + (size_t)r * (size_t)p.D, row_bytes);
}

__device__ __forceinline__ uint32_t word(const uint4& v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}
__device__ __forceinline__ void set_word(uint4& v, int q, uint32_t w) {
    if (q == 0) v.x = w; else if (q == 1) v.y = w; else if (q == 2) v.z = w; else v.w = w;
}

// Shared memory of the block reduction: one (sum, compensation) pair per
// thread, and the certified result broadcast by warp 0.
struct RedScratch {
    float2 part[kMaxThreads];
    float4 result;      // (rounded sum, 1 if certified else 0, its RMS factor, unused)
    float inv_sf[128];  // NVFP4: RN32(y_global_scale / sf) for every E4M3 code sf, 0 for sf = 0
};

// r = 1 / sqrt(S/D + eps), each operation rounded to nearest
__device__ __forceinline__ float rms_factor(float S, int D, float eps) {
    float ms = __fdiv_rn(S, (float)D);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
}

// Block-wide compensated sum of the squares of the row held in v[] (zeros in
// unused slots). Every thread folds its two FP32 lanes into one pair and
// stores it; warp 0 merges the pairs (lane l takes l, l+32, ... in order, then
// a 5-level xor butterfly), certifies the rounding and broadcasts it. The
// other warps run `overlap` while warp 0 merges; warp 0 runs it afterwards.
// Returns true with *out = RN32(exact sum) and *out_r = rms_factor(*out, D,
// eps) (formed once, by thread 0) when certified; false when the exact path
// must decide. The first barrier also orders every store this
// block issued before the call ahead of any load after it.
template <int VPT, class Overlap>
__device__ __forceinline__ bool block_sum_squares(const uint4 (&v)[VPT], float errk, int D, float eps,
                                                  RedScratch* rs, float* out, float* out_r, Overlap overlap) {
    float2 s = make_float2(0.f, 0.f), c = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float2 f = bf2_to_f2(word(v[i], q));
            two_sum_acc2(s, c, mul2_rn(f, f));
        }
    float S = s.x, C = c.x;
    ff_merge(S, C, s.y, c.y);
    rs->part[threadIdx.x] = make_float2(S, C);
    __syncthreads();
    const bool merger = threadIdx.x < 32;
    if (merger) {
        const int nw = blockDim.x >> 5;
        float2 t0 = rs->part[threadIdx.x];
        S = t0.x;
        C = t0.y;
        for (int w = 1; w < nw; ++w) {
            float2 tw = rs->part[threadIdx.x + 32 * w];
            ff_merge(S, C, tw.x, tw.y);
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            float s2 = __shfl_xor_sync(0xFFFFFFFFu, S, off);
            float c2 = __shfl_xor_sync(0xFFFFFFFFu, C, off);
            ff_merge(S, C, s2, c2);
        }
        if (threadIdx.x == 0) {
            float r;
            bool ok = certify_round(S, C, errk, &r);
            // one thread forms the RMS factor of a certified sum for the block
            rs->result = make_float4(r, ok ? 1.0f : 0.0f, ok ? rms_factor(r, D, eps) : 0.0f, 0.0f);
        }
    } else {
        overlap();
    }
    __syncthreads();
    if (merger) overlap();
    const float4 res = rs->result;
    *out = res.x;
    *out_r = res.z;
    return res.y != 0.0f;
}

// h' = bf16(RN32(a + b)) for BF16 a, b, as one packed BF16 add (a single
// rounding of the exact sum). Same result: if the exponents of a and b differ
// by at most 15, a + b fits in 24 bits and RN32 is exact; otherwise
// |b| < 2^-15 |a|, far below half a BF16 ulp of a, and both roundings return a
// (no tie is reachable). Infinities and NaN propagate alike.
__device__ __forceinline__ uint32_t bf2_add(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// FP32 -> E4M3 (OCP E4M3FN), nearest even, saturating; the code in the low byte
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
    uint32_t r;
    asm("{ .reg .b16 t; cvt.rn.satfinite.e4m3x2.f32 t, %1, %2; cvt.u32.u16 %0, t; }" : "=r"(r) : "f"(0.0f), "f"(v));
    return r & 0xFFu;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
    float f;
    const unsigned short b = (unsigned short)code;
    asm("{ .reg .b32 t; .reg .b16 lo, hi; cvt.rn.f16x2.e4m3x2 t, %1; mov.b32 {lo, hi}, t; cvt.f32.f16 %0, lo; }"
        : "=f"(f) : "h"(b));
    return f;
}

// eight FP32 -> eight E2M1 codes, nearest even, saturating: value 2i in the
// low nibble of byte i, value 2i+1 in its high nibble (the pairs are packed
// straight into the word)
__device__ __forceinline__ uint32_t f8_to_e2m1x8(const float2 (&v)[4]) {
    uint32_t r;
    asm("{ .reg .b8 t0, t1, t2, t3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
        "mov.b32 %0, {t0, t1, t2, t3}; }"
        : "=r"(r)
        : "f"(v[0].x), "f"(v[0].y), "f"(v[1].x), "f"(v[1].y), "f"(v[2].x), "f"(v[2].y), "f"(v[3].x),
          "f"(v[3].y));
    return r;
}

// RN32(a / 6) for a BF16 value a >= 0 (at most 8 significant bits) in three
// operations instead of an IEEE division: t = RN32(a c) with c = RN32(1/6) is
// within an ulp of a/6, so r = a - 6 t is exact in one FMA, and one correction
// t + r c (Markstein's correction step for a known divisor) rounds correctly:
// a/6 = (significand / 3) 2^k always lies at least 1/6 ulp from a rounding
// midpoint, far beyond the correction's error. Checked for every non-negative
// finite BF16 value in exact rational arithmetic. For a = +inf, t is +inf
// (a finite a never makes t overflow) and is returned as it is: the correction
// would give inf - inf = NaN.
__device__ __forceinline__ float div6_bf16(float a) {
    const float c = 0x1.555556p-3f;
    const float t = __fmul_rn(a, c);
    const float q = __fmaf_rn(__fmaf_rn(-t, 6.0f, a), c, t);
    return t < INFINITY ? q : t;
}

// h is read and later overwritten by the same thread; this form also keeps
// the read ahead of any later store (the NVFP4 MoE path parks x in the h row)
__device__ __forceinline__ uint4 ld_stream_rw_ordered(const void* p) {
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p), "l"(l2_evict_first()) : "memory");
    return r;
}

// Norm weights staged once per CTA in shared memory by FULL kernels, as BF16
// vectors (ws[vi] = post_w vector vi, ws[nvec + vi] = pre_w vector vi; one
// 16-byte shared load per 8 weights, unpacked at use: measured faster than
// FP32 copies, which need two loads). Other kernels read the BF16 weights from
// global memory (L1-cached) on every row.
__device__ __forceinline__ void stage_weights(const BoundaryParams& p, uint4* ws) {
    for (int vi = threadIdx.x; vi < p.nvec; vi += blockDim.x) {
        ws[vi] = __ldg(reinterpret_cast<const uint4*>(p.post_w) + vi);
        ws[p.nvec + vi] = __ldg(reinterpret_cast<const uint4*>(p.pre_w) + vi);
    }
    __syncthreads();
}

// the 8 weights of vector vi as 4 FP32 pairs, from shared memory (FULL) or global
template <bool FULL>
__device__ __forceinline__ void load_weights(const uint16_t* g, const uint4* ws, int vi, float2 (&w)[4]) {
    const uint4 v = FULL ? ws[vi] : __ldg(reinterpret_cast<const uint4*>(g) + vi);
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = bf2_to_f2(word(v, q));
}

// Everything after the branch x and the stream h of a row are in registers:
// post-norm sum, xn, residual (h' stored over h), pre-norm sum, y (stored).
// `after_s1` runs on every thread right after the post-norm reduction's
// barrier, when every thread has consumed its inputs of this row. FULL: the
// row is exactly NT * VPT vectors (no bounds checks) and ws holds the weights.
template <int VPT, bool MOE, bool FULL, bool QUANT, class AfterS1>
__device__ __forceinline__ void finish_row(const BoundaryParams& p, long long row, uint4 (&xv)[VPT],
                                           uint4 (&hv)[VPT], RedScratch* rs, ExactScratch* sc,
                                           const uint4* ws, AfterS1 after_s1) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const bool force_exact = (p.flags & kFlagForceExact) != 0;
    const size_t base = (size_t)row * (size_t)p.D;
    const float2 c1 = make_float2(p.c1, p.c1), c2 = make_float2(p.c2, p.c2);

    // ---- post-norm sum; while warp 0 merges, the others scale the stream:
    // a = bf16(c1 h) replaces h in registers (it does not depend on r1)
    auto scale_stream = [&]() {
#pragma unroll
        for (int i = 0; i < VPT; ++i)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                set_word(hv[i], q, f2_to_bf2(mul2_rn(c1, bf2_to_f2(word(hv[i], q)))));
    };
    float S1, r1;
    const bool ok1 = block_sum_squares<VPT>(xv, p.errk, p.D, p.eps, rs, &S1, &r1, scale_stream);
    after_s1();
    if (!ok1 || force_exact) {
        // the exact path reads x from global memory: the input row (dense)
        // or, for MoE, the combined x parked in this y row
        const uint16_t* srow = p.x + base;
        if (MOE) {
            // park x in this row of y, or, when y leaves as NVFP4, in the row of
            // h (already in registers; h' overwrites it later)
            uint16_t* park = QUANT ? p.h + base : p.y + base;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int vi = tid + i * nt;
                if (FULL || vi < p.nvec) st_stream(park + (size_t)vi * 8, xv[i]);
            }
            __syncthreads();
            srow = park;
        }
        S1 = exact_row_sum_squares(srow, p.D, sc);
        r1 = rms_factor(S1, p.D, p.eps);
    }
    const float2 r1v = make_float2(r1, r1);

    // ---- xn, b = bf16(c2 xn), h' = a + b (in registers)
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int vi = tid + i * nt;
        if (FULL || vi < p.nvec) {
            float2 pw[4];
            load_weights<FULL>(p.post_w, ws, vi, pw);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float2 xf = bf2_to_f2(word(xv[i], q));
                float2 xn = bf2_to_f2(f2_to_bf2(mul2_rn(mul2_rn(xf, r1v), pw[q])));
                uint32_t b = f2_to_bf2(mul2_rn(c2, xn));
                set_word(hv[i], q, bf2_add(word(hv[i], q), b));
            }
        } else {
            hv[i] = make_uint4(0, 0, 0, 0);
        }
    }

    // ---- pre-norm sum of h'; h' is stored over h while warp 0 merges
    auto store_stream = [&]() {
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int vi = tid + i * nt;
            if (FULL || vi < p.nvec) st_stream(p.h + base + (size_t)vi * 8, hv[i]);
        }
    };
    float S2, r2;
    if (!block_sum_squares<VPT>(hv, p.errk, p.D, p.eps, rs, &S2, &r2, store_stream) || force_exact) {
        __syncthreads();  // warp 0 stored its part of h' after the reduction's last barrier
        S2 = exact_row_sum_squares(p.h + base, p.D, sc);
        r2 = rms_factor(S2, p.D, p.eps);
    }
    const float2 r2v = make_float2(r2, r2);

    // ---- y = bf16((h' r2) pre_w), stored as BF16 or quantised to NVFP4
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int vi = tid + i * nt;
        const bool valid = FULL || vi < p.nvec;
        uint4 yv = make_uint4(0, 0, 0, 0);
        if (valid) {
            float2 qw[4];
            load_weights<FULL>(p.pre_w, ws ? ws + p.nvec : nullptr, vi, qw);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                set_word(yv, q, f2_to_bf2(mul2_rn(mul2_rn(bf2_to_f2(word(hv[i], q)), r2v), qw[q])));
            if (!QUANT) st_stream(p.y + base + (size_t)vi * 8, yv);
        }
        if (QUANT) {
            // a block of 16 is this vector and its neighbour, held by lane ^ 1
            float am = 0.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = bf2_to_f2(word(yv, q));
                am = fmaxf(am, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
            am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
            const uint32_t sfb = f32_to_e4m3(__fmul_rn(div6_bf16(am), p.y_gs));
            uint32_t codes = 0u;
            if (sfb != 0u) {  // code 0 is the only zero scale (the argument is >= 0)
                const float inv = rs->inv_sf[sfb & 0x7Fu];
                const float2 iv = make_float2(inv, inv);
                float2 f[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) f[q] = mul2_rn(bf2_to_f2(word(yv, q)), iv);
                codes = f8_to_e2m1x8(f);
            }
            if (valid) {
                st_stream_u32(p.yq + (base + (size_t)vi * 8) / 2, codes);
                if (!(vi & 1)) st_stream_u8(p.ysf + (base + (size_t)vi * 8) / 16, sfb);
            }
        }
    }
}

struct NoOp {
    __device__ void operator()() const {}
};

// Loads straight to registers (dense x or the MoE combine), optionally asking
// L2 for the inputs of this CTA's row `prefetch_rows` ahead.
template <int VPT, bool MOE, bool FULL, bool QUANT>
__global__ void __launch_bounds__(kMaxThreads) boundary_kernel(const BoundaryParams p) {
    extern __shared__ __align__(16) uint4 ws_dyn[];
    __shared__ RedScratch rs;
    __shared__ ExactScratch sc;
    const int tid = threadIdx.x, nt = blockDim.x;
    const uint4* ws = FULL ? ws_dyn : nullptr;

    // prologue that reads only the norm weights; with a programmatic launch it
    // overlaps the previous kernel on the stream (the caller guarantees that
    // kernel does not write the weights)
    pdl_trigger();
    if (QUANT) {
        // inverse block scales, read after the first row reduction's barrier
        for (int i = tid; i < 128; i += nt) {
            const float sf = e4m3_to_f32((uint32_t)i);
            rs.inv_sf[i] = sf != 0.0f ? __fdiv_rn(p.y_gs, sf) : 0.0f;
        }
    }
    if (FULL) stage_weights(p, ws_dyn);
    // the L2 prefetch of this CTA's first rows: a hint that returns no data (L2
    // is the coherence point), so it may run before the dependency wait
    if (tid == 0)
        for (int k = 0; k < p.prefetch_rows; ++k) prefetch_row<MOE>(p, blockIdx.x + (long long)k * gridDim.x);
    pdl_wait();

    for (long long row = blockIdx.x; row < p.T; row += gridDim.x) {
        const size_t base = (size_t)row * (size_t)p.D;
        uint4 xv[VPT], hv[VPT];
        if (tid == 0 && p.prefetch_rows > 0) prefetch_row<MOE>(p, row + (long long)p.prefetch_rows * gridDim.x);

        if (MOE) {
            // x = bf16(fma chain over the 8 experts, k ascending)
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
                    if (FULL || vi < p.nvec) {
                        uint4 ev = ld_stream_ro(erow + (size_t)k * p.D + (size_t)vi * 8);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            acc[i][q] = __ffma2_rn(w2, bf2_to_f2(word(ev, q)), acc[i][q]);
                    }
                }
            }
            // routing scale applied in the combine (exact when it is 1)
            const float2 rs2 = make_float2(p.route_scale, p.route_scale);
#pragma unroll
            for (int i = 0; i < VPT; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) set_word(xv[i], q, f2_to_bf2(mul2_rn(acc[i][q], rs2)));
        } else {
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int vi = tid + i * nt;
                // x may be h itself, which this kernel writes: x takes the
                // coherent load, not the read-only path (measured the same speed)
                xv[i] = (FULL || vi < p.nvec) ? ld_stream_rw(p.x + base + (size_t)vi * 8) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int vi = tid + i * nt;
            const uint16_t* hp = p.h + base + (size_t)vi * 8;
            hv[i] = (FULL || vi < p.nvec) ? ((MOE && QUANT) ? ld_stream_rw_ordered(hp) : ld_stream_rw(hp))
                                         : make_uint4(0, 0, 0, 0);
        }
        finish_row<VPT, MOE, FULL, QUANT>(p, row, xv, hv, &rs, &sc, ws, NoOp{});
    }
}

// Dense boundary fed by a ring of `stages` shared-memory slots per CTA. Slot s
// holds [x row | h row] of one of this CTA's rows (rows blockIdx.x + i*gridDim.x,
// slot i % stages), filled by two 1-D bulk copies that complete on the slot's
// mbarrier. One thread refills a slot with the row `stages` ahead as soon as
// the post-norm reduction's barrier shows every thread has read it, so up to
// stages-1 rows per CTA are in flight while a row is computed. FULL kernels
// keep the BF16 weights after the ring.
//
// Every slot wait is bounded. The threads vote after each wait: if any wait
// gave up, the CTA stores nothing for that row or any later row of its own
// (h and y keep what they held), records the timeout in the device status
// word, waits (bounded) for the copies it still has in flight, and returns.
// Test hook (kFlagTestWaitTimeout): the copy of each CTA's second row is never
// issued, so that row's wait runs out after test_wait_ns.
template <int VPT, bool FULL>
__global__ void __launch_bounds__(kMaxThreads) boundary_ring_kernel(const BoundaryParams p) {
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ RedScratch rs;
    __shared__ ExactScratch sc;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int S = p.stages;
    const uint32_t row_bytes = (uint32_t)p.D * 2u;
    const long long G = gridDim.x;
    const long long n_iter = (p.T - blockIdx.x + G - 1) / G;  // grid <= T: at least one row
    const bool hook = (p.flags & kFlagTestWaitTimeout) != 0;
    const unsigned long long wait_ns = hook ? p.test_wait_ns : p.wait_ns;
    uint4* ws = FULL ? reinterpret_cast<uint4*>(ring + (size_t)S * 2u * row_bytes) : nullptr;

    auto slot_x = [&](int s) { return ring + (size_t)s * 2u * row_bytes; };
    auto issued = [&](long long i) { return !(hook && i == 1); };
    auto issue = [&](long long i) {  // thread 0 only
        if (!issued(i)) return;
        const int s = (int)(i % S);
        const size_t off = (size_t)(blockIdx.x + i * G) * (size_t)p.D;
        mbar_arrive_expect_tx(&full[s], 2u * row_bytes);
        bulk_load(slot_x(s), p.x + off, row_bytes, &full[s]);
        bulk_load(slot_x(s) + row_bytes, p.h + off, row_bytes, &full[s]);
    };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        mbar_fence_init();
    }
    __syncthreads();
    pdl_trigger();
    if (FULL) stage_weights(p, ws);  // weights only: may overlap the previous kernel
    pdl_wait();
    if (tid == 0)
        for (long long i = 0; i < S && i < n_iter; ++i) issue(i);

    long long dead_from = n_iter;  // first row whose wait gave up (n_iter: none)
    for (long long i = 0; i < n_iter; ++i) {
        const int s = (int)(i % S);
        const uint32_t parity = (uint32_t)((i / S) & 1);
        const bool ok = mbar_wait_bounded(&full[s], parity, wait_ns);
        if (__syncthreads_or(!ok)) {  // block-uniform: every thread leaves the loop here
            dead_from = i;
            break;
        }
        const uint4* xs = reinterpret_cast<const uint4*>(slot_x(s));
        const uint4* hs = reinterpret_cast<const uint4*>(slot_x(s) + row_bytes);
        uint4 xv[VPT], hv[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int vi = tid + j * nt;
            xv[j] = (FULL || vi < p.nvec) ? xs[vi] : make_uint4(0, 0, 0, 0);
            hv[j] = (FULL || vi < p.nvec) ? hs[vi] : make_uint4(0, 0, 0, 0);
        }
        finish_row<VPT, false, FULL, false>(p, blockIdx.x + i * G, xv, hv, &rs, &sc, ws, [&]() {
            if (tid == 0 && i + S < n_iter) issue(i + S);
        });
    }
    // after a timeout: the copies issued for rows dead_from .. dead_from + S - 1
    // may still land; wait for them (bounded) before the shared memory goes
    if (dead_from < n_iter && tid == 0) {
        report_timeout();
        for (long long i = dead_from; i < n_iter && i < dead_from + S; ++i)
            if (issued(i)) mbar_wait_bounded(&full[i % S], (uint32_t)((i / S) & 1), p.wait_ns);
    }
}

}  // namespace beam
