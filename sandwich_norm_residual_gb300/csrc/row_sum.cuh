// Row sum of squares for the two RMSNorms of the fused boundary, sm_103a.
//
// The value returned is S = RN32(sum_j RN32(v_j * v_j)): the exact sum of the
// FP32 squares, rounded once. The pages fix FP32 math for the norms but leave
// the summation order open; this is the one FP32 value that does not depend
// on an order, and so on the launch shape.
//
// Fast path (every row): an error-free compensated sum. Each thread keeps a
// (sum, compensation) pair per FP32 lane, built with Knuth's TwoSum
// (Knuth, TAOCP vol. 2, 4.2.2, theorem B), on packed f32x2 arithmetic; pairs
// are merged with TwoSum across the two lanes, the warp (xor shuffles) and
// the block (shared memory, fixed order). With all terms >= 0 the
// compensation's error has a rigorous bound E = errk * s (errk from the host:
// it depends on the terms per thread and the merge depth). The rounding of
// s + c is certified when [s + c - E, s + c + E] lies strictly inside the
// rounding interval of RN32(s + c); about one row sum in 10^4 is not, and then
// the exact path decides.
//
// Exact path (rare, or forced): the row is re-read from global memory and the
// sum is formed exactly as a 320-bit integer (each FP32 term is m * 2^q *
// 2^-149 with m < 2^24), held as 32-bit chunk sums in 64-bit registers, added
// across the block, carried, and rounded to nearest-even by hand.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace beam {

// ---------------------------------------------------------------- packed helpers

// two BF16 (low half = lower column) -> two FP32, exactly
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// two FP32 -> two BF16, round to nearest even (NaN -> canonical NaN)
__device__ __forceinline__ uint32_t f2_to_bf2(float2 v) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(v.y), "f"(v.x));
    return d;
}

// Packed FP32 pairs in hand-written PTX with explicit .rn rounding. The
// explicit modifier is meant to keep a multiply and a following add as two
// roundings, yet a packed add fed by a packed product was measured to fuse into
// an FMA on sm_103a. So a packed add here only ever takes products that are
// exact in FP32 (squares of BF16 values), where a fused and a separately
// rounded sum give the same bits; products that are not exact feed
// conversions, or scalar __fadd_rn / __fsub_rn, which are never contracted.
#define BEAM_F32X2_OP(NAME, OP)                                                                  \
    __device__ __forceinline__ float2 NAME(float2 a, float2 b) {                                 \
        float2 d;                                                                                \
        asm("{\n\t.reg .b64 ra, rb, rd;\n\t"                                                    \
            "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t" OP " rd, ra, rb;\n\t"          \
            "mov.b64 {%0, %1}, rd;\n\t}"                                                          \
            : "=f"(d.x), "=f"(d.y)                                                               \
            : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                                          \
        return d;                                                                                \
    }
BEAM_F32X2_OP(mul2_rn, "mul.rn.f32x2")
BEAM_F32X2_OP(add2_rn, "add.rn.f32x2")
BEAM_F32X2_OP(sub2_rn, "sub.rn.f32x2")
#undef BEAM_F32X2_OP

// s + c += t, error-free on (s, e) and accumulated into c, both lanes at once
__device__ __forceinline__ void two_sum_acc2(float2& s, float2& c, float2 t) {
    float2 sn = add2_rn(s, t);
    float2 bp = sub2_rn(sn, s);
    float2 ap = sub2_rn(sn, bp);
    float2 db = sub2_rn(t, bp);
    float2 da = sub2_rn(s, ap);
    c = add2_rn(c, add2_rn(da, db));
    s = sn;
}

// (s, c) += (s2, c2)
__device__ __forceinline__ void ff_merge(float& s, float& c, float s2, float c2) {
    float sn = __fadd_rn(s, s2);
    float bp = __fsub_rn(sn, s);
    float e = __fadd_rn(__fsub_rn(s, __fsub_rn(sn, bp)), __fsub_rn(s2, bp));
    c = __fadd_rn(__fadd_rn(c, c2), e);
    s = sn;
}

// Round s + c_exact to FP32 when |c - c_exact| <= errk * s is known to keep the
// rounding decision; returns false when the exact path must decide.
__device__ __forceinline__ bool certify_round(float s, float c, float errk, float* out) {
    if (s == 0.0f) { *out = 0.0f; return true; }  // all terms zero
    if (!(s > 0x1p-100f) || !(s < 0x1p+126f)) return false;  // tiny, huge or not finite
    float r = __fadd_rn(s, c);
    float d = __fadd_rn(__fsub_rn(s, r), c);  // s - r is exact (Sterbenz)
    float m = __fadd_rn(__fmul_rn(errk, s), __fmul_rn(fabsf(d), 0x1p-22f));
    uint32_t rb = __float_as_uint(r);
    float half_up = 0.5f * (__uint_as_float(rb + 1u) - r);   // spacings are powers of 2: exact
    float half_dn = 0.5f * (r - __uint_as_float(rb - 1u));
    *out = r;
    return (__fsub_rn(d, m) > -half_dn) && (__fadd_rn(d, m) < half_up);
}

// ---------------------------------------------------------------- exact path

struct ExactScratch {            // shared memory of the exact path
    unsigned long long limb[32][9];
};

__device__ unsigned long long g_exact_sum_count;  // diagnostics: exact-path row sums

// bits [pos, pos + n) of the 320-bit little-endian integer L, n <= 32
__device__ __forceinline__ uint32_t limb_bits(const uint32_t (&L)[10], int pos, int n) {
    int idx = pos >> 5, off = pos & 31;
    unsigned long long w = L[idx];
    if (idx + 1 < 10) w |= (unsigned long long)L[idx + 1] << 32;
    return (uint32_t)((w >> off) & ((n == 32) ? 0xFFFFFFFFull : ((1ull << n) - 1ull)));
}

// any bit of L below position pos?
__device__ __forceinline__ bool limb_any_below(const uint32_t (&L)[10], int pos) {
    int idx = pos >> 5, off = pos & 31;
    if (off && (L[idx] & ((1u << off) - 1u))) return true;
    for (int i = 0; i < idx; ++i)
        if (L[i]) return true;
    return false;
}

// N * 2^-149 rounded to nearest even FP32
__device__ __forceinline__ float limbs_to_f32(const uint32_t (&L)[10]) {
    int kt = -1;
    for (int i = 9; i >= 0; --i)
        if (L[i]) { kt = i; break; }
    if (kt < 0) return 0.0f;
    int top = 32 * kt + 31 - __clz(L[kt]);
    if (top <= 23) return __uint_as_float(L[0]);  // subnormal or first binade: exact, bits = N
    int lo = top - 23;
    uint32_t m = limb_bits(L, lo, 24);
    uint32_t half = limb_bits(L, lo - 1, 1);
    bool sticky = limb_any_below(L, lo - 1);
    if (half && (sticky || (m & 1u))) ++m;
    if (m == (1u << 24)) { m >>= 1; ++lo; }
    uint32_t eb = (uint32_t)lo + 1u;
    if (eb >= 255u) return __uint_as_float(0x7F800000u);
    return __uint_as_float((eb << 23) | (m & 0x7FFFFFu));
}

// Exact RN32 sum of squares of a BF16 row in global memory. Called by every
// thread of the block (it synchronises the block). The row may have been
// written earlier in this kernel by this block: it is read through L2.
__device__ __noinline__ float exact_row_sum_squares(const uint16_t* row, int D, ExactScratch* sc) {
    unsigned long long acc[9];
#pragma unroll
    for (int L = 0; L < 9; ++L) acc[L] = 0ull;
    int nan = 0, inf = 0;
    for (int j = threadIdx.x; j < D; j += blockDim.x) {
        uint32_t b = __ldcg(reinterpret_cast<const unsigned short*>(row) + j);
        float xf = __uint_as_float(b << 16);
        float t = __fmul_rn(xf, xf);
        uint32_t u = __float_as_uint(t);
        uint32_t E = (u >> 23) & 0xFFu, f = u & 0x7FFFFFu;
        if (E == 0xFFu) {
            if (f) nan = 1; else inf = 1;
            continue;
        }
        uint32_t M = E ? (f | 0x800000u) : f;  // t = M * 2^q * 2^-149
        uint32_t q = E ? E - 1u : 0u;          // q <= 253
        unsigned long long v = (unsigned long long)M << (q & 31u);
        uint32_t k = q >> 5;                   // k <= 7
        uint32_t lo = (uint32_t)v, hi = (uint32_t)(v >> 32);
#pragma unroll
        for (uint32_t L = 0; L < 9; ++L) {
            acc[L] += (L == k) ? lo : 0u;
            acc[L] += (L == k + 1u) ? hi : 0u;
        }
    }
#pragma unroll
    for (int L = 0; L < 9; ++L)
        for (int off = 16; off; off >>= 1) acc[L] += __shfl_xor_sync(0xFFFFFFFFu, acc[L], off);
    const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if ((threadIdx.x & 31) == 0)
        for (int L = 0; L < 9; ++L) sc->limb[warp][L] = acc[L];
    int any_nan = __syncthreads_or(nan);
    int any_inf = __syncthreads_or(inf);
    float result;
    if (any_nan) {
        result = __uint_as_float(0x7FFFFFFFu);
    } else if (any_inf) {
        result = __uint_as_float(0x7F800000u);
    } else {
        uint32_t Lw[10];
        unsigned long long carry = 0ull;
        for (int L = 0; L < 10; ++L) {
            unsigned long long v = carry;
            if (L < 9)
                for (int w = 0; w < nw; ++w) v += sc->limb[w][L];
            Lw[L] = (uint32_t)v;
            carry = v >> 32;
        }
        result = limbs_to_f32(Lw);
    }
    if (threadIdx.x == 0) atomicAdd(&g_exact_sum_count, 1ull);
    __syncthreads();  // the scratch may be reused by the next call
    return result;
}

}  // namespace beam
