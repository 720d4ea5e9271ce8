// Group-limited top-k routing in front of the MoE combine, sm_103a.
//
// Per token (vLLM page, "MoE and residual stream"; SGLang page, "Dense layers
// and grouped MoE routing"), FP32 throughout:
//   s_e = 1 / (1 + exp(-z_e))        sigmoid of the FP32 router logit
//   b_e = s_e + bias_e               biased score, used only to choose experts
//   group score = top1 + top2 of the b_e in the group (the routing matches
//                 DeepSeek-V3, whose group score is the sum of the group's two
//                 best biased scores)
//   keep the topk_group best groups, then the topk best experts among them;
//   ties go to the lower index and the output is in descending b_e
//   w_k = (s_k / sum_k s_k) * scale, the sum taken in output order
//
// One warp per token; lane l holds experts 8l .. 8l+7 (256 experts), so a group
// of 256/n_group experts spans 32/n_group neighbouring lanes. Each top-k round
// is two warp reductions: the largest biased score (as an order-preserving
// unsigned key), then the lowest expert index holding it.
#pragma once

#include <cstdint>

namespace beam {

constexpr int kRouteExperts = 256;
constexpr int kRouteMaxTopk = 16;

struct RouteParams {
    const float* logits;  // [T, 256]
    const float* bias;    // [256]
    int32_t* idx;         // [T, topk]
    float* w;             // [T, topk]
    long long T;
    int n_group, topk_group, topk;
    float scale;
};

// (v1, i1) ranks before (v2, i2): larger value, then lower index
__device__ __forceinline__ bool ranks_before(float v1, int i1, float v2, int i2) {
    return v1 > v2 || (v1 == v2 && i1 < i2);
}

// unsigned key that orders like the float (never 0 for a non-NaN value; -0 and
// +0 differ, but a biased score s + bias is never -0 since s is never -0)
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(256) route_kernel(const RouteParams p) {
    const int lane = threadIdx.x & 31;
    const long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= p.T) return;  // whole warps leave together
    const unsigned full = 0xFFFFFFFFu;

    const float4* z4 = reinterpret_cast<const float4*>(p.logits + t * kRouteExperts + 8 * lane);
    const float4* b4 = reinterpret_cast<const float4*>(p.bias + 8 * lane);
    const float4 za = __ldg(z4), zb = __ldg(z4 + 1), ba = __ldg(b4), bb = __ldg(b4 + 1);
    const float z[8] = {za.x, za.y, za.z, za.w, zb.x, zb.y, zb.z, zb.w};
    const float bias[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
    float s[8], b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        s[i] = __frcp_rn(__fadd_rn(1.0f, expf(-z[i])));  // RN(1 / (1 + e)), as a division
        b[i] = __fadd_rn(s[i], bias[i]);
    }

    // ---- group scores: the two best biased scores of each group
    float m1 = -INFINITY, m2 = -INFINITY;
    int i1 = 0x7FFFFFFF, i2 = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = 8 * lane + i;
        if (ranks_before(b[i], e, m1, i1)) {
            m2 = m1; i2 = i1; m1 = b[i]; i1 = e;
        } else if (ranks_before(b[i], e, m2, i2)) {
            m2 = b[i]; i2 = e;
        }
    }
    const int lpg = 32 / p.n_group;  // lanes per group (a power of two)
    for (int off = lpg >> 1; off; off >>= 1) {
        const float o1 = __shfl_xor_sync(full, m1, off), o2 = __shfl_xor_sync(full, m2, off);
        const int j1 = __shfl_xor_sync(full, i1, off), j2 = __shfl_xor_sync(full, i2, off);
        if (ranks_before(o1, j1, m1, i1)) {  // the other list leads
            if (ranks_before(m1, i1, o2, j2)) { m2 = m1; i2 = i1; } else { m2 = o2; i2 = j2; }
            m1 = o1; i1 = j1;
        } else if (ranks_before(o1, j1, m2, i2)) {
            m2 = o1; i2 = j1;
        }
    }
    const float gscore = __fadd_rn(m1, m2);
    const int my_group = lane / lpg;

    // ---- keep the topk_group best groups
    int rank = 0;
    for (int g = 0; g < p.n_group; ++g) {
        const float sg = __shfl_sync(full, gscore, g * lpg);
        rank += ranks_before(sg, g, gscore, my_group) ? 1 : 0;
    }
    const bool eligible = rank < p.topk_group;

    // ---- topk best biased scores among eligible experts: per round, the best
    // key of each lane (lowest local index among equal keys), the warp's
    // largest key, then the lowest expert index that holds it
    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) key[i] = eligible ? order_key(b[i]) : 0u;  // 0: unavailable
    int sel_i[kRouteMaxTopk];
#pragma unroll
    for (int k = 0; k < kRouteMaxTopk; ++k) {
        if (k >= p.topk) break;
        uint32_t lk = 0u;
        int li = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (key[i] > lk) { lk = key[i]; li = i; }
        const uint32_t m = __reduce_max_sync(full, lk);
        const uint32_t e = __reduce_min_sync(full, (lk == m) ? (uint32_t)(8 * lane + li) : 0xFFFFFFFFu);
        if ((int)(e >> 3) == lane) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i == (int)(e & 7u)) key[i] = 0u;
        }
        sel_i[k] = (int)e;
    }
    // the unbiased score of each pick, from the lane that holds it
    float sel_s[kRouteMaxTopk];
#pragma unroll
    for (int k = 0; k < kRouteMaxTopk; ++k) {
        if (k >= p.topk) break;
        const int e = sel_i[k];
        float mine = s[0];
#pragma unroll
        for (int i = 1; i < 8; ++i)
            if (i == (e & 7)) mine = s[i];
        sel_s[k] = __shfl_sync(full, mine, e >> 3);
    }

    // ---- weights: unbiased scores, renormalised in output order, scaled; lane
    // k < topk writes output k (one division per lane)
    float sum = sel_s[0];
#pragma unroll
    for (int k = 1; k < kRouteMaxTopk; ++k)
        if (k < p.topk) sum = __fadd_rn(sum, sel_s[k]);
    float my_s = sel_s[0];
    int my_i = sel_i[0];
#pragma unroll
    for (int k = 1; k < kRouteMaxTopk; ++k)
        if (k < p.topk && lane == k) { my_s = sel_s[k]; my_i = sel_i[k]; }
    if (lane < p.topk) {
        p.idx[t * p.topk + lane] = my_i;
        p.w[t * p.topk + lane] = __fmul_rn(__fdiv_rn(my_s, sum), p.scale);
    }
}

}  // namespace beam
