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
// unsigned key), then the lowest expert index holding it. The unbiased scores
// wait in shared memory until the picks are known.
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

constexpr int kRouteWarps = 8;  // tokens per 256-thread block

// The topk rounds over NK keys per lane; key i of a lane is expert base + i,
// and 0 marks a key that is not available. Per round: the lane's best key
// (lowest i among equal keys), the warp's largest key, then the lowest expert
// index that holds it. Every lane records every pick; lane k keeps pick k.
template <int NK>
__device__ __forceinline__ void pick_rounds(uint32_t (&key)[NK], uint32_t base, int topk, int lane,
                                            int (&sel_i)[kRouteMaxTopk], int& my_i) {
    const unsigned full = 0xFFFFFFFFu;
#pragma unroll
    for (int k = 0; k < kRouteMaxTopk; ++k) {
        if (k >= topk) break;
        uint32_t lk = 0u;
        int li = 0;
#pragma unroll
        for (int i = 0; i < NK; ++i)
            if (key[i] > lk) { lk = key[i]; li = i; }
        const uint32_t m = __reduce_max_sync(full, lk);
        const uint32_t e = __reduce_min_sync(full, (lk == m) ? base + (uint32_t)li : 0xFFFFFFFFu);
#pragma unroll
        for (int i = 0; i < NK; ++i)
            if (e == base + (uint32_t)i) key[i] = 0u;
        sel_i[k] = (int)e;
        if (lane == k) my_i = (int)e;
    }
}

// The same rounds over 4 keys per lane (expert base + i), sorted once: then a
// lane's best key is its first, and the lane that wins a round shifts its
// list by one. The sort ranks larger keys first and, among equal keys, the
// lower index, so every round picks what pick_rounds would.
__device__ __forceinline__ void pick_rounds_sorted4(uint32_t (&key)[4], uint32_t base, int topk, int lane,
                                                    int (&sel_i)[kRouteMaxTopk], int& my_i) {
    const unsigned full = 0xFFFFFFFFu;
    uint32_t ix[4] = {0u, 1u, 2u, 3u};
    auto order = [&](int a, int b) {  // afterwards (key[a], ix[a]) ranks before (key[b], ix[b])
        const bool sw = key[b] > key[a] || (key[b] == key[a] && ix[b] < ix[a]);
        const uint32_t ka = sw ? key[b] : key[a], kb = sw ? key[a] : key[b];
        const uint32_t ia = sw ? ix[b] : ix[a], ib = sw ? ix[a] : ix[b];
        key[a] = ka; key[b] = kb; ix[a] = ia; ix[b] = ib;
    };
    order(0, 1); order(2, 3); order(0, 2); order(1, 3); order(1, 2);
    uint32_t ixp = ix[0] | (ix[1] << 2) | (ix[2] << 4) | (ix[3] << 6);  // 2 bits per list entry
#pragma unroll
    for (int k = 0; k < kRouteMaxTopk; ++k) {
        if (k >= topk) break;
        const uint32_t mine = base + (ixp & 3u);
        const uint32_t m = __reduce_max_sync(full, key[0]);
        const uint32_t e = __reduce_min_sync(full, (key[0] == m) ? mine : 0xFFFFFFFFu);
        if (e == mine) {
            key[0] = key[1]; key[1] = key[2]; key[2] = key[3]; key[3] = 0u;
            ixp >>= 2;
        }
        sel_i[k] = (int)e;
        if (lane == k) my_i = (int)e;
    }
}

// NG, TG, K: n_group, topk_group and topk fixed at compile time (0: read from
// the parameters). Fixed values unroll every loop and turn the group arithmetic
// into shifts; the arithmetic on the scores is the same either way. When the
// kept groups hold 128 experts, they are first compacted in shared memory to 4
// per lane and sorted within the lane, which makes each topk round two warp
// reductions and a shift.
template <int NG, int TG, int K>
__global__ void __launch_bounds__(256) route_kernel(const RouteParams p) {
    constexpr bool kCompact = NG > 0 && TG > 0 && TG * (kRouteExperts / (NG > 0 ? NG : 1)) == 128;
    __shared__ __align__(16) float s_all[kRouteWarps][kRouteExperts];  // unbiased scores, per warp
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= p.T) return;  // whole warps leave together
    const unsigned full = 0xFFFFFFFFu;
    const int n_group = NG ? NG : p.n_group;
    const int topk_group = TG ? TG : p.topk_group;
    const int topk = K ? K : p.topk;

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
    float4* mine4 = reinterpret_cast<float4*>(&s_all[warp][8 * lane]);
    mine4[0] = make_float4(s[0], s[1], s[2], s[3]);
    mine4[1] = make_float4(s[4], s[5], s[6], s[7]);

    // ---- group scores: the sum of the two largest biased scores of each group.
    // Only the two values matter, not which experts hold them, so a running
    // (largest, second largest) pair of values suffices.
    float m1 = -INFINITY, m2 = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        m2 = fmaxf(m2, fminf(m1, b[i]));
        m1 = fmaxf(m1, b[i]);
    }
    const int lpg = 32 / n_group;  // lanes per group (a power of two)
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        if (off >= lpg) continue;
        const float o1 = __shfl_xor_sync(full, m1, off), o2 = __shfl_xor_sync(full, m2, off);
        m2 = fmaxf(fminf(m1, o1), fmaxf(m2, o2));
        m1 = fmaxf(m1, o1);
    }
    const float gscore = __fadd_rn(m1, m2);
    const int my_group = lane / lpg;

    // ---- keep the topk_group best groups
    int rank = 0;
#pragma unroll
    for (int g = 0; g < 32; ++g) {
        if (g >= n_group) break;
        const float sg = __shfl_sync(full, gscore, g * lpg);
        rank += ranks_before(sg, g, gscore, my_group) ? 1 : 0;
    }
    const bool eligible = rank < topk_group;

    // ---- topk best biased scores among the eligible experts
    int sel_i[kRouteMaxTopk];
    int my_i = 0;
    if constexpr (kCompact) {
        // the 16 lanes of kept groups write their biased scores to slots 0..15
        // in expert order; lane j then holds experts 4j .. 4j+3 of that order
        __shared__ __align__(16) float ck[kRouteWarps][128];
        __shared__ int cb[kRouteWarps][16];
        const unsigned kept = __ballot_sync(full, eligible);
        if (eligible) {
            const int slot = __popc(kept & ((1u << (my_group * lpg)) - 1u)) + (lane & (lpg - 1));
            float4* dst = reinterpret_cast<float4*>(&ck[warp][8 * slot]);
            dst[0] = make_float4(b[0], b[1], b[2], b[3]);
            dst[1] = make_float4(b[4], b[5], b[6], b[7]);
            cb[warp][slot] = 8 * lane;
        }
        __syncwarp();
        const float4 v = reinterpret_cast<const float4*>(ck[warp])[lane];
        uint32_t key[4] = {order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w)};
        pick_rounds_sorted4(key, (uint32_t)(cb[warp][lane >> 1] + 4 * (lane & 1)), topk, lane, sel_i, my_i);
    } else {
        uint32_t key[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) key[i] = eligible ? order_key(b[i]) : 0u;  // 0: unavailable
        pick_rounds<8>(key, (uint32_t)(8 * lane), topk, lane, sel_i, my_i);
    }

    // ---- weights: unbiased scores of the picks, renormalised in output order
    // (the sum reads the same address in every lane), scaled; lane k < topk
    // writes output k (one division per lane)
    __syncwarp();
    const float* sw = s_all[warp];
    float sum = sw[sel_i[0]];
#pragma unroll
    for (int k = 1; k < kRouteMaxTopk; ++k)
        if (k < topk) sum = __fadd_rn(sum, sw[sel_i[k]]);
    if (lane < topk) {
        p.idx[t * topk + lane] = my_i;
        p.w[t * topk + lane] = __fmul_rn(__fdiv_rn(sw[my_i], sum), p.scale);
    }
}

}  // namespace beam
