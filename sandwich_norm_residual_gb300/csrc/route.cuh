// Group-limited top-k routing in front of the MoE combine, sm_103a.
//
// Per token (vLLM page, "MoE and residual stream"; SGLang page, "Dense layers
// and grouped MoE routing"), FP32 throughout:
//   s_e = RN32(1 / (1 + e^-z_e))     sigmoid of the FP32 router logit, the
//                                    correctly rounded value (router_sigmoid.cuh)
//   b_e = s_e + bias_e               biased score, used only to choose experts
//   group score = top1 + top2 of the b_e in the group (the routing matches
//                 DeepSeek-V3, whose group score is the sum of the group's two
//                 best biased scores)
//   keep the topk_group best groups, then the topk best experts among them;
//   ties go to the lower index and the output is in descending b_e
//   w_k = (s_k / sum_k s_k) * scale, the sum taken in output order
// Scores are ranked on one total order: larger first, a NaN below every
// number, equal scores (and NaNs) by index. So exactly topk_group groups and
// topk experts are chosen whatever the logits and the bias hold.
//
// One warp per token; lane l holds experts 8l .. 8l+7 (256 experts), so a group
// of 256/n_group experts spans 32/n_group neighbouring lanes. Each top-k round
// is two warp reductions: the largest biased score (as an order-preserving
// unsigned key), then the lowest expert index holding it. The unbiased scores
// wait in shared memory until the picks are known.
#pragma once

#include <cstdint>

#include "router_sigmoid.cuh"
#include "tma.cuh"

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

// unsigned key that orders like the float, with every NaN at 1, below the key
// of -inf (0x007FFFFF); 0 is left free to mark an unavailable entry. -0 and +0
// differ, but a biased score s + bias is never -0 since s is never -0, and
// neither is a sum of two of them.
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t b = __float_as_uint(v);
    if (v != v) return 1u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// the float of a key (a NaN for key 1)
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
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

// Bound on |b' - b| for a biased score b' = RN32(s' + bias) formed from the
// fast sigmoid s' instead of the exact s: |s' - s| < kFastSigmoidSlack, plus
// two ulps of b for the two roundings of the sum, plus the subnormal spacing.
__device__ __forceinline__ float score_slack(float b) {
    return __fmaf_rn(fabsf(b), 0x1p-22f, kFastSigmoidSlack + 0x1p-148f);
}

// NG, TG, K: n_group, topk_group and topk fixed at compile time (0: read from
// the parameters). Fixed values unroll every loop and turn the group arithmetic
// into shifts; the arithmetic on the scores is the same either way. When the
// kept groups hold 128 experts, they are first compacted in shared memory to 4
// per lane and sorted within the lane, which makes each topk round two warp
// reductions and a shift.
//
// Two passes, the first usually final. Fast pass: every score from the fast
// FP32 sigmoid s' (router_sigmoid_fast, within 2^-19 of the exact sigmoid on
// every float input), so every biased score, group score and pick carries a
// known slack. The choice is accepted when
// the slack cannot change it: every kept group's score interval lies above
// every dropped group's, every pick's above every eligible expert left out,
// and consecutive picks' intervals are disjoint, so the order of the output is
// fixed too. Then only the picks' exact sigmoids are computed (the weights
// need them). Exact pass (a logit or bias is NaN, or an interval test failed,
// for instance on exactly tied scores): every score exact, as defined.
template <int NG, int TG, int K>
__global__ void __launch_bounds__(256, 5) route_kernel(const RouteParams p) {
    constexpr bool kCompact = NG > 0 && TG > 0 && TG * (kRouteExperts / (NG > 0 ? NG : 1)) == 128;
    __shared__ __align__(16) float zs[kRouteWarps][kRouteExperts];  // logits; unbiased scores in the exact pass
    __shared__ __align__(16) float bs[kRouteWarps][kRouteExperts];  // fast biased scores
    __shared__ __align__(16) uint32_t ck[kRouteWarps][128];
    __shared__ int cb[kRouteWarps][16];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    // with a programmatic launch the next kernel on the stream may start its
    // own prologue now; this one reads nothing until the previous kernel is done
    pdl_trigger();
    if (t >= p.T) return;  // whole warps leave together
    const unsigned full = 0xFFFFFFFFu;
    const int n_group = NG ? NG : p.n_group;
    const int topk_group = TG ? TG : p.topk_group;
    const int topk = K ? K : p.topk;
    const int lpg = 32 / n_group;  // lanes per group (a power of two)
    const int my_group = lane / lpg;

    const SigmoidLane lt = sigmoid_lane_table();  // a constant table: readable before the wait
    pdl_wait();
    const float4* z4 = reinterpret_cast<const float4*>(p.logits + t * kRouteExperts + 8 * lane);
    const float4* b4 = reinterpret_cast<const float4*>(p.bias + 8 * lane);
    const float4 za = __ldg(z4), zb = __ldg(z4 + 1), ba = __ldg(b4), bb = __ldg(b4 + 1);
    const float z[8] = {za.x, za.y, za.z, za.w, zb.x, zb.y, zb.z, zb.w};
    const float bias[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
    float4* zrow = reinterpret_cast<float4*>(&zs[warp][8 * lane]);
    zrow[0] = za;
    zrow[1] = zb;

    int sel_i[kRouteMaxTopk];
    int my_i = 0;
    bool eligible = false;
    uint32_t gkey = 0u, rest = 0u;

    // The choice from the keys of this lane's 8 biased scores: group scores
    // (sum of the two largest of each group: only the two values matter, so a
    // running pair of keys suffices), the topk_group best groups on one total
    // order (ties to the lower group), then the topk best eligible experts.
    // Leaves in `rest` the key of the best eligible expert left out (0: none).
    auto choose = [&](const uint32_t (&bk)[8]) {
        uint32_t m1 = 0u, m2 = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            m2 = max(m2, min(m1, bk[i]));
            m1 = max(m1, bk[i]);
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            if (off >= lpg) continue;
            const uint32_t o1 = __shfl_xor_sync(full, m1, off), o2 = __shfl_xor_sync(full, m2, off);
            m2 = max(min(m1, o1), max(m2, o2));
            m1 = max(m1, o1);
        }
        // every group has at least 8 experts (n_group <= 32): m1, m2 are real keys
        gkey = order_key(__fadd_rn(key_value(m1), key_value(m2)));
        // topk_group rounds of two warp reductions: the largest key among the
        // groups not yet kept, then the lowest group index holding it (every
        // lane of a group holds its group's key; keys are never 0)
        eligible = false;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            if (r >= topk_group) break;
            const uint32_t m = __reduce_max_sync(full, eligible ? 0u : gkey);
            const uint32_t gw = __reduce_min_sync(full, (!eligible && gkey == m) ? (uint32_t)my_group : 0xFFFFFFFFu);
            eligible |= (uint32_t)my_group == gw;
        }
        if constexpr (kCompact) {
            // the 16 lanes of kept groups write their keys to slots 0..15 in
            // expert order; lane j then holds experts 4j .. 4j+3 of that order.
            // Exactly 16 lanes are kept (4 whole groups of 4 lanes), so
            // slot < 16; the bound is checked all the same before the writes.
            const unsigned kept = __ballot_sync(full, eligible);
            const int slot = __popc(kept & ((1u << (my_group * lpg)) - 1u)) + (lane & (lpg - 1));
            if (eligible && slot < 16) {
                uint4* dst = reinterpret_cast<uint4*>(&ck[warp][8 * slot]);
                dst[0] = make_uint4(bk[0], bk[1], bk[2], bk[3]);
                dst[1] = make_uint4(bk[4], bk[5], bk[6], bk[7]);
                cb[warp][slot] = 8 * lane;
            }
            __syncwarp();
            const uint4 v = reinterpret_cast<const uint4*>(ck[warp])[lane];
            uint32_t key[4] = {v.x, v.y, v.z, v.w};
            pick_rounds_sorted4(key, (uint32_t)(cb[warp][lane >> 1] + 4 * (lane & 1)), topk, lane, sel_i, my_i);
            rest = __reduce_max_sync(full, key[0]);  // lists stay sorted: the first is the best left
            __syncwarp();                            // ck and cb are reused by a later call
        } else {
            uint32_t key[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) key[i] = eligible ? bk[i] : 0u;  // 0: unavailable
            pick_rounds<8>(key, (uint32_t)(8 * lane), topk, lane, sel_i, my_i);
            uint32_t mk = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) mk = max(mk, key[i]);
            rest = __reduce_max_sync(full, mk);
        }
    };

    // ---- fast pass
    bool finite_in = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) finite_in &= (z[i] == z[i]) && (bias[i] == bias[i]);
    if (__all_sync(full, finite_in)) {
        uint32_t bk[8];
        float bv[8], amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float sf = router_sigmoid_fast(z[i]);
            bv[i] = __fadd_rn(sf, bias[i]);
            bk[i] = order_key(bv[i]);
            amax = fmaxf(amax, fabsf(bv[i]));
        }
        float4* brow = reinterpret_cast<float4*>(&bs[warp][8 * lane]);
        brow[0] = make_float4(bv[0], bv[1], bv[2], bv[3]);
        brow[1] = make_float4(bv[4], bv[5], bv[6], bv[7]);
        choose(bk);
        // groups: the kept ones' score intervals above the dropped ones'
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            if (off >= lpg) continue;
            amax = fmaxf(amax, __shfl_xor_sync(full, amax, off));
        }
        const float g = key_value(gkey);
        const float dg = __fadd_rn(__fmul_rn(2.0f, score_slack(amax)), score_slack(g));
        const float glo = eligible ? __fsub_rn(g, dg) : INFINITY;
        const float ghi = eligible ? -INFINITY : __fadd_rn(g, dg);
        // picks: each pick's interval above the next pick's and above the best
        // eligible expert left out
        __syncwarp();
        const float bsel = lane < topk ? bs[warp][my_i] : 0.0f;
        const float bnext = __shfl_down_sync(full, bsel, 1);
        const float slo = lane < topk ? __fsub_rn(bsel, score_slack(bsel)) : INFINITY;
        const float rv = key_value(rest);
        const float rhi = rest ? __fadd_rn(rv, score_slack(rv)) : -INFINITY;
        bool ok = glo == glo && ghi == ghi && slo == slo && rhi == rhi;
        ok &= (lane + 1 >= topk) || slo > __fadd_rn(bnext, score_slack(bnext));
        const float glo_min = key_value(__reduce_min_sync(full, order_key(glo)));
        const float ghi_max = key_value(__reduce_max_sync(full, order_key(ghi)));
        const float slo_min = key_value(__reduce_min_sync(full, order_key(slo)));
        ok &= glo_min > ghi_max && slo_min > rhi;
        if (__all_sync(full, ok)) {
            // the choice is the exact one: the picks' exact sigmoids give the weights
            const float sk = router_sigmoid(lane < topk ? zs[warp][my_i] : 0.0f, lt);
            float sum = __shfl_sync(full, sk, 0);
#pragma unroll
            for (int k = 1; k < kRouteMaxTopk; ++k)
                if (k < topk) sum = __fadd_rn(sum, __shfl_sync(full, sk, k));
            if (lane < topk) {
                p.idx[t * topk + lane] = my_i;
                p.w[t * topk + lane] = __fmul_rn(__fdiv_rn(sk, sum), p.scale);
            }
            return;
        }
    }

    // ---- exact pass: every score exact
    float sv[8];
    uint32_t bk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        sv[i] = router_sigmoid(z[i], lt);
        bk[i] = order_key(__fadd_rn(sv[i], bias[i]));
    }
    __syncwarp();
    zrow[0] = make_float4(sv[0], sv[1], sv[2], sv[3]);
    zrow[1] = make_float4(sv[4], sv[5], sv[6], sv[7]);
    choose(bk);
    // weights: unbiased scores of the picks, renormalised in output order (the
    // sum reads the same address in every lane), scaled; lane k < topk writes
    // output k (one division per lane)
    __syncwarp();
    const float* sw = zs[warp];
    float sum = sw[sel_i[0]];
#pragma unroll
    for (int k = 1; k < kRouteMaxTopk; ++k)
        if (k < topk) sum = __fadd_rn(sum, sw[sel_i[k]]);
    if (lane < topk) {
        p.idx[t * topk + lane] = my_i;
        p.w[t * topk + lane] = __fmul_rn(__fdiv_rn(sw[my_i], sum), p.scale);
    }
}

// The router's sigmoid alone, elementwise: s[i] = RN32(1 / (1 + e^-z[i])),
// or (fast) the first pass's approximation. Whole warps iterate together (the
// exact sigmoid reads its table by shuffle).
__global__ void __launch_bounds__(256) router_sigmoid_kernel(const float* z, float* s, long long n, int fast) {
    const SigmoidLane lt = sigmoid_lane_table();
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long base = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < n; base += stride) {
        const long long i = base + (threadIdx.x & 31);
        const float zi = i < n ? z[i] : 0.0f;
        const float si = fast ? router_sigmoid_fast(zi) : router_sigmoid(zi, lt);
        if (i < n) s[i] = si;
    }
}

}  // namespace beam
