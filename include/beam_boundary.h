/*
 * libbeamboundary -- the fused sublayer boundary of the Beam decoder on one
 * NVIDIA GB300 (sm_103a) GPU.
 *
 * At each of the decoder's 104 sublayer boundaries (52 layers x attention and
 * feed-forward) three steps run as one kernel:
 *
 *   1. post-RMSNorm of the branch output x                     -> xn (BF16)
 *   2. depth-scaled residual add, n-th add:
 *        h <- bf16( bf16(c1 * h) + bf16(c2 * xn) ),
 *        c1 = RN32(sqrt((n-1)/n)), c2 = RN32(1/sqrt(n))
 *   3. pre-RMSNorm of the new stream for the next sublayer     -> y  (BF16)
 *
 * Sources (Beam blog pages):
 *   - sandwich norm, an RMSNorm before and after every sublayer, and the
 *     residual rule h <- sqrt((n-1)/n) h + x/sqrt(n): vLLM page, "MoE and
 *     residual stream"; SGLang page, "Sandwich normalization and
 *     depth-scaled residual" (which also states that both scaled operands
 *     are rounded to the activation dtype before the add, and that the
 *     unfused transition writes the normalised branch, reads it for the
 *     residual combine and reads the result again for the next input norm);
 *   - one fused kernel with FP32 math and the reference implementation's
 *     BF16 rounding points: vLLM page, "Agent-driven optimization", change 1;
 *   - the MoE variant, where the same norm kernel first combines the top-8
 *     expert outputs: vLLM page, change 3; SGLang page, "Fusion
 *     optimizations" (local expert sum, routing scale and BF16 rounding in
 *     one path) and "Dense layers and grouped MoE routing" (FP32 routing
 *     coefficients, the routing scale carried in the routing weights).
 *
 * Arithmetic, per token row, all FP32 with IEEE round-to-nearest-even:
 *   RMSNorm(v, w)_j = bf16( (v_j * r) * w_j ),  r = 1 / sqrt(S/D + eps),
 *   S = the exact sum of the FP32 squares v_j * v_j, rounded once to FP32.
 *   The pages leave the summation order open and accept FP32 order
 *   differences; this library returns the order-free value (an error-free
 *   compensated sum whose rounding is certified per row, with an exact
 *   integer fallback), so results do not depend on launch shape.
 *   MoE: x_j = bf16(acc_j), acc_j = fma chain over k = 0..7 of w[t,k]*e[t,k,j].
 *
 * Data layout: every tensor is dense, row-major, token-major.
 *   BF16 values are passed as their 16-bit patterns (uint16_t).
 *   h, x, y_out:  [T, D]       expert_out: [T, 8, D]      topk_w: [T, 8] FP32
 *   post_w, pre_w: [D]
 * All pointers are DEVICE pointers on the current device (or managed memory),
 * except in the *_host calls, which also take page-locked host memory. The
 * device calls check no pointer's memory type (that would cost a driver call
 * per launch): pass host memory only to the *_host calls.
 * Every pointer must be 16-byte aligned; D must be a multiple of 8 with
 * 8 <= D <= BEAM_MAX_D.
 *
 * Ownership: the caller owns every buffer. The library allocates no device or
 * host memory in any call and keeps no per-call state. Per device it keeps a
 * small status word and a counter in static device memory (see
 * beam_sync_status).
 *
 * Streams: calls are asynchronous on the given stream (NULL = the legacy
 * default stream). Calls may be made from several host threads.
 *
 * Errors: argument errors are returned before anything is launched and leave
 * every buffer untouched. A failed launch returns BEAM_ERR_CUDA. Errors
 * raised inside a kernel (a bounded wait that gave up) set the device status
 * word, reported by beam_sync_status. No C++ exception crosses this ABI.
 */
#ifndef BEAM_BOUNDARY_H
#define BEAM_BOUNDARY_H

#include <stdint.h>

#if defined(__GNUC__)
#define BEAM_API __attribute__((visibility("default")))
#else
#define BEAM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef struct CUstream_st* beam_stream_t;

typedef enum {
    BEAM_OK = 0,
    BEAM_ERR_NULL = 1,    /* a required pointer is NULL (T > 0) */
    BEAM_ERR_ALIGN = 2,   /* a pointer is not 16-byte aligned */
    BEAM_ERR_SHAPE = 3,   /* T < 0, D not a multiple of 8, D < 8, D > BEAM_MAX_D, T*D too large */
    BEAM_ERR_ARG = 4,     /* n < 1, or eps negative / not finite, or a bad option */
    BEAM_ERR_ALIAS = 5,   /* y_out overlaps another operand, or h partly overlaps an input */
    BEAM_ERR_CUDA = 6,    /* a CUDA runtime call failed (device query, launch, sync) */
    BEAM_ERR_TIMEOUT = 7, /* a bounded device-side wait gave up (see beam_sync_status) */
    BEAM_ERR_DEVICE = 8   /* the current device is not an sm_103 GPU */
} beam_status;

/* Largest supported hidden size. */
#define BEAM_MAX_D 32768
/* Experts combined per token by beam_moe_combine_boundary (top-8 routing). */
#define BEAM_MOE_TOPK 8

/*
 * Dense boundary: post-RMSNorm of x, depth-scaled residual into h (in place),
 * pre-RMSNorm of the new h into y_out.
 *   h      [T, D] BF16, read and overwritten with h'
 *   x      [T, D] BF16 branch output; may be the same pointer as h (then the
 *          branch is the old stream); any other overlap with h is an error
 *   post_w [D] BF16 weight of the post-norm; pre_w [D] BF16 weight of the
 *          next sublayer's pre-norm
 *   n      index of this residual add, n >= 1 (n = 1 makes h' = xn)
 *   eps    RMSNorm epsilon, finite and >= 0
 *   T      token rows (T = 0 returns BEAM_OK and launches nothing; the
 *          pointers are then not checked)
 *   y_out  [T, D] BF16, must not overlap h, x, post_w or pre_w
 */
BEAM_API beam_status beam_boundary_fused(beam_stream_t stream, uint16_t* h, const uint16_t* x,
                                const uint16_t* post_w, const uint16_t* pre_w, int n, float eps,
                                int64_t T, int D, uint16_t* y_out);

/*
 * MoE boundary: x = bf16(sum_k topk_w[t,k] * expert_out[t,k,:]) (FP32 fma
 * chain, k ascending), then the dense boundary on that x.
 *   expert_out [T, 8, D] BF16: the token's 8 routed expert outputs, contiguous
 *   topk_w     [T, 8] FP32 routing weights with the routing scale (2.5 for
 *              Beam) and renormalisation already applied
 *   other arguments as beam_boundary_fused; y_out must not overlap h,
 *   expert_out, topk_w or the weights, and h must not overlap expert_out.
 */
BEAM_API beam_status beam_moe_combine_boundary(beam_stream_t stream, uint16_t* h,
                                      const uint16_t* expert_out, const float* topk_w,
                                      const uint16_t* post_w, const uint16_t* pre_w, int n,
                                      float eps, int64_t T, int D, uint16_t* y_out);

/*
 * MoE boundary with the routing scale applied in the combine (SGLang page,
 * "Dense layers and grouped MoE routing": the scale is applied while the
 * experts are combined, or carried in the weights). topk_w are the
 * renormalised routing weights without the scale;
 *   x = bf16(RN32(route_scale * acc)),  acc as in beam_moe_combine_boundary.
 * With route_scale = 1 this is beam_moe_combine_boundary. route_scale must be
 * finite; other arguments and errors as beam_moe_combine_boundary.
 */
BEAM_API beam_status beam_moe_combine_boundary_scaled(beam_stream_t stream, uint16_t* h,
                                             const uint16_t* expert_out, const float* topk_w,
                                             float route_scale, const uint16_t* post_w,
                                             const uint16_t* pre_w, int n, float eps, int64_t T,
                                             int D, uint16_t* y_out);

/* Router width and the largest top-k of beam_moe_route. */
#define BEAM_ROUTE_EXPERTS 256
#define BEAM_ROUTE_MAX_TOPK 16

/*
 * Group-limited top-k routing in front of the MoE combine (vLLM page, "MoE
 * and residual stream": sigmoid scores plus a correction bias pick the best 4
 * of 8 expert groups, then the top 8 experts, and the renormalised weights are
 * scaled by 2.5; SGLang page, "Dense layers and grouped MoE routing": FP32
 * logits and coefficients). Per token, FP32:
 *   s_e = 1 / (1 + exp(-logit_e)),  b_e = s_e + bias_e
 *   group score = sum of the group's two best b_e (the DeepSeek-V3 rule the
 *   pages say Beam follows); keep the topk_group best of n_group groups;
 *   take the topk best b_e among their experts, in descending order (ties to
 *   the lower index);  topk_w[k] = (s_k / sum of the chosen s) * route_scale,
 *   the sum taken in output order.
 *   logits   [T, E] FP32 router logits, E = BEAM_ROUTE_EXPERTS; 16-byte aligned
 *   bias     [E] FP32 correction bias; 16-byte aligned
 *   n_group  1, 2, 4, 8, 16 or 32 (Beam: 8); topk_group in [1, n_group] (Beam: 4)
 *   topk     in [1, BEAM_ROUTE_MAX_TOPK] and at most topk_group * E / n_group (Beam: 8)
 *   topk_idx [T, topk] int32 expert ids, topk_w [T, topk] FP32; 4-byte aligned,
 *            overlapping neither each other nor the inputs
 * s_e is the correctly rounded FP32 sigmoid (see beam_router_sigmoid), so the
 * chosen experts and the weights are the exact FP32 results of these steps.
 * Scores are ranked on one total order: larger first, a NaN score below every
 * number, equal scores (and NaNs) by index; so exactly topk experts from
 * exactly topk_group groups are chosen whatever the logits and bias hold.
 */
BEAM_API beam_status beam_moe_route(beam_stream_t stream, const float* logits, const float* bias,
                                    int64_t T, int E, int n_group, int topk_group, int topk,
                                    float route_scale, int32_t* topk_idx, float* topk_w);

/*
 * beam_moe_route with BEAM_OPT_* flags: BEAM_OPT_PDL launches the kernel with
 * programmatic stream serialisation, so that it may start while the previous
 * kernel on the stream finishes; it reads its inputs only after that kernel
 * has completed. Any other flag gives BEAM_ERR_ARG.
 */
BEAM_API beam_status beam_moe_route_ex(beam_stream_t stream, const float* logits, const float* bias,
                                       int64_t T, int E, int n_group, int topk_group, int topk,
                                       float route_scale, int32_t* topk_idx, float* topk_w,
                                       uint32_t flags);

/*
 * The router's FP32 sigmoid alone, elementwise (vLLM page, "MoE and residual
 * stream": expert scores are the sigmoid of the router logits; SGLang page,
 * "Dense layers and grouped MoE routing": FP32 routing). s[i] is the float
 * nearest 1 / (1 + e^-z[i]), the exact sigmoid rounded once to nearest-even,
 * for every float input: +-0 -> 0.5, +inf -> 1, -inf -> +0, NaN -> NaN, and a
 * subnormal where the value is one. beam_moe_route scores with this same
 * function.
 *   z, s   [count] FP32 device arrays, 4-byte aligned; s may be z itself
 *          (in place) but must not overlap it otherwise
 *   count  >= 0 (0 launches nothing)
 */
BEAM_API beam_status beam_router_sigmoid(beam_stream_t stream, const float* z, float* s, int64_t count);

/*
 * The fast FP32 sigmoid of beam_moe_route's first pass, elementwise (the
 * pass that chooses the experts when interval tests show the choice cannot
 * change; see beam_moe_route). Not correctly rounded: s[i] lies within 2^-19
 * of the exact sigmoid for every float input, NaN gives NaN. Exposed so that
 * this bound can be checked; arguments and errors as beam_router_sigmoid.
 */
BEAM_API beam_status beam_router_sigmoid_fast(beam_stream_t stream, const float* z, float* s, int64_t count);

/* Head dimension and modes of beam_qk_norm. */
#define BEAM_QK_HEAD_DIM 128
#define BEAM_QK_ROPE 0
#define BEAM_QK_SSMAX 1

/*
 * Per-head Q/K RMSNorm with RoPE or SSMax, in place (vLLM page, "Beam model
 * architecture": Q and K are RMS-normalised per head before RoPE (sliding-
 * window layers) or SSMax (full-attention layers, which scale each query by
 * (1 + p/2048)^0.1, p the 1-based position); 48 query and 8 KV heads of 128).
 * Per head row v, FP32 math:
 *   vn = bf16((v * r) * w), r = 1/sqrt(RN32(exact sum of v^2)/128 + eps), w = q_w or k_w
 *   BEAM_QK_ROPE:  rotate-half pairs (j, j+64) with c = rope_table[pos][j],
 *     s = rope_table[pos][64 + j]: out_j = bf16(RN32(vn_j c) - RN32(vn_{j+64} s)),
 *     out_{j+64} = bf16(RN32(vn_{j+64} c) + RN32(vn_j s)); queries and keys.
 *   BEAM_QK_SSMAX: queries out = bf16(RN32(vn * g)),
 *     g = RN32((1 + (pos + 1)/2048)^0.1) (pos 0-based, correctly rounded;
 *     pos at most 2^24 - 2050); keys out = vn.
 *   q [T, n_q_heads, 128], k [T, n_kv_heads, 128] BF16, overwritten; 16-byte aligned
 *   q_w, k_w [128] BF16 norm weights; pos [T] int32 0-based positions
 *   rope_table [max_pos, 128] FP32 (cos | sin), required for BEAM_QK_ROPE
 *   head_dim must be BEAM_QK_HEAD_DIM; eps finite >= 0.
 * A token whose position is negative, not below max_pos (RoPE) or beyond the
 * SSMax limit is left
 * untouched and beam_sync_status then returns BEAM_ERR_ARG.
 */
BEAM_API beam_status beam_qk_norm(beam_stream_t stream, uint16_t* q, uint16_t* k,
                                  const uint16_t* q_w, const uint16_t* k_w, const int32_t* pos,
                                  const float* rope_table, int64_t max_pos, int64_t T,
                                  int n_q_heads, int n_kv_heads, int head_dim, float eps,
                                  int mode);

/* beam_qk_norm with BEAM_OPT_* flags: BEAM_OPT_FORCE_EXACT_SUM, and BEAM_OPT_PDL
 * (a programmatic dependent launch: the kernel asks L2 for its tokens' rows,
 * a hint that reads no data, then waits for the previous kernel on the stream
 * before it reads q, k or pos). */
BEAM_API beam_status beam_qk_norm_ex(beam_stream_t stream, uint16_t* q, uint16_t* k,
                                     const uint16_t* q_w, const uint16_t* k_w, const int32_t* pos,
                                     const float* rope_table, int64_t max_pos, int64_t T,
                                     int n_q_heads, int n_kv_heads, int head_dim, float eps,
                                     int mode, uint32_t flags);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word. Returns BEAM_OK; BEAM_ERR_TIMEOUT if a kernel's bounded wait gave up
 * since the last read; BEAM_ERR_ARG if beam_qk_norm met a position out of
 * range; or BEAM_ERR_CUDA if the synchronisation failed. The word is shared
 * by all streams and threads using the device.
 */
BEAM_API beam_status beam_sync_status(beam_stream_t stream);

/* Short English text for a status code (static storage, never NULL). */
BEAM_API const char* beam_status_string(beam_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
BEAM_API int beam_version(void);

/* ---------------------------------------------------------------------------
 * Tuning and test hooks. The plain calls above use automatic choices; these
 * variants let benchmarks and tests fix them. Same arguments and errors as the
 * plain calls, plus `opts` (NULL = automatic).
 * ------------------------------------------------------------------------ */
typedef struct {
    uint32_t flags;         /* BEAM_OPT_* bits */
    int32_t vec_per_thread; /* 16-byte vectors per thread per row, 0 = automatic; 1..8 */
    int32_t ctas_per_sm;    /* resident CTAs per SM for the persistent grid, 0 = automatic */
    int32_t prefetch_rows;  /* kernels loading straight to registers: rows ahead (per CTA)
                               whose inputs are bulk-prefetched into L2;
                               0 = automatic, -1 = none, 1..8 */
    int32_t stages;         /* dense boundary: shared-memory ring slots per CTA fed by bulk
                               copies, 2..8; -1 = no ring (loads straight to registers);
                               0 = automatic (no ring, which measured faster at D = 5120,
                               unless BEAM_OPT_TEST_WAIT_TIMEOUT asks for the ring) */
    int32_t reserved[3];    /* must be 0 */
} beam_launch_opts;

/* Take the exact integer row-sum path for every row instead of only for rows
 * whose compensated sum cannot be certified (results are identical). */
#define BEAM_OPT_FORCE_EXACT_SUM 0x1u
/* Test hook for the bounded waits (dense boundary, ring kernel only): the bulk
 * copy of each CTA's second row is never issued, so the wait for that row gives
 * up after 1 ms. The CTA then stores nothing for that row or its later rows
 * (h and y keep what they held), waits for its copies in flight and returns;
 * the device status word records it and beam_sync_status returns
 * BEAM_ERR_TIMEOUT. Each CTA's first row is computed as usual. */
#define BEAM_OPT_TEST_WAIT_TIMEOUT 0x2u
/* Programmatic dependent launch (the following norm loads its weights before
 * its dependency wait: SGLang page, "Fusion optimizations"). The kernel may
 * start while the previous kernel on the stream is still running: it reads
 * post_w and pre_w and asks L2 to prefetch its first rows (a hint that reads
 * no data into the kernel), then waits for that kernel to finish before it
 * reads h, x, expert_out or topk_w, and lets the next kernel start its own
 * prologue early. Use it only when the kernels just before this call on the
 * stream do not write post_w or pre_w. */
#define BEAM_OPT_PDL 0x4u

BEAM_API beam_status beam_boundary_fused_ex(beam_stream_t stream, uint16_t* h, const uint16_t* x,
                                   const uint16_t* post_w, const uint16_t* pre_w, int n,
                                   float eps, int64_t T, int D, uint16_t* y_out,
                                   const beam_launch_opts* opts);

BEAM_API beam_status beam_moe_combine_boundary_ex(beam_stream_t stream, uint16_t* h,
                                         const uint16_t* expert_out, const float* topk_w,
                                         const uint16_t* post_w, const uint16_t* pre_w, int n,
                                         float eps, int64_t T, int D, uint16_t* y_out,
                                         const beam_launch_opts* opts);

/*
 * The dense and MoE boundaries with y leaving as NVFP4 for the next GEMM
 * (SGLang page, "Fusion optimizations": the fusable boundary is extended to
 * NVFP4). The pages give no format; this is NVIDIA's published NVFP4 layout.
 * y is computed as in the BF16 calls, then, per block of 16 consecutive values
 * of a row:
 *   amax = max |y|,  sf = E4M3(RN32(RN32(amax / 6) * y_global_scale))
 *   q_j  = E2M1(RN32(y_j * RN32(y_global_scale / sf))), or 0 when sf is 0
 * (E4M3 = OCP E4M3FN, largest 448; E2M1 values 0, 0.5, 1, 1.5, 2, 3, 4, 6;
 * both nearest-even and saturating; signs kept).
 *   y_fp4   [T, D/2] bytes: element 2i in the low nibble, 2i+1 in the high; 16-byte aligned
 *   y_scale [T, D/16] bytes: one E4M3 scale per block, row-major (no swizzle)
 *   y_global_scale finite > 0; D a multiple of 16; no BF16 y is written.
 * Other arguments and errors as beam_boundary_fused_ex / beam_moe_combine_boundary_ex;
 * opts may be NULL; options of the shared-memory ring (stages > 0, the wait
 * timeout hook) give BEAM_ERR_ARG. y_fp4 and y_scale overlap neither each other
 * nor any other operand.
 * Non-finite y: the block amax skips NaN values; an infinite amax gives the
 * saturated scale 448 (0x7E) and infinite values the codes +-6; a NaN value's
 * code is +6 (0x7), since E2M1 has no NaN.
 */
BEAM_API beam_status beam_boundary_fused_nvfp4(beam_stream_t stream, uint16_t* h, const uint16_t* x,
                                      const uint16_t* post_w, const uint16_t* pre_w, int n,
                                      float eps, int64_t T, int D, float y_global_scale,
                                      uint8_t* y_fp4, uint8_t* y_scale,
                                      const beam_launch_opts* opts);

BEAM_API beam_status beam_moe_combine_boundary_nvfp4(beam_stream_t stream, uint16_t* h,
                                            const uint16_t* expert_out, const float* topk_w,
                                            const uint16_t* post_w, const uint16_t* pre_w, int n,
                                            float eps, int64_t T, int D, float y_global_scale,
                                            uint8_t* y_fp4, uint8_t* y_scale,
                                            const beam_launch_opts* opts);

/*
 * The dense and MoE boundaries on a batch that lives in host memory. Any
 * operand may be page-locked host memory (cudaHostAlloc, cudaHostRegister),
 * device memory of the current device, or managed memory; pageable host memory
 * only on a device that reads it through the host's page tables. The kernels
 * read and write host operands directly over the CPU-GPU link: no staging
 * copy and no device memory. On a Grace node that link is coherent NVLink-C2C,
 * and the boundary runs at link speed with both directions busy at once.
 * This is an addition of this library; the pages have no host-memory path.
 * Results are bit-identical to beam_boundary_fused / beam_moe_combine_boundary.
 * The launch uses the register kernels without L2 prefetch.
 * Asynchronous on `stream`: touch no host operand until the stream is
 * synchronised. Same arguments and errors as the device calls, checked before
 * any CUDA call; then BEAM_ERR_ARG for an operand the device cannot address
 * (pageable memory without pageable access, another device's memory).
 */
BEAM_API beam_status beam_boundary_fused_host(beam_stream_t stream, uint16_t* h, const uint16_t* x,
                                     const uint16_t* post_w, const uint16_t* pre_w, int n,
                                     float eps, int64_t T, int D, uint16_t* y_out);

BEAM_API beam_status beam_moe_combine_boundary_host(beam_stream_t stream, uint16_t* h,
                                           const uint16_t* expert_out, const float* topk_w,
                                           const uint16_t* post_w, const uint16_t* pre_w, int n,
                                           float eps, int64_t T, int D, uint16_t* y_out);

/*
 * Synchronises `stream` and returns in *count the number of row sums (two per
 * row: the post-norm and the pre-norm sum) that took the exact integer path on
 * the current device since the last reset; reset != 0 zeroes the counter.
 */
BEAM_API beam_status beam_exact_sum_count(beam_stream_t stream, uint64_t* count, int reset);

#ifdef __cplusplus
}
#endif

#endif /* BEAM_BOUNDARY_H */
