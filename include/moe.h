/*
 * moe.h -- C ABI of the single-GPU Mixture-of-Experts layer for GB300 (sm_103a).
 *
 * The layer: top-k router gating, padding-free token dispatch (per-expert histogram,
 * exclusive scan, permute-gather into one contiguous expert-ordered buffer with no
 * per-expert padding, optional capacity dropping), a grouped SwiGLU expert FFN over
 * the ragged expert segments, and a weighted un-permute/combine, with the matching
 * backward.
 *
 * Where each operation is defined (page title, then section / figure / field):
 *   - "MoE Training Optimization with Primus" (AMD blog), Figure 7 dataflow: router
 *     top-k per token; a permutation into expert order; the grouped gate/up projection
 *     (FC1), SwiGLU and the grouped down projection (FC2); a last step that un-permutes
 *     the rows, scales them by the gate weights and sums each token's k of them.
 *     MegaMoE section: the backward mirrors dispatch and combine, and adds the two
 *     weight-gradient GEMMs whose K is each expert's row count.  JAX section: a single
 *     grouped-GEMM launch covers all expert groups, each of its own length; the token
 *     counts never leave the GPU (no host synchronisation).
 *   - X-MoE verdict page (pith.science, arXiv 2508.13337), "key machinery": the
 *     padding-free token buffer -- only the routed tokens, stored contiguously per
 *     expert, plus side arrays giving each row's source token, its expert, the rows per
 *     expert and the combine weight; referee minor comment on section 4.1.1 Listing 1:
 *     max_token_count and c = 1.25; major comment on section 5.6: an assignment is
 *     dropped only when its expert is over capacity.
 *
 * Conventions shared by every call
 *   - Every pointer argument is a DEVICE pointer owned by the caller, except the
 *     moe_config_t pointer and the size_t/int32_t out-parameters of the host-only
 *     helpers, which are host pointers.  The library never allocates or frees
 *     device memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls only
 *     enqueue work and never synchronise with the host (the token counts stay on
 *     the device), except moe_status(), which synchronises `stream`.
 *   - Arguments are validated on the host before anything is enqueued; an invalid
 *     call returns MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED with nothing enqueued.
 *   - Anomalies seen on the device (a NaN logit, an out-of-range index in an input
 *     index array, inconsistent segment offsets, a pipeline wait that gave up) set
 *     bits in an error word at the start of `ws`; kernels never trap.  Read and
 *     clear it with moe_status().
 *   - Dtypes: logits fp32; activations, weights and their gradients bf16 (raw 16-bit
 *     patterns, `void*` here); gate weights and dlogits fp32; indices int32.
 *     Matrix products accumulate in fp32.
 *   - Layouts are row-major.  W1 is [E, 2f, d] (rows 0..f-1 gate, f..2f-1 up, i.e.
 *     nn.Linear (out, in)), W2 is [E, d, f]; the shared expert's W1s [2fs, d] and
 *     W2s [d, fs].  Every buffer indexed by an expert-ordered row ("xp", "ab", ...)
 *     is sized for T*k rows; the live row count is offsets[E] on the device.
 *   - Alignment: every device pointer 16-byte aligned.
 *   - Limits: 1 <= k <= 8, k <= E <= 256, 1 <= T, T*k < 2^31, d and f (and fs if
 *     non-zero) multiples of 64.  Anything else returns MOE_ERR_UNSUPPORTED.
 *   - Thread safety: calls on different streams with disjoint buffers may run
 *     concurrently; the library keeps no mutable state of its own between calls
 *     (the error word lives in the caller's `ws`) -- except the fixed scratch behind
 *     moe_route_noalloc, whose own comment says how it is shared.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, k > E, ... (nothing enqueued) */
    MOE_ERR_UNSUPPORTED = 2,   /* valid but outside the limits above (nothing enqueued)  */
    MOE_ERR_CUDA = 3,          /* a CUDA runtime call failed                             */
    MOE_ERR_DEVICE_FLAG = 4,   /* moe_status(): a device-side anomaly was flagged        */
    MOE_ERR_TIMEOUT = 5        /* moe_status(): a device pipeline wait gave up           */
} moe_status_t;

typedef enum {
    MOE_GATE_SOFTMAX_TOPK = 0, /* w_j = exp(l_j) / sum_{i in top-k} exp(l_i)            */
    MOE_GATE_SIGMOID_TOPK = 1  /* w_j = route_scale * sigma(l_j) / sum_{i in top-k} sigma(l_i) */
} moe_gate_t;

/* Device error bits reported by moe_status() through *flags. */
#define MOE_DEVERR_NAN_LOGIT   0x1   /* a router logit was NaN (it ranks below -inf)      */
#define MOE_DEVERR_BAD_INDEX   0x2   /* an index array held an out-of-range entry        */
#define MOE_DEVERR_TIMEOUT     0x4   /* a GEMM pipeline wait exceeded its bound          */
#define MOE_DEVERR_BAD_OFFSETS 0x8   /* segment offsets not monotone or past capacity    */

typedef struct {
    int64_t T;            /* tokens                                                    */
    int32_t d;            /* model width                                               */
    int32_t E;            /* routed experts                                            */
    int32_t k;            /* experts per token                                         */
    int32_t ffn;          /* routed expert SwiGLU width f                              */
    int32_t ffn_shared;   /* shared (always-on) expert width fs; 0 = none              */
    int32_t gate;         /* moe_gate_t                                                */
    float route_scale;    /* 1.0 for softmax; the sigmoid gate's scale (e.g. 2.5)      */
    int32_t capacity;     /* per-expert capacity; 0 = unlimited                        */
    /* Routing variants and memory trade-off (zero-initialise for the plain layer): */
    const float *select_bias; /* [E] device fp32, or NULL: added (fp32) to the logits for the
                                 top-k choice only -- the gate weights use the raw logits
                                 (a DeepSeek-V3-style balancing bias)                     */
    int32_t drop_negative;    /* 1: an assignment whose raw logit is negative is dropped
                                 before the capacity ranking and is not counted (DeepSpeed-
                                 MoE's rule, X-MoE verdict page, major comment on 5.6)    */
    int32_t recompute;        /* 1: selective rematerialisation -- ctx keeps neither ab nor
                                 h (nor ab_s, h_s); moe_layer_bwd recomputes FC1 from the
                                 saved xp (MegaScale-MoE notes: selective activation
                                 rematerialisation).  Results are bit-identical.         */
    int32_t drop_by_score;    /* 1 (with capacity > 0): an expert over capacity keeps the
                                 assignments with the largest raw logit (ties: lower token)
                                 instead of the earliest tokens; kept rows stay in token
                                 order inside its segment.  Needs (E+1 + T*k)*4 more bytes
                                 of ws.                                                   */
    int32_t mxfp8;            /* 1: the routed experts' forward GEMMs run on MXFP8 operands
                                 (moe_layer_fwd_mx), and with moe_layer_bwd_mx the data-
                                 gradient GEMMs of the backward too; needs d and ffn
                                 multiples of 128 and more ws for the quantised
                                 activations.  The weight gradients stay bf16.
                                 2: as 1, and the weight gradients too: their operands
                                 (dyp, h, dab, xp) are quantised along each segment's
                                 tokens, in 32-row blocks from the segment's first row
                                 (the Primus MoE blog, FP8 section: permuted tokens padded
                                 to the quantisation block boundary); needs about
                                 (2d + 3ffn) * (T*k + 128*E) * 33/32 more bytes of ws.
                                 0, 1, 2 only.                                            */
} moe_config_t;

/* Index of each saved tensor inside the forward context `ctx` (see moe_ctx_offsets). */
typedef enum {
    MOE_CTX_TOPK_IDX = 0,  /* int32 [T,k]                                               */
    MOE_CTX_TOPK_W,        /* fp32  [T,k]                                               */
    MOE_CTX_COUNTS,        /* int32 [E]                                                 */
    MOE_CTX_KEPT,          /* int32 [E]                                                 */
    MOE_CTX_OFFSETS,       /* int32 [E+1]                                               */
    MOE_CTX_DEST_ROW,      /* int32 [T,k]  (-1 = dropped)                               */
    MOE_CTX_SRC_TOK,       /* int32 [T*k]                                               */
    MOE_CTX_SRC_SLOT,      /* int32 [T*k]                                               */
    MOE_CTX_DROP_MASK,     /* uint8 [T,k]                                               */
    MOE_CTX_XP,            /* bf16  [T*k, d]   permuted tokens                          */
    MOE_CTX_AB,            /* bf16  [T*k, 2f]  FC1 output [a | b] (pre-activation)      */
    MOE_CTX_H,             /* bf16  [T*k, f]   silu(a) * b                              */
    MOE_CTX_YP,            /* bf16  [T*k, d]   FC2 output                               */
    MOE_CTX_AB_S,          /* bf16  [T, 2fs]   shared expert FC1 output (fs > 0)        */
    MOE_CTX_H_S,           /* bf16  [T, fs]                                             */
    MOE_CTX_YS,            /* bf16  [T, d]     shared expert output                     */
    MOE_CTX_NFIELDS
} moe_ctx_field_t;

/* floor(c * T * k / E): the per-expert capacity (max_token_count) for factor c
 * (X-MoE verdict page, referee minor comment on section 4.1.1 Listing 1).
 * Host-only.  Returns 0 (unlimited) for c <= 0 and -1 for invalid T, k, E. */
int32_t moe_capacity_from_factor(int64_t T, int32_t k, int32_t E, double c);

/* Bytes of the workspace `ws` (scratch + error word; one block serves every call)
 * and of the forward context `ctx` (tensors saved for the backward).  Host-only;
 * both out-pointers may be NULL. */
moe_status_t moe_workspace_size(const moe_config_t *cfg, size_t *ws_bytes, size_t *ctx_bytes);

/* Byte offset of every saved tensor inside `ctx`; offsets[MOE_CTX_NFIELDS]. Host-only. */
moe_status_t moe_ctx_offsets(const moe_config_t *cfg, size_t *offsets);

/* Clear the error word at the start of `ws` (enqueued on `stream`).  Call once on a
 * freshly allocated workspace. */
moe_status_t moe_ws_init(void *ws, void *stream);

/*
 * F1 + F2: route.  Primus MoE blog, Figure 7 dataflow (router top-k); X-MoE verdict
 * page, key machinery (padding-free buffer side arrays), referee comments on section
 * 4.1.1 Listing 1 and section 5.6 (capacity, drop only on overflow).
 *   logits   [T,E] fp32 in.
 *   topk_idx [T,k] out: the k best experts per token, by logit descending, ties to
 *            the lower id, NaN below -inf.  topk_w [T,k] out: gate weights computed
 *            over all k before any drop.
 *   counts [E] (assignments routed to e that were not dropped for a negative score),
 *            kept [E] = min(counts, capacity), offsets [E+1] = exclusive scan of
 *            kept; dest_row [T,k] = offsets[e] + (rank of t among e's tokens by
 *            ascending t), or -1 if that rank >= capacity; src_tok [T*k] / src_slot
 *            [T*k] (= t*k+j) invert dest_row (-1 past offsets[E]); drop_mask [T,k].
 *   Every integer output is deterministic (no atomics decide an order).
 */
moe_status_t moe_route(const moe_config_t *cfg, const float *logits, int32_t *topk_idx,
                       float *topk_w, int32_t *counts, int32_t *kept, int32_t *offsets,
                       int32_t *dest_row, int32_t *src_tok, int32_t *src_slot,
                       uint8_t *drop_mask, void *ws, void *stream);

/* Size of the fixed device scratch behind moe_route_noalloc (per GPU). */
#define MOE_NOALLOC_ROUTE_SCRATCH_BYTES (1u << 20)

/*
 * moe_route_noalloc -- the routing step (same outputs, same kernels as moe_route) for
 * callers that cannot allocate device memory, so cannot provide `ws`.  There is no
 * counterpart of this entry point in the paper; it exists for deployment reasons.
 *
 * Who needs it: a plugin running inside a host framework that owns all device memory
 * through its own pool and does not allow other code to call cudaMalloc, or a
 * latency-critical caller that cannot accept the device-wide synchronisation that
 * cudaMalloc / cudaFree may cause.  This call allocates nothing: the routing histogram
 * lives in a fixed __device__ array of MOE_NOALLOC_ROUTE_SCRATCH_BYTES compiled into
 * the library, which every GPU that loads the library holds until the process exits.
 *
 *   Arguments as for moe_route, except that `ws` is replaced by dev_flags_or_null: an
 *   optional device int32 that receives the MOE_DEVERR_* bits (NaN logits); with NULL
 *   those flags are dropped.
 *   Limit: the routing scratch must fit in MOE_NOALLOC_ROUTE_SCRATCH_BYTES.  With
 *   up(n) = n rounded up to a multiple of 256, it takes
 *       up(ceil(T/32) * E * 4)                                  bytes, plus, only when
 *       drop_by_score is set with a capacity,  up((E+1) * 4) + up(T * k * 4)  bytes
 *   (each expert's base and one 32-bit word per assignment for the score ranking).
 *   Examples that fit: plain or token-order capacity routing up to T = 32768 with
 *   E = 256 (exactly 1 MiB); drop-by-score routing with T = 16384, E = 64, k = 6
 *   (128 KiB + 512 B + 384 KiB).  T = 32768, E = 256 with drop_by_score does not fit.
 *   Larger shapes return MOE_ERR_UNSUPPORTED with nothing enqueued.
 *   Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call before any
 *   stream capture.  Only a successful lookup is remembered: if it fails (the call
 *   returns MOE_ERR_CUDA, nothing enqueued), the next call on that device tries again.
 *   Sharing: every call on a device uses the same array and leaves its contents behind
 *   (the kernels overwrite every entry they read, so nothing has to be cleared between
 *   calls); calls whose execution overlaps on the GPU -- e.g. on two streams without an
 *   ordering between them -- race on it and must be serialised by the caller.
 */
moe_status_t moe_route_noalloc(const moe_config_t *cfg, const float *logits, int32_t *topk_idx,
                               float *topk_w, int32_t *counts, int32_t *kept, int32_t *offsets,
                               int32_t *dest_row, int32_t *src_tok, int32_t *src_slot,
                               uint8_t *drop_mask, int32_t *dev_flags_or_null, void *stream);

/*
 * F3: permute-gather into expert order (Primus MoE blog, Figure 7, the permutation step
 * before FC1; X-MoE padding-free buffer).
 *   xp[p] = x[src_tok[p]] for p < offsets[E]; rows past offsets[E] are not written.
 *   x [T,d] bf16 in, xp [T*k,d] bf16 out.  A pure bit copy.
 */
moe_status_t moe_permute(const moe_config_t *cfg, const void *x, const int32_t *src_tok,
                         const int32_t *offsets, void *xp, void *ws, void *stream);

/*
 * F4 + F5: grouped SwiGLU expert FFN over the ragged segments given by offsets
 * (Primus MoE blog, Figure 7 FC1 / SwiGLU / FC2; JAX section: one launch over
 * ragged variable-M groups).  For every row p of expert e:
 *   [a | b] = xp[p] W1[e]^T  -> ab[p] (bf16, saved for the backward)
 *   h[p]    = silu(a) * b    (from the bf16 a, b; bf16)
 *   yp[p]   = h[p] W2[e]^T   (bf16)
 *   xp [T*k,d], ab [T*k,2f], h [T*k,f], yp [T*k,d]; only rows < offsets[E] written.
 */
moe_status_t moe_grouped_ffn(const moe_config_t *cfg, const void *xp, const int32_t *offsets,
                             const void *W1, const void *W2, void *ab, void *h, void *yp,
                             void *ws, void *stream);

/*
 * F3 + F4 + F5 fused: moe_grouped_ffn with the permute folded into FC1's operand loads
 * (Primus MoE blog, MegaMoE section: the dispatch fused into the FC1 grouped GEMM, here
 * on one GPU: tensor-memory-accelerator gathers of the token rows, no xp buffer).
 *   Row p of expert e is computed from x[src_tok[p]]; outputs as moe_grouped_ffn.
 *   x [T,d] bf16, src_tok [T*k] int32 (entries < offsets[E] must lie in [0,T); a bad one
 *   sets MOE_DEVERR_BAD_INDEX and row 0 is read instead).
 */
moe_status_t moe_grouped_ffn_gather(const moe_config_t *cfg, const void *x,
                                    const int32_t *src_tok, const int32_t *offsets,
                                    const void *W1, const void *W2, void *ab, void *h, void *yp,
                                    void *ws, void *stream);

/*
 * F7: combine = unpermute and scale (Primus MoE blog, Figure 7, last step).
 *   y[t] = sum_{j = 0..k-1, dest_row[t,j] >= 0} topk_w[t,j] * yp[dest_row[t,j]]
 *          (+ ys[t] if ys_or_null is not NULL), fp32 accumulation, bf16 out [T,d].
 */
moe_status_t moe_combine(const moe_config_t *cfg, const void *yp, const int32_t *dest_row,
                         const float *topk_w, const void *ys_or_null, void *y, void *ws,
                         void *stream);

/*
 * B1: backward of combine and of the gate (Primus MoE blog, MegaMoE section: the
 * dispatch of the upstream gradient dy).  For each kept slot (t,j) with row p = dest_row[t,j]:
 *   dyp[p] = bf16(topk_w[t,j] * dy[t]);  dw[t,j] = <dy[t], yp[p]> (0 if dropped)
 *   softmax gate: dlogits[t,e_j] = w_j (dw_j - sum_i w_i dw_i)
 *   sigmoid gate: S = sum_i s_i, s_i = sigma(l_i):
 *                 dlogits[t,e_j] = scale (dw_j / S - sum_i s_i dw_i / S^2) s_j (1 - s_j)
 *   dlogits [T,E] fp32 out, zero for unselected experts.  Both are evaluated in the
 *   equal pairwise form sum_i u_i (dw_j - dw_i) (u_i the normalised scores, summing to 1),
 *   which keeps its precision when one score carries almost all the weight.
 */
moe_status_t moe_combine_bwd(const moe_config_t *cfg, const void *dy, const void *yp,
                             const float *logits, const int32_t *topk_idx, const float *topk_w,
                             const int32_t *dest_row, void *dyp, float *dlogits, void *ws,
                             void *stream);

/*
 * B2..B5: backward of the grouped SwiGLU FFN (Primus MoE blog, MegaMoE section and
 * JAX section: data-gradient grouped GEMMs plus the two variable-K weight-gradient
 * grouped GEMMs).  For the rows of expert e (K of the weight gradients = the
 * segment's row count, which may be 0):
 *   dh = dyp W2[e];  da = dh * b * silu'(a);  db = dh * silu(a)  -> dab [T*k,2f] bf16
 *   dW2[e] = dyp_e^T h_e  [d,f] bf16;   dxp = dab W1[e]  [T*k,d] bf16;
 *   dW1[e] = dab_e^T xp_e [2f,d] bf16  (all fp32-accumulated).
 */
moe_status_t moe_grouped_ffn_bwd(const moe_config_t *cfg, const void *dyp, const void *xp,
                                 const int32_t *offsets, const void *W1, const void *W2,
                                 const void *ab, const void *h, void *dab, void *dxp, void *dW1,
                                 void *dW2, void *ws, void *stream);

/*
 * B2..B5 with the FC1 weight gradient gathering its operand from x: as
 * moe_grouped_ffn_bwd with xp[p] = x[src_tok[p]] read straight from x
 * (dW1[e] = dab_e^T x[src_tok]_e); no xp buffer exists.  Same index rules as
 * moe_grouped_ffn_gather.
 */
moe_status_t moe_grouped_ffn_bwd_gather(const moe_config_t *cfg, const void *dyp, const void *x,
                                        const int32_t *src_tok, const int32_t *offsets,
                                        const void *W1, const void *W2, const void *ab,
                                        const void *h, void *dab, void *dxp, void *dW1,
                                        void *dW2, void *ws, void *stream);

/*
 * B1's dispatch of dy fused into B2 (Primus MoE blog, MegaMoE section: the dispatch of the
 * upstream gradient folded into the FC2 data-gradient grouped GEMM).  As
 * moe_grouped_ffn_bwd, except that the FC2 data-gradient takes its rows straight from dy:
 * for row p of expert e, t = src_tok[p], s = src_slot[p],
 *   dh = topk_w[s] * (dy[t] W2[e])      (fp32: the gate weight is applied to the product
 *                                         in the GEMM's epilogue, so w * dy is never rounded
 *                                         to bf16 on this path)
 *   da, db from dh as in moe_grouped_ffn_bwd -> dab [T*k,2f] bf16
 * dy [T,d] bf16 and topk_w [T,k] fp32 as moe_combine_bwd takes them; src_tok / src_slot
 * [T*k] int32 from moe_route (entries < offsets[E] must lie in [0,T) and [0,T*k); a bad
 * one sets MOE_DEVERR_BAD_INDEX, row 0 of dy / a weight of 0 is used instead).
 * The FC2 weight gradient still contracts the rows dyp = bf16(w dy) that moe_combine_bwd
 * writes, so dyp is an input here; dxp, dW1 and dW2 are as in moe_grouped_ffn_bwd.
 */
moe_status_t moe_grouped_ffn_bwd_dispatch(const moe_config_t *cfg, const void *dy,
                                          const float *topk_w, const int32_t *src_tok,
                                          const int32_t *src_slot, const void *dyp,
                                          const void *xp, const int32_t *offsets,
                                          const void *W1, const void *W2, const void *ab,
                                          const void *h, void *dab, void *dxp, void *dW1,
                                          void *dW2, void *ws, void *stream);

/*
 * B6: un-permute reduce (Primus MoE blog, MegaMoE section: the reduction of each
 * token's rows after the FC1 data gradient).
 *   dx[t] = sum_{j kept} dxp[dest_row[t,j]] (+ dxs[t] if dxs_or_null), fp32 accumulation,
 *   gathered per token (deterministic, no atomics); bf16 [T,d] out.
 */
moe_status_t moe_unpermute_reduce(const moe_config_t *cfg, const void *dxp,
                                  const int32_t *dest_row, const void *dxs_or_null, void *dx,
                                  void *ws, void *stream);

/*
 * ---- MXFP8 forward of the routed experts (Primus MoE blog, FP8 section: the MXFP8 recipe
 * with OCP E4M3 elements for the expert grouped GEMMs, weight-quantisation caching;
 * MegaMoE section: the SwiGLU step quantises its own output).  MX rule (OCP Microscaling
 * formats v1.0): blocks of 32 consecutive elements along the contraction axis share the
 * scale 2^X, X = floor(log2(max |v|)) - 8 clamped to [-127, 127] (-127 for an all-zero
 * block), stored as the E8M0 code X + 127; elements are E4M3(v / 2^X), rounded to
 * nearest (ties to even) and saturated at +-448.  d and ffn must be multiples of 128.
 */

/* Bytes of the quantised-weight blob for cfg's routed experts, and the byte offsets of its
 * eight parts: offsets[0] W1 codes [E][2f][d] E4M3, offsets[1] W1 scales, offsets[2] W2
 * codes [E][d][f], offsets[3] W2 scales (the forward's, quantised along d and f);
 * offsets[4] W2^T codes [E][f][d] quantised along d, offsets[5] their scales, offsets[6]
 * W1^T codes [E][d][2f] quantised along 2f, offsets[7] their scales (the backward's data
 * gradients).  The transposes' scale atoms ((e*ceil(C/256) + nt)*(K/128) + kb)*2 + half
 * cover rows e*C + nt*256 + half*128 + m of the transpose (C = f or d rows per expert,
 * K = d or 2f).  The scales are stored in 512-byte atoms: atom
 * ((e*(f/128) + nb)*(d/128) + kb)*2 + half holds, at byte 16*(m%32) + 4*(m/32) + j, the
 * scale of W1 row e*2f + half*f + nb*128 + m, elements 32*(4*kb + j) .. +31; W2 atom
 * ((e*ceil(d/256) + nt)*(f/128) + kb)*2 + half covers W2 row e*d + nt*256 + half*128 + m.
 * Atom bytes of rows past an expert's end hold 127.  Host-only; offsets (8 entries) may be
 * NULL. */
moe_status_t moe_mx_weights_size(const moe_config_t *cfg, size_t *bytes, size_t *offsets);

/* Bytes of an activation scale array for contraction length K (d for x, ffn for h).
 * Activation scales are stored in 512-byte atoms tiled by 128 rows inside each expert
 * segment: for row p of expert e, local row l = p - offsets[e], m = l % 128, the scale of
 * elements 32*(4*kb + j) .. +31 sits in atom ((offsets[e] >> 7) + e + l/128) * (K/128) + kb
 * at byte 16*(m%32) + 4*(m/32) + j; bytes of rows past a segment's end are unspecified.
 * Size: ((T*k >> 7) + E + 1) * (K/128) * 512.  Host-only. */
moe_status_t moe_mx_act_scales_size(const moe_config_t *cfg, int32_t K, size_t *bytes);

/* Quantise W1 [E,2f,d] and W2 [E,d,f] (bf16) into the blob (device, 256-byte aligned,
 * moe_mx_weights_size bytes).  The caller keeps the blob while the weights are unchanged
 * (weight-quantisation caching). */
moe_status_t moe_mx_quantize_weights(const moe_config_t *cfg, const void *W1, const void *W2,
                                     void *wq, void *stream);

/* F3 with MXFP8 output: for p < offsets[E], xq[p] = E4M3 codes of x[src_tok[p]] ([T*k][d]
 * bytes) and its E8M0 scales into x_sf (activation atoms, moe_mx_act_scales_size(cfg, d)
 * bytes); with xp_or_null also the bf16 copy xp[p] = x[src_tok[p]] (the backward's saved
 * input). */
moe_status_t moe_mx_permute_quant(const moe_config_t *cfg, const void *x,
                                  const int32_t *src_tok, const int32_t *offsets,
                                  void *xp_or_null, void *xq, uint8_t *x_sf, void *ws,
                                  void *stream);

/* F4 + F5 on MXFP8 operands (block-scaled tensor-core MMAs, fp32 accumulation):
 *   [a|b] = bf16(deq(xq) deq(W1q[e])^T) -> ab;  h = bf16(silu(a) b) -> h;
 *   hq, h_sf = MX(h) along f (the SwiGLU epilogue quantises its bf16 output);
 *   yp = bf16(deq(hq) deq(W2q[e])^T).
 * Shapes as moe_grouped_ffn; hq [T*k][f] bytes; x_sf and h_sf are activation atoms
 * (moe_mx_act_scales_size with K = d and K = ffn). */
moe_status_t moe_grouped_ffn_mx(const moe_config_t *cfg, const void *xq, const uint8_t *x_sf,
                                const int32_t *offsets, const void *wq, void *ab, void *h,
                                uint8_t *hq, uint8_t *h_sf, void *yp, void *ws, void *stream);

/* Whole forward with the routed experts in MXFP8 (cfg->mxfp8 = 1): route -> permute and
 * quantise -> MXFP8 grouped FFN -> (bf16 shared expert) -> combine.  ctx receives the same
 * tensors as moe_layer_fwd (xp, ab, h, yp in bf16), so moe_layer_bwd runs unchanged; the
 * quantised activations live in ws.  wq: the blob of moe_mx_quantize_weights. */
moe_status_t moe_layer_fwd_mx(const moe_config_t *cfg, const float *logits, const void *x,
                              const void *wq, const void *W1s, const void *W2s, void *y,
                              void *ctx, void *ws, void *stream);

/* B2..B5 with the data-gradient GEMMs on MXFP8 operands (cfg->mxfp8 = 1 or 2): dyp is
 * quantised along d; dh = deq(MX(dyp)) deq(W2^T codes), the SwiGLU backward gives dab
 * (bf16 out) which is quantised along 2f; dxp = bf16(deq(MX(dab)) deq(W1^T codes)).  With
 * cfg->mxfp8 = 1 the weight gradients dW1, dW2 are computed from the bf16 xp, h, dyp and
 * dab as in moe_grouped_ffn_bwd; with 2, dW2[e] = bf16(deq(Q(dyp_e))^T deq(Q(h_e))) and
 * dW1[e] = bf16(deq(Q(dab_e))^T deq(Q(xp_e))), Q quantising each column of the segment's
 * rows in 32-row blocks from its first row (an expert without rows gets zeros).
 * wq: the blob of moe_mx_quantize_weights.  The quantised operands live in ws. */
moe_status_t moe_grouped_ffn_bwd_mx(const moe_config_t *cfg, const void *dyp, const void *xp,
                                    const int32_t *offsets, const void *wq, const void *ab,
                                    const void *h, void *dab, void *dxp, void *dW1, void *dW2,
                                    void *ws, void *stream);

/* Whole backward with the routed experts' data gradients in MXFP8 (cfg->mxfp8 = 1; with 2
 * their weight gradients too, as in moe_grouped_ffn_bwd_mx); as moe_layer_bwd otherwise
 * (the shared expert stays bf16). */
moe_status_t moe_layer_bwd_mx(const moe_config_t *cfg, const void *ctx, const float *logits,
                              const void *x, const void *dy, const void *wq, const void *W1s,
                              const void *W2s, void *dx, void *dW1, void *dW2, void *dW1s,
                              void *dW2s, float *dlogits, void *ws, void *stream);

/*
 * Whole forward: route -> permute -> grouped FFN -> (shared expert) -> combine.
 *   logits [T,E] fp32, x [T,d], W1, W2 (W1s, W2s if ffn_shared > 0, else may be NULL)
 *   y [T,d] out.  ctx (moe_workspace_size bytes) receives the saved tensors listed in
 *   moe_ctx_field_t; ws is scratch.  No host synchronisation.
 */
moe_status_t moe_layer_fwd(const moe_config_t *cfg, const float *logits, const void *x,
                           const void *W1, const void *W2, const void *W1s, const void *W2s,
                           void *y, void *ctx, void *ws, void *stream);

/*
 * Whole backward from the forward's ctx and the upstream gradient dy [T,d]:
 *   dx [T,d], dW1 [E,2f,d], dW2 [E,d,f] (dW1s, dW2s if ffn_shared > 0), dlogits [T,E].
 *   x and logits are the forward's inputs (not copied into ctx).
 */
moe_status_t moe_layer_bwd(const moe_config_t *cfg, const void *ctx, const float *logits,
                           const void *x, const void *dy, const void *W1, const void *W2,
                           const void *W1s, const void *W2s, void *dx, void *dW1, void *dW2,
                           void *dW1s, void *dW2s, float *dlogits, void *ws, void *stream);

/*
 * Diagnostics: exercises the device-side failure path without a GPU fault.  Enqueues one
 * small kernel that waits on an mbarrier nothing will ever complete, with the same bounded
 * wait the grouped GEMM uses, limited to `budget_cycles` SM clock cycles (clamped to
 * 2e9, about one second).  When the wait gives up it sets MOE_DEVERR_TIMEOUT in the error
 * word of `ws` and returns normally, so moe_status() then reports MOE_ERR_TIMEOUT and
 * the context stays usable.  (Not part of the layer; there is no counterpart on the
 * pages.)
 */
moe_status_t moe_selftest_wait_timeout(void *ws, int64_t budget_cycles, void *stream);

/*
 * Diagnostics: the SM clock the grouped GEMMs' mainloops ran at.  Under the power cap the
 * clock that sampling tools report between samples can differ from the one the tensor-core
 * loops see, which decides the peak their throughput is measured against.  While tracing
 * is on, the MMA-issuing warp of every bf16 and MXFP8 grouped-GEMM CTA (the leader of a
 * CTA pair) adds, once per launch, the SM cycles (clock64) and the nanoseconds
 * (%globaltimer) of its tile loop to device-side sums; cycles / ns is that loop's clock.
 * The cost is a flag load and two timer reads per CTA and launch, plus three atomics per
 * CTA and launch while on.  (Not part of the layer; there is no counterpart on the pages.)
 *
 * moe_gemm_clock_trace(1) zeroes the sums and turns tracing on; moe_gemm_clock_trace(0)
 * turns it off and keeps them.  moe_gemm_clock_read() returns the sums: *cycles and *ns
 * over *loops loops (NULL pointers: MOE_ERR_INVALID_ARG).  Both are synchronous host
 * calls on the current device, ordered with the legacy default stream only: call them
 * with no grouped GEMM in flight (after a device or stream synchronisation).  Tracing
 * state is per device and shared by every caller in the process.
 */
moe_status_t moe_gemm_clock_trace(int enable);
moe_status_t moe_gemm_clock_read(uint64_t *cycles, uint64_t *ns, uint64_t *loops);

/* Synchronise `stream`, then read and clear the device error word in `ws`.
 * Returns MOE_OK, MOE_ERR_DEVICE_FLAG or MOE_ERR_TIMEOUT (MOE_DEVERR_TIMEOUT set),
 * or MOE_ERR_CUDA; *flags (may be NULL) receives the MOE_DEVERR_* bits. */
moe_status_t moe_status(void *ws, void *stream, int32_t *flags);

/* Human-readable name of a status code.  Host-only; never NULL. */
const char *moe_status_string(moe_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
