/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) routed mixture-of-experts
 * expert layer.
 *
 * The layer (flashinfer.fused_moe.cute_dsl_fused_moe_bf16, summary formula):
 *
 *   out[t] = sum_j w[t,j] * ffn(x[t]; e[t,j]),
 *   ffn(x; e) = (silu(x . W1_gate[e]^T) * (x . W1_up[e]^T)) . W2[e]^T
 *
 * computed as route -> sort -> gather -> FC1+SwiGLU -> FC2 -> finalize, every
 * step in a hand-written CUDA kernel.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers, owned by the caller, row-major
 *     and contiguous.  bf16 tensors are passed as moe_bf16 (the 16-bit
 *     pattern).  The library never allocates device memory, never frees a
 *     caller pointer and never synchronises the host inside a launch.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *   - Every call returns MOE_OK (0) or a negative MOE_ERR_* code; on an error
 *     nothing has been enqueued.  moe_status_string() describes a code.
 *   - Expert weights are the LOCAL bank of an expert-parallel shard
 *     (cute_dsl_fused_moe_bf16, Parameters): W1 [L, 2I, H] holds, for local
 *     expert i (global id local_offset + i), the I "up" rows followed by the
 *     I "gate" rows (the canonical [up | gate] order of
 *     flashinfer.fused_moe.cake / cake_cute, Host plan); W2 [L, H, I].
 *     Routes to global ids outside [local_offset, local_offset + L)
 *     contribute zero (cute_dsl_fused_moe_bf16, Supported configuration).
 *   - Arithmetic: bf16 operands, fp32 accumulation, bf16 output
 *     (cute_dsl_fused_moe_bf16, Supported configuration).
 *   - Device-side problems that the host cannot see (a pre-routed id outside
 *     [0, E), a bounded wait that gave up) are reported by OR-ing MOE_DEV_*
 *     bits into a caller-provided int32 status word in device memory.  The
 *     launch chain clears it first; read it after the stream has finished.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef uint16_t moe_bf16; /* bfloat16 bit pattern */

/* ---- return codes --------------------------------------------------------- */
#define MOE_OK 0
#define MOE_ERR_NULL (-1)        /* a required pointer is NULL                 */
#define MOE_ERR_SHAPE (-2)       /* a size is out of range or not a supported multiple */
#define MOE_ERR_ALIGN (-3)       /* a pointer is not 16-byte aligned           */
#define MOE_ERR_WORKSPACE (-4)   /* workspace NULL or smaller than required    */
#define MOE_ERR_MODE (-5)        /* routing inputs: give logits XOR (ids, weights) */
#define MOE_ERR_CUDA (-6)        /* a CUDA runtime call or launch failed       */
#define MOE_ERR_DEVICE (-7)      /* no device, or the device is not sm_103     */
#define MOE_ERR_TENSOR_MAP (-8)  /* the driver rejected a TMA tensor map       */
#define MOE_ERR_STATE (-9)       /* call not valid for this plan's state       */

/* ---- device status bits ---------------------------------------------------- */
#define MOE_DEV_BAD_EXPERT 1u    /* a routed id outside [0, E): route dropped  */
#define MOE_DEV_TIMEOUT 2u       /* a bounded in-kernel wait gave up           */

/* ---- limits ------------------------------------------------------------------ */
#define MOE_MAX_EXPERTS 1024     /* E and L                                    */
#define MOE_MAX_TOP_K 16

/* Describe a return code (static string, never NULL). */
MOE_API const char *moe_status_string(int code);

/* Version of this ABI (major * 100 + minor). */
MOE_API int moe_abi_version(void);

/* ---- S1 route ----------------------------------------------------------------
 * Renormalised top-k routing ("Renormalize top-k":
 * flashinfer.experimental.cake_stepfun_moe, opening paragraphs; routing read
 * from logits, RoutingInputMode.FromLogits, Unified MoE API opt-in).
 *   logits   [T, E] fp32 (read)
 *   topk_ids [T, top_k] int32 (written): the top_k experts of each token by
 *            logit, descending, equal logits ordered by lower expert id.
 *   topk_w   [T, top_k] fp32 (written): softmax restricted to the chosen
 *            experts, w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0).
 * Sizes: T >= 0, 1 <= E <= MOE_MAX_EXPERTS, 1 <= top_k <= min(E, MOE_MAX_TOP_K).
 * One warp per token.  T == 0 is a no-op. */
MOE_API int moe_route(const float *logits, int T, int E, int top_k, int32_t *topk_ids,
              float *topk_w, void *stream);

/* ---- S2 sort -------------------------------------------------------------------
 * Stable counting sort of the T*top_k routes by local expert (the
 * consecutive-row groups of Cake ragged BF16 grouped GEMM, operation table;
 * expanded_idx_to_permuted_idx of flashinfer.experimental.cake_stepfun_moe,
 * Prepared launches).  Expanded index r = t*top_k + j.
 *   topk_ids    [T, top_k] int32 global ids (read)
 *   m_indptr    [L+1] int32 (written): m_indptr[0] = 0, group i = permuted
 *               rows [m_indptr[i], m_indptr[i+1]); M = m_indptr[L].
 *   perm_to_exp [T*top_k] int32 (written, first M valid): expanded index of
 *               each permuted row; ascending r inside a group.
 *   exp_to_perm [T*top_k] int32 (written): permuted row of each route, -1 for
 *               a route whose id is not local or outside [0, E).
 *   workspace   >= moe_sort_workspace_size(T, top_k, L) bytes (may be NULL
 *               when that size is 0).
 *   status      optional int32 word: cleared, then MOE_DEV_BAD_EXPERT if any
 *               id is outside [0, E).
 * Sizes: 0 <= local_offset, 1 <= L, local_offset + L <= E <= MOE_MAX_EXPERTS. */
MOE_API size_t moe_sort_workspace_size(int T, int top_k, int num_local);
MOE_API int moe_sort(const int32_t *topk_ids, int T, int top_k, int E, int local_offset,
             int num_local, int32_t *m_indptr, int32_t *perm_to_exp,
             int32_t *exp_to_perm, void *workspace, size_t workspace_bytes,
             int32_t *status, void *stream);

/* ---- S2 sort without a workspace ----------------------------------------------
 * The pages have no counterpart of this entry point.  It is moe_sort for
 * callers that cannot allocate device memory: a plugin whose host framework
 * hands it only its input and output buffers, or a runtime that plans all
 * device memory up front and forbids allocating afterwards.  The same kernels
 * run; the per-chunk table that moe_sort keeps in the caller's workspace lives
 * instead in a fixed 1 MiB array inside the library's device memory, held on
 * every device that loads the library until the process exits.  Nothing is
 * allocated and no workspace is passed; arguments and outputs are those of
 * moe_sort.
 *   Limit: ceil(T*top_k / 4096) * num_local <= 262144 table entries (T*top_k
 *   <= 2048 uses no table at all); larger problems return MOE_ERR_WORKSPACE
 *   before anything is enqueued.
 *   The array's device address is looked up, with the calling device
 *   current, on every call made outside stream capture; a call being captured
 *   reuses the address of the last such lookup on its device, so make one call
 *   on each device before any stream capture (a captured call without one
 *   returns MOE_ERR_CUDA).
 *   All calls share the array: calls whose kernels overlap on the GPU (for
 *   example on two streams) race on it and must be serialised by the caller.
 *   The kernels write every entry they read, so no clearing is needed. */
MOE_API int moe_sort_no_alloc(const int32_t *topk_ids, int T, int top_k, int E,
                              int local_offset, int num_local, int32_t *m_indptr,
                              int32_t *perm_to_exp, int32_t *exp_to_perm,
                              int32_t *status, void *stream);

/* ---- S3 gather -------------------------------------------------------------------
 * xp[p, :] = x[perm_to_exp[p] / top_k, :] for p < M = m_indptr[L] (the
 * expanded per-route activations; cute_dsl_fused_moe_bf16, Parameters,
 * use_fused_finalize).  Rows p >= M of xp are not written.
 *   x [T, H] bf16, xp [T*top_k, H] bf16.  H % 8 == 0. */
MOE_API int moe_gather(const moe_bf16 *x, const int32_t *perm_to_exp,
               const int32_t *m_indptr, int T, int H, int top_k, int num_local,
               moe_bf16 *xp, void *stream);

/* ---- S4 FC1 + SwiGLU -----------------------------------------------------------
 * For permuted row p of group i: u = xp[p] . W1[i, 0:I]^T,
 * g = xp[p] . W1[i, I:2I]^T (fp32), h[p] = bf16_rne(silu(g) * u)
 * (cute_dsl_fused_moe_bf16, summary formula; SwiGLU fused into GEMM1,
 * Supported configuration).  tcgen05 grouped GEMM, persistent, TMA-fed.
 *   xp [max_rows, H] bf16, w1 [L, 2I, H] bf16, m_indptr [L+1] (device),
 *   h [max_rows, I] bf16 (rows >= M untouched).
 *   max_rows bounds M (e.g. T*top_k).  H % 64 == 0, I % 64 == 0. */
MOE_API int moe_fc1_swiglu(const moe_bf16 *xp, const moe_bf16 *w1,
                   const int32_t *m_indptr, int max_rows, int H, int I,
                   int num_local, moe_bf16 *h, void *stream);

/* ---- S3 + S4 fused: FC1 + SwiGLU reading its rows through the permutation --------
 * h[p] = bf16_rne(silu(g) * u) for permuted row p < M with the activations
 * taken straight from x: row p is x[perm_to_exp[p] / top_k] (no xp buffer).
 * Three gather warps (one per ring slot) copy the rows with 16-byte
 * cp.async into the swizzled layout of a TMA box.  Bitwise the same result as
 * moe_gather followed by moe_fc1_swiglu, without the [T*top_k, H] buffer of
 * gathered rows, but slower: the copies of one slot take longer to land than
 * the tensor cores take for the other two (FC1 measured 1.95 ms against
 * 1.26 ms + 0.02 ms for the gather at T=4096, H=4096, I=14336, E=8, top-2,
 * and 4.63 ms against 3.10 ms + 0.26 ms at T=8192, H=7168, I=2048, E=256,
 * top-8).  moe_forward uses the gather kernel unless the plan sets
 * MOE_PLAN_FUSED_GATHER.
 *   x [T, H] bf16, perm_to_exp [T*top_k], m_indptr [L+1], w1 [L, 2I, H],
 *   h [T*top_k, I] bf16.  H % 64 == 0, I % 128 == 0. */
MOE_API int moe_fc1_swiglu_gathered(const moe_bf16 *x, const int32_t *perm_to_exp,
                                    const int32_t *m_indptr, int T, int top_k,
                                    const moe_bf16 *w1, int H, int I, int num_local,
                                    moe_bf16 *h, void *stream);

/* ---- S4 with the StepFun epilogue ---------------------------------------------------
 * moe_fc1_swiglu with SwiGLUStep(limit): GEMM1's outputs are clamped before
 * the activation, g' = min(g, limit[i]), u' = min(max(u, -limit[i]), limit[i]),
 * h[p] = bf16_rne(silu(g') * u') for permuted rows p of local expert i (the
 * StepFun SwiGLUStep activation with one clamp limit per expert,
 * flashinfer.experimental.cake_stepfun_moe, opening paragraph; the per-expert
 * gemm1_clamp_limit of Unified MoE API opt-in).  This clamp is the library's
 * reading: the page names the activation and the per-expert limit only.
 *   clamp_limit [L] fp32 (device), one limit per local expert; +inf leaves an
 *   expert's SwiGLU unclamped (bitwise moe_fc1_swiglu).  Other arguments as
 *   moe_fc1_swiglu.  The prepared launch takes the same limits through
 *   moe_forward_desc.clamp_limit on every path. */
MOE_API int moe_fc1_swiglu_step(const moe_bf16 *xp, const moe_bf16 *w1, const float *clamp_limit,
                                const int32_t *m_indptr, int max_rows, int H, int I,
                                int num_local, moe_bf16 *h, void *stream);

/* ---- S4 / S5 with E4M3 operands (the fp8 per-tensor family, MOE_WEIGHTS_E4M3) --------
 * moe_fc1_swiglu_e4m3: hq[p] = e4m3( swiglu_step(g * sc, u * sc, limit[i]) * RN(1 / h_scale) )
 *   with u, g = xq[p] . W1q[i, up / gate rows]^T (fp32) and sc = x_scale * w1_scale[i]
 *   (the product with the correctly rounded reciprocal is within one fp32 ulp of the
 *   quotient by h_scale);
 *   xq [max_rows, H], w1q [L, 2I, H], hq [max_rows, I] E4M3 codes (uint8);
 *   clamp_limit [L] or NULL (plain SwiGLU).
 * moe_fc2_e4m3: y[p] = (hq[p] . W2q[i]^T) * (h_scale * w2_scale[i]), fp32;
 *   w2q [L, H, I] E4M3 codes, y [max_rows, H] fp32.
 * H % 128 == 0, I % 128 == 0; m_indptr [L+1] on the device. */
MOE_API int moe_fc1_swiglu_e4m3(const uint8_t *xq, const uint8_t *w1q, const float *w1_scale,
                                float x_scale, float h_scale, const float *clamp_limit,
                                const int32_t *m_indptr, int max_rows, int H, int I,
                                int num_local, uint8_t *hq, void *stream);
MOE_API int moe_fc2_e4m3(const uint8_t *hq, const uint8_t *w2q, const float *w2_scale,
                         float h_scale, const int32_t *m_indptr, int max_rows, int H, int I,
                         int num_local, float *y, void *stream);

/* ---- S5 FC2 ------------------------------------------------------------------------
 * y[p] = h[p] . W2[i]^T, fp32, unscaled and unrounded (cute_dsl_fused_moe_bf16,
 * Parameters, use_fused_finalize=False).
 *   h [max_rows, I] bf16, w2 [L, H, I] bf16, y [max_rows, H] fp32.
 *   H % 64 == 0, I % 64 == 0. */
MOE_API int moe_fc2(const moe_bf16 *h, const moe_bf16 *w2, const int32_t *m_indptr,
            int max_rows, int H, int I, int num_local, float *y, void *stream);

/* ---- S7 decode-form FC1 / FC2 ------------------------------------------------------
 * The same products as moe_fc1_swiglu / moe_fc2, computed with the operands
 * swapped for few rows per expert (the swap-AB small-token forms of
 * flashinfer.fused_moe.cake / cake_cute, Generated kernels): 128 weight rows
 * take the MMA's M side and the expert's rows its N side (16/32/64), so each
 * weight byte is streamed from HBM once.  max_group_rows is the expected
 * largest group (it picks the N tile; larger groups are still correct, in
 * several N tiles).  Arguments and layouts otherwise as moe_fc1_swiglu /
 * moe_fc2.  moe_forward uses these for T <= 64 tokens (MOE_PATH_AUTO). */
MOE_API int moe_fc1_swiglu_swapab(const moe_bf16 *xp, const moe_bf16 *w1,
                                  const int32_t *m_indptr, int max_rows,
                                  int max_group_rows, int H, int I, int num_local,
                                  moe_bf16 *h, void *stream);
MOE_API int moe_fc2_swapab(const moe_bf16 *h, const moe_bf16 *w2, const int32_t *m_indptr,
                           int max_rows, int max_group_rows, int H, int I,
                           int num_local, float *y, void *stream);

/* ---- S6 finalize --------------------------------------------------------------------
 * out[t] = bf16_rne( sum_{j=0..top_k-1, exp_to_perm[t*top_k+j] >= 0}
 *                    topk_w[t,j] * y[exp_to_perm[t*top_k+j]] ), summed in fp32
 * in ascending j with no atomics, so replays are bitwise identical
 * (cute_dsl_fused_moe_bf16, Parameters, use_fused_finalize=False).
 *   y [*, H] fp32, exp_to_perm [T*top_k], topk_w [T, top_k] fp32,
 *   out [T, H] bf16.  H % 8 == 0. */
MOE_API int moe_finalize(const float *y, const int32_t *exp_to_perm,
                 const float *topk_w, int T, int top_k, int H, moe_bf16 *out,
                 void *stream);

/* ---- S8 ragged grouped GEMM forward ---------------------------------------------------
 * Y[offs[e-1]:offs[e]] = X[offs[e-1]:offs[e]] . W[e]^T (offs[-1] = 0), bf16
 * output, fp32 accumulation (Cake ragged BF16 grouped GEMM, operation table,
 * fwd).  offs [E] int32 cumulative group ends, read on the device only; groups
 * may be empty or any size.  X [sum_m, K], W [E, N, K], Y [sum_m, N].
 * Rows of Y outside [0, offs[E-1]) are not written.
 * N % 64 == 0, K % 64 == 0, 1 <= E <= MOE_MAX_EXPERTS, offs[E-1] <= sum_m. */
MOE_API int grouped_gemm_fwd(const moe_bf16 *X, const moe_bf16 *W, const int32_t *offs,
                     int sum_m, int E, int N, int K, moe_bf16 *Y, void *stream);
/* The same with plan flags; MOE_PLAN_NO_TAIL_TILES is the only one it reads. */
MOE_API int grouped_gemm_fwd_flags(const moe_bf16 *X, const moe_bf16 *W, const int32_t *offs,
                                   int sum_m, int E, int N, int K, moe_bf16 *Y, int flags,
                                   void *stream);
/* The same with the small-group kernel beside the CTA-pair kernel: when
 * counters is not NULL (and the shape takes the pair kernel, N % 256 == 0,
 * with tail tiles), the groups of at most 64 rows are streamed by a one-CTA
 * swap-AB kernel on 24 SMs while the pair kernel takes the others, both
 * claiming tiles at run time through the counters (see
 * MOE_PLAN_NO_SMALL_GROUP_KERNEL).  counters: device int32
 * [MOE_GROUPED_GEMM_COUNTERS], 16-byte aligned, owned by the caller and
 * cleared on the stream by every call; calls that overlap on the GPU need
 * counters of their own.  Y is bitwise the same as without it.  NULL counters:
 * grouped_gemm_fwd_flags.  It pays where the GEMM is tensor-bound (active
 * groups averaging well over 280 rows) with some small groups; where weight
 * streaming bounds the GEMM it only takes SMs from the pair kernel. */
#define MOE_GROUPED_GEMM_COUNTERS 4
MOE_API int grouped_gemm_fwd_ex(const moe_bf16 *X, const moe_bf16 *W, const int32_t *offs,
                                int sum_m, int E, int N, int K, moe_bf16 *Y, int flags,
                                int32_t *counters, void *stream);

/* ---- ragged grouped GEMM backward ---------------------------------------------------------
 * The dgrad and wgrad rows of Cake ragged BF16 grouped GEMM, operation table
 * (and its Autograd section: x.grad from dgrad, w.grad from wgrad), groups as
 * in grouped_gemm_fwd (offs [E] cumulative ends read on the device; groups may
 * be empty or any size; no padding, no host synchronisation).  bf16 operands,
 * fp32 accumulation in a fixed order, no atomics: replays are bitwise equal.
 *
 * grouped_gemm_dgrad: dX[offs[e-1]:offs[e]] = G[offs[e-1]:offs[e]] . W[e],
 *   W used in place.  G [sum_m, N], W [E, N, K], dX [sum_m, K] bf16 (rows
 *   outside [0, offs[E-1]) are not written).
 * grouped_gemm_wgrad: dW[e] = G[offs[e-1]:offs[e]]^T . X[offs[e-1]:offs[e]]
 *   for every e, exactly zero for an empty group.  G [sum_m, N], X [sum_m, K],
 *   dW [E, N, K] fp32 (dw_fp32 != 0) or bf16 (one rounding of the fp32 sum).
 * N % 64 == 0, K % 64 == 0, 1 <= E <= MOE_MAX_EXPERTS, offs[E-1] <= sum_m;
 * pointers 16-byte aligned.  sum_m == 0: dgrad does nothing, wgrad zeroes dW. */
MOE_API int grouped_gemm_dgrad(const moe_bf16 *G, const moe_bf16 *W, const int32_t *offs,
                               int sum_m, int E, int N, int K, moe_bf16 *dX, void *stream);
MOE_API int grouped_gemm_wgrad(const moe_bf16 *G, const moe_bf16 *X, const int32_t *offs,
                               int sum_m, int E, int N, int K, void *dW, int dw_fp32,
                               void *stream);

/* ---- BGMV LoRA-MoE shrink + expand ------------------------------------------------------------
 * LoRA deltas of the routed (token, expert) pairs of an MoE layer
 * (flashinfer.fused_moe.prepare_bgmv_moe, description and Parameters).  For
 * routed pair p: t = sorted_token_ids[p], e = expert_ids[p], l = lora_indices[t].
 * For every slice s (rank R; A_s = lora_a[s] [num_loras, E, R, H],
 * B_s = lora_b[s] [num_loras, E, feat_out[s], R], bf16):
 *   shrink_out[s, p, r] = bf16( A_s[l, e, r, :] . x[t, :] )      (fp32 sum)
 *   y_accum[t, off_s + f] = sum over the pairs p of token t, in ascending p,
 *                           of topk_weights[p] * (B_s[l, e, f, :] . shrink_out[s, p, :])
 * in fp32 (off_s = feat_out[0] + .. + feat_out[s-1]).  Each output element is
 * written by one owner that adds the token's pairs in that fixed order, so
 * replays are bitwise identical; a token without pairs gets zeros.  The
 * library's readings: y_accum is overwritten (not added to), and the shrink
 * values are rounded to bf16 (the weight dtype of the page's shrink
 * workspace) before the expand.
 *   x [T, H] bf16 (H % 8 == 0); lora_a, lora_b, feat_out: HOST arrays of
 *   num_slices (1..8) device pointers / sizes (feat_out[s] % 8 == 0);
 *   rank in {8, 16, 32, 64}; sorted_token_ids, expert_ids, topk_weights
 *   [num_pairs]; lora_indices [T]; shrink_out [num_slices, num_pairs, rank]
 *   bf16; y_accum [T, ld_y] fp32, ld_y >= sum feat_out (it may be a column
 *   slice of a wider row-major buffer).
 *   contiguous_top_k = k > 0 (k <= MOE_MAX_TOP_K): the pairs are token-major,
 *   pair p of token p / k (num_pairs == T * k); 0: any order (e.g. sorted by
 *   expert), through a per-token route index.
 *   The pairs are grouped by (LoRA, expert), so each A and B block is read
 *   once per group (the page's pair-grouped pipeline): while groups x pairs
 *   <= 2^22 by a scan (one CTA per group), else, up to MOE_MAX_EXPERTS
 *   groups, by the routes' stable counting sort; the expand writes fp32
 *   per-pair partials that one owner per token adds in ascending pair order.
 *   Otherwise one CTA per pair (shrink) and one per token (expand).
 *   workspace: moe_bgmv_workspace_size(T, num_pairs, contiguous_top_k,
 *   num_loras, E, sum feat_out) bytes (route index, grouping, partials).
 *   A pair whose token, expert or LoRA index is out of range (or, with
 *   contiguous_top_k, whose token is not p / k) contributes nothing and raises
 *   MOE_DEV_BAD_EXPERT in *status (cleared first; optional).
 * No allocation, no host synchronisation: capturable in a CUDA graph. */
MOE_API size_t moe_bgmv_workspace_size(int T, int num_pairs, int contiguous_top_k, int num_loras,
                                       int E, int total_feat_out);
MOE_API int moe_bgmv(const moe_bf16 *x, int T, int H, const moe_bf16 *const *lora_a,
                     const moe_bf16 *const *lora_b, int num_slices, const int *feat_out, int rank,
                     int num_loras, int E, const int32_t *sorted_token_ids,
                     const int32_t *expert_ids, const int32_t *lora_indices,
                     const float *topk_weights, int num_pairs, int contiguous_top_k,
                     moe_bf16 *shrink_out, float *y_accum, int ld_y, void *workspace,
                     size_t workspace_bytes, int32_t *status, void *stream);

/* ---- whole layer (one shot) --------------------------------------------------------------
 * Routing inputs: exactly one of
 *   logits [T, E] fp32                      (RoutingInputMode.FromLogits), or
 *   topk_ids [T, top_k] int32 + topk_w [T, top_k] fp32, weights normalised
 *   by the caller                           (UnpackedPrecomputed;
 *   cute_dsl_fused_moe_bf16, Parameters token_selected_experts /
 *   token_final_scales).
 * x [T, H] bf16, w1 [L, 2I, H], w2 [L, H, I], out [T, H] bf16.
 * workspace >= moe_workspace_size(...) bytes, 256-byte aligned.
 * T == 0 is a no-op (cute_dsl_fused_moe_bf16, Supported configuration).
 * H % 64 == 0, I % 64 == 0. */
MOE_API size_t moe_workspace_size(int T, int H, int I, int E, int top_k, int num_local);
MOE_API int moe_forward(const moe_bf16 *x, const float *logits, const int32_t *topk_ids,
                const float *topk_w, const moe_bf16 *w1, const moe_bf16 *w2,
                int T, int H, int I, int E, int top_k, int local_offset,
                int num_local, moe_bf16 *out, void *workspace,
                size_t workspace_bytes, int32_t *status, void *stream);

/* ---- prepared launch ------------------------------------------------------------------------
 * Prepare once, launch many (flashinfer.experimental.cake_stepfun_moe,
 * Prepared launches; Cake ragged BF16 grouped GEMM, Prepared launches):
 * moe_forward_prepare validates the descriptor, lays out the workspace and
 * encodes the TMA tensor maps (host memory only).  moe_plan_launch then only
 * enqueues work: no allocation, no host synchronisation, capturable in a
 * CUDA graph, and valid for new VALUES written into the bound buffers.  Every
 * launch first clears the status word (if given) on the launch stream, before
 * any kernel of the launch can report into it: with cudaMemsetAsync, or, for
 * the decode chain in one launch, with a one-CTA kernel that also zeroes the
 * counters the chain keeps in the workspace.  A grouped-path launch that runs
 * the small-group kernel beside the CTA-pair GEMMs (MOE_PLAN_SMALL_GROUP_KERNEL
 * below) likewise zeroes the GEMMs' tile-claim counters in the workspace with
 * one more cudaMemsetAsync first, so plans may share a workspace.  The
 * workspace is every launch's scratch: launches of one plan (or of plans
 * sharing a workspace) must run one after another (one stream, or streams
 * ordered by events).
 */
#define MOE_PATH_AUTO 0    /* decided from the shape                         */
#define MOE_PATH_GROUPED 1 /* route/sort/gather + tcgen05 grouped GEMMs       */
#define MOE_PATH_DECODE 2  /* weight-streaming kernels for few tokens         */

#define MOE_PLAN_STAGE_TIMING 1 /* record CUDA events around each stage     */
#define MOE_PLAN_ONE_CTA_GEMM 2 /* grouped path: one-CTA GEMM kernels instead of
                                   the CTA-pair (2-SM MMA) kernels (comparison) */
#define MOE_PLAN_DECODE_CHAIN 4 /* decode path, T*top_k <= 1024: always the
                                   chain (sort, gather and finalize folded into
                                   the GEMM kernels) as two kernels; without a
                                   decode flag the chain runs as one launch for
                                   T*top_k <= 32, where it measured faster */
#define MOE_PLAN_DECODE_SEPARATE 8 /* decode path: always the five separate
                                      kernels (sort, gather, FC1, FC2, finalize) */
#define MOE_PLAN_FUSED_GATHER 16 /* grouped path, CTA-pair GEMMs: FC1 copies its
                                    token rows straight from x (no gather kernel,
                                    no permuted copy of x; measured slower, see
                                    moe_fc1_swiglu_gathered) */
#define MOE_PLAN_DECODE_ONE_LAUNCH 32 /* decode path, T*top_k <= 1024: always the
                                         chain as one kernel; CTAs without FC1 work
                                         stream their W2 tile while FC1 runs and wait
                                         (bounded) until the FC1 tiles of its expert
                                         are done.  The kernel takes at most one CTA
                                         per SM; if other work holds SMs for longer
                                         than the wait limit, the launch reports
                                         MOE_DEV_TIMEOUT in the status word. */
#define MOE_PLAN_NO_TAIL_TILES 128 /* CTA-pair GEMMs: a group's last rows run as a
                                     main tile (256 token rows, the rows past the
                                     group computed and not stored) instead of a
                                     swap-AB tail tile (weights on the MMA's M
                                     side, the group's rows on N) */
#define MOE_PLAN_NO_SMALL_GROUP_KERNEL 256 /* grouped path, CTA-pair GEMMs: the
                                             pair kernel takes every group.
                                             Without this flag, when the plan's
                                             routes average at most 512 per local
                                             expert, each GEMM runs as two kernels
                                             at once: a one-CTA kernel on 24 SMs
                                             streams the groups of at most 64
                                             rows (weights on the MMA's M side,
                                             the group's rows on N), the pair
                                             kernel takes the others; both claim
                                             tiles at run time.  The outputs are
                                             bitwise the same either way. */
#define MOE_PLAN_SMALL_GROUP_KERNEL 512 /* grouped path, CTA-pair GEMMs: the two
                                          kernels whatever the average group */
#define MOE_PLAN_TEST_UNREACHABLE_WAIT 64 /* test hook, not for production: the
                                             decode chain in one launch seeds its
                                             per-expert counts of finished FC1 tiles
                                             with -1 instead of 0, so every FC2 tile's
                                             wait for them runs out; the launch then
                                             ends with MOE_DEV_TIMEOUT in the status
                                             word (and a wrong output).  Used with
                                             moe_plan_set_wait_limit to test that a
                                             bounded wait returns and reports. */

typedef struct moe_forward_desc {
    const moe_bf16 *x;
    const float *logits;     /* NULL in pre-routed mode */
    const int32_t *topk_ids; /* NULL in logits mode     */
    const float *topk_w;     /* NULL in logits mode     */
    const moe_bf16 *w1;
    const moe_bf16 *w2;
    moe_bf16 *out;
    void *workspace;
    size_t workspace_bytes;
    int32_t *status;         /* optional */
    int T, H, I, E, top_k, local_offset, num_local;
    int path;                /* MOE_PATH_* */
    int flags;               /* MOE_PLAN_* */
    const float *clamp_limit; /* [L] fp32 SwiGLUStep limits per local expert
                                 (moe_fc1_swiglu_step), or NULL for SwiGLU */
    int weight_format;        /* MOE_WEIGHTS_BF16 or MOE_WEIGHTS_E4M3         */
    const float *w1_scale;    /* E4M3: [L] fp32 scale of each expert's W1      */
    const float *w2_scale;    /* E4M3: [L] fp32 scale of each expert's W2      */
    float x_scale;            /* E4M3: per-tensor scale of x (FC1 input)       */
    float h_scale;            /* E4M3: per-tensor scale of h (FC2 input)       */
} moe_forward_desc;

/* Weight families of the prepared launch (flashinfer.experimental.
 * cake_stepfun_moe, opening paragraph: bf16 and fp8 (per-tensor) among the
 * families served).  MOE_WEIGHTS_E4M3, the library's reading of the fp8
 * per-tensor family: w1 / w2 hold E4M3 codes (uint8, the same [L, 2I, H] /
 * [L, H, I] layouts) with one fp32 scale per expert and tensor (w1_scale,
 * w2_scale); x enters FC1 as e4m3(x / x_scale) and h enters FC2 as
 * e4m3(h / h_scale) (the requantisation between the GEMMs; h is not rounded
 * to bf16), codes rounded to nearest even and saturated at 448; FC1's
 * accumulator is dequantised by x_scale * w1_scale[e] before the SwiGLU(Step),
 * FC2's by h_scale * w2_scale[e]; the combine and out are as in the bf16
 * family.  E4M3 plans run the grouped path with one-CTA tcgen05 kernels
 * (kind::f8f6f4) for any T; H % 128 == 0, I % 128 == 0; MOE_PATH_DECODE is
 * refused (MOE_ERR_SHAPE). */
#define MOE_WEIGHTS_BF16 0
#define MOE_WEIGHTS_E4M3 1

typedef struct moe_plan moe_plan;

/* Device pointers to the intermediates a launch leaves in the workspace
 * (the do_finalize=False outputs of flashinfer.experimental.cake_stepfun_moe,
 * Prepared launches, plus the sort and FC1 results). */
typedef struct moe_plan_buffers {
    int32_t *topk_ids;    /* [T*top_k]; the caller's in pre-routed mode   */
    float *topk_w;        /* [T*top_k]                                     */
    int32_t *m_indptr;    /* [L+1]                                         */
    int32_t *perm_to_exp; /* [T*top_k]                                     */
    int32_t *exp_to_perm; /* [T*top_k]                                     */
    moe_bf16 *xp;         /* [T*top_k, H] (grouped path)                   */
    moe_bf16 *h;          /* [T*top_k, I]                                  */
    float *y;             /* [T*top_k, H]                                  */
    int path;             /* the path the plan runs                        */
} moe_plan_buffers;

MOE_API int moe_forward_prepare(const moe_forward_desc *desc, moe_plan **plan);
MOE_API int moe_plan_launch(moe_plan *plan, void *stream);
MOE_API int moe_plan_buffers_get(const moe_plan *plan, moe_plan_buffers *out);
/* Longest a single wait inside this plan's kernels may take before the kernel
 * gives up, raises MOE_DEV_TIMEOUT in the status word and returns (every
 * in-kernel wait is bounded: on a TMA copy, an MMA, a ring slot or another
 * CTA's count).  Default 4 s.  MOE_WAIT_LIMIT_MIN_NS <= limit_ns <=
 * MOE_WAIT_LIMIT_MAX_NS, else MOE_ERR_SHAPE.  Takes effect at the next launch
 * (a CUDA graph keeps the limit it was captured with).  A limit shorter than a
 * kernel's normal waits makes a correct launch report a timeout. */
#define MOE_WAIT_LIMIT_MIN_NS 1000ull
#define MOE_WAIT_LIMIT_MAX_NS 600000000000ull
MOE_API int moe_plan_set_wait_limit(moe_plan *plan, unsigned long long limit_ns);
/* Stage timing (plans prepared with MOE_PLAN_STAGE_TIMING): the number of
 * stages and their names; moe_plan_stage_times waits for the recorded events
 * and returns, per stage, the summed milliseconds over the launches since
 * the last reset (at most 1024 launches are recorded). */
MOE_API int moe_plan_stage_count(const moe_plan *plan);
MOE_API const char *moe_plan_stage_name(const moe_plan *plan, int stage);
MOE_API int moe_plan_stage_times(moe_plan *plan, float *ms, int max_stages,
                         int *n_launches);
MOE_API int moe_plan_stage_reset(moe_plan *plan);
/* Number of kernels one moe_plan_launch enqueues (depends on the path, the
 * shape and the plan flags only; memsets are not counted).  On the grouped
 * path with the small-group kernel, each GEMM counts two kernels. */
MOE_API int moe_plan_kernels_per_launch(const moe_plan *plan);
MOE_API int moe_plan_destroy(moe_plan *plan);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
