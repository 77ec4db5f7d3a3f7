/*
 * CPU oracle for the routed MoE expert-layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library: every step below is written out plainly, in the order the
 * documentation pages state it, with no blocking, fusion or reordering.
 *
 * Sources (page title, section):
 *   [P4] "flashinfer.fused_moe.cute_dsl_fused_moe_bf16", summary formula:
 *        out[t] = sum_k scale[t,k] * ffn(x[t]; e[t,k]),
 *        ffn(x; e) = (silu(x . W1_gate[e]^T) * (x . W1_up[e]^T)) . W2[e]^T
 *   [P4] same page, "Supported configuration": bf16 operands, fp32
 *        accumulation; EP via num_local_experts / local_expert_offset with
 *        routes outside the local shard contributing zero.
 *   [P4] same page, "Parameters", use_fused_finalize=False: GEMM2 leaves
 *        unscaled rows per (token, slot); the combine applies the scales and
 *        sums in fp32 in a fixed order with one final rounding.
 *   [P1] "flashinfer.experimental.cake_stepfun_moe", opening paragraphs:
 *        routing is "Renormalize top-k" (softmax, top-k, renormalise).
 *   [P2] "flashinfer.fused_moe.cake / cake_cute (MXFP4 SiTU routed MoE)",
 *        "Host plan": the canonical W1 bank holds the up rows, then the gate
 *        rows ([up | gate]).
 *   [P1] same page, opening paragraph and "Unified MoE API opt-in": the
 *        StepFun activation SwiGLUStep(limit) with a per-expert clamp limit
 *        (gemm1_clamp_limit).
 *   [P5] "flashinfer.fused_moe.prepare_bgmv_moe": BGMV LoRA shrink + expand
 *        over routed (token, expert) pairs, one owner per output that
 *        accumulates routes in fixed input order, FP32 output accumulator.
 *   [P1] same page, opening paragraph: the fp8 (per-tensor) weight family.
 *   [P3] "Cake ragged BF16 grouped GEMM (experimental)", operation table:
 *        Y[offs[e-1]:offs[e]] = X[offs[e-1]:offs[e]] . W[e]^T, offs holding
 *        cumulative group end offsets, groups may be empty; dgrad
 *        dX = G . W[e] (W in place, bf16 out) and wgrad dW[e] = G^T . X
 *        (bf16 or fp32 out, exact zeros for an empty group) per group.
 *
 * Precision: the pages fix fp32 accumulation with bf16 inputs and outputs, so
 * the oracle computes in fp32.  The only roundings to bf16 are the SwiGLU
 * intermediate h and the final output (and the grouped GEMM output Y).  Every
 * sum runs sequentially in index order.  Build with -ffp-contract=off so that
 * a*b+c is never fused into one rounding on any host.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - top-k is chosen on the logits (softmax is strictly increasing, so the
 *     chosen set is the same), ordered by value descending, ties to the lower
 *     expert id;
 *   - the renormalised weight of slot j is exp(l_j - l_0) / sum_i exp(l_i - l_0)
 *     over the chosen k only (the full softmax denominator cancels);
 *   - silu(g) = g / (1 + exp(-g)) in fp32; u and g are not rounded, h is;
 *   - SwiGLUStep(limit) clamps GEMM1's two outputs before the activation:
 *     the gate from above at limit, the up projection to [-limit, limit];
 *     h = bf16(silu(min(g, limit)) * clamp(u, -limit, limit)), limit taken
 *     per local expert; no limit (or +inf) is the plain SwiGLU;
 *   - the unscaled GEMM2 rows y stay fp32;
 *   - the pre-routed mode takes ids and weights as given (the caller
 *     normalised them); ids outside [0, E) are dropped and flagged.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BAD_EXPERT 1

/* ---- bf16 <-> fp32 from the IEEE-754 binary32 layout -------------------- */

/* bf16 is the upper 16 bits of a binary32, so widening is exact. */
static float bf16_to_float(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to even.  The dropped low half
 * is compared against one half of the bf16 ulp (0x8000); at exactly one half
 * the kept part is rounded to even.  NaN maps to a quiet NaN. */
static uint16_t float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t hi = u >> 16;
    uint32_t lo = u & 0xffffu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u)))
        hi += 1u;
    return (uint16_t)hi;
}

/* ---- FP8 E4M3 (the OCP 8-bit format "E4M3FN") ---------------------------
 * Bits s eeee mmm, exponent bias 7.  e = 0: subnormal, (m / 8) * 2^-6;
 * otherwise (1 + m / 8) * 2^(e - 7).  The largest finite magnitude is
 * 1.75 * 2^8 = 448 (code 0x7E); 0x7F and 0xFF are NaN; there is no infinity. */
static float e4m3_to_float(uint8_t b) {
    int e = (b >> 3) & 15, m = b & 7;
    float v = e == 0 ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
    return (b & 0x80) ? -v : v;
}

/* fp32 -> E4M3, round to nearest, ties to even code, magnitudes above 448
 * saturating to 448 (finite inputs).  Subnormal range: q = round(|f| * 2^9)
 * is the code itself (q = 8 is the smallest normal, code 0x08); normal range:
 * |f| = mant * 2^e with mant in [1, 2), q = round(mant * 8) in [8, 16]. */
static uint8_t float_to_e4m3(float f) {
    uint8_t s = signbit(f) ? 0x80 : 0x00;
    float a = fabsf(f);
    if (a >= 448.0f) return (uint8_t)(s | 0x7E);
    if (a < ldexpf(1.0f, -6)) {
        float q = nearbyintf(ldexpf(a, 9)); /* default rounding: nearest, ties even */
        return (uint8_t)(s | (uint8_t)q);
    }
    int k;
    float fr = frexpf(a, &k);       /* a = fr * 2^k, fr in [0.5, 1) */
    int e = k - 1;                  /* a = mant * 2^e, mant in [1, 2) */
    float q = nearbyintf(ldexpf(fr, 4)); /* mant * 8 = fr * 16 */
    if (q == 16.0f) {
        q = 8.0f;
        e += 1;
    }
    int code = ((e + 7) << 3) | ((int)q - 8);
    if (code > 0x7E) code = 0x7E;
    return (uint8_t)(s | (uint8_t)code);
}

uint8_t oracle_float_to_e4m3(float f) { return float_to_e4m3(f); }
float oracle_e4m3_to_float(uint8_t b) { return e4m3_to_float(b); }

uint16_t oracle_float_to_bf16(float f) { return float_to_bf16(f); }
float oracle_bf16_to_float(uint16_t b) { return bf16_to_float(b); }

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* ---- routing: softmax -> top-k -> renormalise  [P1 opening; P4 params] -- */

/* logits [T, E] fp32 row-major -> ids [T, k] int32, w [T, k] fp32. */
void oracle_route(const float *logits, int T, int E, int k, int32_t *ids,
                  float *w, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        char *taken = (char *)calloc((size_t)E, 1);
        int32_t *sel = ids + (size_t)t * k;
        /* k rounds of "largest remaining logit"; scanning ids upwards with a
         * strict '>' keeps the lowest id among equal values. */
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            sel[j] = best;
        }
        free(taken);
        /* softmax over the chosen k: exp(l_j - max) / sum */
        float m = l[sel[0]];
        float ex[64];
        float s = 0.0f;
        for (int j = 0; j < k; ++j) {
            ex[j] = expf(l[sel[j]] - m);
            s = s + ex[j];
        }
        for (int j = 0; j < k; ++j) w[(size_t)t * k + j] = ex[j] / s;
    }
}

/* ---- sort / permute by expert  [P3 operation table; P1 prepared launches] -
 *
 * Routes are indexed by the expanded index r = t*k + j.  Local experts are the
 * ids in [off, off+L).  m_indptr[L+1] has a leading zero; group i (global
 * expert off+i) is permuted rows [m_indptr[i], m_indptr[i+1]).  Inside a group
 * rows keep ascending r (a stable counting sort).  perm_to_exp[p] = r for
 * p < M = m_indptr[L]; exp_to_perm[r] = p, or -1 for a route that is not local
 * (or whose id is outside [0, E)).  Returns ORACLE_BAD_EXPERT when any id is
 * outside [0, E). */
int oracle_sort(const int32_t *ids, int T, int k, int E, int off, int L,
                int32_t *m_indptr, int32_t *perm_to_exp, int32_t *exp_to_perm) {
    int status = 0;
    long R = (long)T * k;
    int32_t *cnt = (int32_t *)calloc((size_t)L + 1, sizeof(int32_t));
    for (long r = 0; r < R; ++r) {
        int e = ids[r];
        if (e < 0 || e >= E) { status |= ORACLE_BAD_EXPERT; continue; }
        if (e >= off && e < off + L) cnt[e - off] += 1;
    }
    m_indptr[0] = 0;
    for (int i = 0; i < L; ++i) m_indptr[i + 1] = m_indptr[i] + cnt[i];
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * ((size_t)L + 1));
    for (int i = 0; i < L; ++i) next[i] = m_indptr[i];
    for (long r = 0; r < R; ++r) {
        int e = ids[r];
        if (e < 0 || e >= E || e < off || e >= off + L) {
            exp_to_perm[r] = -1;
            continue;
        }
        int p = next[e - off]++;
        perm_to_exp[p] = (int32_t)r;
        exp_to_perm[r] = p;
    }
    free(next);
    free(cnt);
    return status;
}

/* ---- SwiGLU and SwiGLUStep(limit)  [P4 formula; P1 SwiGLUStep reading] ----
 *
 * silu(g) * u in fp32 after clamping g from above at `limit` and u to
 * [-limit, limit]; with limit = +inf both comparisons are false and this is
 * the plain SwiGLU of the summary formula. */
static float swiglu_step(float g, float u, float limit) {
    if (g > limit) g = limit;
    if (u > limit) u = limit;
    if (u < -limit) u = -limit;
    float silu_g = g / (1.0f + expf(-g));
    return silu_g * u;
}

/* per-expert limit of local expert e, +inf without limits */
static float limit_of(const float *clamp, int e) {
    return clamp ? clamp[e] : INFINITY;
}

/* ---- one expert's FFN on one row  [P4 formula; P2 host plan for W1 rows] --
 *
 * x_row [H] bf16; w1e [2I, H] bf16 with rows 0..I-1 = up, I..2I-1 = gate;
 * w2e [H, I] bf16; limit the expert's SwiGLUStep clamp (+inf: none).
 * Writes h [I] bf16 and y [H] fp32 (unscaled, unrounded). */
static void expert_ffn_row(const uint16_t *x_row, const uint16_t *w1e,
                           const uint16_t *w2e, int H, int I, float limit,
                           uint16_t *h, float *y) {
    for (int n = 0; n < I; ++n) {
        const uint16_t *up_row = w1e + (size_t)n * H;
        const uint16_t *gate_row = w1e + (size_t)(I + n) * H;
        float u = 0.0f, g = 0.0f;
        for (int c = 0; c < H; ++c) {
            float xv = bf16_to_float(x_row[c]);
            u = u + xv * bf16_to_float(up_row[c]);
            g = g + xv * bf16_to_float(gate_row[c]);
        }
        h[n] = float_to_bf16(swiglu_step(g, u, limit));
    }
    for (int c = 0; c < H; ++c) {
        const uint16_t *w2_row = w2e + (size_t)c * I;
        float acc = 0.0f;
        for (int n = 0; n < I; ++n)
            acc = acc + bf16_to_float(h[n]) * bf16_to_float(w2_row[n]);
        y[c] = acc;
    }
}

/* ---- the combine of one token  [P4 Parameters, use_fused_finalize=False] --
 * out[c] = bf16( sum over the local slots j, ascending, of w[j] * y[j][c] ),
 * fp32 with one final rounding. */
static void combine_row(const float *w, const float *y, const char *local, int k, int H,
                        uint16_t *out) {
    for (int c = 0; c < H; ++c) {
        float acc = 0.0f;
        for (int j = 0; j < k; ++j)
            if (local[j])
                acc = acc + w[j] * y[(size_t)j * H + c];
        out[c] = float_to_bf16(acc);
    }
}

/* ---- whole layer for a list of tokens  [P4 formula, EP rule, combine] -----
 *
 * x [T, H] bf16; ids, w [T, k]; w1 [L, 2I, H]; w2 [L, H, I] (local experts,
 * local index = global id - off).  tokens[n_tok] selects which tokens to
 * evaluate; out [n_tok, H] bf16 row i belongs to token tokens[i].
 * Optional h_out [n_tok*k, I] bf16 and y_out [n_tok*k, H] fp32 receive the
 * per-route intermediates in (token, slot) order; rows of routes that are not
 * local are left untouched.  clamp [L] (or NULL) holds each local expert's
 * SwiGLUStep limit.  Returns ORACLE_BAD_EXPERT if any selected route has an
 * id outside [0, E). */
int oracle_moe_tokens(const uint16_t *x, const int32_t *ids, const float *w,
                      const uint16_t *w1, const uint16_t *w2, int T, int H,
                      int I, int E, int k, int off, int L,
                      const int32_t *tokens, int n_tok, uint16_t *out,
                      uint16_t *h_out, float *y_out, int nthreads,
                      const float *clamp) {
    (void)T;
    int status = 0;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int i = 0; i < n_tok; ++i) {
        int t = tokens[i];
        uint16_t *h = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)I);
        float *y = (float *)malloc(sizeof(float) * (size_t)H * (size_t)k);
        char *local = (char *)calloc((size_t)k, 1);
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            if (e < 0 || e >= E) { status |= ORACLE_BAD_EXPERT; continue; }
            if (e < off || e >= off + L) continue; /* contributes zero */
            local[j] = 1;
            const uint16_t *w1e = w1 + (size_t)(e - off) * 2 * I * H;
            const uint16_t *w2e = w2 + (size_t)(e - off) * H * I;
            expert_ffn_row(x + (size_t)t * H, w1e, w2e, H, I,
                           limit_of(clamp, e - off), h, y + (size_t)j * H);
            if (h_out)
                memcpy(h_out + ((size_t)i * k + j) * I, h, sizeof(uint16_t) * I);
            if (y_out)
                memcpy(y_out + ((size_t)i * k + j) * H, y + (size_t)j * H,
                       sizeof(float) * H);
        }
        combine_row(w + (size_t)t * k, y, local, k, H, out + (size_t)i * H);
        free(local);
        free(y);
        free(h);
    }
    return status;
}

/* ---- stages on permuted rows (for stage-by-stage comparisons) ------------
 *
 * The permuted layout: group i of the L local experts is rows
 * [group_end[i-1], group_end[i]) (group_end[-1] = 0)  [P3 operation table]. */
static int group_of_row(const int32_t *group_end, int L, int p) {
    for (int i = 0; i < L; ++i)
        if (p < group_end[i]) return i;
    return -1;
}

/* FC1 + SwiGLU on selected permuted rows: xp [*, H] bf16, w1 [L, 2I, H],
 * rows[n_rows] -> h_rows [n_rows, I] bf16; clamp [L] or NULL as above. */
void oracle_fc1_swiglu_rows(const uint16_t *xp, const uint16_t *w1,
                            const int32_t *group_end, int L, int H, int I,
                            const int32_t *rows, int n_rows, uint16_t *h_rows,
                            int nthreads, const float *clamp) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n_rows; ++q) {
        int p = rows[q];
        int g = group_of_row(group_end, L, p);
        const uint16_t *xr = xp + (size_t)p * H;
        const uint16_t *w1e = w1 + (size_t)g * 2 * I * H;
        for (int n = 0; n < I; ++n) {
            float u = 0.0f, gt = 0.0f;
            for (int c = 0; c < H; ++c) {
                float xv = bf16_to_float(xr[c]);
                u = u + xv * bf16_to_float(w1e[(size_t)n * H + c]);
                gt = gt + xv * bf16_to_float(w1e[(size_t)(I + n) * H + c]);
            }
            h_rows[(size_t)q * I + n] =
                float_to_bf16(swiglu_step(gt, u, limit_of(clamp, g)));
        }
    }
}

/* FC2 on selected permuted rows: h [*, I] bf16, w2 [L, H, I] ->
 * y_rows [n_rows, H] fp32 (unrounded). */
void oracle_fc2_rows(const uint16_t *h, const uint16_t *w2,
                     const int32_t *group_end, int L, int H, int I,
                     const int32_t *rows, int n_rows, float *y_rows,
                     int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n_rows; ++q) {
        int p = rows[q];
        int g = group_of_row(group_end, L, p);
        const uint16_t *hr = h + (size_t)p * I;
        const uint16_t *w2e = w2 + (size_t)g * H * I;
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int n = 0; n < I; ++n)
                acc = acc + bf16_to_float(hr[n]) *
                                bf16_to_float(w2e[(size_t)c * I + n]);
            y_rows[(size_t)q * H + c] = acc;
        }
    }
}

/* Combine: out[t] = bf16( sum_j w[t,j] * y[exp_to_perm[t*k+j]] ), j ascending,
 * skipping slots with exp_to_perm == -1  [P4 params, deterministic path]. */
void oracle_finalize(const float *y, const int32_t *exp_to_perm,
                     const float *w, int T, int k, int H, uint16_t *out,
                     int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                int p = exp_to_perm[(size_t)t * k + j];
                if (p < 0) continue;
                acc = acc + w[(size_t)t * k + j] * y[(size_t)p * H + c];
            }
            out[(size_t)t * H + c] = float_to_bf16(acc);
        }
    }
}

/* Ragged grouped GEMM forward on selected rows  [P3 operation table, fwd]:
 * X [sum_m, K] bf16, W [E, N, K] bf16, offs[E] cumulative ends.  Row p of
 * group e: Y[p, n] = bf16( sum_c X[p,c] * W[e,n,c] ). */
void oracle_grouped_gemm_rows(const uint16_t *X, const uint16_t *W,
                              const int32_t *offs, int E, int N, int K,
                              const int32_t *rows, int n_rows,
                              uint16_t *Y_rows, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n_rows; ++q) {
        int p = rows[q];
        int e = group_of_row(offs, E, p);
        const uint16_t *xr = X + (size_t)p * K;
        const uint16_t *we = W + (size_t)e * N * K;
        for (int n = 0; n < N; ++n) {
            float acc = 0.0f;
            for (int c = 0; c < K; ++c)
                acc = acc + bf16_to_float(xr[c]) *
                                bf16_to_float(we[(size_t)n * K + c]);
            Y_rows[(size_t)q * N + n] = float_to_bf16(acc);
        }
    }
}

/* ---- ragged grouped GEMM backward  [P3 operation table: dgrad, wgrad] -----
 *
 * Groups as in the forward: group e is rows [offs[e-1], offs[e]) of the
 * packed activations (offs[-1] = 0).
 *
 * dgrad, W used in place: dX[p, c] = bf16( sum_{n=0..N-1} G[p,n] * W[e,n,c] )
 * for row p of group e; G [sum_m, N], W [E, N, K], the sum sequential in n
 * in fp32.  Writes the listed rows into dX_rows [n_rows, K]. */
void oracle_grouped_gemm_dgrad_rows(const uint16_t *G, const uint16_t *W,
                                    const int32_t *offs, int E, int N, int K,
                                    const int32_t *rows, int n_rows,
                                    uint16_t *dX_rows, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n_rows; ++q) {
        int p = rows[q];
        int e = group_of_row(offs, E, p);
        const uint16_t *gr = G + (size_t)p * N;
        const uint16_t *we = W + (size_t)e * N * K;
        for (int c = 0; c < K; ++c) {
            float acc = 0.0f;
            for (int n = 0; n < N; ++n)
                acc = acc + bf16_to_float(gr[n]) *
                                bf16_to_float(we[(size_t)n * K + c]);
            dX_rows[(size_t)q * K + c] = float_to_bf16(acc);
        }
    }
}

/* wgrad: dW[e, n, c] = sum over the rows p of group e, ascending, of
 * G[p,n] * X[p,c] in fp32 (an empty group gives exactly 0); G [sum_m, N],
 * X [sum_m, K].  For each listed (e, n) pair q writes the K values of row n
 * of dW[e] into dW_f32 [n_sel, K] (fp32, when not NULL) and dW_bf16
 * [n_sel, K] (one bf16 rounding of the fp32 sum, when not NULL). */
void oracle_grouped_gemm_wgrad_rows(const uint16_t *G, const uint16_t *X,
                                    const int32_t *offs, int E, int N, int K,
                                    const int32_t *sel_e, const int32_t *sel_n,
                                    int n_sel, float *dW_f32, uint16_t *dW_bf16,
                                    int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n_sel; ++q) {
        int e = sel_e[q], n = sel_n[q];
        int start = e == 0 ? 0 : offs[e - 1];
        int end = offs[e];
        for (int c = 0; c < K; ++c) {
            float acc = 0.0f;
            for (int p = start; p < end; ++p)
                acc = acc + bf16_to_float(G[(size_t)p * N + n]) *
                                bf16_to_float(X[(size_t)p * K + c]);
            if (dW_f32) dW_f32[(size_t)q * K + c] = acc;
            if (dW_bf16) dW_bf16[(size_t)q * K + c] = float_to_bf16(acc);
        }
    }
}

/* ---- BGMV LoRA-MoE shrink + expand  [P5 prepare_bgmv_moe: description and
 * Parameters] -------------------------------------------------------------
 *
 * Routed pairs p = 0..P-1 (any order): token t = tok[p], expert e = eid[p],
 * LoRA l = lora[t], routing weight w[p].  For every slice s of the S slices
 * (rank R; A_s [num_loras, E, R, H], B_s [num_loras, E, F_s, R], bf16):
 *
 *   shrink[s, p, r] = bf16( sum_h A_s[l, e, r, h] * x[t, h] )
 *                     (fp32, sequential in h; the shrink workspace holds the
 *                     weight dtype)
 *   y[t, off_s + f] = sum over the pairs p of token t, in ascending p, of
 *                     w[p] * ( sum_r B_s[l, e, f, r] * shrink[s, p, r] )
 *                     (fp32, sequential; "each output has one owner that
 *                     accumulates routes in fixed input order")
 *
 * where off_s = F_0 + .. + F_{s-1} and y has ld_y >= sum F_s floats per row.
 * A token without pairs gets zeros.  A pair whose token, expert or LoRA index
 * is out of range is dropped (its shrink rows are zero) and the call returns
 * ORACLE_BAD_EXPERT (the page treats routing indices out of range as invalid
 * inputs). */
int oracle_bgmv(const uint16_t *x, int T, int H, const uint16_t *const *lora_a,
                const uint16_t *const *lora_b, int S, const int *feat_out,
                int num_loras, int E, int R, const int32_t *tok,
                const int32_t *eid, const int32_t *lora, const float *w, int P,
                uint16_t *shrink, float *y, int ld_y, int nthreads) {
    int status = 0;
    char *ok = (char *)malloc((size_t)(P > 0 ? P : 1));
    for (int p = 0; p < P; ++p) {
        int t = tok[p];
        int good = t >= 0 && t < T && eid[p] >= 0 && eid[p] < E;
        if (good) good = lora[t] >= 0 && lora[t] < num_loras;
        ok[p] = (char)good;
        if (!good) status |= ORACLE_BAD_EXPERT;
    }
    set_threads(nthreads);
    /* shrink, pair by pair */
    for (int sl = 0; sl < S; ++sl) {
#pragma omp parallel for schedule(dynamic, 16)
        for (int p = 0; p < P; ++p) {
            uint16_t *out = shrink + ((size_t)sl * P + p) * R;
            if (!ok[p]) {
                for (int r = 0; r < R; ++r) out[r] = 0;
                continue;
            }
            int t = tok[p];
            const uint16_t *a = lora_a[sl] +
                                (((size_t)lora[t] * E + eid[p]) * R) * (size_t)H;
            for (int r = 0; r < R; ++r) {
                float acc = 0.0f;
                for (int h = 0; h < H; ++h)
                    acc = acc + bf16_to_float(a[(size_t)r * H + h]) *
                                    bf16_to_float(x[(size_t)t * H + h]);
                out[r] = float_to_bf16(acc);
            }
        }
    }
    /* the pairs of each token in ascending p */
    int *cnt = (int *)calloc((size_t)T + 1, sizeof(int));
    int *list = (int *)malloc(sizeof(int) * (size_t)(P > 0 ? P : 1));
    for (int p = 0; p < P; ++p)
        if (ok[p]) cnt[tok[p] + 1]++;
    for (int t = 0; t < T; ++t) cnt[t + 1] += cnt[t];
    int *fill = (int *)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
    for (int t = 0; t < T; ++t) fill[t] = cnt[t];
    for (int p = 0; p < P; ++p)
        if (ok[p]) list[fill[tok[p]]++] = p;
    /* expand: one owner per output row */
#pragma omp parallel for schedule(dynamic, 4)
    for (int t = 0; t < T; ++t) {
        int col = 0;
        for (int sl = 0; sl < S; ++sl) {
            int F = feat_out[sl];
            for (int f = 0; f < F; ++f) {
                float acc = 0.0f;
                for (int q = cnt[t]; q < cnt[t + 1]; ++q) {
                    int p = list[q];
                    const uint16_t *b = lora_b[sl] +
                                        (((size_t)lora[t] * E + eid[p]) * F + f) * (size_t)R;
                    const uint16_t *sp = shrink + ((size_t)sl * P + p) * R;
                    float v = 0.0f;
                    for (int r = 0; r < R; ++r)
                        v = v + bf16_to_float(b[r]) * bf16_to_float(sp[r]);
                    acc = acc + w[p] * v;
                }
                y[(size_t)t * ld_y + col + f] = acc;
            }
            col += F;
        }
    }
    free(fill);
    free(list);
    free(cnt);
    free(ok);
    return status;
}

/* ---- FP8 per-tensor weight family  [P1 "flashinfer.experimental.
 * cake_stepfun_moe", opening paragraph: the fp8 (per-tensor) weight family]
 *
 * Reading: W1q [L, 2I, H] and W2q [L, H, I] hold E4M3 codes with one fp32
 * scale per local expert and weight tensor (s1[e], s2[e]); the activations
 * entering each GEMM are quantised to E4M3 with one static fp32 scale per
 * tensor (a1 for x, a2 for h, the requantisation between FC1 and FC2):
 *   xq = e4m3(x / a1)
 *   u, g = (sum_c xq * W1q) * (a1 * s1[e])        fp32, sequential in c
 *   hq = e4m3(swiglu_step(g, u, limit) / a2)      (no bf16 rounding of h)
 *   y  = (sum_n hq * W2q) * (a2 * s2[e])          fp32, sequential in n
 *   out = bf16(sum_j w_j * y_j)                    as in the bf16 family
 * Products of two E4M3 values are exact in fp32. */
static void expert_ffn_row_fp8(const uint8_t *xq, const uint8_t *w1e, const uint8_t *w2e,
                               int H, int I, float scale1, float a2, float scale2,
                               float limit, uint8_t *hq, float *y) {
    for (int n = 0; n < I; ++n) {
        const uint8_t *up_row = w1e + (size_t)n * H;
        const uint8_t *gate_row = w1e + (size_t)(I + n) * H;
        float u = 0.0f, g = 0.0f;
        for (int c = 0; c < H; ++c) {
            float xv = e4m3_to_float(xq[c]);
            u = u + xv * e4m3_to_float(up_row[c]);
            g = g + xv * e4m3_to_float(gate_row[c]);
        }
        u = u * scale1;
        g = g * scale1;
        hq[n] = float_to_e4m3(swiglu_step(g, u, limit) / a2);
    }
    for (int c = 0; c < H; ++c) {
        const uint8_t *w2_row = w2e + (size_t)c * I;
        float acc = 0.0f;
        for (int n = 0; n < I; ++n)
            acc = acc + e4m3_to_float(hq[n]) * e4m3_to_float(w2_row[n]);
        y[c] = acc * scale2;
    }
}

/* x bf16 [n, H] -> xq E4M3 codes [n, H] with scale a1. */
void oracle_quantize_e4m3(const uint16_t *x, long n, float a1, uint8_t *xq) {
    for (long i = 0; i < n; ++i) xq[i] = float_to_e4m3(bf16_to_float(x[i]) / a1);
}

/* The layer with FP8 weights for the listed tokens (arguments as
 * oracle_moe_tokens; w1q, w2q E4M3 codes; s1, s2 [L]; a1, a2 scalars).
 * hq_out [n_tok*k, I] E4M3 codes and y_out [n_tok*k, H] fp32 optional. */
int oracle_moe_tokens_fp8(const uint16_t *x, const int32_t *ids, const float *w,
                          const uint8_t *w1q, const uint8_t *w2q, const float *s1,
                          const float *s2, float a1, float a2, int T, int H, int I,
                          int E, int k, int off, int L, const int32_t *tokens,
                          int n_tok, uint16_t *out, uint8_t *hq_out, float *y_out,
                          int nthreads, const float *clamp) {
    (void)T;
    int status = 0;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int i = 0; i < n_tok; ++i) {
        int t = tokens[i];
        uint8_t *xq = (uint8_t *)malloc((size_t)H);
        uint8_t *hq = (uint8_t *)malloc((size_t)I);
        float *y = (float *)malloc(sizeof(float) * (size_t)H * (size_t)k);
        char *local = (char *)calloc((size_t)k, 1);
        for (int c = 0; c < H; ++c) xq[c] = float_to_e4m3(bf16_to_float(x[(size_t)t * H + c]) / a1);
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            if (e < 0 || e >= E) { status |= ORACLE_BAD_EXPERT; continue; }
            if (e < off || e >= off + L) continue;
            local[j] = 1;
            int le = e - off;
            const uint8_t *w1e = w1q + (size_t)le * 2 * I * H;
            const uint8_t *w2e = w2q + (size_t)le * H * I;
            expert_ffn_row_fp8(xq, w1e, w2e, H, I, a1 * s1[le], a2, a2 * s2[le],
                               limit_of(clamp, le), hq, y + (size_t)j * H);
            if (hq_out) memcpy(hq_out + ((size_t)i * k + j) * I, hq, (size_t)I);
            if (y_out)
                memcpy(y_out + ((size_t)i * k + j) * H, y + (size_t)j * H, sizeof(float) * H);
        }
        combine_row(w + (size_t)t * k, y, local, k, H, out + (size_t)i * H);
        free(local);
        free(y);
        free(hq);
        free(xq);
    }
    return status;
}

/* FC1 + SwiGLU + requantisation on selected permuted rows of xq (E4M3). */
void oracle_fc1_fp8_rows(const uint8_t *xq, const uint8_t *w1q, const float *s1, float a1,
                         float a2, const int32_t *group_end, int L, int H, int I,
                         const int32_t *rows, int n_rows, uint8_t *hq_rows, int nthreads,
                         const float *clamp) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n_rows; ++q) {
        int p = rows[q];
        int g = group_of_row(group_end, L, p);
        const uint8_t *xr = xq + (size_t)p * H;
        const uint8_t *w1e = w1q + (size_t)g * 2 * I * H;
        for (int n = 0; n < I; ++n) {
            float u = 0.0f, gt = 0.0f;
            for (int c = 0; c < H; ++c) {
                float xv = e4m3_to_float(xr[c]);
                u = u + xv * e4m3_to_float(w1e[(size_t)n * H + c]);
                gt = gt + xv * e4m3_to_float(w1e[(size_t)(I + n) * H + c]);
            }
            float sc = a1 * s1[g];
            hq_rows[(size_t)q * I + n] =
                float_to_e4m3(swiglu_step(gt * sc, u * sc, limit_of(clamp, g)) / a2);
        }
    }
}

/* FC2 with the dequantisation on selected permuted rows of hq (E4M3) ->
 * y_rows [n_rows, H] fp32. */
void oracle_fc2_fp8_rows(const uint8_t *hq, const uint8_t *w2q, const float *s2, float a2,
                         const int32_t *group_end, int L, int H, int I, const int32_t *rows,
                         int n_rows, float *y_rows, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < n_rows; ++q) {
        int p = rows[q];
        int g = group_of_row(group_end, L, p);
        const uint8_t *hr = hq + (size_t)p * I;
        const uint8_t *w2e = w2q + (size_t)g * H * I;
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int n = 0; n < I; ++n)
                acc = acc + e4m3_to_float(hr[n]) * e4m3_to_float(w2e[(size_t)c * I + n]);
            y_rows[(size_t)q * H + c] = acc * (a2 * s2[g]);
        }
    }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
