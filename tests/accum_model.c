/*
 * accum_model.c -- two more CPU evaluations of the routed MoE layer, used only
 * to derive the end-to-end acceptance floor of the parity tests.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library loads this file; it shares
 * no code with the oracle (oracle/) or with the CUDA path.  The layer is the
 * one of flashinfer.fused_moe.cute_dsl_fused_moe_bf16 (summary formula):
 *   out[t] = bf16( sum_j w[t,j] * y_j ),  y_j = h_j . W2[e]^T,
 *   h_j = bf16( silu(x[t] . W1_gate[e]^T) * (x[t] . W1_up[e]^T) ),
 * with W1 rows [up | gate], fp32 sums, h rounded to bf16 once, y in fp32, the
 * combine sequential in fp32 over j, one final bf16 rounding.  The two
 * evaluations differ from the oracle only in how each dot product's fp32 sum
 * is accumulated:
 *
 *   mode 0 (blocked fp32): the K products are taken in consecutive blocks of
 *     16; each block is summed sequentially in fp32 (round to nearest even),
 *     and the block sum is added to the running fp32 sum.  A correct fp32
 *     implementation that only sums in another order than the oracle.
 *
 *   mode 1 (tensor-core accumulation model): blocks of 16 consecutive products
 *     (the K of one bf16 MMA step) are added to the fp32 accumulator together:
 *     the 16 exact products and the accumulator are aligned to the largest
 *     magnitude among them, every term is cut toward zero to 2 bits below the
 *     fp32 precision of that magnitude (25 bits), the cut terms are summed
 *     exactly, and the sum is cut toward zero to fp32.  This is the kind of
 *     fixed-point block accumulation described for tensor cores by Fasi,
 *     Higham, Mikaitis and Pranesh, "Numerical behavior of NVIDIA tensor
 *     cores", PeerJ Computer Science 7:e330 (2021); block length and guard
 *     bits are the choice this file makes.
 *
 * Products of two bf16 values are exact in double, and the cut terms of one
 * block are multiples of one power of two below 2^31 of them, so every double
 * sum here is exact; only the stated cuts and roundings lose information.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define BLOCK 16
#define GUARD_BITS 2

static float am_bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* bf16 round to nearest even (finite inputs). */
static uint16_t am_float_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  const uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* fp32 nearest to x toward zero. */
static float am_round_toward_zero(double x) {
  float f = (float)x;
  if (fabs((double)f) > fabs(x)) f = nextafterf(f, 0.0f);
  return f;
}

/* One dot product a . b of bf16 vectors (stride 1), accumulated per `mode`. */
double am_dot(const uint16_t *a, const uint16_t *b, int K, int mode) {
  float acc = 0.0f;
  for (int k0 = 0; k0 < K; k0 += BLOCK) {
    const int n = K - k0 < BLOCK ? K - k0 : BLOCK;
    double p[BLOCK + 1];
    for (int i = 0; i < n; ++i)
      p[i] = (double)am_bf16_to_float(a[k0 + i]) * (double)am_bf16_to_float(b[k0 + i]);
    if (mode == 0) {
      float s = 0.0f;
      for (int i = 0; i < n; ++i) s = s + (float)p[i]; /* each product is exact in fp32 */
      acc = acc + s;
      continue;
    }
    p[n] = (double)acc;
    double big = 0.0;
    for (int i = 0; i <= n; ++i)
      if (fabs(p[i]) > big) big = fabs(p[i]);
    if (big == 0.0) continue;
    const int e = ilogb(big);                         /* 2^e <= big < 2^(e+1) */
    const double up = ldexp(1.0, 23 + GUARD_BITS - e);  /* terms in units of the cut */
    double s = 0.0;
    for (int i = 0; i <= n; ++i) s += trunc(p[i] * up);
    acc = am_round_toward_zero(s / up);
  }
  return (double)acc;
}

/* out[m*N + n] = a[m] . b[n] for A [M, K], B [N, K] (bf16 bits), per `mode`. */
void am_dots(const uint16_t *A, const uint16_t *B, int M, int N, int K, int mode, double *out) {
#pragma omp parallel for schedule(static)
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) out[(size_t)m * N + n] = am_dot(A + (size_t)m * K, B + (size_t)n * K, K, mode);
}

/* The layer for the listed tokens.  x [T,H], ids/w [T,k], w1 [L,2I,H],
 * w2 [L,H,I] (bf16 bits); routes to ids outside [off, off+L) contribute zero.
 * out [n_tok, H] bf16 bits; h_out (optional) [n_tok*k, I] bf16 bits; clamp
 * (optional) [L] per-local-expert SwiGLUStep limits (gate clamped from above,
 * up to [-limit, limit], before silu(g) * u).
 * Returns 0, 1 if an id is outside [0, E), 2 if host memory ran out. */
int am_moe_tokens(const uint16_t *x, const int32_t *ids, const float *w, const uint16_t *w1,
                  const uint16_t *w2, int T, int H, int I, int E, int k, int off, int L,
                  const int32_t *tokens, int n_tok, uint16_t *out, uint16_t *h_out, int mode,
                  int nthreads, const float *clamp) {
  (void)T;
  int bad = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int i = 0; i < n_tok; ++i) {
    const int t = tokens[i];
    const uint16_t *xt = x + (size_t)t * H;
    /* per route: h (bf16) then y (fp32 per column) */
    float *ys = (float *)malloc(sizeof(float) * (size_t)k * H);
    uint16_t *hb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)I);
    if (!ys || !hb) {
      free(ys);
      free(hb);
      bad |= 2;
      continue;
    }
    int local[16];
    for (int j = 0; j < k; ++j) {
      const int g = ids[(size_t)t * k + j];
      local[j] = 0;
      if (g < 0 || g >= E) {
        bad = 1;
        continue;
      }
      if (g < off || g >= off + L) continue;
      local[j] = 1;
      const int e = g - off;
      const uint16_t *W1 = w1 + (size_t)e * 2 * I * H;
      const uint16_t *W2 = w2 + (size_t)e * H * I;
      const float lim = clamp ? clamp[e] : INFINITY;
      for (int c = 0; c < I; ++c) {
        float u = (float)am_dot(xt, W1 + (size_t)c * H, H, mode);
        float gt = (float)am_dot(xt, W1 + (size_t)(I + c) * H, H, mode);
        gt = gt > lim ? lim : gt;
        u = u > lim ? lim : (u < -lim ? -lim : u);
        const float silu = gt / (1.0f + expf(-gt));
        hb[c] = am_float_to_bf16(silu * u);
      }
      if (h_out) memcpy(h_out + ((size_t)i * k + j) * I, hb, sizeof(uint16_t) * (size_t)I);
      for (int c = 0; c < H; ++c) ys[(size_t)j * H + c] = (float)am_dot(hb, W2 + (size_t)c * I, I, mode);
    }
    for (int c = 0; c < H; ++c) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j)
        if (local[j]) acc = acc + w[(size_t)t * k + j] * ys[(size_t)j * H + c];
      out[(size_t)i * H + c] = am_float_to_bf16(acc);
    }
    free(ys);
    free(hb);
  }
  return bad;
}

/* ---- the fp8 per-tensor family (E4M3 operands) --------------------------
 * xq = e4m3(x / a1); u, g = model dot of xq and W1q rows times a1 * s1[e];
 * hq = e4m3(swiglu(limit) / a2); y = model dot of hq and W2q rows times
 * a2 * s2[e]; the combine as above.  In mode 1 the blocks are 32 products
 * (the K of one E4M3 MMA); products of two E4M3 values are exact. */
static float am_e4m3_to_float(uint8_t b) {
  const int e = (b >> 3) & 15, m = b & 7;
  const float v = e == 0 ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
  return (b & 0x80) ? -v : v;
}

/* nearest E4M3 code by search over the 127 magnitudes, ties to the even code,
 * above 448 saturating */
static uint8_t am_float_to_e4m3(float f) {
  const uint8_t s = signbit(f) ? 0x80 : 0;
  const float a = fabsf(f);
  if (a >= 448.0f) return s | 0x7E;
  int best = 0;
  float bd = a;
  for (int c = 1; c <= 0x7E; ++c) {
    const float d = fabsf(am_e4m3_to_float((uint8_t)c) - a);
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  return (uint8_t)(s | best);
}

static double am_dot_q(const uint8_t *a, const uint8_t *b, int K, int mode) {
  enum { QB = 32 };
  float acc = 0.0f;
  for (int k0 = 0; k0 < K; k0 += QB) {
    const int n = K - k0 < QB ? K - k0 : QB;
    double p[QB + 1];
    for (int i = 0; i < n; ++i) p[i] = (double)am_e4m3_to_float(a[k0 + i]) * (double)am_e4m3_to_float(b[k0 + i]);
    if (mode == 0) {
      float s = 0.0f;
      for (int i = 0; i < n; ++i) s = s + (float)p[i];
      acc = acc + s;
      continue;
    }
    p[n] = (double)acc;
    double big = 0.0;
    for (int i = 0; i <= n; ++i)
      if (fabs(p[i]) > big) big = fabs(p[i]);
    if (big == 0.0) continue;
    const double up = ldexp(1.0, 23 + GUARD_BITS - ilogb(big));
    double s = 0.0;
    for (int i = 0; i <= n; ++i) s += trunc(p[i] * up);
    acc = am_round_toward_zero(s / up);
  }
  return (double)acc;
}

int am_moe_tokens_e4m3(const uint16_t *x, const int32_t *ids, const float *w, const uint8_t *w1q,
                       const uint8_t *w2q, const float *s1, const float *s2, float a1, float a2, int T,
                       int H, int I, int E, int k, int off, int L, const int32_t *tokens, int n_tok,
                       uint16_t *out, int mode, int nthreads, const float *clamp) {
  (void)T;
  int bad = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int i = 0; i < n_tok; ++i) {
    const int t = tokens[i];
    uint8_t *xq = (uint8_t *)malloc((size_t)H);
    uint8_t *hq = (uint8_t *)malloc((size_t)I);
    float *ys = (float *)malloc(sizeof(float) * (size_t)k * H);
    if (!xq || !hq || !ys) {
      free(xq);
      free(hq);
      free(ys);
      bad |= 2;
      continue;
    }
    for (int c = 0; c < H; ++c) xq[c] = am_float_to_e4m3(am_bf16_to_float(x[(size_t)t * H + c]) / a1);
    int local[16];
    for (int j = 0; j < k; ++j) {
      const int g = ids[(size_t)t * k + j];
      local[j] = 0;
      if (g < 0 || g >= E) {
        bad |= 1;
        continue;
      }
      if (g < off || g >= off + L) continue;
      local[j] = 1;
      const int e = g - off;
      const uint8_t *W1 = w1q + (size_t)e * 2 * I * H;
      const uint8_t *W2 = w2q + (size_t)e * H * I;
      const float sc1 = a1 * s1[e], sc2 = a2 * s2[e];
      const float lim = clamp ? clamp[e] : INFINITY;
      for (int c = 0; c < I; ++c) {
        float u = (float)am_dot_q(xq, W1 + (size_t)c * H, H, mode) * sc1;
        float gt = (float)am_dot_q(xq, W1 + (size_t)(I + c) * H, H, mode) * sc1;
        gt = gt > lim ? lim : gt;
        u = u > lim ? lim : (u < -lim ? -lim : u);
        hq[c] = am_float_to_e4m3((gt / (1.0f + expf(-gt))) * u / a2);
      }
      for (int c = 0; c < H; ++c) ys[(size_t)j * H + c] = (float)am_dot_q(hq, W2 + (size_t)c * I, I, mode) * sc2;
    }
    for (int c = 0; c < H; ++c) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j)
        if (local[j]) acc = acc + w[(size_t)t * k + j] * ys[(size_t)j * H + c];
      out[(size_t)i * H + c] = am_float_to_bf16(acc);
    }
    free(xq);
    free(hq);
    free(ys);
  }
  return bad;
}

int am_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
