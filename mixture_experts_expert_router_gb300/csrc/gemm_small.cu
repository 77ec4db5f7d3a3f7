// S4 / S5 / S8 for the groups of at most 64 rows, beside the CTA-pair grouped GEMM.
//
// A group of r <= 64 rows reads its whole weight block once for very little
// MMA work, so its speed is how fast an SM can stream weights.  Inside the
// CTA-pair kernel such a group runs as swap-AB tail tiles at about 57 GB/s of
// weights per SM, which takes SM time from the tensor-bound tiles of the large
// groups.  This kernel streams those groups on a few SMs of their own, at the
// same time as the pair kernel works through the larger groups' tiles
// (launch order, claims and completion: launch_gemm in gemm.cu).  Both
// kernels take tiles at run time from counters in device memory: this one
// takes only small-group tiles, the pair kernel takes its main tiles first and
// then whatever small-group tiles are left, so the two finish together
// whatever the mix of group sizes.
//
// The MMAs are swap-AB, one CTA: the tile's 256 weight rows are two M = 128
// operands (FC1: the 128 up rows and the matching 128 gate rows; FC2 and the
// grouped GEMM forward: two halves of 128 output columns), the group's r
// token rows the N side
// (N = 16, 32 or 64).  Each half has its own accumulator and its own issuing
// thread: a thread issues a small-N MMA on a new weight tile only about every
// 83 ns, so two threads stream about twice as many bytes.  With the weights
// on N instead (M = 128 token rows) an SM streamed twice as fast alone, but
// computing 128 token rows for groups of mostly 16 or fewer drew enough power
// to pull every SM's clock down by about 14 % while the pair kernel ran.
//
// Tiles: (small group j, n-block n) numbered j * n_tiles + n, the small
// groups in group order (cute_dsl_fused_moe_bf16 and the Cake ragged BF16
// grouped GEMM both define the rows of group g as one contiguous range given
// by the cumulative group ends).
//
// CTA organisation (256 threads, one CTA per SM, clusters of two CTAs so that
// the kernel holds whole SM pairs and leaves the others to CTA-pair clusters;
// the two CTAs do not cooperate):
//   warp 0   claims tiles and publishes them in a shared-memory queue; loads
//            the token box (16 / 32 / 64 rows) and the first 128 weight rows;
//   warp 6   loads the other 128 weight rows;
//   warps 1, 7  MMA issuers, one per half (M = 128, N = 16..64, K = 16 bf16
//            or 32 E4M3 per instruction); warp 1 owns the TMEM allocation;
//   warps 2..5  epilogue (TMEM lane quarter warp % 4 = weight rows; columns
//            are the tile's tokens).
// A ring slot is 32 KB of weights (two boxes of 128 rows) and an 8 KB token
// box; five slots.
#include <cuda_bf16.h>

#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int SM_BM = 128;                     // MMA M: weight rows of one half of the tile
constexpr int SM_W_HALF = SM_BM * 128;         // one half's weight rows of a k-block (16 KB)
constexpr int SM_T_BYTES = 64 * 128;           // token box slot: up to 64 rows of 128 bytes
constexpr int SM_STAGE = 2 * SM_W_HALF + SM_T_BYTES;
constexpr int SM_STAGES = 5;
// two tiles in flight x two halves x up to 64 token columns
constexpr uint32_t SM_TMEM_COLS = 256;
constexpr int SM_QD = 8;                   // tile queue slots
constexpr int kSmallThreads = 256;
constexpr int kSmallMax = 64;              // largest group this kernel takes
// queue readers besides the claiming thread: warp 6, two MMA threads, 4 epilogue warps
constexpr int SM_Q_READERS = 7;
constexpr int SM_NBARS = 2 * SM_STAGES + 5 + 2 * SM_QD;
constexpr int SM_BAR_OFF = SM_STAGES * SM_STAGE;
constexpr int SM_MISC_OFF = SM_BAR_OFF + SM_NBARS * 8;
constexpr int SM_TQ_OFF = SM_MISC_OFF + 16;
constexpr int SM_TAB_OFF = SM_TQ_OFF + SM_QD * 4;

struct SmallArgs {
  CUtensorMap map_t[3];  // tokens, box {128 bytes, 16 / 32 / 64 rows}
  CUtensorMap map_b;     // weights [G * b_rows, K], box {128 bytes, 128 rows}
  const int32_t *group_end;
  void *out;
  int32_t *status;
  int32_t *sched;        // [1] small-tile claims, [2] start flag, [3] CTAs done
  unsigned long long wait_ns;
  const float *clamp;    // SwiGLU: [G] SwiGLUStep limits, or null
  const float *wscale;   // E4M3: [G] weight scales
  float ascale, oscale;  // E4M3: activation scale of A, requantisation scale of h
  long max_rows;
  int G, K, n_out, b_rows, n_tiles, small_max;
};

// 16 consecutive TMEM columns of this warp's 32 lanes (one value per lane and column).
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void st_release_gpu(int32_t *p, int32_t v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <int EPI, int Q>
__global__ void __launch_bounds__(kSmallThreads, 1) small_group_gemm_kernel(const __grid_constant__ SmallArgs args) {
  constexpr bool kSwiGLU = EPI == (int)Epi::kSwiGLU;
  constexpr int KE = Q ? 128 : 64;  // elements per k-block (128 bytes of a row either way)
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_base + SM_BAR_OFF;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (SM_STAGES + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * SM_STAGES + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * SM_STAGES + 2 + a); };
  const uint32_t drain_bar = bar_base + 8u * (2 * SM_STAGES + 4);
  auto qfull_bar = [&](int j) { return bar_base + 8u * (2 * SM_STAGES + 5 + j); };
  auto qempty_bar = [&](int j) { return bar_base + 8u * (2 * SM_STAGES + 5 + SM_QD + j); };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + SM_MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM_MISC_OFF + 4);
  volatile int *n_small_s = reinterpret_cast<volatile int *>(smem + SM_MISC_OFF + 8);
  volatile int *tq = reinterpret_cast<volatile int *>(smem + SM_TQ_OFF);
  int *gend = reinterpret_cast<int *>(smem + SM_TAB_OFF);  // [G]
  int *small_g = gend + args.G;                             // [G]: the small groups in order

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = args.G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SM_STAGES; ++s) {
      mbar_init(full_bar(s), 2);   // both producers arm their bytes
      mbar_init(empty_bar(s), 2);  // both MMA threads commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 2);
      mbar_init(tempty_bar(a), 4);  // one arrival per epilogue warp
    }
    mbar_init(drain_bar, 2);
    for (int j = 0; j < SM_QD; ++j) {
      mbar_init(qfull_bar(j), 1);
      mbar_init(qempty_bar(j), SM_Q_READERS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < 3; ++i) tma_prefetch_desc(&args.map_t[i]);
    tma_prefetch_desc(&args.map_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), SM_TMEM_COLS);
    tmem_relinquish();
  }
  // Once every CTA of this kernel runs, the CTA-pair kernel may launch (it
  // then holds the other SMs while this kernel holds these).
  pdl_launch_dependents();
  // The gather (and before it the sort) has finished: tell the CTA-pair
  // kernel, which starts behind this one without waiting for it to end.
  pdl_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0) st_release_gpu(args.sched + 2, 1);
  for (int g = threadIdx.x; g < G; g += kSmallThreads) {
    long e = args.group_end[g];
    e = e < 0 ? 0 : (e > args.max_rows ? args.max_rows : e);
    gend[g] = (int)e;
  }
  __syncthreads();
  if (warp == 0) {  // small_g = the groups with 1..small_max rows, in group order
    int carry = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      bool small = false;
      if (g < G) {
        const int cnt = gend[g] - (g == 0 ? 0 : gend[g - 1]);
        small = cnt > 0 && cnt <= args.small_max;
      }
      const uint32_t m = __ballot_sync(0xffffffffu, small);
      if (small) small_g[carry + __popc(m & ((1u << lane) - 1u))] = g;
      carry += __popc(m);
    }
    if (lane == 0) *n_small_s = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_holder;
  const int total = *n_small_s * args.n_tiles;
  const int num_kb = args.K / KE;

  // i-th tile of this CTA from the queue (single-thread readers); -1 = none.
  auto queue_read = [&](int i) -> int {
    const int j = i % SM_QD;
    if (!mbar_wait(qfull_bar(j), (uint32_t)(i / SM_QD) & 1u, abort_flag, args.status, args.wait_ns)) return -1;
    const int t = tq[j];
    mbar_arrive(qempty_bar(j));
    return t;
  };
  struct SmallTile {
    int g, n, row0, r, box;  // box: token rows 16 << box
    int w0, w1;              // first weight row of each half
  };
  auto tile_of = [&](int t) -> SmallTile {
    SmallTile c;
    const int j = t / args.n_tiles;
    c.n = t - j * args.n_tiles;
    c.g = small_g[j];
    c.row0 = c.g == 0 ? 0 : gend[c.g - 1];
    c.r = gend[c.g] - c.row0;
    c.box = c.r <= 16 ? 0 : (c.r <= 32 ? 1 : 2);
    if (kSwiGLU) {  // up rows and the matching gate rows
      c.w0 = c.g * args.b_rows + c.n * SM_BM;
      c.w1 = c.w0 + args.b_rows / 2;
    } else {  // output columns n * 256 .. + 127 and + 128 .. + 255
      c.w0 = c.g * args.b_rows + c.n * 2 * SM_BM;
      c.w1 = c.w0 + SM_BM;
    }
    return c;
  };
  const uint64_t pol_w = policy_evict_first();  // weights of a small group are read once
  const uint64_t pol_t = policy_evict_normal();

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------- claims + token box + first weight half --
      int it = 0;
      bool ok = true;
      // The queue runs one tile ahead of this thread, and each claim is made
      // one tile before it is published (the counter's round trip overlaps a
      // tile's copies), after the publication before it (a release, which
      // would otherwise wait for the round trip).
      int pend = atomicAdd(args.sched + 1, 1);
      auto publish = [&](int i, int t) -> int {
        const int j = i % SM_QD;
        if (t >= 0 && !mbar_wait(qempty_bar(j), ((uint32_t)(i / SM_QD) & 1u) ^ 1u, abort_flag, args.status,
                                 args.wait_ns))
          t = -1;
        tq[j] = t;
        mbar_arrive(qfull_bar(j));  // release: the readers see tq[j]
        if (t >= 0) pend = atomicAdd(args.sched + 1, 1);  // the claim for the tile after it
        return t;
      };
      int cur = publish(0, pend < total ? pend : -1);
      for (int i = 0;; ++i) {
        const int t = cur;
        if (t < 0) break;
        cur = publish(i + 1, ok && pend < total ? pend : -1);
        const SmallTile c = tile_of(t);
        const uint32_t t_bytes = (16u << c.box) * 128u;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % SM_STAGES;
          const uint32_t ph = (uint32_t)(it / SM_STAGES) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, args.status, args.wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t dst = smem_base + s * SM_STAGE;
          mbar_arrive_expect_tx_relaxed(full_bar(s), SM_W_HALF + t_bytes);
          tma_load_2d(dst, &args.map_b, full_bar(s), kb * KE, c.w0, pol_w);
          tma_load_2d(dst + 2 * SM_W_HALF, &args.map_t[c.box], full_bar(s), kb * KE, c.row0, pol_t);
        }
      }
      for (int j = it > SM_STAGES ? it - SM_STAGES : 0; j < it; ++j)
        mbar_wait(full_bar(j % SM_STAGES), (uint32_t)(j / SM_STAGES) & 1u, nullptr, args.status, args.wait_ns);
    }
  } else if (warp == 6) {
    if (lane == 0) {
      // ------------------------------------------------------ second weight half --
      int it = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int t = queue_read(i);
        if (t < 0) break;
        const SmallTile c = tile_of(t);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % SM_STAGES;
          const uint32_t ph = (uint32_t)(it / SM_STAGES) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, args.status, args.wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t dst = smem_base + s * SM_STAGE + SM_W_HALF;
          mbar_arrive_expect_tx_relaxed(full_bar(s), SM_W_HALF);
          tma_load_2d(dst, &args.map_b, full_bar(s), kb * KE, c.w1, pol_w);
        }
      }
      for (int j = it > SM_STAGES ? it - SM_STAGES : 0; j < it; ++j)
        mbar_wait(full_bar(j % SM_STAGES), (uint32_t)(j / SM_STAGES) & 1u, nullptr, args.status, args.wait_ns);
    }
  } else if (warp == 1 || warp == 7) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuers, one per half --
      // One thread's MMAs on a new weight tile issue about every 83 ns; two
      // threads with their own accumulators stream about twice as many bytes.
      const int half = warp == 1 ? 0 : 1;
      int it = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int t = queue_read(i);
        if (t < 0) break;
        const SmallTile c = tile_of(t);
        const uint32_t n_tok = 16u << c.box;
        const uint32_t idesc = Q ? idesc_e4m3_f32(SM_BM, n_tok) : idesc_bf16_f32(SM_BM, n_tok);
        const int acc = i & 1;
        if (!mbar_wait(tempty_bar(acc), ((uint32_t)(i >> 1) & 1u) ^ 1u, abort_flag, args.status, args.wait_ns))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * 128 + half * 64);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % SM_STAGES;
          if (!mbar_wait(full_bar(s), (uint32_t)(it / SM_STAGES) & 1u, abort_flag, args.status, args.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_base + s * SM_STAGE;
          const uint64_t w = smem_desc_k_sw128(st + half * SM_W_HALF);
          const uint64_t tk = smem_desc_k_sw128(st + 2 * SM_W_HALF);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // 32 bytes of each row per instruction
            if (Q) umma_e4m3(d, w + 2u * k, tk + 2u * k, idesc, (kb | k) != 0);
            else umma_bf16(d, w + 2u * k, tk + 2u * k, idesc, (kb | k) != 0);
          }
          umma_commit(empty_bar(s));  // the slot is free once both threads' MMAs have read it
        }
        if (ok) umma_commit(tfull_bar(acc));
      }
      umma_commit(drain_bar);
      mbar_wait(drain_bar, 0, nullptr, args.status, args.wait_ns);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------------ epilogue --
    const int quarter = warp & 3;
    const int r_in_tile = quarter * 32 + lane;
    for (int i = 0;; ++i) {
      int t = -1;
      if (lane == 0) t = queue_read(i);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t < 0) break;
      const SmallTile c = tile_of(t);
      const int acc = i & 1;
      int got = 1;
      if (lane == 0)
        got = mbar_wait(tfull_bar(acc), (uint32_t)(i >> 1) & 1u, abort_flag, args.status, args.wait_ns) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      tc_fence_after();
      {
        // lanes: weight row wr of each half; columns: the tile's tokens
        const int wr = quarter * 32 + lane;
        const uint32_t t0 = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * 128), t1 = t0 + 64;
        const float sc = Q ? __fmul_rn(args.ascale, __ldg(args.wscale + c.g)) : 1.f;
        const float lim = step_limit(args.clamp, c.g);
#pragma unroll 1
        for (int c0 = 0; c0 < c.r; c0 += 16) {
          uint32_t a[16], b[16];
          tmem_ld_x16(t0 + (uint32_t)c0, a);
          tmem_ld_x16(t1 + (uint32_t)c0, b);
          tmem_ld_wait();
          const long row = (long)c.row0 + c0;
          if (kSwiGLU) {  // h[token][n * 128 + wr] from up (a) and gate (b)
            const long col = (long)c.n * SM_BM + wr;
            if (Q) {
              const float inv = __frcp_rn(args.oscale);
              uint8_t *h = reinterpret_cast<uint8_t *>(args.out);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < c.r) {
                  const float uu = __fmul_rn(__uint_as_float(a[j]), sc);
                  const float gg = __fmul_rn(__uint_as_float(b[j]), sc);
                  h[(row + j) * args.n_out + col] =
                      (uint8_t)(e4m3x2(__fmul_rn(swiglu_step(gg, uu, lim), inv), 0.f) & 0xFFu);
                }
            } else {
              __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(args.out);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < c.r)
                  h[(row + j) * args.n_out + col] =
                      __float2bfloat16_rn(swiglu_step(__uint_as_float(b[j]), __uint_as_float(a[j]), lim));
            }
          } else if (EPI == (int)Epi::kF32) {  // y[token][n * 256 + wr] and [.. + 128 + wr]
            float *y = reinterpret_cast<float *>(args.out);
            const long col = (long)c.n * 2 * SM_BM + wr;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j < c.r) {
                float *yr = y + (row + j) * args.n_out + col;
                yr[0] = Q ? __fmul_rn(__uint_as_float(a[j]), sc) : __uint_as_float(a[j]);
                yr[SM_BM] = Q ? __fmul_rn(__uint_as_float(b[j]), sc) : __uint_as_float(b[j]);
              }
          } else {  // the grouped GEMM forward: Y rounded to bf16
            __nv_bfloat16 *y = reinterpret_cast<__nv_bfloat16 *>(args.out);
            const long col = (long)c.n * 2 * SM_BM + wr;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j < c.r) {
                __nv_bfloat16 *yr = y + (row + j) * args.n_out + col;
                yr[0] = __float2bfloat16_rn(__uint_as_float(a[j]));
                yr[SM_BM] = __float2bfloat16_rn(__uint_as_float(b[j]));
              }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, SM_TMEM_COLS);
  }
  if (threadIdx.x == 0) {  // this CTA's rows are written: count it done
    __threadfence();
    atomicAdd(args.sched + 3, 1);
  }
}

}  // namespace

size_t small_gemm_smem(int G) { return 1024 + SM_TAB_OFF + (size_t)(2 * G) * 4; }

int small_gemm_max_rows() { return kSmallMax; }

cudaError_t small_gemm_configure(Epi epi, int q, size_t smem) {
  if (q) {
    if (epi == Epi::kSwiGLU)
      return raise_smem_limit(small_group_gemm_kernel<(int)Epi::kSwiGLU, 1>, smem);
    return raise_smem_limit(small_group_gemm_kernel<(int)Epi::kF32, 1>, smem);
  }
  if (epi == Epi::kSwiGLU) return raise_smem_limit(small_group_gemm_kernel<(int)Epi::kSwiGLU, 0>, smem);
  if (epi == Epi::kF32) return raise_smem_limit(small_group_gemm_kernel<(int)Epi::kF32, 0>, smem);
  return raise_smem_limit(small_group_gemm_kernel<(int)Epi::kBf16, 0>, smem);
}

cudaError_t launch_small_gemm(const GemmPlan &p, const Launch &l) {
  SmallArgs a;
  for (int i = 0; i < 3; ++i) a.map_t[i] = p.map_t[i + 1];  // boxes of 16, 32, 64 rows
  a.map_b = p.map_b;
  a.group_end = p.group_end;
  a.out = p.out;
  a.status = p.status;
  a.sched = p.sched;
  a.wait_ns = p.wait_ns;
  a.clamp = p.clamp;
  a.wscale = p.wscale;
  a.ascale = p.ascale;
  a.oscale = p.oscale;
  a.max_rows = p.max_rows;
  a.G = p.G;
  a.K = p.K;
  a.n_out = p.n_out;
  a.b_rows = p.b_rows;
  a.n_tiles = p.n_tiles;
  a.small_max = p.small_max;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.side_ctas);
  cfg.blockDim = dim3(kSmallThreads);
  cfg.dynamicSmemBytes = small_gemm_smem(p.G);
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = l.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (p.q) {
    if (p.epi == Epi::kSwiGLU) return cudaLaunchKernelEx(&cfg, small_group_gemm_kernel<(int)Epi::kSwiGLU, 1>, a);
    return cudaLaunchKernelEx(&cfg, small_group_gemm_kernel<(int)Epi::kF32, 1>, a);
  }
  if (p.epi == Epi::kSwiGLU) return cudaLaunchKernelEx(&cfg, small_group_gemm_kernel<(int)Epi::kSwiGLU, 0>, a);
  if (p.epi == Epi::kF32) return cudaLaunchKernelEx(&cfg, small_group_gemm_kernel<(int)Epi::kF32, 0>, a);
  return cudaLaunchKernelEx(&cfg, small_group_gemm_kernel<(int)Epi::kBf16, 0>, a);
}

}  // namespace moe
