// S7 for few tokens as a chain: FC1 and FC2 of the decode regime with the
// sort, the gather and the finalize folded in, as two kernels or as one.
//
// For T*top_k <= kChainMaxRoutes routes each CTA sorts the routes itself in shared
// memory (the same stable counting sort as sort.cu: ascending expanded index
// inside each local expert), so no sort kernel runs.  Both phases are swap-AB
// weight-streaming GEMMs (decode.cu): 128 weight rows on the MMA's M side,
// the expert's tokens on N.
//
//   FC1  the producer warp gathers the expert's token rows straight from x
//        (four rows per TMA row-gather), the epilogue writes
//        h[p] = bf16(silu(g) * u); the first CTA also publishes the sort
//        (m_indptr, perm_to_exp, exp_to_perm).
//   FC2  streams W2 (the first ring of weight boxes before h is ready),
//        writes the unscaled fp32 rows y, and combines: every (token, 128-col
//        block) has a counter; the tile that brings it to the token's number
//        of local routes sums the token's rows in ascending slot order,
//        out = bf16(sum_j w_j * y_j), exactly the finalize kernel's
//        arithmetic, so the result does not depend on which tile is last.
//
// Two kernels: FC2 waits for FC1 by programmatic dependent launch, and FC1's
// first CTA zeroes the combine counters.  One launch: every CTA runs its FC1
// tiles first and then its FC2 tiles; an FC2 tile loads h once the count of
// finished FC1 tiles of its expert is complete (a bounded wait on a counter
// that FC1 epilogues raise after their h stores).  Every launch first runs a
// one-CTA kernel that zeroes the counters and clears the status word
// (chain_clear_kernel); the chain follows it by programmatic dependent launch
// and touches neither before its griddepcontrol.wait, so no state carries over
// from another launch or from another plan that shares the workspace.  With
// at most one CTA per SM and
// no more CTAs than SMs, every CTA that others wait for has an SM, and FC1
// tiles wait for nothing.
//
// The k-loop runs as two half-pipelines (even / odd k-blocks, each with its
// own producer, MMA thread and TMEM accumulator; the epilogue adds the two),
// as in decode.cu.
//
// Programmatic dependent launch: each kernel reads only the layer's inputs
// (and, in logits mode, the routing kernel's output, waited for) before its
// griddepcontrol.wait; it writes nothing before it.
#include <cuda_bf16.h>

#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BK = 64;
// warps: 0 / 6 producers of the even / odd k-blocks, 1 / 7 their MMA issuers
// (1 also owns TMEM), 2..5 epilogue
constexpr int kThreads = 256;
constexpr int kProd1Warp = 6;
constexpr int kMma1Warp = 7;
constexpr int kEpiThreads = 128;

// Kernel modes: the two kernels of the chain, or both phases in one launch.
constexpr int kModeFc2 = 0, kModeFc1 = 1, kModeBoth = 2;

struct ChainArgs {
  CUtensorMap map_w1;  // W1 [L*2I, H] box {64, 64}
  CUtensorMap map_x;   // x [T, H] box {64, 1} (row gathers)
  CUtensorMap map_w2;  // W2 [L*H, I] box {64, 128}
  CUtensorMap map_h;   // h [R, I] box {64, BNT}
  const int32_t *ids;  // [T*k] global expert ids
  const float *w;      // [T*k] routing weights
  uint16_t *h;         // [R, I] bf16: FC1 writes, FC2 reads
  float *y;            // [R, H] fp32: FC2
  uint16_t *out;       // [T, H] bf16: FC2
  int32_t *comb;       // [T * m_tiles2] combine counters
  int32_t *done1;      // one launch: [L] finished FC1 tiles per expert
  int32_t *m_indptr_out, *p2e_out, *e2p_out;  // published by the first CTA of FC1
  int32_t *status;
  unsigned long long wait_ns;  // bounded-wait limit of this launch
  const float *clamp;         // SwiGLU epilogue: [groups] SwiGLUStep limits, or null
  int T, k, E, off, L, H, I, m_tiles1, m_tiles2, ids_early;
};

template <int BNT>
struct ChainCfg {
  static constexpr int A_BYTES = 128 * BK * 2;
  static constexpr int B_BYTES = BNT * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BNT == 64 ? 6 : 8;  // two private halves, one per half-pipeline
  static_assert(STAGES % 2 == 0, "the ring splits evenly between the half-pipelines");
  static constexpr int NBARS = 2 * STAGES + 6;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;         // tmem base, abort, bad flag
  static constexpr int SG_OFF = (MISC_OFF + 16 + 15) & ~15;    // [BNT][64] fp32 (FC1) / flags (FC2)
  static constexpr int TAB_OFF = SG_OFF + BNT * 64 * 4;
  static constexpr uint32_t TMEM_COLS = 4 * BNT;  // [tile buffer][half-pipeline] accumulators
  static constexpr uint32_t IDESC = idesc_bf16_f32(128, BNT);
  // tables: m_indptr [L+1], next [L+1], tile_start [L+1], p2e [R], e2p [R], tok_n [T]
  static size_t smem_bytes(int L, int R, int T) {
    return 1024 + TAB_OFF + (size_t)(3 * (L + 1) + 2 * R + T + 8) * 4;
  }
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ bool epi_bar_any(bool flag) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)flag)
      : "memory");
  return r != 0;
}

// Stable counting sort of the R routes by local expert, in shared memory; all
// threads of the CTA call it.  m_indptr[L+1], p2e[R] (first M valid),
// e2p[R] (-1 for a route that is not local or has a bad id).
__device__ void cta_sort(const int32_t *ids, int R, int E, int off, int L, int *m_indptr, int *next,
                         int *p2e, int *e2p, volatile int *bad) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int x = tid; x < L; x += kThreads) m_indptr[x] = 0;
  if (tid == 0) *bad = 0;
  __syncthreads();
  for (int r = tid; r < R; r += kThreads) {
    const int g = ids[r];
    if (g < 0 || g >= E) *bad = 1;
    else if (g >= off && g < off + L) atomicAdd(&m_indptr[g - off], 1);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the counts; m_indptr[L] = M
    int carry = 0;
    for (int base = 0; base < L; base += 32) {
      const int x = base + lane;
      const int v = x < L ? m_indptr[x] : 0;
      int inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (x < L) {
        m_indptr[x] = carry + inc - v;
        next[x] = carry + inc - v;
      }
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) m_indptr[L] = carry;
    __syncwarp();
    // placement, 32 routes at a time in ascending r
    for (int base = 0; base < R; base += 32) {
      const int r = base + lane;
      int e = -1;
      if (r < R) {
        const int g = ids[r];
        if (g >= off && g < off + L && g < E) e = g - off;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (e >= 0) {
        const int p = next[e] + rank;
        p2e[p] = r;
        e2p[r] = p;
      } else if (r < R) {
        e2p[r] = -1;
      }
      __syncwarp();
      if (e >= 0 && rank == 0) next[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
}

struct Tile {
  int g, m, n;
};

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Tile t of a list with m_tiles weight tiles per row block of each expert:
// nbp is the prefix of the experts' row-block counts; tiles run expert by
// expert, then weight tile, then row block.
__device__ __forceinline__ Tile decode_tile(int t, const int *nbp, int L, int m_tiles) {
  int lo = 0, hi = L;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (m_tiles * nbp[mid] <= t) lo = mid;
    else hi = mid;
  }
  Tile c;
  c.g = lo;
  const int local = t - m_tiles * nbp[lo];
  const int nt = nbp[lo + 1] - nbp[lo];
  c.m = local / nt;
  c.n = local - c.m * nt;
  return c;
}

// One work item: a weight tile (128 weight rows) times a block of BNT
// permuted rows of one expert, from FC1 or from FC2.
struct Item {
  bool fc1;
  Tile c;
};

template <int BNT, int MODE>
__global__ void __launch_bounds__(kThreads, 1) chain_kernel(const __grid_constant__ ChainArgs a) {
  using C = ChainCfg<BNT>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_base + C::BAR_OFF;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int x) { return bar_base + 8u * (2 * C::STAGES + x); };
  auto tempty_bar = [&](int x) { return bar_base + 8u * (2 * C::STAGES + 2 + x); };
  auto drain_bar = [&](int q) { return bar_base + 8u * (2 * C::STAGES + 4 + q); };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
  volatile int *bad = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 8);
  float *sg = reinterpret_cast<float *>(smem + C::SG_OFF);
  int *sflag = reinterpret_cast<int *>(smem + C::SG_OFF);  // FC2: last-arriver tokens [BNT]
  const int L = a.L, T = a.T, R = a.T * a.k;
  int *m_indptr = reinterpret_cast<int *>(smem + C::TAB_OFF);
  int *next = m_indptr + (L + 1);
  int *nbp = next + (L + 1);  // prefix of the experts' row blocks ceil(rows / BNT)
  int *p2e = nbp + (L + 1);
  int *e2p = p2e + R;
  int *tok_n = e2p + R;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(tfull_bar(x), 2);  // both MMA issuers commit
      mbar_init(tempty_bar(x), kEpiThreads);
      mbar_init(drain_bar(x), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (MODE != kModeFc2) {
      tma_prefetch_desc(&a.map_w1);
      tma_prefetch_desc(&a.map_x);
    }
    if (MODE != kModeFc1) {
      tma_prefetch_desc(&a.map_w2);
      tma_prefetch_desc(&a.map_h);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (!a.ids_early) pdl_wait();  // the routing kernel wrote ids and weights

  // Early weights.  With T <= BNT every active expert has exactly one row
  // block (an expert gets at most one route per token), so a CTA's first item
  // follows from the rank of its expert among the distinct local experts of
  // the routes, in ascending order.  For at most 32 routes each producer warp
  // works that out from the ids and issues the weight boxes of its first
  // k-blocks (the first use of its ring slots) before the sort below; the
  // item's token boxes go out once the sort is done.
  constexpr int HS0 = C::STAGES / 2;
  int n_early = 0;
  if ((warp == 0 || warp == kProd1Warp) && T <= BNT && R <= 32) {
    asm volatile("bar.sync 2, 64;" ::: "memory");  // warp 6 sees the barriers warp 0 initialised
    const int q = warp == 0 ? 0 : 1;
    int g = -1;
    if (lane < R) {
      const int id = a.ids[lane];
      if (id >= a.off && id < a.off + L) g = id - a.off;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, g);
    const bool first = g >= 0 && (peers & ((1u << lane) - 1u)) == 0u;
    // one row block per expert also needs at most BNT routes per expert (more
    // only with repeated ids inside a token's routes): otherwise no early issue
    const bool one_block = __all_sync(0xffffffffu, g < 0 || __popc(peers) <= BNT);
    int rank = 0;  // distinct local experts below g
    for (int j = 0; j < 32; ++j) {
      const int gj = __shfl_sync(0xffffffffu, g, j);
      const bool fj = __shfl_sync(0xffffffffu, first ? 1 : 0, j) != 0;
      if (fj && gj < g) ++rank;
    }
    const int n_act = __popc(__ballot_sync(0xffffffffu, first));
    const int t1 = MODE == kModeFc2 ? 0 : a.m_tiles1 * n_act;
    const int t2 = MODE == kModeFc1 ? 0 : a.m_tiles2 * n_act;
    const int w = (int)blockIdx.x;
    if (one_block && w < t1 + t2) {
      const bool fc1 = w < t1;
      const int e = fc1 ? w / a.m_tiles1 : (w - t1) / a.m_tiles2;
      const int m = fc1 ? w - e * a.m_tiles1 : (w - t1) - e * a.m_tiles2;
      const unsigned sel = __ballot_sync(0xffffffffu, first && rank == e);
      const int ge = __shfl_sync(0xffffffffu, g, sel ? __ffs(sel) - 1 : 0);
      const int wrow = fc1 ? ge * 2 * a.I + m * 64 : ge * a.H + m * 128;
      const int nkb = (fc1 ? a.H : a.I) / BK;
      const uint64_t pol_w = policy_evict_first();
      for (int kb = q; kb < nkb && n_early < HS0 && sel != 0u; kb += 2, ++n_early) {
        const int s = q * HS0 + n_early;
        const uint32_t a_dst = smem_base + s * C::STAGE_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
          if (fc1) {
            tma_load_2d(a_dst, &a.map_w1, full_bar(s), kb * BK, wrow, pol_w);
            tma_load_2d(a_dst + 64 * 128, &a.map_w1, full_bar(s), kb * BK, wrow + a.I, pol_w);
          } else {
            tma_load_2d(a_dst, &a.map_w2, full_bar(s), kb * BK, wrow, pol_w);
          }
        }
      }
    }
  }

  cta_sort(a.ids, R, a.E, a.off, L, m_indptr, next, p2e, e2p, bad);
  if (MODE != kModeFc1) {
    for (int t = threadIdx.x; t < T; t += kThreads) {
      int n = 0;
      for (int j = 0; j < a.k; ++j) n += e2p[t * a.k + j] >= 0;
      tok_n[t] = n;
    }
  }
  if (warp == 0) {  // row blocks per non-empty expert: ceil(cnt / BNT)
    int carry = 0;
    if (lane == 0) nbp[0] = 0;
    for (int base = 0; base < L; base += 32) {
      const int g = base + lane;
      int nb = 0;
      if (g < L) nb = (m_indptr[g + 1] - m_indptr[g] + BNT - 1) / BNT;
      int inc = nb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (g < L) nbp[g + 1] = carry + inc;
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();

  const uint32_t tmem_base = *tmem_holder;
  // FC1 tiles: I / 64 weight tiles (64 up + 64 gate rows) per row block; FC2
  // tiles: H / 128 weight tiles per row block.  In one launch the FC1 items
  // come first, so a CTA finishes all its FC1 items before its first FC2 item.
  const int total1 = MODE == kModeFc2 ? 0 : a.m_tiles1 * nbp[L];
  const int total2 = MODE == kModeFc1 ? 0 : a.m_tiles2 * nbp[L];
  const int total = total1 + total2;
  auto item = [&](int w) {
    Item it;
    it.fc1 = w < total1;
    it.c = it.fc1 ? decode_tile(w, nbp, L, a.m_tiles1) : decode_tile(w - total1, nbp, L, a.m_tiles2);
    return it;
  };
  // Each half-pipeline owns half of the ring (slots q * HS .. q * HS + HS - 1),
  // so a slot is only ever filled and drained by one producer / MMA pair and
  // every wait on it is for the phase right after the one it last saw.
  constexpr int HS = C::STAGES / 2;
  const int M = m_indptr[L];

  if ((warp == 0 || warp == kProd1Warp)) {
    // --------------------------------------------------------------- producers --
    // Producer q (warp 0: q = 0, warp 6: q = 1) loads the k-blocks kb % 2 == q
    // of every item; FC1's token rows come from the lanes, four rows each.
    // FC2's h rows are written by FC1: by the previous kernel of the chain
    // (programmatic dependent launch) or, in one launch, by other CTAs, which
    // count each finished FC1 tile per expert.  Until they are there the
    // weight boxes go out and the h boxes are listed, then loaded once h is
    // ready; a producer never waits on a slot that holds a listed box.
    const int q = warp == 0 ? 0 : 1;
    const uint64_t pol_w = policy_evict_first();  // each weight byte is read once
    const uint64_t pol_x = policy_evict_last();
    int iq = n_early;  // this pipeline's k-blocks so far: its private ring slots q * HS + iq % HS
    bool ok = true;
    int pend_s[HS], pend_kb[HS];
    int n_pend = 0;
    bool pdl_done = false;
    // one launch: the clear kernel before this one zeroes the counters and the
    // status word; no wait below may report into the status word before it
    if (MODE == kModeBoth) pdl_wait();
    for (int wi = blockIdx.x; wi < total && ok; wi += gridDim.x) {
      const Item it = item(wi);
      const Tile c = it.c;
      const int num_kb = (it.fc1 ? a.H : a.I) / BK;
      const int wrow = it.fc1 ? c.g * 2 * a.I + c.m * 64 : c.g * a.H + c.m * 128;
      const int xrow = m_indptr[c.g] + c.n * BNT;
      // h of this item may be loaded: always for FC1; for FC2 once the chain's
      // first kernel has finished, or in one launch once every FC1 tile of the
      // expert has
      bool dep_ok = it.fc1 || (MODE == kModeFc2 && pdl_done);
      const int need = a.m_tiles1 * (nbp[c.g + 1] - nbp[c.g]);
      auto finish = [&]() {
        pdl_wait();
        pdl_done = true;
        int w_ok = 1;
        if (MODE == kModeBoth && lane == 0)
          w_ok = counter_wait(a.done1 + c.g, need, abort_flag, a.status, a.wait_ns) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) ok = false;
        if (MODE == kModeBoth) fence_proxy_async_global();
        // the listed boxes go out even after a failed wait (their reads stay in
        // bounds), so that every armed slot completes and the drain below ends
        if (lane == 0)
          for (int j = 0; j < n_pend; ++j)
            tma_load_2d(smem_base + pend_s[j] * C::STAGE_BYTES + C::A_BYTES, &a.map_h, full_bar(pend_s[j]),
                        pend_kb[j] * BK, xrow, pol_x);
        n_pend = 0;
        dep_ok = true;
      };
      int tr0 = 0, tr1 = 0, tr2 = 0, tr3 = 0;  // FC1: this lane's four token rows of x
      const bool tok_lane = it.fc1 && lane < BNT / 4;
      if (tok_lane) {
        int tr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int p = xrow + 4 * lane + i;
          tr[i] = p < M ? p2e[p] / a.k : 0;
        }
        tr0 = tr[0];
        tr1 = tr[1];
        tr2 = tr[2];
        tr3 = tr[3];
      }
      // the first item's early k-blocks: their weight boxes are out; now
      // their token boxes (FC1) or h boxes (FC2, listed until h is ready)
      const int early = wi == (int)blockIdx.x ? n_early : 0;
      for (int j = 0; j < early; ++j) {
        const int s = q * HS + j, kb = q + 2 * j;
        const uint32_t a_dst = smem_base + s * C::STAGE_BYTES;
        if (it.fc1) {
          if (tok_lane)
            tma_gather4(a_dst + C::A_BYTES + lane * 512, &a.map_x, full_bar(s), kb * BK, tr0, tr1, tr2, tr3, pol_x);
        } else if (dep_ok) {
          if (lane == 0) tma_load_2d(a_dst + C::A_BYTES, &a.map_h, full_bar(s), kb * BK, xrow, pol_x);
        } else {
          pend_s[n_pend] = s;
          pend_kb[n_pend] = kb;
          ++n_pend;
        }
      }
      for (int kb = 0; kb < num_kb && ok; ++kb) {
        if ((kb & 1) != q) continue;
        if (kb < q + 2 * early) continue;  // issued early
        if (!dep_ok && n_pend == HS) {  // the next slot holds a listed box
          finish();
          if (!ok) break;
        }
        const int s = q * HS + iq % HS;
        const uint32_t ph = (uint32_t)(iq / HS) & 1u;
        ++iq;
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, a.status, a.wait_ns) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        const uint32_t a_dst = smem_base + s * C::STAGE_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
          if (it.fc1) {
            tma_load_2d(a_dst, &a.map_w1, full_bar(s), kb * BK, wrow, pol_w);
            tma_load_2d(a_dst + 64 * 128, &a.map_w1, full_bar(s), kb * BK, wrow + a.I, pol_w);
          } else {
            tma_load_2d(a_dst, &a.map_w2, full_bar(s), kb * BK, wrow, pol_w);
          }
        }
        __syncwarp();
        if (it.fc1) {
          if (tok_lane)
            tma_gather4(a_dst + C::A_BYTES + lane * 512, &a.map_x, full_bar(s), kb * BK, tr0, tr1, tr2,
                        tr3, pol_x);
        } else if (dep_ok) {
          if (lane == 0) tma_load_2d(a_dst + C::A_BYTES, &a.map_h, full_bar(s), kb * BK, xrow, pol_x);
        } else {
          pend_s[n_pend] = s;
          pend_kb[n_pend] = kb;
          ++n_pend;
        }
      }
      if (ok && !dep_ok) finish();
    }
    if (lane == 0)  // let this pipeline's last copies land
      for (int j = iq > HS ? iq - HS : 0; j < iq; ++j)
        mbar_wait(full_bar(q * HS + j % HS), (uint32_t)(j / HS) & 1u, nullptr, a.status, a.wait_ns);
  } else if ((warp == 1 || warp == kMma1Warp) && lane == 0) {
    // ------------------------------------------------------------- MMA issuers --
    // Issuer q multiplies the k-blocks kb % 2 == q into accumulator q of the
    // item's buffer; both commit every item.
    const int q = warp == 1 ? 0 : 1;
    int iq = 0, tc = 0;
    bool ok = true;
    if (MODE == kModeBoth) pdl_wait();  // as for the producers
    for (int wi = blockIdx.x; wi < total && ok; wi += gridDim.x, ++tc) {
      const int num_kb = (wi < total1 ? a.H : a.I) / BK;
      const int acc = tc & 1;
      const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
      if (!mbar_wait(tempty_bar(acc), aph ^ 1u, abort_flag, a.status, a.wait_ns)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)((2 * acc + q) * BNT);
      bool first = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        if ((kb & 1) != q) continue;
        const int s = q * HS + iq % HS;
        const uint32_t ph = (uint32_t)(iq / HS) & 1u;
        ++iq;
        if (!mbar_wait(full_bar(s), ph, abort_flag, a.status, a.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_base + s * C::STAGE_BYTES;
        const uint64_t a_desc = smem_desc_k_sw128(a_addr);
        const uint64_t b_desc = smem_desc_k_sw128(a_addr + C::A_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_bf16(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, C::IDESC, (first && kk == 0) ? 0u : 1u);
        first = false;
        umma_commit(empty_bar(s));
      }
      if (ok) umma_commit(tfull_bar(acc));
    }
    umma_commit(drain_bar(q));
    mbar_wait(drain_bar(q), 0, nullptr, a.status, a.wait_ns);
  } else if (warp >= 2 && warp <= 5) {
    // ---------------------------------------------------------------- epilogue --
    pdl_wait();  // the previous kernel may still read what this one writes
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // weight row inside the tile (TMEM lane)
    const int etid = threadIdx.x - 64;  // 0..127
    if (blockIdx.x == 0) {
      if (MODE != kModeFc2) {
        // the launch clears the status word on the stream before this kernel
        // runs; a kernel only ORs bits into it
        if (etid == 0 && a.status && *bad)
          atomicOr(reinterpret_cast<unsigned int *>(a.status), MOE_DEV_BAD_EXPERT);
        for (int x = etid; x <= L; x += kEpiThreads) a.m_indptr_out[x] = m_indptr[x];
        for (int x = etid; x < R; x += kEpiThreads) {
          a.e2p_out[x] = e2p[x];
          if (x < M) a.p2e_out[x] = p2e[x];
        }
        // the chain's second kernel counts from zero (one launch resets its
        // counters when it ends instead)
        if (MODE == kModeFc1)
          for (int x = etid; x < T * a.m_tiles2; x += kEpiThreads) a.comb[x] = 0;
      }
      if (MODE != kModeFc1) {  // tokens with no local route: their output row is zero
        for (int t = 0; t < T; ++t)
          if (tok_n[t] == 0)
            for (int x = etid; x < a.H; x += kEpiThreads) a.out[(long)t * a.H + x] = 0;
      }
    }
    int tc = 0;
    for (int wi = blockIdx.x; wi < total; wi += gridDim.x, ++tc) {
      const Item it = item(wi);
      const Tile c = it.c;
      const int num_kb = (it.fc1 ? a.H : a.I) / BK;
      const int xrow = m_indptr[c.g] + c.n * BNT;
      const int valid = m_indptr[c.g + 1] - xrow;  // rows of this item (> 0)
      const int acc = tc & 1;
      const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
      const bool got = mbar_wait(tfull_bar(acc), aph, abort_flag, a.status, a.wait_ns);
      if (epi_bar_any(!got)) break;
      float v[BNT];
      tc_fence_after();
      const uint32_t lane_addr = tmem_base + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
      for (int c0 = 0; c0 < BNT; c0 += 16) {
        uint32_t qv[16];
        tmem_ld_x16(lane_addr + (uint32_t)(2 * acc * BNT + c0), qv);
        if (num_kb > 1) {  // the odd k-blocks' accumulator
          uint32_t q1[16];
          tmem_ld_x16(lane_addr + (uint32_t)((2 * acc + 1) * BNT + c0), q1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            qv[i] = __float_as_uint(__fadd_rn(__uint_as_float(qv[i]), __uint_as_float(q1[i])));
        }
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) v[c0 + i] = __uint_as_float(qv[i]);
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      if (it.fc1) {
        if (r >= 64) {
#pragma unroll
          for (int j = 0; j < BNT; ++j) sg[j * 64 + (r - 64)] = v[j];
        }
        epi_bar();
        if (r < 64) {
          __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(a.h);
          const long col = (long)c.m * 64 + r;
          const float lim = step_limit(a.clamp, c.g);
#pragma unroll
          for (int j = 0; j < BNT; ++j)
            if (j < valid)
              h[(long)(xrow + j) * a.I + col] = __float2bfloat16_rn(swiglu_step(sg[j * 64 + r], v[j], lim));
        }
        if (MODE == kModeBoth) __threadfence();  // h before the expert's count
        epi_bar();
        if (MODE == kModeBoth && etid == 0) atomicAdd(a.done1 + c.g, 1);
      } else {
        const int col = c.m * 128 + r;
        if (col < a.H) {
#pragma unroll
          for (int j = 0; j < BNT; ++j)
            if (j < valid) a.y[(long)(xrow + j) * a.H + col] = v[j];
        }
        __threadfence();
        epi_bar();
        // one counter per (token, column block): the tile that completes it combines
        if (etid < BNT) {
          int last = -1;
          if (etid < valid) {
            const int tkn = p2e[xrow + etid] / a.k;
            const int old = atomicAdd(&a.comb[tkn * a.m_tiles2 + c.m], 1);
            if (old == tok_n[tkn] - 1) last = tkn;
          }
          sflag[etid] = last;
        }
        epi_bar();
        __threadfence();
#pragma unroll 1
        for (int j = 0; j < BNT && j < valid; ++j) {
          const int tkn = sflag[j];
          if (tkn < 0 || col >= a.H) continue;
          float sum = 0.f;
          for (int s = 0; s < a.k; ++s) {
            const int pp = e2p[tkn * a.k + s];
            if (pp < 0) continue;
            sum = __fadd_rn(sum, __fmul_rn(a.w[tkn * a.k + s], __ldcg(a.y + (long)pp * a.H + col)));
          }
          reinterpret_cast<__nv_bfloat16 *>(a.out)[(long)tkn * a.H + col] = __float2bfloat16_rn(sum);
        }
        epi_bar();
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int encode(CUtensorMap *map, const void *ptr, long rows, int K, int box_rows) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return MOE_ERR_DEVICE;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_TENSOR_MAP;
}

template <int BNT>
cudaError_t configure(size_t smem) {
  cudaError_t e = raise_smem_limit(chain_kernel<BNT, kModeFc1>, smem);
  if (e == cudaSuccess) e = raise_smem_limit(chain_kernel<BNT, kModeFc2>, smem);
  if (e == cudaSuccess) e = raise_smem_limit(chain_kernel<BNT, kModeBoth>, smem);
  return e;
}

template <int BNT, int MODE>
cudaError_t launch_inst(const ChainPlan &p, const Launch &l) {
  ChainArgs a;
  a.map_w1 = p.map_w1;
  a.map_x = p.map_x;
  a.map_w2 = p.map_w2;
  a.map_h = p.map_h;
  a.ids = p.ids;
  a.w = p.w;
  a.h = p.h;
  a.y = p.y;
  a.out = p.out;
  a.comb = p.comb;
  a.done1 = p.done1;
  a.m_indptr_out = p.m_indptr;
  a.p2e_out = p.p2e;
  a.e2p_out = p.e2p;
  a.status = p.status;
  a.wait_ns = p.wait_ns;
  a.clamp = p.clamp;
  a.T = p.T;
  a.k = p.k;
  a.E = p.E;
  a.off = p.off;
  a.L = p.L;
  a.H = p.H;
  a.I = p.I;
  a.m_tiles1 = p.I / 64;
  a.m_tiles2 = (p.H + 127) / 128;
  a.ids_early = p.ids_early && l.pdl ? 1 : 0;
  const int grid = MODE == kModeFc1 ? p.grid1 : (MODE == kModeFc2 ? p.grid2 : p.grid_one);
  return launch_kernel(chain_kernel<BNT, MODE>, dim3(grid), dim3(kThreads), p.smem, l, a);
}

template <int BNT>
cudaError_t launch_bnt(const ChainPlan &p, int part, const Launch &l) {
  if (part == 1) return launch_inst<BNT, kModeFc1>(p, l);
  if (part == 2) return launch_inst<BNT, kModeFc2>(p, l);
  return launch_inst<BNT, kModeBoth>(p, l);
}

}  // namespace

size_t chain_comb_ints(int T, int H) { return (size_t)T * ((H + 127) / 128); }

int chain_prepare(ChainPlan &p) {
  if ((long)p.T * p.k > kChainMaxRoutes || p.I % 64 || p.H % 64) return MOE_ERR_SHAPE;
  p.bnt = p.T <= 16 ? 16 : (p.T <= 32 ? 32 : 64);
  int rc = encode(&p.map_w1, p.w1, (long)p.L * 2 * p.I, p.H, 64);
  if (rc == MOE_OK) rc = encode(&p.map_x, p.x, p.T, p.H, 1);
  if (rc == MOE_OK) rc = encode(&p.map_w2, p.w2, (long)p.L * p.H, p.I, 128);
  if (rc == MOE_OK) rc = encode(&p.map_h, p.h, (long)p.T * p.k, p.I, p.bnt);
  if (rc != MOE_OK) return rc;
  const long R = (long)p.T * p.k;
  p.smem = p.bnt == 16 ? ChainCfg<16>::smem_bytes(p.L, (int)R, p.T)
                       : (p.bnt == 32 ? ChainCfg<32>::smem_bytes(p.L, (int)R, p.T)
                                      : ChainCfg<64>::smem_bytes(p.L, (int)R, p.T));
  if (p.smem > 227 * 1024) return MOE_ERR_SHAPE;
  const long groups = p.L < R ? p.L : R;
  const long sms = device_sm_count();
  const long t1 = (long)(p.I / 64) * ((R + p.bnt - 1) / p.bnt + groups);
  const long t2 = (long)((p.H + 127) / 128) * ((R + p.bnt - 1) / p.bnt + groups);
  p.grid1 = (int)(t1 < sms ? t1 : sms);
  p.grid2 = (int)(t2 < sms ? t2 : sms);
  // one launch: at most one CTA per SM (each takes most of an SM's shared
  // memory), so every CTA whose FC1 tiles others wait for gets an SM
  p.grid_one = (int)(t1 + t2 < sms ? t1 + t2 : sms);
  cudaError_t e = p.bnt == 16 ? configure<16>(p.smem) : (p.bnt == 32 ? configure<32>(p.smem) : configure<64>(p.smem));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

namespace {

// Zeroes the one-launch kernel's counters (comb, then done1: consecutive in
// the workspace) and the status word, and lets the chain kernel start at once
// (programmatic dependent launch): the chain touches neither before its
// griddepcontrol.wait.  unreachable: done1 is filled with -1 instead.
__global__ void __launch_bounds__(256) chain_clear_kernel(int32_t *lo, int n, const int32_t *done1, int32_t *status,
                                                          int unreachable) {
  // The chain behind this kernel may launch at once (its prologue then runs
  // while the previous launch's chain ends); this kernel clears only once the
  // kernel before it in the stream has finished with the counters.
  pdl_launch_dependents();
  pdl_wait();
  for (int i = threadIdx.x; i < n; i += blockDim.x) lo[i] = unreachable && lo + i >= done1 ? -1 : 0;
  if (threadIdx.x == 0 && status) *status = 0;
}

}  // namespace

cudaError_t launch_chain_clear(const ChainPlan &p, bool unreachable, const Launch &l) {
  // the plan lays out done1 right after comb (256-byte aligned), so one range
  // from comb to the end of done1 covers both
  const int n = (int)(p.done1 + p.L + 1 - p.comb);
  return launch_kernel(chain_clear_kernel, dim3(1), dim3(256), 0, l, p.comb, n, (const int32_t *)p.done1,
                       p.status, unreachable ? 1 : 0);
}

cudaError_t launch_chain(const ChainPlan &p, int part, const Launch &l) {
  if (p.bnt == 16) return launch_bnt<16>(p, part, l);
  if (p.bnt == 32) return launch_bnt<32>(p, part, l);
  return launch_bnt<64>(p, part, l);
}

}  // namespace moe
