// S4 / S5 / S8 on CTA pairs: the persistent ragged grouped GEMM issued as
// 2-SM tensor-core MMAs (tcgen05.mma.cta_group::2, M = 256).
//
// A cluster of two CTAs shares one tcgen05 MMA stream.  Each group's rows are
// covered by two kinds of tiles, both 256 x (columns of one n-block):
//
//   main tile  256 token rows: each CTA stages 128 token rows (A) and half of
//              the 256 weight rows (B); D = tokens x weights, each CTA's TMEM
//              holding its own 128 token rows.
//   tail tile  the group's last r <= 128 rows (r = rows mod 256, groups of at
//              most 128 rows are a tail only): operands swapped, the 256
//              weight rows take the M side (128 staged by each CTA) and the r
//              token rows the N side (N = 16, 32, 64 or 128, half staged by
//              each CTA); D = weights x tokens, each CTA's TMEM holding its own
//              128 weight rows for all N tokens.  The MMA work scales with r.
//              In a group that also has main tiles, the weight rows are the
//              ones its main tiles of the same n-block read, so they come from
//              L2; a group of at most 128 rows streams its weights from HBM.
//
// A group with 128 < r < 256 rows left over gets one more main tile whose
// second CTA is only partly used.  Tiles past a group's rows are computed but
// never stored.
//
// For FC1 (SwiGLU) a main tile's weights are 128 up rows (first CTA) and the
// matching 128 gate rows (second CTA), so D columns 0..127 are u and 128..255
// are g for the same outputs; a tail tile's weights are, in each CTA, 64 up
// rows followed by the matching 64 gate rows, and the gate half hands its
// values to the up half through shared memory.
//
// E4M3 operands (the fp8 per-tensor family, Q = 1): a k-block is 128 codes,
// the same 128 bytes per row as 64 bf16 values, so stages, boxes and
// descriptor steps are unchanged; the MMAs are kind::f8f6f4 (K = 32); the
// epilogues dequantise by ascale * wscale[group], and FC1 requantises h to
// E4M3 codes e4m3(h * RN(1 / oscale)), as the one-CTA kernel does.  The
// product differs from the quotient h / oscale by at most one fp32 ulp, so a
// code can change only where that ulp straddles an E4M3 rounding boundary;
// the multiply keeps FC1's epilogue under the E4M3 MMAs (a correctly rounded
// division per element held FC1 at 0.87 ms instead of 0.74 ms at the
// few-large-experts shape).
//
// Synchronisation across the pair:
//   full[s]   leader only; both CTAs' TMA loads signal it (the leader arms the
//             transaction bytes of both);
//   empty[s]  each CTA; arrived by the leader's commit, multicast to both;
//   tfull[a]  each CTA; arrived by the leader's commit, multicast to both;
//   tempty[a] leader only; one arrival per epilogue warp of both CTAs.
// Every wait is bounded (see ptx.cuh); the pair meets at cluster barriers
// before any CTA touches the other's shared memory and before it exits.
#include <cuda_bf16.h>

#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;  // token (main) or weight (tail) rows per CTA
constexpr int BN = 256;  // main tile MMA N (weight rows per pair; 128 staged by each CTA)
constexpr int BK = 64;  // k-block: one 128-byte-wide TMA box, four K = 16 MMAs
// A ring stage holds KH k-blocks: one wait, 4 * KH MMAs and one commit per
// stage.  In a stand-alone loop a stage round (producer wait, arm, copies; MMA
// thread wait, MMAs, commit) cost of the order of 200 ns, enough to hold one
// k-block per round at about 84 ns per MMA against the 66 ns the tensor pipe
// needs; here two k-blocks per stage (three stages) shortened FC1 at the
// default workload by about 2 %.
constexpr int KH = 2;
// warps: 0 token producer, 1 TMEM owner + MMA issuer, 2..5 epilogue (TMEM
// lane quarters warp % 4), 6 weight producer; in gather mode warps 7..9 copy
// the token rows (one ring slot each) and warp 0 only drains the ring.  With
// E4M3 operands warps 7..10 are a second epilogue group: they take the upper
// half of a SwiGLU main tile's h columns (the requantising epilogue would
// otherwise outlast the tile's E4M3 MMAs) and only release the accumulator
// of the other tiles.
constexpr int kThreads = 224;
constexpr int kWeightWarp = 6;
constexpr int kGatherWarp0 = 7;
constexpr int kThreadsGather = 320;
constexpr int kEpiWarp1 = 7;
constexpr int kThreadsQ = 352;
constexpr int A_BYTES = BM * BK * 2;        // one k-block of the M-side operand
constexpr int B_BYTES = (BN / 2) * BK * 2;  // one k-block of this CTA's half of the N side
constexpr int A_STAGE = KH * A_BYTES;
constexpr int STAGE_BYTES = KH * (A_BYTES + B_BYTES);  // per CTA: [A k-blocks][B k-blocks]
constexpr int STG_BYTES = BM * 32 * 4;                 // fp32 store staging: 128 rows x 32 columns

// Shared-memory layout per epilogue kind (the fp32 form adds one store-staging
// buffer).
// Tiles claimed at run time (beside the small-group kernel) reach every role
// of both CTAs through a queue of this many slots in each CTA.  A slot is 64
// bits, the entry's sequence number (index + 1) above the tile number, so a
// reader needs only the slot itself: it spins on its own CTA's copy, with no
// acquire, and then counts itself done on the leader's empty barrier, with no
// release (the leader refills a slot once all readers have counted).  Waits and
// arrivals with cluster-scope acquire or release at every tile boundary cost
// the kernel about 7 % at 17 us tiles.
constexpr int kPairQD = 8;

template <int EPI>
struct PairLayout {
  static constexpr int STAGES = 3;
  static constexpr int NBARS = 2 * STAGES + 5 + kPairQD;  // ring, accumulators, drain, queue slots free
  static constexpr int STG_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = STG_OFF + (EPI == (int)Epi::kF32 ? STG_BYTES : 0);
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
  static constexpr int TQ_OFF = MISC_OFF + 16;  // tile queue [kPairQD] x 64 bits
  static constexpr int SG_OFF = TQ_OFF + kPairQD * 8;  // tail gate hand-off [16][64] fp32
  static constexpr int TAB_OFF = SG_OFF + 16 * 64 * 4;  // tile_start [G+1], gend [G], small groups [G]
};
constexpr uint32_t TMEM_COLS = 2 * BN;

struct PairArgs {
  CUtensorMap map_a;      // tokens [rows, K], box {64, 128}
  CUtensorMap map_b;      // weights [G * b_rows, K], box {64, 128}
  CUtensorMap map_w64;    // weights, box {64, 64} (FC1 tail tiles)
  CUtensorMap map_t[4];   // tokens, box {64, 8 / 16 / 32 / 64} (tail tiles, N = 16..128)
  CUtensorMap map_y;      // fp32 output [rows, n_out], box {32, 128}, 128-byte swizzle (TMA stores)
  const uint16_t *x;      // gather mode: token rows x [x_rows, K]
  const int32_t *p2e;     // gather mode: permuted row -> expanded index
  long x_rows;
  int gather_k;           // gather mode: top_k (token = p2e[row] / top_k); 0 = rows given directly
  const int32_t *group_end;
  void *out;
  int32_t *status;
  unsigned long long wait_ns;  // bounded-wait limit of this launch
  const float *clamp;         // SwiGLU epilogue: [groups] SwiGLUStep limits, or null
  const float *wscale;        // E4M3: [groups] weight scales
  float ascale, oscale;       // E4M3: activation scale of A, requantisation scale of h
  long max_rows;
  int G, K, n_out, b_rows, n_tiles, m_major;
  int tail_max;               // remainders of up to this many rows run as swap-AB tail tiles (0: none)
  // Beside the small-group kernel (null: static round-robin over all groups):
  // [0] main-tile claims, [1] small-tile claims (shared with it), [2] its
  // start flag, [3] its CTAs done.  Groups of 1..small_max rows are its tiles.
  int32_t *sched;
  int small_max, side_ctas;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// The second epilogue group's own barrier (E4M3): ORs a flag across its four warps.
__device__ __forceinline__ bool epi1_bar_any(bool flag) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 3, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)flag)
      : "memory");
  return r != 0;
}

// Barrier over the four epilogue warps of this CTA that ORs a flag across them.
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

// Waits (bounded, like mbar_wait) until the 64-bit queue slot holds sequence
// number seq and returns its tile number in *t; false on abort or timeout.
__device__ __forceinline__ bool queue_wait(volatile unsigned long long *slot, uint32_t seq, volatile int *abort,
                                           int32_t *status, unsigned long long limit_ns, int *t) {
  unsigned long long v = *slot;
  if ((uint32_t)(v >> 32) == seq) {
    *t = (int)(uint32_t)v;
    return true;
  }
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    v = *slot;
    if ((uint32_t)(v >> 32) == seq) {
      *t = (int)(uint32_t)v;
      return true;
    }
    if ((it & 63u) == 0u) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort = 1;
        if (status) atomicOr(reinterpret_cast<unsigned int *>(status), MOE_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// Tail tile N for r tail rows (1..128): the smallest of 16, 32, 64, 128.
__device__ __forceinline__ int tail_n(int r) { return r <= 16 ? 16 : (r <= 32 ? 32 : (r <= 64 ? 64 : 128)); }
__device__ __forceinline__ int tail_map(int n) { return n == 16 ? 0 : (n == 32 ? 1 : (n == 64 ? 2 : 3)); }

struct PairTile {
  int g, mp, n;   // group, m-pair index inside the group, n-block
  int gstart;     // first row of the group
  int tail;       // 0: main tile; else the tail's row count r (1..128)
};

// Per group: full pairs cnt / 256 plus one more tile when rows are left.
__device__ __forceinline__ int group_pairs(int cnt) { return cnt > 0 ? (cnt + 2 * BM - 1) / (2 * BM) : 0; }

// Tile order: group-major; inside a group the m-pairs or the n-blocks run
// innermost as chosen on the host.  tile_start[g] is the prefix of the
// groups' pair counts.  (Spreading the tiles of the groups of at most 128 rows
// evenly among the others was measured slower: their once-read weight
// streams then evict the large groups' reused weight blocks from L2.)
__device__ __forceinline__ PairTile decode_pair_tile(int t, const int *tile_start, const int *gend, int G,
                                                     int n_tiles, int m_major, int tail_max) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_start[mid] * n_tiles <= t) lo = mid;
    else hi = mid;
  }
  PairTile c;
  c.g = lo;
  const int mp = tile_start[lo + 1] - tile_start[lo];
  const int local = t - tile_start[lo] * n_tiles;
  if (m_major) {
    c.mp = local / n_tiles;
    c.n = local - c.mp * n_tiles;
  } else {
    c.n = local / mp;
    c.mp = local - c.n * mp;
  }
  c.gstart = lo == 0 ? 0 : gend[lo - 1];
  const int r = gend[lo] - c.gstart - c.mp * 2 * BM;  // rows from this tile's first row to the group's end
  c.tail = (r > 0 && r <= tail_max) ? r : 0;
  return c;
}

// E4M3 SwiGLU main tile, h columns [col_lo, col_hi) of this thread's token
// row: u and g dequantised by ascale * wscale[g], SwiGLU(Step), h requantised
// as h times RN(1 / h_scale).
template <int BNT>
__device__ __forceinline__ void epi_swiglu_e4m3(const PairArgs &args, uint32_t taddr, long orow, bool row_ok,
                                                int g, int n_blk, int col_lo, int col_hi) {
  uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(args.out) + orow * args.n_out +
                                         (long)n_blk * (BNT / 2));
  const float lim = step_limit(args.clamp, g);
  const float sc = __fmul_rn(args.ascale, __ldg(args.wscale + g));
  const float inv = __frcp_rn(args.oscale);  // h / h_scale as h times RN(1 / h_scale)
#pragma unroll 1
  for (int col = col_lo; col < col_hi; col += 32) {
    uint32_t u[32], gv[32];
    tmem_ld_32x32b_x32(taddr + col, u);
    tmem_ld_32x32b_x32(taddr + BNT / 2 + col, gv);
    tmem_ld_wait();
    uint32_t packed[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float hv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float uu = __fmul_rn(__uint_as_float(u[4 * i + q]), sc);
        const float gg = __fmul_rn(__uint_as_float(gv[4 * i + q]), sc);
        hv[q] = __fmul_rn(swiglu_step(gg, uu, lim), inv);
      }
      packed[i] = e4m3x2(hv[0], hv[1]) | (e4m3x2(hv[2], hv[3]) << 16);
    }
    if (row_ok) {
      dst[col / 16] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      dst[col / 16 + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    }
  }
}

// This CTA's operand boxes for a tile: the token box (rows tok_row ..
// tok_row + tok_rows) and the weight box(es), and the bytes both bring per
// k-block.
struct PairOperands {
  int tok_row, tok_rows, tmap, w_row, w_row2;
  uint32_t bytes;    // token + weight box bytes per k-block
  uint32_t w_bytes;  // weight box bytes per k-block
};

template <bool SWIGLU>
__device__ __forceinline__ PairOperands pair_operands(const PairTile &c, uint32_t rank, int b_rows) {
  PairOperands o;
  o.w_row2 = 0;
  o.tmap = 0;
  if (!c.tail) {
    o.tok_row = c.gstart + (2 * c.mp + (int)rank) * BM;
    if (SWIGLU)  // leader stages the up rows, the peer the gate rows
      o.w_row = c.g * b_rows + c.n * (BN / 2) + (int)rank * (b_rows / 2);
    else
      o.w_row = c.g * b_rows + c.n * BN + (int)rank * (BN / 2);
    o.bytes = A_BYTES + B_BYTES;
    o.w_bytes = B_BYTES;
    o.tok_rows = BM;
  } else {
    const int n = tail_n(c.tail);
    o.tmap = tail_map(n);
    if (SWIGLU) {  // 64 up rows then the matching 64 gate rows
      o.w_row = c.g * b_rows + c.n * (BN / 2) + (int)rank * 64;
      o.w_row2 = o.w_row + b_rows / 2;
    } else {
      o.w_row = c.g * b_rows + c.n * BN + (int)rank * BM;
    }
    o.tok_row = c.gstart + c.mp * 2 * BM + (int)rank * (n / 2);
    o.bytes = A_BYTES + (uint32_t)(n / 2) * BK * 2;
    o.w_bytes = A_BYTES;
    o.tok_rows = n / 2;
  }
  return o;
}

template <int EPI, bool GATH, int Q>
__global__ void __launch_bounds__(GATH ? kThreadsGather : (Q ? kThreadsQ : kThreads), 1)
    pair_gemm_kernel(const __grid_constant__ PairArgs args) {
  static_assert(!Q || (!GATH && EPI != (int)Epi::kBf16), "E4M3: FC1 and FC2 epilogues, token rows by TMA");
  constexpr int KE = Q ? 128 : BK;  // elements per k-block (128 bytes of a row either way)
  using Lay = PairLayout<EPI>;
  constexpr int STAGES = Lay::STAGES;
  static_assert(kThreadsGather / 32 - kGatherWarp0 == STAGES, "one gather warp per ring slot");
  constexpr int BAR_OFF = Lay::BAR_OFF;
  constexpr int MISC_OFF = Lay::MISC_OFF;
  constexpr int SG_OFF = Lay::SG_OFF;
  constexpr int TAB_OFF = Lay::TAB_OFF;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_base + BAR_OFF;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 4);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + MISC_OFF + 4);
  volatile int *n_small_s = reinterpret_cast<volatile int *>(smem + MISC_OFF + 8);
  volatile unsigned long long *tq = reinterpret_cast<volatile unsigned long long *>(smem + Lay::TQ_OFF);
  float *sg = reinterpret_cast<float *>(smem + SG_OFF);
  int *tile_start = reinterpret_cast<int *>(smem + TAB_OFF);
  int *gend = tile_start + (args.G + 1);
  int *small_g = gend + args.G;
  // Run-time tile claims (beside the small-group kernel): the leader's weight
  // producer claims each tile and publishes it to both CTAs' queues.
  const bool dyn = !GATH && args.sched != nullptr;
  auto qempty_bar = [&](int j) { return bar_base + 8u * (2 * STAGES + 5 + j); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = leader
  const int G = args.G;
  constexpr bool kSwiGLU = EPI == (int)Epi::kSwiGLU;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // gather mode: the leader's weight arm plus one arrival per CTA's gather warp
      mbar_init(full_bar(s), GATH ? 3 : 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), Q ? 16 : 8);  // 4 (E4M3: 8) epilogue warps x 2 CTAs
    }
    mbar_init(drain_bar, 1);
    // queue readers: token producer and epilogue warps of both CTAs, the MMA
    // thread, the peer's weight producer
    const uint32_t readers = 2u * (1u + 4u + (Q ? 4u : 0u)) + 2u;
    for (int j = 0; j < kPairQD; ++j) {
      mbar_init(qempty_bar(j), readers);
      tq[j] = 0ull;  // sequence 0: nothing published
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&args.map_a);
    tma_prefetch_desc(&args.map_b);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (dyn) {
    // Launched behind the small-group kernel, which sets the flag once the
    // gather and the sort have finished (waiting for the whole previous grid
    // here would wait for that kernel to end).
    if (threadIdx.x == 0 && counter_wait(args.sched + 2, 1, abort_flag, args.status, args.wait_ns))
      fence_proxy_async_global();  // the rows the flag releases are read by TMA
    __syncthreads();
  } else {
    pdl_wait();
  }
  for (int g = threadIdx.x; g < G; g += (int)blockDim.x) {
    long e = args.group_end[g];
    e = e < 0 ? 0 : (e > args.max_rows ? args.max_rows : e);
    gend[g] = (int)e;
  }
  __syncthreads();
  if (warp == 0) {
    // tile_start = prefix of per-group tile counts (per n-block); with claims
    // at run time the groups of 1..small_max rows are listed apart (small_g)
    int carry = 0, scarry = 0;
    if (lane == 0) tile_start[0] = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int mp = 0;
      bool small = false;
      if (g < G) {
        const int cnt = gend[g] - (g == 0 ? 0 : gend[g - 1]);
        small = dyn && cnt > 0 && cnt <= args.small_max;
        mp = small ? 0 : group_pairs(cnt);
      }
      int inc = mp;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (g < G) tile_start[g + 1] = carry + inc;
      carry += __shfl_sync(0xffffffffu, inc, 31);
      const uint32_t m = __ballot_sync(0xffffffffu, small);
      if (small) small_g[scarry + __popc(m & ((1u << lane) - 1u))] = g;
      scarry += __popc(m);
    }
    if (lane == 0) *n_small_s = scarry;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers and TMEM exist before any cross-CTA traffic
  tc_fence_after();
  pdl_launch_dependents();

  const uint32_t tmem_base = *tmem_holder;
  const bool dead = *abort_flag != 0;  // the start flag never came: no tiles
  const int total = dead ? 0 : tile_start[G] * args.n_tiles;  // tiles numbered 0 .. total - 1 first
  const int total_small = dead ? 0 : *n_small_s * args.n_tiles;  // then small-group tiles
  // Claims at run time only when there are small-group tiles to share: without
  // them the small-group kernel leaves at once and this grid's late clusters
  // start a few microseconds late, which costs less than the claims.
  const bool claims = dyn && total_small > 0;
  const int num_kb = args.K / KE;
  const int n_rounds = (num_kb + KH - 1) / KH;  // ring stages per tile
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;

  // Tile number -> coordinates: the main numbering, then (claims at run time
  // only) the small groups' tiles, each a tail-only group.
  auto tile_of = [&](int t) -> PairTile {
    if (t < total) return decode_pair_tile(t, tile_start, gend, G, args.n_tiles, args.m_major, args.tail_max);
    PairTile c;
    const int s = t - total;
    const int j = s / args.n_tiles;
    c.n = s - j * args.n_tiles;
    c.g = small_g[j];
    c.mp = 0;
    c.gstart = c.g == 0 ? 0 : gend[c.g - 1];
    c.tail = gend[c.g] - c.gstart;
    return c;
  };
  // The i-th tile of this cluster for one reader thread (-1: no more).
  // Static: round-robin over the clusters.  Run time: the queue entry, whose
  // slot the reader then releases on the leader's qempty barrier.
  auto seq_tile = [&](int i) -> int {
    if (!claims) {
      const int t = cluster + i * nclusters;
      return t < total ? t : -1;
    }
    const int j = i % kPairQD;
    int t;
    if (!queue_wait(tq + j, (uint32_t)(i + 1), abort_flag, args.status, args.wait_ns, &t)) return -1;
    // t came from the slot (the wait ended on it), so the arrival cannot pass the read
    if (rank == 0) mbar_arrive_relaxed(qempty_bar(j));
    else mbar_arrive_relaxed_cluster(mapa_shared(qempty_bar(j), 0));
    return t;
  };

  if (warp == 0) {
    // --------------------------------------------------------- token producer --
    // Lane 0 waits, arms the leader's barrier and loads the token box.  In
    // gather mode the gather warps fill the token boxes and the weight
    // producer arms; this warp only counts the rounds for the final drain.
    const uint64_t pol_first = policy_evict_first(), pol_last = policy_evict_last();
    int it = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      int t = -1;
      if (lane == 0) t = seq_tile(i);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t < 0) break;
      if (GATH) {
        it += n_rounds;
        continue;
      }
      const PairTile c = tile_of(t);
      const uint64_t pol = (c.tail && c.mp == 0) ? pol_first : pol_last;
      const PairOperands o = pair_operands<kSwiGLU>(c, rank, args.b_rows);
      const CUtensorMap *tok_map = c.tail ? &args.map_t[o.tmap] : &args.map_a;
      for (int kr = 0; kr < n_rounds; ++kr, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
        const int nk = min(KH, num_kb - kr * KH);
        if (lane == 0) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, args.status, args.wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t leader_full = mapa_shared(full_bar(s), 0);
          if (rank == 0) mbar_arrive_expect_tx(full_bar(s), 2 * o.bytes * (uint32_t)nk);
          for (int h = 0; h < nk; ++h) {
            const int kx = (kr * KH + h) * KE;
            const uint32_t t_dst = smem_base + s * STAGE_BYTES + (c.tail ? A_STAGE + h * B_BYTES : h * A_BYTES);
            tma_load_2d_pair(t_dst, tok_map, leader_full, kx, o.tok_row, pol);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0 && rank == 0) {  // let both CTAs' last copies land (they all signal the leader)
      for (int j = it > STAGES ? it - STAGES : 0; j < it; ++j)
        mbar_wait(full_bar(j % STAGES), (uint32_t)(j / STAGES) & 1u, nullptr, args.status, args.wait_ns);
    }
  } else if (warp == kWeightWarp) {
    // -------------------------------------------------------- weight producer --
    // A second issuing thread: one thread's TMA copies run at about half of
    // what an SM can take in, so weights and tokens are issued separately.
    if (lane == 0) {
      const uint64_t pol_first = policy_evict_first(), pol_last = policy_evict_last();
      int it = 0;
      bool ok = true;
      // Claims (leader, run time): main tiles while any are left, then
      // small-group tiles.  The queue runs one tile ahead of this thread (the
      // peer's producers find the next tile published when they reach it),
      // and each claim is made one tile before it is published (the counter's
      // round trip overlaps a tile's copies), after the publication before
      // it (a release, which would otherwise wait for the round trip).
      bool main_left = true, pend_main = true;
      int pend = 0, cur = -1;
      auto resolve = [&]() -> int {  // the pending claim as a tile number, -1 when none is left
        if (pend_main && pend >= total) {
          main_left = false;
          pend_main = false;
          pend = atomicAdd(args.sched + 1, 1);
        }
        return pend_main ? pend : (pend < total_small ? total + pend : -1);
      };
      auto publish = [&](int i, int t) -> int {  // queue slot of the cluster's i-th tile, in both CTAs
        const int j = i % kPairQD;
        if (t >= 0 && !mbar_wait<false, true>(qempty_bar(j), ((uint32_t)(i / kPairQD) & 1u) ^ 1u, abort_flag,
                                              args.status, args.wait_ns))
          t = -1;
        const unsigned long long v = ((unsigned long long)(uint32_t)(i + 1) << 32) | (uint32_t)t;
        tq[j] = v;
        asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(mapa_shared(smem_u32((const void *)(tq + j)), 1)),
                     "l"(v)
                     : "memory");
        if (t >= 0) {  // the claim for the tile after it
          pend_main = main_left;
          pend = atomicAdd(args.sched + (main_left ? 0 : 1), 1);
        }
        return t;
      };
      if (claims && rank == 0) {
        pend = atomicAdd(args.sched + 0, 1);
        cur = publish(0, resolve());
      }
      for (int i = 0;; ++i) {
        int t;
        if (claims && rank == 0) {
          t = cur;
          if (t < 0) break;
          cur = publish(i + 1, ok ? resolve() : -1);  // -1 ends every role's loop
        } else {
          if (!ok) break;
          t = seq_tile(i);
        }
        if (t < 0) break;
        const PairTile c = tile_of(t);
        // L2: a group that is only this tail reads its weights once (stream them
        // through); everything else is read again by neighbouring tiles (keep it)
        const uint64_t pol = (c.tail && c.mp == 0) ? pol_first : pol_last;
        const PairOperands o = pair_operands<kSwiGLU>(c, rank, args.b_rows);
        for (int kr = 0; kr < n_rounds; ++kr, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          const int nk = min(KH, num_kb - kr * KH);
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, args.status, args.wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t leader_full = mapa_shared(full_bar(s), 0);
          // gather mode: only the weight boxes are counted as transaction bytes
          if (GATH && rank == 0) mbar_arrive_expect_tx(full_bar(s), 2 * o.w_bytes * (uint32_t)nk);
          for (int h = 0; h < nk; ++h) {
            const int kx = (kr * KH + h) * KE;
            const uint32_t w_dst = smem_base + s * STAGE_BYTES + (c.tail ? h * A_BYTES : A_STAGE + h * B_BYTES);
            if (c.tail && kSwiGLU) {  // 64 up rows then the matching 64 gate rows
              tma_load_2d_pair(w_dst, &args.map_w64, leader_full, kx, o.w_row, pol);
              tma_load_2d_pair(w_dst + 64 * 128, &args.map_w64, leader_full, kx, o.w_row2, pol);
            } else {
              tma_load_2d_pair(w_dst, &args.map_b, leader_full, kx, o.w_row, pol);
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ----------------------------------------------------- MMA issuer (leader) --
      int it = 0;
      bool ok = true;
      for (int tc = 0; ok; ++tc) {
        const int t = seq_tile(tc);
        if (t < 0) break;
        const PairTile c = tile_of(t);
        const uint32_t n_mma = c.tail ? (uint32_t)tail_n(c.tail) : (uint32_t)BN;
        const uint32_t idesc = Q ? idesc_e4m3_f32(2 * BM, n_mma) : idesc_bf16_f32(2 * BM, n_mma);
        const int acc = tc & 1;
        const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
        if (!mbar_wait(tempty_bar(acc), aph ^ 1u, abort_flag, args.status, args.wait_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kr = 0; kr < n_rounds; ++kr, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          const int nk = min(KH, num_kb - kr * KH);
          if (!mbar_wait<GATH>(full_bar(s), ph, abort_flag, args.status, args.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_base + s * STAGE_BYTES;
          for (int h = 0; h < nk; ++h) {
            const uint64_t a_desc = smem_desc_k_sw128(st + h * A_BYTES);
            const uint64_t b_desc = smem_desc_k_sw128(st + A_STAGE + h * B_BYTES);
#pragma unroll
            for (int k = 0; k < 4; ++k) {  // 32 bytes of each row per MMA: 16 bf16 or 32 E4M3 values
              if (Q) umma_e4m3_pair(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, (kr | h | k) != 0);
              else umma_bf16_pair(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, (kr | h | k) != 0);
            }
          }
          umma_commit_pair(empty_bar(s), 0x3);
        }
        if (ok) umma_commit_pair(tfull_bar(acc), 0x3);
      }
      umma_commit_pair(drain_bar, 0x1);
      mbar_wait(drain_bar, 0, nullptr, args.status, args.wait_ns);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------------ epilogue --
    const int quarter = warp & 3;
    const int r_in_tile = quarter * 32 + lane;  // TMEM lane: token row (main) or weight row (tail)
    const uint32_t leader_tempty0 = mapa_shared(tempty_bar(0), 0);
    const uint32_t leader_tempty1 = mapa_shared(tempty_bar(1), 0);
    for (int tc = 0;; ++tc) {
      int t = -1;
      if (lane == 0) t = seq_tile(tc);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (epi_bar_any(t < 0)) break;  // all four warps stop together
      const PairTile c = tile_of(t);
      const int acc = tc & 1;
      const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
      const bool got = mbar_wait(tfull_bar(acc), aph, abort_flag, args.status, args.wait_ns);
      if (epi_bar_any(!got)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      if (!c.tail) {
        const int row0 = c.gstart + (2 * c.mp + (int)rank) * BM;
        const int valid = gend[c.g] - row0;  // may be <= 0 for the second CTA's rows
        const bool row_ok = r_in_tile < valid;
        const long orow = (long)row0 + r_in_tile;
        if (kSwiGLU && Q) {
          // E4M3: the lower half of the h columns (the second group takes the upper half)
          epi_swiglu_e4m3<BN>(args, taddr, orow, row_ok, c.g, c.n, 0, BN / 4);
        } else if (kSwiGLU) {
          uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(args.out) +
                                                 orow * args.n_out + (long)c.n * (BN / 2));
          const float lim = step_limit(args.clamp, c.g);
#pragma unroll 1
          for (int col = 0; col < BN / 2; col += 32) {
            uint32_t u[32], g[32];
            tmem_ld_32x32b_x32(taddr + col, u);
            tmem_ld_32x32b_x32(taddr + BN / 2 + col, g);
            tmem_ld_wait();
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              packed[i] = pack_bf16x2(swiglu_step(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i]), lim),
                                      swiglu_step(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1]), lim));
            if (row_ok) {
#pragma unroll
              for (int v = 0; v < 4; ++v)
                dst[col / 8 + v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                              packed[4 * v + 3]);
            }
          }
        } else if (EPI == (int)Epi::kF32) {
          // E4M3: y dequantised by ascale * wscale[g]
          const float sc = Q ? __fmul_rn(args.ascale, __ldg(args.wscale + c.g)) : 1.f;
          if (valid >= BM) {
            // full tile: 32-column chunks staged in swizzled shared memory and
            // written by TMA stores (whole 128-byte rows)
            const int etid = threadIdx.x - 64;
#pragma unroll 1
            for (int col = 0; col < BN; col += 32) {
              if (col > 0) {  // the previous chunk's store has read the staging buffer
                if (etid == 0) bulk_wait_read<0>();
                epi_bar();
              }
              uint32_t r[32];
              tmem_ld_32x32b_x32(taddr + col, r);
              tmem_ld_wait();
              if (Q) {
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[i]), sc));
              }
              const uint32_t row_addr = smem_base + Lay::STG_OFF + r_in_tile * 128;
#pragma unroll
              for (int v = 0; v < 8; ++v)
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 row_addr + (uint32_t)((v ^ (r_in_tile & 7)) * 16)),
                             "r"(r[4 * v]), "r"(r[4 * v + 1]), "r"(r[4 * v + 2]), "r"(r[4 * v + 3])
                             : "memory");
              fence_proxy_async_smem();
              epi_bar();
              if (etid == 0) {
                tma_store_2d(&args.map_y, smem_base + Lay::STG_OFF, c.n * BN + col, row0);
                bulk_commit();
              }
            }
            if (etid == 0) bulk_wait_read<0>();
            epi_bar();
          } else {
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<float *>(args.out) +
                                                   orow * args.n_out + (long)c.n * BN);
#pragma unroll 1
            for (int col = 0; col < BN; col += 32) {
              uint32_t r[32];
              tmem_ld_32x32b_x32(taddr + col, r);
              tmem_ld_wait();
              if (Q) {
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[i]), sc));
              }
              if (row_ok) {
#pragma unroll
                for (int v = 0; v < 8; ++v)
                  dst[col / 4 + v] = make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
              }
            }
          }
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(args.out) +
                                                 orow * args.n_out + (long)c.n * BN);
#pragma unroll 1
          for (int col = 0; col < BN; col += 32) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + col, r);
            tmem_ld_wait();
            if (row_ok) {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 o;
                o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                dst[col / 8 + v] = o;
              }
            }
          }
        }
      } else {
        // tail tile: lanes are weight rows, columns are the tail's tokens
        const int n = tail_n(c.tail);
        const long tok0 = (long)c.gstart + c.mp * 2 * BM;
        const float lim = step_limit(args.clamp, c.g);
        const float sc = Q ? __fmul_rn(args.ascale, __ldg(args.wscale + c.g)) : 1.f;  // E4M3 dequantisation
#pragma unroll 1
        for (int c0 = 0; c0 < n; c0 += 16) {
          uint32_t r[16];
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
              "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
              : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
                "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
              : "r"(taddr + (uint32_t)c0));
          tmem_ld_wait();
          if (kSwiGLU) {
            if (r_in_tile >= 64) {
#pragma unroll
              for (int j = 0; j < 16; ++j) sg[j * 64 + (r_in_tile - 64)] = __uint_as_float(r[j]);
            }
            epi_bar();
            if (r_in_tile < 64) {
              const long col = (long)c.n * (BN / 2) + (int)rank * 64 + r_in_tile;
              if (Q) {
                uint8_t *h = reinterpret_cast<uint8_t *>(args.out);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (c0 + j < c.tail) {
                    const float uu = __fmul_rn(__uint_as_float(r[j]), sc);
                    const float gg = __fmul_rn(sg[j * 64 + r_in_tile], sc);
                    h[(tok0 + c0 + j) * args.n_out + col] =
                        (uint8_t)(e4m3x2(__fmul_rn(swiglu_step(gg, uu, lim), __frcp_rn(args.oscale)), 0.f) & 0xFFu);
                  }
              } else {
                __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(args.out);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (c0 + j < c.tail)
                    h[(tok0 + c0 + j) * args.n_out + col] =
                        __float2bfloat16_rn(swiglu_step(sg[j * 64 + r_in_tile], __uint_as_float(r[j]), lim));
              }
            }
            epi_bar();
          } else {
            const long col = (long)c.n * BN + (int)rank * BM + r_in_tile;
            if (EPI == (int)Epi::kF32) {
              float *y = reinterpret_cast<float *>(args.out);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < c.tail)
                  y[(tok0 + c0 + j) * args.n_out + col] = Q ? __fmul_rn(__uint_as_float(r[j]), sc) : __uint_as_float(r[j]);
            } else {
              __nv_bfloat16 *y = reinterpret_cast<__nv_bfloat16 *>(args.out);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < c.tail)
                  y[(tok0 + c0 + j) * args.n_out + col] = __float2bfloat16_rn(__uint_as_float(r[j]));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? leader_tempty1 : leader_tempty0);
    }
  } else if (Q && warp >= kEpiWarp1 && warp < kEpiWarp1 + 4) {
    // ------------------------------------------------ second epilogue group (E4M3) --
    const int quarter = warp & 3;
    const int r_in_tile = quarter * 32 + lane;
    const uint32_t leader_tempty0 = mapa_shared(tempty_bar(0), 0);
    const uint32_t leader_tempty1 = mapa_shared(tempty_bar(1), 0);
    for (int tc = 0;; ++tc) {
      int t = -1;
      if (lane == 0) t = seq_tile(tc);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (epi1_bar_any(t < 0)) break;  // all four warps of the group stop together
      const PairTile c = tile_of(t);
      const int acc = tc & 1;
      const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
      const bool got = mbar_wait(tfull_bar(acc), aph, abort_flag, args.status, args.wait_ns);
      if (epi1_bar_any(!got)) break;
      tc_fence_after();
      if (kSwiGLU && !c.tail) {
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
        const int row0 = c.gstart + (2 * c.mp + (int)rank) * BM;
        const int valid = gend[c.g] - row0;
        epi_swiglu_e4m3<BN>(args, taddr, (long)row0 + r_in_tile, r_in_tile < valid, c.g, c.n, BN / 4, BN / 2);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? leader_tempty1 : leader_tempty0);
    }
  } else if (GATH && warp >= kGatherWarp0) {
    // -------------------------------------------------------- token row gather --
    // Gather warp j fills the token boxes of ring slot j only, straight from x:
    // row q of a box is x[p2e[p] / top_k] for its permuted row p.  Per k-block
    // lane l copies 16-byte chunk l % 8 of rows l / 8, l / 8 + 4, ... into the
    // 128-byte-swizzled layout a TMA box has (chunk c of row q at q * 128 +
    // ((c ^ (q % 8)) * 16)).  Once its copies have landed the warp makes them
    // visible to the tensor cores and arrives on the leader's full barrier.
    // (Rows past the last routed row read row 0 of x; their results are
    // never stored.)
    const int j = warp - kGatherWarp0;
    const uint64_t pol = policy_evict_last();  // each token row is read by top_k groups
    const int m_total = G > 0 ? gend[G - 1] : 0;
    const int sub = lane >> 3, chunk = lane & 7;
    const char *xb = reinterpret_cast<const char *>(args.x) + chunk * 16;
    const long row_bytes = (long)args.K * 2;
    const uint32_t leader_full = mapa_shared(full_bar(j), 0);
    int it = 0;
    bool ok = true;
    for (int t = cluster; t < total && ok; t += nclusters) {
      const PairTile c = decode_pair_tile(t, tile_start, gend, G, args.n_tiles, args.m_major, args.tail_max);
      const PairOperands o = pair_operands<kSwiGLU>(c, rank, args.b_rows);
      const int r4 = o.tok_rows / 4;  // rows per lane: 2 .. 32
      int tok[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        tok[i] = 0;
        if (i < r4) {
          const int p = o.tok_row + sub + 4 * i;
          const int tk = p < m_total ? args.p2e[p] / args.gather_k : 0;
          tok[i] = (tk < 0 || tk >= args.x_rows) ? 0 : tk;
        }
      }
      for (int kr = 0; kr < n_rounds; ++kr, ++it) {
        if (it % STAGES != j) continue;
        const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
        const int nk = min(KH, num_kb - kr * KH);
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait(empty_bar(j), ph ^ 1u, abort_flag, args.status, args.wait_ns) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        for (int h = 0; h < nk; ++h) {
          const long kx_bytes = (long)(kr * KH + h) * BK * 2;
          const uint32_t dst0 = smem_base + j * STAGE_BYTES + (c.tail ? A_STAGE + h * B_BYTES : h * A_BYTES) +
                                (uint32_t)sub * 128;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i < r4) {
              // row q = sub + 4 i, so q % 8 = sub + 4 (i % 2)
              const uint32_t dst = dst0 + (uint32_t)i * 512 + (uint32_t)((chunk ^ (sub + 4 * (i & 1))) << 4);
              cp_async_16(dst, xb + (long)tok[i] * row_bytes + kx_bytes, pol);
            }
          }
        }
        cp_async_commit();
        cp_async_wait_all();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(leader_full);
      }
    }
  }

  if (EPI == (int)Epi::kF32 && threadIdx.x == 64) bulk_wait_all();  // TMA stores complete
  // Beside the small-group kernel: this grid ends only after that kernel's
  // CTAs have written their rows, so whatever waits for this grid (the next
  // kernel's dependent-launch wait) also sees those rows.
  if (dyn && blockIdx.x == 0 && threadIdx.x == 0)
    counter_wait(args.sched + 3, args.side_ctas, abort_flag, args.status, args.wait_ns);
  __syncthreads();
  cluster_sync();  // the peer no longer reads this CTA's shared memory or TMEM
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
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

// uint8 [rows, K] (E4M3 codes): box {128, box_rows}, 128-byte swizzle.
int encode_u8(CUtensorMap *map, const void *ptr, long rows, int K, int box_rows) {
  void *p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return MOE_ERR_DEVICE;
  EncodeTiledFn fn = reinterpret_cast<EncodeTiledFn>(p);
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_TENSOR_MAP;
}

// fp32 [rows, cols] row-major for TMA stores: box {32, 128}, 128-byte swizzle.
int encode_f32_store(CUtensorMap *map, void *ptr, long rows, int cols) {
  EncodeTiledFn fn = nullptr;
  {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return MOE_ERR_DEVICE;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {32, (cuuint32_t)BM};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_TENSOR_MAP;
}

}  // namespace

size_t pair_gemm_smem(Epi epi, int G) {
  const int tab = epi == Epi::kF32 ? PairLayout<(int)Epi::kF32>::TAB_OFF : PairLayout<(int)Epi::kBf16>::TAB_OFF;
  return 1024 + tab + (size_t)(3 * G + 1) * 4;
}

bool pair_gemm_supported(Epi epi, int n_out) {
  return epi == Epi::kSwiGLU ? (n_out % (BN / 2) == 0) : (n_out % BN == 0);
}

int pair_gemm_encode_extra(GemmPlan &p, const uint16_t *A, long a_rows, const uint16_t *B,
                           long b_rows_total, int K) {
  int rc = encode(&p.map_w64, B, b_rows_total, K, 64);
  for (int i = 0; i < 4 && rc == MOE_OK; ++i) rc = encode(&p.map_t[i], A, a_rows, K, 8 << i);
  if (rc == MOE_OK && p.epi == Epi::kF32) rc = encode_f32_store(&p.map_y, p.out, p.max_rows, p.n_out);
  return rc;
}

int pair_gemm_encode_u8(GemmPlan &p, const uint8_t *A, long a_rows, const uint8_t *B, long b_rows_total, int K) {
  int rc = encode_u8(&p.map_a, A, a_rows, K, BM);
  if (rc == MOE_OK) rc = encode_u8(&p.map_b, B, b_rows_total, K, BN / 2);
  if (rc == MOE_OK) rc = encode_u8(&p.map_w64, B, b_rows_total, K, 64);
  for (int i = 0; i < 4 && rc == MOE_OK; ++i) rc = encode_u8(&p.map_t[i], A, a_rows, K, 8 << i);
  if (rc == MOE_OK && p.epi == Epi::kF32) rc = encode_f32_store(&p.map_y, p.out, p.max_rows, p.n_out);
  return rc;
}

cudaError_t pair_gemm_configure(Epi epi, size_t smem, int q) {
  if (q) {
    if (epi == Epi::kSwiGLU) return raise_smem_limit(pair_gemm_kernel<(int)Epi::kSwiGLU, false, 1>, smem);
    return raise_smem_limit(pair_gemm_kernel<(int)Epi::kF32, false, 1>, smem);
  }
  if (epi == Epi::kSwiGLU) {
    const cudaError_t e = raise_smem_limit(pair_gemm_kernel<(int)Epi::kSwiGLU, false, 0>, smem);
    if (e != cudaSuccess) return e;
    return raise_smem_limit(pair_gemm_kernel<(int)Epi::kSwiGLU, true, 0>, smem);
  }
  if (epi == Epi::kF32) return raise_smem_limit(pair_gemm_kernel<(int)Epi::kF32, false, 0>, smem);
  return raise_smem_limit(pair_gemm_kernel<(int)Epi::kBf16, false, 0>, smem);
}

cudaError_t launch_pair_gemm(const GemmPlan &p, const Launch &l) {
  PairArgs a;
  a.map_a = p.map_a;
  a.map_b = p.map_b;
  a.map_w64 = p.map_w64;
  for (int i = 0; i < 4; ++i) a.map_t[i] = p.map_t[i];
  a.x = p.gather_x;
  a.map_y = p.map_y;
  a.p2e = p.gather_p2e;
  a.x_rows = p.gather_rows;
  a.gather_k = p.gather_k;
  a.group_end = p.group_end;
  a.out = p.out;
  a.status = p.status;
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
  a.m_major = p.m_major;
  a.tail_max = p.tail_max;
  a.sched = p.sched;
  a.small_max = p.small_max;
  a.side_ctas = p.side_ctas;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  const bool gath = p.gather_k > 0 && p.epi == Epi::kSwiGLU;
  cfg.blockDim = dim3(gath ? kThreadsGather : (p.q ? kThreadsQ : kThreads));
  cfg.dynamicSmemBytes = p.smem;
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
    if (p.epi == Epi::kSwiGLU) return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<(int)Epi::kSwiGLU, false, 1>, a);
    return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<(int)Epi::kF32, false, 1>, a);
  }
  if (gath) return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<(int)Epi::kSwiGLU, true, 0>, a);
  if (p.epi == Epi::kSwiGLU) return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<(int)Epi::kSwiGLU, false, 0>, a);
  if (p.epi == Epi::kF32) return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<(int)Epi::kF32, false, 0>, a);
  return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<(int)Epi::kBf16, false, 0>, a);
}

}  // namespace moe
