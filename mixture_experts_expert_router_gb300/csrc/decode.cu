// S7: the decode regime (few tokens per expert): weight-streaming GEMMs on the
// tensor cores with the operands swapped.
//
// When an expert receives only a handful of tokens, a 128-row token tile is
// almost all padding and the layer is bound by reading each active expert's
// weights once from HBM.  Here the WEIGHT rows take the MMA's M side (128 rows)
// and the expert's tokens its N side (16, 32 or 64 columns), the "swap-AB"
// small-token forms of flashinfer.fused_moe.cake / cake_cute (Generated
// kernels, gemm1_swapab / gemm2_swapab).  Every weight byte is read once; the
// tokens' rows are re-read from L2.
//
//   FC1: D[128 x n] = [W1 up rows n0..n0+63 ; W1 gate rows n0..n0+63] . xp^T
//        h[p, n0 + r] = bf16(silu(D[64 + r, p]) * D[r, p])
//   FC2: D[128 x n] = W2 rows c0..c0+127 . h^T,  y[p, c0 + r] = D[r, p] (fp32)
//
// The k-loop runs as two half-pipelines: the even k-blocks are loaded by one
// producer thread and multiplied by one MMA thread into accumulator 0, the odd
// k-blocks by another pair into accumulator 1; the epilogue adds the two.  Each
// half owns its own half of the mbarrier ring, so every slot always passes
// between the same producer and consumer and its phase parity cannot alias
// whatever the number of k-blocks per tile.  (A weight-streaming MMA here has a tiny N, and one
// issuing thread starts a new-operand tcgen05.mma only about every 80 ns, which
// caps one thread near 50 GB/s of weights per SM; two get about twice that.)
// Two TMEM accumulator pairs alternate between tiles.  The epilogue copies its
// accumulators to registers and releases TMEM at once; for FC1 the gate half
// is handed to the up half through shared memory.
//
// In a prepared chain (sort -> gather -> FC1 -> FC2) the group offsets were
// written two kernels earlier, so a kernel started early by programmatic
// dependent launch may read them and stream its first weight tiles before it
// waits for its predecessor; it waits before touching the activations.
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

struct SwapArgs {
  CUtensorMap map_w;  // weights [G * w_rows, K] bf16, box {64, 64 (FC1) or 128 (FC2)}
  CUtensorMap map_x;  // activations [max_rows, K] bf16, box {64, BNT}
  const int32_t *group_end;
  void *out;
  int32_t *status;
  unsigned long long wait_ns;  // bounded-wait limit of this launch
  const float *clamp;         // SwiGLU epilogue: [groups] SwiGLUStep limits, or null
  long max_rows;
  int G, K, n_out, w_rows, m_tiles, early;
};

template <int BNT>
struct SwapCfg {
  static constexpr int A_BYTES = 128 * BK * 2;
  static constexpr int B_BYTES = BNT * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BNT == 64 ? 8 : 10;  // two private halves, one per half-pipeline
  static_assert(STAGES % 2 == 0, "the ring splits evenly between the half-pipelines");
  static constexpr int TILE_BYTES = STAGES * STAGE_BYTES;
  static constexpr int NBARS = 2 * STAGES + 6;
  static constexpr int BAR_OFF = TILE_BYTES;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
  static constexpr int SG_OFF = (MISC_OFF + 16 + 15) & ~15;        // gate hand-off [BNT][64] fp32
  static constexpr int TAB_OFF = SG_OFF + BNT * 64 * 4;
  static constexpr uint32_t TMEM_COLS = 4 * BNT;  // [tile buffer][half-pipeline] accumulators
  static constexpr uint32_t IDESC = idesc_bf16_f32(128, BNT);
  static size_t smem_bytes(int G) { return 1024 + TAB_OFF + (size_t)(2 * G + 2) * 4; }
};

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
  static_assert(N % 16 == 0, "16-column granules");
#pragma unroll
  for (int c = 0; c < N; c += 16) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr + (uint32_t)c));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[c + i] = __uint_as_float(r[i]);
  }
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Barrier over the four epilogue warps that also ORs a flag across them, so
// that all of them take the same branch after it.
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

struct Tile {
  int g, m, n;
};

__device__ __forceinline__ Tile decode_swap_tile(int t, const int *tile_start, const int *gend, int G,
                                                 int m_tiles) {
  int lo = 0, hi = G;  // largest g with tile_start[g] <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_start[mid] <= t) lo = mid;
    else hi = mid;
  }
  Tile c;
  c.g = lo;
  const int local = t - tile_start[lo];
  const int nt = (tile_start[lo + 1] - tile_start[lo]) / m_tiles;  // token tiles of the group
  c.m = local / nt;
  c.n = local - c.m * nt;
  return c;
}

template <int BNT, bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1) swapab_kernel(const __grid_constant__ SwapArgs args) {
  using C = SwapCfg<BNT>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_base + C::BAR_OFF;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * C::STAGES + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * C::STAGES + 2 + a); };
  auto drain_bar = [&](int q) { return bar_base + 8u * (2 * C::STAGES + 4 + q); };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
  float *sg = reinterpret_cast<float *>(smem + C::SG_OFF);
  int *tile_start = reinterpret_cast<int *>(smem + C::TAB_OFF);
  int *gend = tile_start + (args.G + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = args.G;
  const int rows_per_tile = SWIGLU ? 64 : 128;  // weight rows per TMA box

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 2);  // both MMA issuers commit
      mbar_init(tempty_bar(a), kEpiThreads);
      mbar_init(drain_bar(a), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&args.map_w);
    tma_prefetch_desc(&args.map_x);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (!args.early) pdl_wait();

  // Tile table: per group (cnt > 0) m_tiles x ceil(cnt / BNT) tiles.
  for (int g = threadIdx.x; g < G; g += kThreads) {
    long e = __ldcg(args.group_end + g);
    e = e < 0 ? 0 : (e > args.max_rows ? args.max_rows : e);
    gend[g] = (int)e;
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    if (lane == 0) tile_start[0] = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int nt = 0;
      if (g < G) {
        const int cnt = gend[g] - (g == 0 ? 0 : gend[g - 1]);
        nt = cnt > 0 ? ((cnt + BNT - 1) / BNT) * args.m_tiles : 0;
      }
      int inc = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (g < G) tile_start[g + 1] = carry + inc;
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // The next kernel of a prepared chain only needs this kernel's tile table
  // inputs to be final (they are: they were written two kernels back), so it
  // may start streaming its own weights now; it waits for this kernel to
  // finish before it reads what this kernel writes.
  pdl_launch_dependents();

  const uint32_t tmem_base = *tmem_holder;
  const int total = tile_start[G];
  const int num_kb = args.K / BK;
  // Each half-pipeline owns half of the ring (slots q * HS .. q * HS + HS - 1),
  // so a slot is only ever filled and drained by one producer / MMA pair and
  // every wait on it is for the phase right after the one it last saw.
  constexpr int HS = C::STAGES / 2;

  if ((warp == 0 || warp == kProd1Warp) && lane == 0) {
    // ------------------------------------------------------------ producers --
    // Producer q loads the k-blocks kb with kb % 2 == q of every tile.
    const int q = warp == 0 ? 0 : 1;
    const uint64_t pol_w = policy_evict_first();  // weights are read once
    const uint64_t pol_x = policy_evict_last();   // token rows are re-read
    int iq = 0;  // this pipeline's k-blocks so far: its private ring slots q * HS + iq % HS
    bool ok = true;
    // In early mode the weight boxes of the first ring's worth of k-blocks go
    // out before the wait for the predecessor; their activation boxes (listed
    // here) follow it.  Every producer flushes its list before its first wait
    // on a ring slot, so no slot waits on a k-block whose tokens are held back.
    int pend_s[C::STAGES], pend_kb[C::STAGES], pend_row[C::STAGES];
    int n_pend = 0;
    bool waited = !args.early;
    auto finish_wait = [&]() {
      pdl_wait();
      waited = true;
      for (int j = 0; j < n_pend; ++j)
        tma_load_2d(smem_base + pend_s[j] * C::STAGE_BYTES + C::A_BYTES, &args.map_x, full_bar(pend_s[j]),
                    pend_kb[j] * BK, pend_row[j], pol_x);
      n_pend = 0;
    };
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile c = decode_swap_tile(t, tile_start, gend, G, args.m_tiles);
      const int wrow = c.g * args.w_rows + c.m * rows_per_tile;
      const int xrow = (c.g == 0 ? 0 : gend[c.g - 1]) + c.n * BNT;
      for (int kb = 0; kb < num_kb; ++kb) {
        if ((kb & 1) != q) continue;
        const int s = q * HS + iq % HS;
        const uint32_t ph = (uint32_t)(iq / HS) & 1u;
        ++iq;
        if (!waited && iq > HS) finish_wait();  // this pipeline's ring is full of early loads
        if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, args.status, args.wait_ns)) {
          ok = false;
          break;
        }
        const uint32_t a_dst = smem_base + s * C::STAGE_BYTES;
        mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
        if (SWIGLU) {
          tma_load_2d(a_dst, &args.map_w, full_bar(s), kb * BK, wrow, pol_w);
          tma_load_2d(a_dst + 64 * 128, &args.map_w, full_bar(s), kb * BK, wrow + args.w_rows / 2,
                      pol_w);
        } else {
          tma_load_2d(a_dst, &args.map_w, full_bar(s), kb * BK, wrow, pol_w);
        }
        if (waited) {
          tma_load_2d(a_dst + C::A_BYTES, &args.map_x, full_bar(s), kb * BK, xrow, pol_x);
        } else {
          pend_s[n_pend] = s;
          pend_kb[n_pend] = kb;
          pend_row[n_pend] = xrow;
          ++n_pend;
        }
      }
    }
    if (!waited) finish_wait();  // fewer k-blocks in total than ring stages
    // let this pipeline's last copies land
    for (int j = iq > HS ? iq - HS : 0; j < iq; ++j)
      mbar_wait(full_bar(q * HS + j % HS), (uint32_t)(j / HS) & 1u, nullptr, args.status, args.wait_ns);
  } else if ((warp == 1 || warp == kMma1Warp) && lane == 0) {
    // ----------------------------------------------------------- MMA issuers --
    // Issuer q multiplies the k-blocks kb % 2 == q into accumulator q of the
    // tile's buffer and commits the tile once its last one is issued.
    const int q = warp == 1 ? 0 : 1;
    int iq = 0, tc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
      const int acc = tc & 1;
      const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
      if (!mbar_wait(tempty_bar(acc), aph ^ 1u, abort_flag, args.status, args.wait_ns)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)((2 * acc + q) * BNT);
      bool first = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        if ((kb & 1) != q) continue;
        const int s = q * HS + iq % HS;
        const uint32_t ph = (uint32_t)(iq / HS) & 1u;
        ++iq;
        if (!mbar_wait(full_bar(s), ph, abort_flag, args.status, args.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_base + s * C::STAGE_BYTES;
        const uint64_t a_desc = smem_desc_k_sw128(a_addr);
        const uint64_t b_desc = smem_desc_k_sw128(a_addr + C::A_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          umma_bf16(d_tmem, a_desc + 2u * k, b_desc + 2u * k, C::IDESC, (first && k == 0) ? 0u : 1u);
        first = false;
        umma_commit(empty_bar(s));
      }
      if (ok) umma_commit(tfull_bar(acc));
    }
    umma_commit(drain_bar(q));
    mbar_wait(drain_bar(q), 0, nullptr, args.status, args.wait_ns);
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------------ epilogue --
    if (args.early) pdl_wait();
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // weight row inside the tile (TMEM lane)
    int tc = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
      const Tile c = decode_swap_tile(t, tile_start, gend, G, args.m_tiles);
      const int xrow = (c.g == 0 ? 0 : gend[c.g - 1]) + c.n * BNT;
      const int valid = gend[c.g] - xrow;  // tokens of this tile (> 0)
      const int acc = tc & 1;
      const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
      const bool got = mbar_wait(tfull_bar(acc), aph, abort_flag, args.status, args.wait_ns);
      if (epi_bar_any(!got)) break;  // a wait gave up somewhere: all four warps stop together
      float v[BNT];
      tc_fence_after();
      const uint32_t lane_addr = tmem_base + ((uint32_t)(quarter * 32) << 16);
      tmem_ld_cols<BNT>(lane_addr + (uint32_t)(2 * acc * BNT), v);
      if (num_kb > 1) {  // the odd k-blocks' accumulator
        float v1[BNT];
        tmem_ld_cols<BNT>(lane_addr + (uint32_t)((2 * acc + 1) * BNT), v1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < BNT; ++j) v[j] = __fadd_rn(v[j], v1[j]);
      }
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      if (SWIGLU) {
        // the gate half (rows 64..127) hands its values to the up half
        if (r >= 64) {
#pragma unroll
          for (int j = 0; j < BNT; ++j) sg[j * 64 + (r - 64)] = v[j];
        }
        epi_bar();
        if (r < 64) {
          __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(args.out);
          const long col = (long)c.m * 64 + r;
          const float lim = step_limit(args.clamp, c.g);
#pragma unroll
          for (int j = 0; j < BNT; ++j) {
            if (j < valid) {
              const float gg = sg[j * 64 + r];
              h[(long)(xrow + j) * args.n_out + col] = __float2bfloat16_rn(swiglu_step(gg, v[j], lim));
            }
          }
        }
        epi_bar();
      } else {
        float *y = reinterpret_cast<float *>(args.out);
        const long col = (long)c.m * 128 + r;
        if (col < args.n_out) {
#pragma unroll
          for (int j = 0; j < BNT; ++j)
            if (j < valid) y[(long)(xrow + j) * args.n_out + col] = v[j];
        }
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

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

int encode(CUtensorMap *map, const void *ptr, long rows, int K, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MOE_ERR_DEVICE;
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

template <int BNT, bool SW>
size_t inst_smem(int G) {
  return SwapCfg<BNT>::smem_bytes(G);
}

template <int BNT, bool SW>
cudaError_t inst_configure(size_t smem) {
  return raise_smem_limit(swapab_kernel<BNT, SW>, smem);
}

template <int BNT, bool SW>
cudaError_t inst_launch(const SwapPlan &p, const Launch &l) {
  SwapArgs a;
  a.map_w = p.map_w;
  a.map_x = p.map_x;
  a.group_end = p.group_end;
  a.out = p.out;
  a.status = p.status;
  a.wait_ns = p.wait_ns;
  a.clamp = p.clamp;
  a.max_rows = p.max_rows;
  a.G = p.G;
  a.K = p.K;
  a.n_out = p.n_out;
  a.w_rows = p.w_rows;
  a.m_tiles = p.m_tiles;
  a.early = (p.early && l.pdl) ? 1 : 0;
  return launch_kernel(swapab_kernel<BNT, SW>, dim3(p.grid), dim3(kThreads), p.smem, l, a);
}

template <bool SW>
cudaError_t dispatch_configure(const SwapPlan &p) {
  if (p.bnt == 16) return inst_configure<16, SW>(p.smem);
  if (p.bnt == 32) return inst_configure<32, SW>(p.smem);
  return inst_configure<64, SW>(p.smem);
}

}  // namespace

int swap_prepare(SwapPlan &p, bool swiglu, const uint16_t *W, int G, int w_rows, int K,
                 const uint16_t *X, long max_rows, int n_out, const int32_t *group_end,
                 long max_group_rows, void *out, int32_t *status, bool early) {
  p = SwapPlan();
  p.swiglu = swiglu;
  p.G = G;
  p.K = K;
  p.n_out = n_out;
  p.w_rows = w_rows;
  p.group_end = group_end;
  p.max_rows = max_rows;
  p.out = out;
  p.status = status;
  p.early = early;
  p.bnt = max_group_rows <= 16 ? 16 : (max_group_rows <= 32 ? 32 : 64);
  p.m_tiles = swiglu ? n_out / 64 : (n_out + 127) / 128;
  int rc = encode(&p.map_w, W, (long)G * w_rows, K, swiglu ? 64 : 128);
  if (rc != MOE_OK) return rc;
  rc = encode(&p.map_x, X, max_rows, K, p.bnt);
  if (rc != MOE_OK) return rc;
  p.smem = p.bnt == 16 ? inst_smem<16, true>(G) : (p.bnt == 32 ? inst_smem<32, true>(G) : inst_smem<64, true>(G));
  const long groups = G < max_rows ? G : max_rows;
  const long max_tiles = (long)p.m_tiles * ((max_rows + p.bnt - 1) / p.bnt + groups);
  const long sms = device_sm_count();
  p.grid = (int)(max_tiles < sms ? (max_tiles > 0 ? max_tiles : 1) : sms);
  const cudaError_t e = swiglu ? dispatch_configure<true>(p) : dispatch_configure<false>(p);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

cudaError_t launch_swap(const SwapPlan &p, const Launch &l) {
  if (p.swiglu) {
    if (p.bnt == 16) return inst_launch<16, true>(p, l);
    if (p.bnt == 32) return inst_launch<32, true>(p, l);
    return inst_launch<64, true>(p, l);
  }
  if (p.bnt == 16) return inst_launch<16, false>(p, l);
  if (p.bnt == 32) return inst_launch<32, false>(p, l);
  return inst_launch<64, false>(p, l);
}

}  // namespace moe
