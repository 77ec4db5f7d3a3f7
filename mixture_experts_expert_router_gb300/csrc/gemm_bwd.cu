// Backward of the ragged grouped GEMM (Cake ragged BF16 grouped GEMM,
// operation table, dgrad and wgrad rows) on the 5th-generation tensor cores:
//
//   dgrad  dX[rows of g] = G[rows of g] . W[g]          W [E, N, K] in place, bf16 out
//   wgrad  dW[g] = G[rows of g]^T . X[rows of g]        fp32 or bf16 out; zeros for an empty g
//
// with the groups given by cumulative end offsets read on the device (no host
// synchronisation), fp32 accumulation in tensor memory and a fixed reduction
// order (no atomics), so replays are bitwise identical.
//
// Both products contract over a dimension that is NOT contiguous in one or
// both operands, so those operands are fed to tcgen05 "MN-major": a TMA
// SWIZZLE_128B box of 64 contiguous elements (the output dimension) by 64
// rows of the contraction dimension lands as 8-row x 128-byte swizzle atoms;
// the descriptor's leading byte offset steps between 64-element chunks of the
// output dimension (8 KB apart, one box each) and its stride byte offset
// between 8-row groups of the contraction dimension (1 KB), and the
// instruction descriptor marks the operand as transposed.
//   dgrad: A = G rows (K-major, as in the forward), B = W[g] MN-major.
//   wgrad: A = G^T and B = X, both MN-major, contracting over the group's rows.
//
// wgrad's contraction runs over the rows of one group, which start and end
// anywhere: a k-block of 64 rows that passes the group's end holds rows of
// the next group, so a masking warp zeroes those rows of both operands in
// shared memory (the whole 128-byte row: the swizzle only permutes 16-byte
// pieces inside a row) before the MMA may read the slot.  Rows past the
// tensor's end arrive as TMA zero fill.
//
// CTA (224 threads, one per SM, persistent): warp 0 TMA producer, warp 1 TMEM
// owner and MMA issuer (M = 128, N = 256, K = 16), warps 2..5 epilogue, warp 6
// the masking warp (wgrad).  Two 256-column TMEM accumulators alternate so the
// epilogue of one tile overlaps the main loop of the next.  wgrad's output
// (dW, [E, N, K], the larger part of its traffic) leaves the epilogue as
// 128-byte-wide column chunks of the tile staged in 128-byte-swizzled shared
// memory (four chunks in rotation) and written by TMA bulk stores through a
// 3-D [E, N, K] tensor map, which clips a partial tile at N instead of
// writing into the next expert's rows.  Every wait is bounded (the plan's wait limit); a timeout raises
// MOE_DEV_TIMEOUT.
#include <cuda_bf16.h>

#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;   // rows of the output tile (dX rows / dW rows)
constexpr int BN = 256;   // columns of the output tile
constexpr int BK = 64;    // contraction per k-block
constexpr int kThreads = 224;
constexpr int kEpiThreads = 128;
constexpr int kMaskWarp = 6;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB: two 8 KB chunks when MN-major
constexpr int B_BYTES = BN * BK * 2;          // 32 KB: four 8 KB chunks
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int CHUNK = 64 * BK * 2;            // one 64 x 64 box: 8 KB
constexpr int STG_BYTES = BM * 128;           // one 128-row x 128-byte staging chunk
constexpr uint32_t TMEM_COLS = 2 * BN;

enum Mode : int { kDgrad = 0, kWgradF32 = 1, kWgradBf16 = 2 };

// Shared memory per mode.  wgrad's contraction over one group is short (a few
// k-blocks per tile) and its output is the bulk of its traffic, so it trades a
// ring stage for four staging chunks: while one chunk of a tile is written
// the TMA stores of the previous three are still reading theirs.
template <int MODE>
struct BwdLayout {
  static constexpr int STAGES = MODE == kDgrad ? 4 : 3;
  static constexpr int NSTG = MODE == kDgrad ? 0 : 4;
  static constexpr int NBARS = 3 * STAGES + 5;   // full, ready, empty, tfull[2], tempty[2], drain
  static constexpr int STG_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = STG_OFF + NSTG * STG_BYTES;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base, abort flag
  static constexpr int TAB_OFF = MISC_OFF + 16;
};

struct BwdArgs {
  CUtensorMap map_a;   // dgrad: G [sum_m, N] box {64, 128}; wgrad: G [sum_m, N] box {64, 64}
  CUtensorMap map_b;   // dgrad: W [E*N, K] box {64, 64};   wgrad: X [sum_m, K] box {64, 64}
  CUtensorMap map_o;   // wgrad: dW [E, N, K] store map, box {128 bytes of K, 128, 1}
  const int32_t *group_end;
  void *out;           // dgrad: dX [sum_m, K] bf16; wgrad: dW [E, N, K]
  int32_t *status;
  unsigned long long wait_ns;
  long sum_m;
  int E, N, K;
  int n_tiles;         // column tiles: ceil(K / BN)
  int m_tiles_w;       // wgrad: row tiles of dW per group, ceil(N / BM)
};

// MN-major operand with the 128-byte swizzle: chunks of 64 elements of the
// output dimension `lbo` bytes apart, 8-row groups of the contraction 1 KB apart.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// kind::f16 instruction descriptor bits marking A / B as MN-major.
constexpr uint32_t kTransposeA = 1u << 15;
constexpr uint32_t kTransposeB = 1u << 16;

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// True on every epilogue thread when `flag` is set on any of the 128 (the
// epilogue leaves its loop together, so no named barrier waits for a thread
// that has gone).
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

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

struct Tile {
  int g, m, n;
};

// dgrad: tiles run group by group (m-tiles of 128 rows, column blocks innermost);
// wgrad: E * m_tiles_w * n_tiles tiles, every group (an empty one writes zeros).
template <int MODE>
__device__ __forceinline__ Tile decode(int t, const int *tile_start, int G, const BwdArgs &a) {
  Tile c;
  if (MODE == kDgrad) {
    int lo = 0, hi = G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tile_start[mid] * a.n_tiles <= t) lo = mid;
      else hi = mid;
    }
    c.g = lo;
    const int local = t - tile_start[lo] * a.n_tiles;
    c.m = local / a.n_tiles;
    c.n = local - c.m * a.n_tiles;
  } else {
    const int per = a.m_tiles_w * a.n_tiles;
    c.g = t / per;
    const int local = t - c.g * per;
    c.m = local / a.n_tiles;
    c.n = local - c.m * a.n_tiles;
  }
  return c;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) grouped_bwd_kernel(const __grid_constant__ BwdArgs a) {
  constexpr bool kW = MODE != kDgrad;
  using Lay = BwdLayout<MODE>;
  constexpr int STAGES = Lay::STAGES;
  constexpr int BAR_OFF = Lay::BAR_OFF, MISC_OFF = Lay::MISC_OFF, TAB_OFF = Lay::TAB_OFF;
  constexpr int NSTG = Lay::NSTG > 0 ? Lay::NSTG : 1;  // wgrad's staging chunks (dgrad has none)
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_base + BAR_OFF;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto ready_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto empty_bar = [&](int s) { return bar_base + 8u * (2 * STAGES + s); };
  auto tfull_bar = [&](int x) { return bar_base + 8u * (3 * STAGES + x); };
  auto tempty_bar = [&](int x) { return bar_base + 8u * (3 * STAGES + 2 + x); };
  const uint32_t drain_bar = bar_base + 8u * (3 * STAGES + 4);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + MISC_OFF + 4);
  const int G = a.E;
  int *gend = reinterpret_cast<int *>(smem + TAB_OFF);  // [G] clamped group ends
  int *tile_start = gend + G;                            // dgrad: [G + 1] m-tile prefix

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(ready_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(tfull_bar(x), 1);
      mbar_init(tempty_bar(x), kEpiThreads);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.map_a);
    tma_prefetch_desc(&a.map_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
    tmem_relinquish();
  }
  pdl_wait();  // the offsets and operands may come from the previous kernel

  for (int g = threadIdx.x; g < G; g += kThreads) {
    long e = a.group_end[g];
    e = e < 0 ? 0 : (e > a.sum_m ? a.sum_m : e);
    gend[g] = (int)e;
  }
  __syncthreads();
  if (!kW && warp == 0) {  // exclusive prefix of per-group m-tile counts
    int carry = 0;
    if (lane == 0) tile_start[0] = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int mt = 0;
      if (g < G) {
        const int cnt = gend[g] - (g == 0 ? 0 : gend[g - 1]);
        mt = cnt > 0 ? (cnt + BM - 1) / BM : 0;
      }
      int inc = mt;
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
  pdl_launch_dependents();

  const uint32_t tmem_base = *tmem_holder;
  const int total = kW ? G * a.m_tiles_w * a.n_tiles : tile_start[G] * a.n_tiles;
  auto gstart = [&](int g) { return g == 0 ? 0 : gend[g - 1]; };
  // k-blocks of a tile: dgrad contracts over N, wgrad over the group's rows
  auto num_kb = [&](const Tile &c) {
    return kW ? (gend[c.g] - gstart(c.g) + BK - 1) / BK : a.N / BK;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer --
      const uint64_t pol = policy_evict_normal();
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile c = decode<MODE>(t, tile_start, G, a);
        const int nk = num_kb(c);
        const int col0 = c.n * BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, a.status, a.wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = smem_base + s * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          mbar_arrive_expect_tx(full_bar(s), STAGE_BYTES);
          if (kW) {
            const int r0 = gstart(c.g) + kb * BK;
            const int m0 = c.m * BM;
            tma_load_2d(a_dst, &a.map_a, full_bar(s), m0, r0, pol);
            tma_load_2d(a_dst + CHUNK, &a.map_a, full_bar(s), m0 + 64, r0, pol);
#pragma unroll
            for (int q = 0; q < 4; ++q) tma_load_2d(b_dst + q * CHUNK, &a.map_b, full_bar(s), col0 + 64 * q, r0, pol);
          } else {
            const int row0 = gstart(c.g) + c.m * BM;
            tma_load_2d(a_dst, &a.map_a, full_bar(s), kb * BK, row0, pol);
            const int wrow = c.g * a.N + kb * BK;
#pragma unroll
            for (int q = 0; q < 4; ++q) tma_load_2d(b_dst + q * CHUNK, &a.map_b, full_bar(s), col0 + 64 * q, wrow, pol);
          }
        }
      }
      // every copy this thread started lands before the CTA may exit
      for (int j = it > STAGES ? it - STAGES : 0; j < it; ++j)
        mbar_wait(full_bar(j % STAGES), (uint32_t)(j / STAGES) & 1u, nullptr, a.status, a.wait_ns);
    }
  } else if (warp == kMaskWarp) {
    // ------------------------------------------------- masking (wgrad only) --
    // Passes every slot on from "full" to "ready"; in a group's last k-block
    // it first zeroes the rows at and past the group's end in all six chunks.
    if (kW) {
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile c = decode<MODE>(t, tile_start, G, a);
        const int nk = num_kb(c);
        const int rows = gend[c.g] - gstart(c.g);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          int w_ok = 1;
          if (lane == 0) w_ok = mbar_wait(full_bar(s), ph, abort_flag, a.status, a.wait_ns) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
            ok = false;
            break;
          }
          const int valid = rows - kb * BK;  // > 0
          if (valid < BK) {
            unsigned char *st = smem + s * STAGE_BYTES;
            const int n16 = (BK - valid) * 8;  // 16-byte pieces per chunk to clear
            for (int ch = 0; ch < 6; ++ch) {
              uint4 *base = reinterpret_cast<uint4 *>(st + ch * CHUNK + valid * 128);
              for (int x = lane; x < n16; x += 32) base[x] = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();  // the MMA reads shared memory through the async proxy
            __syncwarp();
          }
          if (lane == 0) mbar_arrive(ready_bar(s));
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer --
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN) | kTransposeB | (kW ? kTransposeA : 0u);
      int it = 0, tc = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
        const Tile c = decode<MODE>(t, tile_start, G, a);
        const int nk = num_kb(c);
        const int acc = tc & 1;
        const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
        if (!mbar_wait(tempty_bar(acc), aph ^ 1u, abort_flag, a.status, a.wait_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait(kW ? ready_bar(s) : full_bar(s), ph, abort_flag, a.status, a.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_base + s * STAGE_BYTES;
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {  // K = 16 per MMA
            const uint64_t ad = kW ? smem_desc_mn_sw128(a_addr + 2048u * k, CHUNK)
                                   : smem_desc_k_sw128(a_addr) + 2u * k;
            const uint64_t bd = smem_desc_mn_sw128(b_addr + 2048u * k, CHUNK);
            umma_bf16(d_tmem, ad, bd, IDESC, (kb | k) != 0);
          }
          umma_commit(empty_bar(s));
        }
        if (ok) umma_commit(tfull_bar(acc));
      }
      umma_commit(drain_bar);  // every MMA done before TMEM is released
      mbar_wait(drain_bar, 0, nullptr, a.status, a.wait_ns);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------------ epilogue --
    const int quarter = warp & 3;
    const int r_in_tile = quarter * 32 + lane;
    int tc = 0;
    int n_stg = 0;  // wgrad: staging chunks used so far (the ring position)
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
      const Tile c = decode<MODE>(t, tile_start, G, a);
      const int acc = tc & 1;
      const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
      const bool got = mbar_wait(tfull_bar(acc), aph, abort_flag, a.status, a.wait_ns);
      if (epi_bar_any(!got)) break;  // all four warps stop together
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      const int col0 = c.n * BN;
      if (!kW) {
        const int row0 = gstart(c.g) + c.m * BM;
        const bool row_ok = r_in_tile < gend[c.g] - row0;
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) +
                                               (long)(row0 + r_in_tile) * a.K + col0);
#pragma unroll 1
        for (int col = 0; col < BN; col += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + col, r);
          tmem_ld_wait();
          if (row_ok && col0 + col < a.K) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[col / 8 + v] = make_uint4(pack2(__uint_as_float(r[8 * v]), __uint_as_float(r[8 * v + 1])),
                                            pack2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                                            pack2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                                            pack2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
          }
        }
      } else {
        // dW[g] rows c.m * BM .., columns col0 ..: 128-byte column chunks
        // (32 fp32 or 64 bf16) staged swizzled, then one TMA store each
        constexpr int CW = MODE == kWgradF32 ? 32 : 64;  // columns per chunk
        const bool empty = gend[c.g] <= gstart(c.g);
        const int etid = threadIdx.x - 64;
#pragma unroll 1
        for (int col = 0; col < BN && col0 + col < a.K; col += CW, ++n_stg) {
          const uint32_t stg = smem_base + Lay::STG_OFF + (uint32_t)((n_stg % NSTG) * STG_BYTES);
          const uint32_t row_addr = stg + r_in_tile * 128;
          uint32_t v[32];  // this row's 128 bytes of the chunk
          if (empty) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0u;  // +0.0
          } else if (MODE == kWgradF32) {
            tmem_ld_32x32b_x32(taddr + col, v);
            tmem_ld_wait();
          } else {
            uint32_t r0[32], r1[32];
            tmem_ld_32x32b_x32(taddr + col, r0);
            tmem_ld_32x32b_x32(taddr + col + 32, r1);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              v[j] = pack2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1]));
              v[16 + j] = pack2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1]));
            }
          }
          // the store that used this staging chunk NSTG chunks ago has read it
          if (etid == 0) bulk_wait_read<NSTG - 1>();
          epi_bar();
#pragma unroll
          for (int q = 0; q < 8; ++q)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             row_addr + (uint32_t)((q ^ (r_in_tile & 7)) * 16)),
                         "r"(v[4 * q]), "r"(v[4 * q + 1]), "r"(v[4 * q + 2]), "r"(v[4 * q + 3])
                         : "memory");
          fence_proxy_async_smem();
          epi_bar();
          if (etid == 0) {
            tma_store_3d(&a.map_o, stg, col0 + col, c.m * BM, c.g);
            bulk_commit();
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
    }
  }

  if (kW && threadIdx.x == 64) bulk_wait_all();  // the last stores are done before the CTA exits
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// bf16 [rows, cols] row-major, box {64, box_rows}, 128-byte swizzle, zero fill.
int encode(CUtensorMap *map, const void *ptr, long rows, int cols, int box_rows) {
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
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_TENSOR_MAP;
}

// dW [E, N, K] (fp32 or bf16) as a 3-D store map: box {128 bytes of K, 128 rows, 1 expert}.
int encode_dw(CUtensorMap *map, void *ptr, int E, int N, int K, bool f32) {
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
  const int esz = f32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)N, (cuuint64_t)E};
  cuuint64_t strides[2] = {(cuuint64_t)K * esz, (cuuint64_t)N * K * esz};
  cuuint32_t box[3] = {(cuuint32_t)(128 / esz), (cuuint32_t)BM, 1u};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_TENSOR_MAP;
}

template <int MODE>
cudaError_t launch_mode(const BwdPlan &p, const Launch &l) {
  BwdArgs a;
  a.map_a = p.map_a;
  a.map_b = p.map_b;
  a.map_o = p.map_o;
  a.group_end = p.group_end;
  a.out = p.out;
  a.status = p.status;
  a.wait_ns = p.wait_ns;
  a.sum_m = p.sum_m;
  a.E = p.E;
  a.N = p.N;
  a.K = p.K;
  a.n_tiles = (p.K + BN - 1) / BN;
  a.m_tiles_w = (p.N + BM - 1) / BM;
  return launch_kernel(grouped_bwd_kernel<MODE>, dim3(p.grid), dim3(kThreads), p.smem, l, a);
}

}  // namespace

int bwd_prepare(BwdPlan &p, bool wgrad, bool out_f32, const uint16_t *G, const uint16_t *B, const int32_t *offs,
                long sum_m, int E, int N, int K, void *out, int32_t *status) {
  if (sum_m < 0 || E < 1 || E > MOE_MAX_EXPERTS || N <= 0 || K <= 0 || N % 64 || K % 64) return MOE_ERR_SHAPE;
  p = BwdPlan();
  p.mode = wgrad ? (out_f32 ? kWgradF32 : kWgradBf16) : kDgrad;
  p.group_end = offs;
  p.out = out;
  p.status = status;
  p.sum_m = sum_m;
  p.E = E;
  p.N = N;
  p.K = K;
  int rc;
  if (wgrad) {
    rc = encode(&p.map_a, G, sum_m, N, 64);            // G^T: boxes of 64 dW rows x 64 group rows
    if (rc == MOE_OK) rc = encode(&p.map_b, B, sum_m, K, 64);  // X
    if (rc == MOE_OK) rc = encode_dw(&p.map_o, out, E, N, K, out_f32);
  } else {
    rc = encode(&p.map_a, G, sum_m, N, BM);             // G rows, K-major
    if (rc == MOE_OK) rc = encode(&p.map_b, B, (long)E * N, K, 64);  // W in place
  }
  if (rc != MOE_OK) return rc;
  const int tab_off = wgrad ? BwdLayout<kWgradF32>::TAB_OFF : BwdLayout<kDgrad>::TAB_OFF;
  p.smem = 1024 + tab_off + (size_t)(2 * E + 2) * 4;
  const long n_tiles = (K + BN - 1) / BN;
  const long tiles = wgrad ? (long)E * ((N + BM - 1) / BM) * n_tiles
                           : ((sum_m + BM - 1) / BM + E) * n_tiles;
  const long sms = device_sm_count();
  p.grid = (int)(tiles < sms ? (tiles > 0 ? tiles : 1) : sms);
  cudaError_t e = cudaSuccess;
  switch (p.mode) {
    case kDgrad: e = raise_smem_limit(grouped_bwd_kernel<kDgrad>, p.smem); break;
    case kWgradF32: e = raise_smem_limit(grouped_bwd_kernel<kWgradF32>, p.smem); break;
    default: e = raise_smem_limit(grouped_bwd_kernel<kWgradBf16>, p.smem); break;
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

cudaError_t launch_bwd(const BwdPlan &p, const Launch &l) {
  switch (p.mode) {
    case kDgrad: return launch_mode<kDgrad>(p, l);
    case kWgradF32: return launch_mode<kWgradF32>(p, l);
    default: return launch_mode<kWgradBf16>(p, l);
  }
}

}  // namespace moe
