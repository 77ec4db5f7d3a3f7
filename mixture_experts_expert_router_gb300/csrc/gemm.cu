// S4 / S5 / S8: persistent ragged grouped GEMM on the 5th-generation tensor
// cores (tcgen05), fed by TMA through a shared-memory ring, accumulating in
// tensor memory (TMEM).
//
//   Y[rows of group g] = A[rows of group g] . B[g]^T          (fp32 accumulate)
//
// Groups are consecutive row ranges given by cumulative end offsets that the
// kernel reads on the device (Cake ragged BF16 grouped GEMM, operation table):
// no host synchronisation, no padding, empty groups and ragged tails allowed.
// Three epilogues share the main loop:
//   kBf16   - Y rounded to bf16 (the grouped GEMM forward);
//   kSwiGLU - B tile = [up rows | gate rows] of W1; h = bf16(silu(g) * u)
//             (GEMM1 with the SwiGLU fused, cute_dsl_fused_moe_bf16,
//             Supported configuration);
//   kF32    - Y stored as fp32, unrounded (GEMM2 of the deterministic path).
// With Q = 1 the operands are E4M3 codes (the fp8 per-tensor weight family of
// flashinfer.experimental.cake_stepfun_moe, opening paragraph): a k-block is
// 128 codes (still one 128-byte swizzled row), the MMA is kind::f8f6f4 with
// K = 32, the accumulator is dequantised by ascale * wscale[group], and the
// SwiGLU epilogue writes E4M3 h = e4m3(h * RN(1 / oscale)) (the
// requantisation between FC1 and FC2; the product is within one fp32 ulp of
// the quotient h / oscale).
//
// CTA organisation (192 threads, one CTA per SM, persistent):
//   warp 0      TMA producer: one thread streams A and B k-blocks into a
//               STAGES-deep ring, signalling "full" mbarriers;
//   warp 1      owns the TMEM allocation; one thread issues tcgen05.mma
//               (M=128, N=BN, K=16) and commits to "empty" (frees a ring slot)
//               and "tmem_full" (a finished accumulator);
//   warps 2..5  epilogue: TMEM -> registers (tcgen05.ld, one row per thread)
//               -> activation -> global stores; then "tmem_empty".
// Two TMEM accumulators of BN fp32 columns alternate between tiles, so the
// epilogue of one tile overlaps the main loop of the next.
//
// Tiles: 128 rows of one group x one column block.  Tile order is group-major;
// inside a group either the m-tiles or the column blocks run innermost,
// whichever keeps the re-read operand in L2 (chosen on the host from shapes).
//
// Shared memory tiles use the 128-byte swizzle that TMA writes and the MMA
// descriptors read: each k-block is 64 bf16 (128 bytes) wide.
#include <cuda_bf16.h>

#include <cstdio>

#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;

struct GemmArgs {
  CUtensorMap map_a;
  CUtensorMap map_b;
  const int32_t *group_end;
  void *out;
  int32_t *status;
  unsigned long long wait_ns;  // bounded-wait limit of this launch
  const float *clamp;         // SwiGLU epilogue: [groups] SwiGLUStep limits, or null
  const float *wscale;        // E4M3: [groups] weight scales
  float ascale, oscale;       // E4M3: activation scale of A, requantisation scale of h
  long max_rows;
  int G;
  int K;
  int n_out;
  int b_rows;
  int n_tiles;
  int m_major;
};

template <int BN>
struct Cfg {
  static constexpr int STAGES = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TILE_BYTES = STAGES * STAGE_BYTES;
  static constexpr int NBARS = 2 * STAGES + 5;  // full, empty, tfull[2], tempty[2], drain
  static constexpr int BAR_OFF = TILE_BYTES;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base, abort flag
  static constexpr int TAB_OFF = MISC_OFF + 16;
  static constexpr uint32_t TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
  static size_t smem_bytes(int G) { return 1024 + TAB_OFF + (size_t)(2 * G + 2) * 4; }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// Which (group, m-tile, column block) tile number t is.
struct TileCoord {
  int g, m, n;
};

__device__ __forceinline__ TileCoord decode_tile(int t, const int *tile_start, int G, int n_tiles,
                                                 int m_major) {
  int lo = 0, hi = G;  // largest g with tile_start[g] * n_tiles <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_start[mid] * n_tiles <= t) lo = mid;
    else hi = mid;
  }
  TileCoord c;
  c.g = lo;
  const int mt = tile_start[lo + 1] - tile_start[lo];
  const int local = t - tile_start[lo] * n_tiles;
  if (m_major) {
    c.m = local / n_tiles;
    c.n = local - c.m * n_tiles;
  } else {
    c.n = local / mt;
    c.m = local - c.n * mt;
  }
  return c;
}

template <int BN, int EPI, int Q>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmArgs args) {
  using C = Cfg<BN>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_base + C::BAR_OFF;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * C::STAGES + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * C::STAGES + 2 + a); };
  const uint32_t drain_bar = bar_base + 8u * (2 * C::STAGES + 4);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
  int *tile_start = reinterpret_cast<int *>(smem + C::TAB_OFF);  // [G+1]
  int *gend = tile_start + (args.G + 1);                          // [G] clamped ends

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = args.G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kEpiThreads);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&args.map_a);
    tma_prefetch_desc(&args.map_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
    tmem_relinquish();
  }

  // Everything below reads what the previous kernel wrote.
  pdl_wait();

  for (int g = threadIdx.x; g < G; g += kThreads) {
    long e = args.group_end[g];
    e = e < 0 ? 0 : (e > args.max_rows ? args.max_rows : e);
    gend[g] = (int)e;
  }
  __syncthreads();
  if (warp == 0) {  // tile_start = exclusive prefix of per-group m-tile counts
    int carry = 0;
    if (lane == 0) tile_start[0] = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int mt = 0;
      if (g < G) {
        const int start = g == 0 ? 0 : gend[g - 1];
        const int cnt = gend[g] - start;
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
  const int total = tile_start[G] * args.n_tiles;
  constexpr int KB = Q ? 128 : BK;  // elements per k-block (128 bytes either way)
  const int num_kb = args.K / KB;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer --
      const uint64_t pol = policy_evict_normal();
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileCoord c = decode_tile(t, tile_start, G, args.n_tiles, args.m_major);
        const int row0 = (c.g == 0 ? 0 : gend[c.g - 1]) + c.m * BM;
        int brow0, brow1 = 0;
        if (EPI == (int)Epi::kSwiGLU) {
          brow0 = c.g * args.b_rows + c.n * (BN / 2);  // up rows
          brow1 = brow0 + args.b_rows / 2;             // matching gate rows
        } else {
          brow0 = c.g * args.b_rows + c.n * BN;
        }
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, args.status, args.wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = smem_base + s * C::STAGE_BYTES;
          const uint32_t b_dst = a_dst + C::A_BYTES;
          mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
          tma_load_2d(a_dst, &args.map_a, full_bar(s), kb * KB, row0, pol);
          if (EPI == (int)Epi::kSwiGLU) {
            tma_load_2d(b_dst, &args.map_b, full_bar(s), kb * KB, brow0, pol);
            tma_load_2d(b_dst + (BN / 2) * 128, &args.map_b, full_bar(s), kb * KB, brow1, pol);
          } else {
            tma_load_2d(b_dst, &args.map_b, full_bar(s), kb * KB, brow0, pol);
          }
        }
      }
      // Let every copy this thread started land before the CTA can exit.
      for (int j = it > C::STAGES ? it - C::STAGES : 0; j < it; ++j)
        mbar_wait(full_bar(j % C::STAGES), (uint32_t)(j / C::STAGES) & 1u, nullptr, args.status, args.wait_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer --
      int it = 0, tc = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
        const int acc = tc & 1;
        const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
        if (!mbar_wait(tempty_bar(acc), aph ^ 1u, abort_flag, args.status, args.wait_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
          if (!mbar_wait(full_bar(s), ph, abort_flag, args.status, args.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_base + s * C::STAGE_BYTES;
          const uint64_t a_desc = smem_desc_k_sw128(a_addr);
          const uint64_t b_desc = smem_desc_k_sw128(a_addr + C::A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)  // K = 16 per MMA: +32 bytes in the swizzled row
            if (Q)  // K = 32 E4M3 codes per MMA: the same 32 bytes of the swizzled row
              umma_e4m3(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc_e4m3_f32(BM, BN), (kb | k) != 0);
            else
              umma_bf16(d_tmem, a_desc + 2u * k, b_desc + 2u * k, C::IDESC, (kb | k) != 0);
          umma_commit(empty_bar(s));
        }
        if (ok) umma_commit(tfull_bar(acc));
      }
      // Wait for every MMA this thread issued before TMEM can be released.
      umma_commit(drain_bar);
      mbar_wait(drain_bar, 0, nullptr, args.status, args.wait_ns);
    }
  } else {
    // ------------------------------------------------------------------ epilogue --
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    const int r_in_tile = quarter * 32 + lane;
    int tc = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
      const TileCoord c = decode_tile(t, tile_start, G, args.n_tiles, args.m_major);
      const int row0 = (c.g == 0 ? 0 : gend[c.g - 1]) + c.m * BM;
      const int valid = gend[c.g] - row0;
      const int acc = tc & 1;
      const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
      if (!mbar_wait(tfull_bar(acc), aph, abort_flag, args.status, args.wait_ns)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      const bool row_ok = r_in_tile < valid;
      const long orow = (long)row0 + r_in_tile;
      if (Q && EPI == (int)Epi::kSwiGLU) {
        // E4M3: u, g dequantised by ascale * wscale[g], SwiGLU(Step), h requantised
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(args.out) +
                                               orow * args.n_out + (long)c.n * (BN / 2));
        const float lim = step_limit(args.clamp, c.g);
        const float sc = __fmul_rn(args.ascale, __ldg(args.wscale + c.g));
        const float inv = __frcp_rn(args.oscale);  // h / h_scale as h times RN(1 / h_scale)
#pragma unroll 1
        for (int col = 0; col < BN / 2; col += 32) {
          uint32_t u[32], g[32];
          tmem_ld_32x32b_x32(taddr + col, u);
          tmem_ld_32x32b_x32(taddr + BN / 2 + col, g);
          tmem_ld_wait();
          uint32_t packed[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float hv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float uu = __fmul_rn(__uint_as_float(u[4 * i + q]), sc);
              const float gg = __fmul_rn(__uint_as_float(g[4 * i + q]), sc);
              hv[q] = __fmul_rn(swiglu_step(gg, uu, lim), inv);
            }
            packed[i] = e4m3x2(hv[0], hv[1]) | (e4m3x2(hv[2], hv[3]) << 16);
          }
          if (row_ok) {
            dst[col / 16] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[col / 16 + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
          }
        }
      } else if (Q && EPI == (int)Epi::kF32) {
        // E4M3: y dequantised by ascale * wscale[g]
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<float *>(args.out) +
                                               orow * args.n_out + (long)c.n * BN);
        const float sc = __fmul_rn(args.ascale, __ldg(args.wscale + c.g));
#pragma unroll 1
        for (int col = 0; col < BN; col += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + col, r);
          tmem_ld_wait();
          if (row_ok) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[col / 4 + v] = make_uint4(__float_as_uint(__fmul_rn(__uint_as_float(r[4 * v]), sc)),
                                            __float_as_uint(__fmul_rn(__uint_as_float(r[4 * v + 1]), sc)),
                                            __float_as_uint(__fmul_rn(__uint_as_float(r[4 * v + 2]), sc)),
                                            __float_as_uint(__fmul_rn(__uint_as_float(r[4 * v + 3]), sc)));
          }
        }
      } else if (EPI == (int)Epi::kSwiGLU) {
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
          for (int i = 0; i < 16; ++i) {
            float hv[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const float uu = __uint_as_float(u[2 * i + q]);
              const float gg = __uint_as_float(g[2 * i + q]);
              hv[q] = swiglu_step(gg, uu, lim);
            }
            packed[i] = pack_bf16x2(hv[0], hv[1]);
          }
          if (row_ok) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[col / 8 + v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                            packed[4 * v + 3]);
          }
        }
      } else if (EPI == (int)Epi::kF32) {
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<float *>(args.out) +
                                               orow * args.n_out + (long)c.n * BN);
#pragma unroll 1
        for (int col = 0; col < BN; col += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + col, r);
          tmem_ld_wait();
          if (row_ok) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[col / 4 + v] = make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
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
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side --
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

// 2-D bf16 tensor [rows, K] (row stride K elements), box {64, box_rows},
// 128-byte swizzle, out-of-bounds elements read as zero.
int encode_2d(CUtensorMap *map, const void *ptr, long rows, int K, int box_rows) {
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

template <int BN, int EPI, int Q = 0>
cudaError_t configure_inst(const GemmPlan &p) {
  return raise_smem_limit(grouped_gemm_kernel<BN, EPI, Q>, p.smem);
}

template <int BN, int EPI, int Q = 0>
cudaError_t launch_inst(const GemmPlan &p, const Launch &l) {
  auto kern = grouped_gemm_kernel<BN, EPI, Q>;
  GemmArgs a;
  a.map_a = p.map_a;
  a.map_b = p.map_b;
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
  return launch_kernel(kern, dim3(p.grid), dim3(kThreads), p.smem, l, a);
}

}  // namespace

static cudaError_t configure_gemm(const GemmPlan &p);

int gemm_prepare(GemmPlan &p, Epi epi, const uint16_t *A, long a_rows, const uint16_t *B, int G,
                 int b_rows, int K, int n_out, const int32_t *group_end, long max_rows, void *out,
                 int32_t *status, bool allow_pair) {
  p = GemmPlan();
  p.epi = epi;
  p.G = G;
  p.K = K;
  p.n_out = n_out;
  p.b_rows = b_rows;
  p.group_end = group_end;
  p.max_rows = max_rows;
  p.out = out;
  p.status = status;
  int box_b;
  if (epi == Epi::kSwiGLU) {
    const int half = (n_out % 128 == 0) ? 128 : 64;
    p.bn = 2 * half;
    p.n_tiles = n_out / half;
    box_b = half;
  } else {
    p.bn = (n_out % 256 == 0) ? 256 : ((n_out % 128 == 0) ? 128 : 64);
    p.n_tiles = n_out / p.bn;
    box_b = p.bn;
  }
  p.pair = (allow_pair && pair_gemm_supported(epi, n_out)) ? 1 : 0;
  if (p.pair) {  // each CTA of the pair stages 128 of the 256 B rows
    p.bn = 256;
    p.n_tiles = epi == Epi::kSwiGLU ? n_out / 128 : n_out / 256;
    box_b = 128;
  }
  int rc = encode_2d(&p.map_a, A, a_rows, K, BM);
  if (rc != MOE_OK) return rc;
  rc = encode_2d(&p.map_b, B, (long)G * b_rows, K, box_b);
  if (rc != MOE_OK) return rc;
  if (p.pair) {
    rc = pair_gemm_encode_extra(p, A, a_rows, B, (long)G * b_rows, K);
    if (rc != MOE_OK) return rc;
  }
  // Keep the operand that the inner tile loop re-reads in L2: when one
  // group's weights fit comfortably, run column blocks innermost (m-major).
  const double b_group_bytes = (double)b_rows * K * 2.0;
  p.m_major = b_group_bytes <= 64.0 * 1024 * 1024 ? 1 : 0;
  switch (p.bn) {
    case 256: p.smem = Cfg<256>::smem_bytes(G); break;
    case 128: p.smem = Cfg<128>::smem_bytes(G); break;
    default: p.smem = Cfg<64>::smem_bytes(G); break;
  }
  const long sms = device_sm_count();
  if (p.pair) {
    p.smem = pair_gemm_smem(epi, G);
    const long max_pairs = ((max_rows + 2 * BM - 1) / (2 * BM) + G) * (long)p.n_tiles;
    const long clusters = sms / 2;
    p.grid = 2 * (int)(max_pairs < clusters ? (max_pairs > 0 ? max_pairs : 1) : clusters);
    return pair_gemm_configure(epi, p.smem) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  const long max_tiles = ((max_rows + BM - 1) / BM + G) * (long)p.n_tiles;
  p.grid = (int)(max_tiles < sms ? (max_tiles > 0 ? max_tiles : 1) : sms);
  return configure_gemm(p) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Raise the kernel's dynamic shared-memory limit (host, outside any capture).
static cudaError_t configure_gemm(const GemmPlan &p) {
  if (p.epi == Epi::kSwiGLU) {
    if (p.bn == 256) return configure_inst<256, (int)Epi::kSwiGLU>(p);
    return configure_inst<128, (int)Epi::kSwiGLU>(p);
  }
  if (p.epi == Epi::kF32) {
    if (p.bn == 256) return configure_inst<256, (int)Epi::kF32>(p);
    if (p.bn == 128) return configure_inst<128, (int)Epi::kF32>(p);
    return configure_inst<64, (int)Epi::kF32>(p);
  }
  if (p.bn == 256) return configure_inst<256, (int)Epi::kBf16>(p);
  if (p.bn == 128) return configure_inst<128, (int)Epi::kBf16>(p);
  return configure_inst<64, (int)Epi::kBf16>(p);
}

// uint8 [rows, K] (E4M3 codes), box {128, box_rows}, 128-byte swizzle, zero fill.
static int encode_2d_u8(CUtensorMap *map, const void *ptr, long rows, int K, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MOE_ERR_DEVICE;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_TENSOR_MAP;
}

int gemm_prepare_e4m3(GemmPlan &p, Epi epi, const uint8_t *A, long a_rows, const uint8_t *B, int G,
                      int b_rows, int K, int n_out, const int32_t *group_end, long max_rows,
                      void *out, int32_t *status, bool allow_pair) {
  if (K % 128 != 0 || epi == Epi::kBf16) return MOE_ERR_SHAPE;
  p = GemmPlan();
  p.q = 1;
  p.epi = epi;
  p.G = G;
  p.K = K;
  p.n_out = n_out;
  p.b_rows = b_rows;
  p.group_end = group_end;
  p.max_rows = max_rows;
  p.out = out;
  p.status = status;
  int box_b;
  if (epi == Epi::kSwiGLU) {
    if (n_out % 128 != 0) return MOE_ERR_SHAPE;  // 32 h codes per epilogue step, 128 per tile half
    p.bn = 256;
    p.n_tiles = n_out / 128;
    box_b = 128;
  } else {
    p.bn = (n_out % 256 == 0) ? 256 : ((n_out % 128 == 0) ? 128 : 64);
    p.n_tiles = n_out / p.bn;
    box_b = p.bn;
  }
  const double b_group_bytes = (double)b_rows * K;
  p.m_major = b_group_bytes <= 64.0 * 1024 * 1024 ? 1 : 0;
  const long sms = device_sm_count();
  if (allow_pair && pair_gemm_supported(epi, n_out)) {  // CTA pairs: 128 of the 256 B rows per CTA
    p.pair = 1;
    p.bn = 256;
    p.n_tiles = epi == Epi::kSwiGLU ? n_out / 128 : n_out / 256;
    if (int rc = pair_gemm_encode_u8(p, A, a_rows, B, (long)G * b_rows, K)) return rc;
    p.smem = pair_gemm_smem(epi, G);
    const long max_pairs = ((max_rows + 2 * BM - 1) / (2 * BM) + G) * (long)p.n_tiles;
    const long clusters = sms / 2;
    p.grid = 2 * (int)(max_pairs < clusters ? (max_pairs > 0 ? max_pairs : 1) : clusters);
    return pair_gemm_configure(epi, p.smem, 1) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  int rc = encode_2d_u8(&p.map_a, A, a_rows, K, BM);
  if (rc == MOE_OK) rc = encode_2d_u8(&p.map_b, B, (long)G * b_rows, K, box_b);
  if (rc != MOE_OK) return rc;
  switch (p.bn) {
    case 256: p.smem = Cfg<256>::smem_bytes(G); break;
    case 128: p.smem = Cfg<128>::smem_bytes(G); break;
    default: p.smem = Cfg<64>::smem_bytes(G); break;
  }
  const long max_tiles = ((max_rows + BM - 1) / BM + G) * (long)p.n_tiles;
  p.grid = (int)(max_tiles < sms ? (max_tiles > 0 ? max_tiles : 1) : sms);
  cudaError_t e;
  if (epi == Epi::kSwiGLU) e = configure_inst<256, (int)Epi::kSwiGLU, 1>(p);
  else if (p.bn == 256) e = configure_inst<256, (int)Epi::kF32, 1>(p);
  else if (p.bn == 128) e = configure_inst<128, (int)Epi::kF32, 1>(p);
  else e = configure_inst<64, (int)Epi::kF32, 1>(p);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int gemm_prepare_gather(GemmPlan &p, const uint16_t *x, long x_rows, const int32_t *p2e, int k,
                        const uint16_t *W1, int G, int I, int H, const int32_t *group_end,
                        long max_rows, void *h, int32_t *status) {
  if (!pair_gemm_supported(Epi::kSwiGLU, I) || k < 1) return MOE_ERR_SHAPE;
  // the direct-row maps still need a valid base: point them at x
  int rc = gemm_prepare(p, Epi::kSwiGLU, x, x_rows, W1, G, 2 * I, H, I, group_end, max_rows, h,
                        status, true);
  if (rc != MOE_OK) return rc;
  p.gather_x = x;
  p.gather_p2e = p2e;
  p.gather_rows = x_rows;
  p.gather_k = k;
  return pair_gemm_encode_extra(p, x, x_rows, W1, (long)G * 2 * I, H);
}

int gemm_attach_small(GemmPlan &p, int32_t *sched, int ctas) {
  if (!p.pair || p.gather_k > 0 || (p.q && p.epi == Epi::kBf16) || !sched || ctas < 2 || ctas % 2 ||
      p.tail_max < small_gemm_max_rows())
    return MOE_ERR_SHAPE;
  p.sched = sched;
  p.side_ctas = ctas;
  p.small_max = small_gemm_max_rows();
  return small_gemm_configure(p.epi, p.q, small_gemm_smem(p.G)) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

cudaError_t launch_gemm(const GemmPlan &p, const Launch &l) {
  if (p.pair && p.side_ctas > 0) {
    // The small-group kernel first: the pair kernel launches once all of its
    // CTAs are running (they signal dependents at once), so both hold SMs
    // together; the pair kernel starts on that kernel's flag, not on a
    // dependent-launch wait.
    if (cudaError_t e = launch_small_gemm(p, l)) return e;
    Launch behind = l;
    behind.pdl = true;
    return launch_pair_gemm(p, behind);
  }
  if (p.pair) return launch_pair_gemm(p, l);
  if (p.q) {
    if (p.epi == Epi::kSwiGLU)
      return p.bn == 256 ? launch_inst<256, (int)Epi::kSwiGLU, 1>(p, l) : launch_inst<128, (int)Epi::kSwiGLU, 1>(p, l);
    if (p.bn == 256) return launch_inst<256, (int)Epi::kF32, 1>(p, l);
    if (p.bn == 128) return launch_inst<128, (int)Epi::kF32, 1>(p, l);
    return launch_inst<64, (int)Epi::kF32, 1>(p, l);
  }
  if (p.epi == Epi::kSwiGLU) {
    if (p.bn == 256) return launch_inst<256, (int)Epi::kSwiGLU>(p, l);
    return launch_inst<128, (int)Epi::kSwiGLU>(p, l);
  }
  if (p.epi == Epi::kF32) {
    if (p.bn == 256) return launch_inst<256, (int)Epi::kF32>(p, l);
    if (p.bn == 128) return launch_inst<128, (int)Epi::kF32>(p, l);
    return launch_inst<64, (int)Epi::kF32>(p, l);
  }
  if (p.bn == 256) return launch_inst<256, (int)Epi::kBf16>(p, l);
  if (p.bn == 128) return launch_inst<128, (int)Epi::kBf16>(p, l);
  return launch_inst<64, (int)Epi::kBf16>(p, l);
}

}  // namespace moe
