// S3 gather and S6 finalize: the two row-copy / row-combine passes around the
// grouped GEMMs.  Both are HBM-bound streams of 16-byte vector accesses.
//
// Gather builds the expanded per-route activations (one row per (token, slot)
// in expert order) that GEMM1 reads: either row by row through perm_to_exp
// (moe_gather, the decode path) or token by token through exp_to_perm, which
// reads each token row of x once for all its routes (the grouped path).  Finalize is the deterministic combine of
// flashinfer.fused_moe.cute_dsl_fused_moe_bf16 (Parameters,
// use_fused_finalize=False): each output row has one owner that sums its
// top_k unscaled GEMM2 rows, scaled by the routing weights, in fp32 in
// ascending slot order, then rounds once to bf16.  No atomics.
#include <cuda_bf16.h>

#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256)
    gather_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ p2e,
                  const int32_t *__restrict__ m_total, int vec, int k, uint4 *__restrict__ xp) {
  pdl_wait();
  const long M = *m_total;
  const int lane = threadIdx.x & 31;
  const long warp = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
  pdl_launch_dependents();
  for (long p = warp; p < M; p += nwarps) {
    const long t = p2e[p] / k;
    const uint4 *src = x + t * vec;
    uint4 *dst = xp + p * vec;
    int i = lane;
    // eight 16-byte loads in flight per lane; xp is written once and read by
    // the next kernel, so the stores stream past L1
    for (; i + 224 < vec; i += 256) {
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __ldg(src + i + 32 * j);
#pragma unroll
      for (int j = 0; j < 8; ++j) __stcs(dst + i + 32 * j, v[j]);
    }
    for (; i < vec; i += 32) __stcs(dst + i, __ldg(src + i));
  }
}

// The same copy driven by the tokens: each warp reads one token row of x
// once and writes it to the permuted rows of all its local routes
// (exp_to_perm, negative for routes outside the shard).  x is read from HBM
// once instead of once per route.
__global__ void __launch_bounds__(256)
    gather_tokens_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ e2p, int T, int k,
                         int vec, long max_rows, uint4 *__restrict__ xp) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long warp = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
  pdl_launch_dependents();
  for (long t = warp; t < T; t += nwarps) {
    const int my_p = lane < k ? e2p[t * k + lane] : -1;
    const uint4 *src = x + t * vec;
    // warp-uniform loop bounds: every lane reaches each shuffle
    int b = 0;
    for (; b + 256 <= vec; b += 256) {
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __ldg(src + b + lane + 32 * j);
      for (int s = 0; s < k; ++s) {
        const int p = __shfl_sync(0xffffffffu, my_p, s);
        if (p < 0 || p >= max_rows) continue;
        uint4 *dst = xp + (long)p * vec + b + lane;
#pragma unroll
        for (int j = 0; j < 8; ++j) __stcs(dst + 32 * j, v[j]);
      }
    }
    for (; b < vec; b += 32) {
      const int i = b + lane;
      const bool in = i < vec;
      const uint4 v = in ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
      for (int s = 0; s < k; ++s) {
        const int p = __shfl_sync(0xffffffffu, my_p, s);
        if (p >= 0 && p < max_rows && in) __stcs(xp + (long)p * vec + i, v);
      }
    }
  }
}

// The token-major copy for E4M3 activations: each element of x is divided by
// the per-tensor scale (fp32, correctly rounded) and converted to E4M3
// (nearest even, saturating at 448); a lane turns 16 bf16 values (32 bytes)
// into 16 codes (one 16-byte store per route row).
__global__ void __launch_bounds__(256)
    gather_tokens_q_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ e2p, int T, int k,
                           int vec16, float scale, long max_rows, uint4 *__restrict__ xq) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long warp = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
  pdl_launch_dependents();
  for (long t = warp; t < T; t += nwarps) {
    const int my_p = lane < k ? e2p[t * k + lane] : -1;
    const uint4 *src = x + t * 2 * vec16;
    for (int b = 0; b < vec16; b += 32) {  // warp-uniform bounds: every lane reaches each shuffle
      const int i = b + lane;
      const bool in = i < vec16;
      uint4 q = make_uint4(0, 0, 0, 0);
      if (in) {
        const uint4 v0 = __ldg(src + 2 * i), v1 = __ldg(src + 2 * i + 1);
        const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t c[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t a = u[2 * j], bb = u[2 * j + 1];
          const uint32_t lo = e4m3x2(__fdiv_rn(__uint_as_float(a << 16), scale),
                                     __fdiv_rn(__uint_as_float(a & 0xFFFF0000u), scale));
          const uint32_t hi = e4m3x2(__fdiv_rn(__uint_as_float(bb << 16), scale),
                                     __fdiv_rn(__uint_as_float(bb & 0xFFFF0000u), scale));
          c[j] = lo | (hi << 16);
        }
        q = make_uint4(c[0], c[1], c[2], c[3]);
      }
      for (int s = 0; s < k; ++s) {
        const int p = __shfl_sync(0xffffffffu, my_p, s);
        if (p >= 0 && p < max_rows && in) __stcs(xq + (long)p * vec16 + i, q);
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

__global__ void __launch_bounds__(256)
    finalize_kernel(const float4 *__restrict__ y, const int32_t *__restrict__ e2p,
                    const float *__restrict__ w, int T, int k, int H, uint4 *__restrict__ out) {
  __shared__ int sp[MOE_MAX_TOP_K];
  __shared__ float sw[MOE_MAX_TOP_K];
  pdl_wait();
  const int c8n = H >> 3;  // 8 output columns per thread step
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    if (threadIdx.x < k) {
      sp[threadIdx.x] = e2p[(size_t)t * k + threadIdx.x];
      sw[threadIdx.x] = w[(size_t)t * k + threadIdx.x];
    }
    __syncthreads();
    for (int c8 = threadIdx.x; c8 < c8n; c8 += blockDim.x) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int j = 0; j < k; ++j) {
        const int p = sp[j];
        if (p < 0) continue;
        const float wj = sw[j];
        const float4 *row = y + (size_t)p * (H >> 2) + c8 * 2;
        const float4 a = __ldg(row), b = __ldg(row + 1);
        acc[0] = __fadd_rn(acc[0], __fmul_rn(wj, a.x));
        acc[1] = __fadd_rn(acc[1], __fmul_rn(wj, a.y));
        acc[2] = __fadd_rn(acc[2], __fmul_rn(wj, a.z));
        acc[3] = __fadd_rn(acc[3], __fmul_rn(wj, a.w));
        acc[4] = __fadd_rn(acc[4], __fmul_rn(wj, b.x));
        acc[5] = __fadd_rn(acc[5], __fmul_rn(wj, b.y));
        acc[6] = __fadd_rn(acc[6], __fmul_rn(wj, b.z));
        acc[7] = __fadd_rn(acc[7], __fmul_rn(wj, b.w));
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      out[(size_t)t * c8n + c8] = o;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_gather(const uint16_t *x, const int32_t *p2e, const int32_t *m_total, int H,
                          int k, long max_rows, uint16_t *xp, const Launch &l) {
  if (max_rows <= 0) return cudaSuccess;
  const long want_blocks = (max_rows + 7) / 8;  // 8 warps per block, one row per warp
  const long cap = (long)device_sm_count() * 8;
  const int blocks = (int)(want_blocks < cap ? want_blocks : cap);
  return launch_kernel(gather_kernel, dim3(blocks), dim3(256), 0, l,
                       reinterpret_cast<const uint4 *>(x), p2e, m_total, H / 8, k,
                       reinterpret_cast<uint4 *>(xp));
}

cudaError_t launch_gather_tokens_q(const uint16_t *x, const int32_t *e2p, int T, int H, int k,
                                   float scale, long max_rows, uint8_t *xq, const Launch &l) {
  if (T <= 0) return cudaSuccess;
  const long want_blocks = ((long)T + 7) / 8;
  const long cap = (long)device_sm_count() * 8;
  const int blocks = (int)(want_blocks < cap ? want_blocks : cap);
  return launch_kernel(gather_tokens_q_kernel, dim3(blocks), dim3(256), 0, l,
                       reinterpret_cast<const uint4 *>(x), e2p, T, k, H / 16, scale, max_rows,
                       reinterpret_cast<uint4 *>(xq));
}

cudaError_t launch_gather_tokens(const uint16_t *x, const int32_t *e2p, int T, int H, int k,
                                 long max_rows, uint16_t *xp, const Launch &l) {
  if (T <= 0) return cudaSuccess;
  const long want_blocks = ((long)T + 7) / 8;  // 8 warps per block, one token per warp
  const long cap = (long)device_sm_count() * 8;
  const int blocks = (int)(want_blocks < cap ? want_blocks : cap);
  return launch_kernel(gather_tokens_kernel, dim3(blocks), dim3(256), 0, l,
                       reinterpret_cast<const uint4 *>(x), e2p, T, k, H / 8, max_rows,
                       reinterpret_cast<uint4 *>(xp));
}

cudaError_t launch_finalize(const float *y, const int32_t *e2p, const float *w, int T, int k,
                            int H, uint16_t *out, const Launch &l) {
  if (T <= 0) return cudaSuccess;
  const long cap = (long)device_sm_count() * 16;
  const int blocks = (int)(T < cap ? T : cap);
  const int threads = (H / 8) < 256 ? ((H / 8 + 31) / 32) * 32 : 256;
  return launch_kernel(finalize_kernel, dim3(blocks), dim3(threads), 0, l,
                       reinterpret_cast<const float4 *>(y), e2p, w, T, k, H,
                       reinterpret_cast<uint4 *>(out));
}

}  // namespace moe
