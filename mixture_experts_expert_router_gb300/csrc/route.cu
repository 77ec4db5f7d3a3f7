// S1: renormalised top-k routing, one warp per token.
//
// "Renormalize top-k" (flashinfer.experimental.cake_stepfun_moe, opening
// paragraphs): softmax over the E logits, keep the top_k, renormalise.  The
// kept set is chosen on the logits directly (softmax is strictly increasing),
// ordered by logit descending with equal logits ordered by lower expert id, and
// the renormalised weights are the softmax over the kept logits only:
// w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0), summed in ascending j.
#include <cfloat>

#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// Lexicographic (value descending, id ascending) "a is before b".
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

template <int VPL>  // logits held per lane: lane l holds experts l, l+32, ...
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, int T, int E,
                                                    int k, int32_t *__restrict__ ids,
                                                    float *__restrict__ w) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int tok = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (tok >= T) return;
  const float *row = logits + (size_t)tok * E;
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldg(row + e) : -FLT_MAX;
  }
  uint32_t taken = 0;
  float my_v = 0.f;   // lane j keeps the j-th chosen (value, id)
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    // best remaining entry of this lane (ids grow with i, so '>' keeps the lower id)
    float bv = -FLT_MAX;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (!((taken >> i) & 1u) && e < E && (bi == 0x7fffffff || v[i] > bv)) {
        bv = v[i];
        bi = e;
      }
    }
    // warp arg-best under the same order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi != 0x7fffffff && (bi == 0x7fffffff || before(ov, oi, bv, bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_v = bv;
      my_id = bi;
    }
  }
  const float m = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = expf(my_v - m);
  float s = 0.f;
  for (int j = 0; j < k; ++j) s = __fadd_rn(s, __shfl_sync(0xffffffffu, ex, j));
  if (lane < k) {
    ids[(size_t)tok * k + lane] = my_id;
    w[(size_t)tok * k + lane] = __fdiv_rn(ex, s);
  }
}

}  // namespace

cudaError_t launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                         const Launch &l) {
  if (T <= 0) return cudaSuccess;
  const dim3 block(256);
  const dim3 grid((unsigned)(((long)T * 32 + 255) / 256));
  if (E <= 32) return launch_kernel(route_kernel<1>, grid, block, 0, l, logits, T, E, k, ids, w);
  if (E <= 64) return launch_kernel(route_kernel<2>, grid, block, 0, l, logits, T, E, k, ids, w);
  if (E <= 128) return launch_kernel(route_kernel<4>, grid, block, 0, l, logits, T, E, k, ids, w);
  if (E <= 256) return launch_kernel(route_kernel<8>, grid, block, 0, l, logits, T, E, k, ids, w);
  if (E <= 512) return launch_kernel(route_kernel<16>, grid, block, 0, l, logits, T, E, k, ids, w);
  return launch_kernel(route_kernel<32>, grid, block, 0, l, logits, T, E, k, ids, w);
}

}  // namespace moe
