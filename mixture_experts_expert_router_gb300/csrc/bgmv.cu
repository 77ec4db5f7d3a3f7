// BGMV LoRA-MoE shrink + expand (flashinfer.fused_moe.prepare_bgmv_moe):
// LoRA deltas of the routed (token, expert) pairs of an MoE layer.
//
//   shrink[s, p, :] = bf16( A_s[l, e] . x[t] )                  rank R values per pair
//   y[t, off_s + f] = sum over the pairs p of token t, ascending p,
//                     of w_p * ( B_s[l, e, f, :] . shrink[s, p, :] )   (fp32)
//
// with t = sorted_token_ids[p], e = expert_ids[p], l = lora_indices[t].  The
// ranks are small (8..64), so both steps stream weights and are bound by
// memory, not by arithmetic: they run on the CUDA cores with 16-byte loads.
//
//   shrink  one CTA per (pair, slice): each of the 8 warps takes rank rows
//           r = warp, warp + 8, ...; a lane sums a strided share of the row in
//           fp32 and the warp adds the 32 partial sums in a fixed butterfly.
//   expand  one CTA per token, the owner of its output row: the token's pairs
//           are taken in ascending pair index, each thread owning output
//           columns f and adding w_p * (B row f . shrink) in pair order, so
//           every replay is bitwise identical and nothing uses atomics.
//
// Pair layouts: "contiguous top-k" (pair p belongs to token p / k, the layout
// the page's fast path serves) needs no index.  Any other order (for example
// pairs sorted by expert) goes through a route index built by one kernel: up
// to kSlots pair numbers per token, in arbitrary slot order, which the expand
// CTA sorts ascending; a token with more pairs than slots scans all pairs in
// order (exact, slower).  Pairs with an out-of-range token, expert or LoRA
// index contribute nothing and raise MOE_DEV_BAD_EXPERT.
#include <cuda_bf16.h>

#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kShrinkThreads = 256;
constexpr int kExpandThreads = 256;
constexpr int kSlots = 16;

struct BgmvArgs {
  const uint16_t *x;
  const uint16_t *a[kBgmvMaxSlices];
  const uint16_t *b[kBgmvMaxSlices];
  int f[kBgmvMaxSlices];
  int off[kBgmvMaxSlices];
  const int32_t *tok, *eid, *lora;
  const float *w;
  uint16_t *shrink;  // [S, P, R]
  float *y;          // [T, ld_y]
  int32_t *cnt;      // general layout: [T] pairs per token
  int32_t *idx;      // general layout: [T, kSlots] pair numbers
  int32_t *status;
  int T, H, R, S, L, E, P, k, ld_y;
};

__device__ __forceinline__ bool pair_ok(const BgmvArgs &a, int p) {
  const int t = a.tok[p];
  if (t < 0 || t >= a.T) return false;
  const int e = a.eid[p];
  if (e < 0 || e >= a.E) return false;
  const int l = a.lora[t];
  return l >= 0 && l < a.L;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float (&o)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(u[i] << 16);
    o[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// General layout: route index, one thread per pair.
__global__ void bgmv_index_kernel(const __grid_constant__ BgmvArgs a) {
  pdl_wait();
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p < a.P && pair_ok(a, p)) {
    const int t = a.tok[p];
    const int slot = atomicAdd(a.cnt + t, 1);
    if (slot < kSlots) a.idx[(long)t * kSlots + slot] = p;
  }
  pdl_launch_dependents();
}

__global__ void __launch_bounds__(kShrinkThreads) bgmv_shrink_kernel(const __grid_constant__ BgmvArgs a) {
  pdl_wait();
  const int p = blockIdx.x, s = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint16_t *out = a.shrink + ((long)s * a.P + p) * a.R;
  if (!pair_ok(a, p)) {
    for (int r = threadIdx.x; r < a.R; r += kShrinkThreads) out[r] = 0;
    if (threadIdx.x == 0 && a.status) atomicOr(reinterpret_cast<unsigned int *>(a.status), MOE_DEV_BAD_EXPERT);
    pdl_launch_dependents();
    return;
  }
  const int t = a.tok[p];
  const long wrow = ((long)a.lora[t] * a.E + a.eid[p]) * a.R;
  const uint4 *xr = reinterpret_cast<const uint4 *>(a.x + (long)t * a.H);
  const int nv = a.H / 8;  // 16-byte vectors per row
  for (int r = warp; r < a.R; r += kShrinkThreads / 32) {
    const uint4 *ar = reinterpret_cast<const uint4 *>(a.a[s] + (wrow + r) * a.H);
    float acc = 0.f;
    for (int v = lane; v < nv; v += 32) {
      float xf[8], af[8];
      bf16x8_to_f32(__ldg(xr + v), xf);
      bf16x8_to_f32(__ldcs(ar + v), af);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = __fmaf_rn(af[i], xf[i], acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) out[r] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
  }
  pdl_launch_dependents();
}

__global__ void __launch_bounds__(kExpandThreads) bgmv_expand_kernel(const __grid_constant__ BgmvArgs a) {
  __shared__ int pairs[kSlots];
  __shared__ int n_pairs;
  __shared__ float sh[64];   // the current pair's shrink values (R <= 64)
  pdl_wait();
  const int t = blockIdx.x;
  // this token's pairs in ascending pair index
  int scan = 0;  // 1: more pairs than slots, walk all pairs in order
  if (threadIdx.x == 0) {
    int n = 0;
    if (a.k > 0) {  // contiguous top-k (k <= kSlots): pairs t*k .. t*k + k - 1
      bool mismatch = false;
      for (int j = 0; j < a.k; ++j) {
        const int p = t * a.k + j;
        if (p >= a.P) break;
        if (a.tok[p] != t) mismatch = true;
        else if (pair_ok(a, p)) pairs[n++] = p;
      }
      if (mismatch && a.status) atomicOr(reinterpret_cast<unsigned int *>(a.status), MOE_DEV_BAD_EXPERT);
    } else {
      n = a.cnt[t];
      if (n <= kSlots) {
        for (int i = 0; i < n; ++i) pairs[i] = a.idx[(long)t * kSlots + i];
        for (int i = 1; i < n; ++i) {  // insertion sort: at most 16 entries
          const int v = pairs[i];
          int j = i - 1;
          while (j >= 0 && pairs[j] > v) {
            pairs[j + 1] = pairs[j];
            --j;
          }
          pairs[j + 1] = v;
        }
      } else {
        n = -1;
      }
    }
    n_pairs = n;
  }
  __syncthreads();
  const int n = n_pairs;
  if (n < 0) scan = 1;
  const int nv = a.R / 8;
  for (int s = 0; s < a.S; ++s) {
    const int F = a.f[s];
    float *yrow = a.y + (long)t * a.ld_y + a.off[s];
    const uint16_t *shr = a.shrink + (long)s * a.P * a.R;
    // each thread owns columns f = tid + 256 * i (at most 32 of them kept in registers)
    for (int f0 = 0; f0 < F; f0 += kExpandThreads * 32) {
      float acc[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = 0.f;
      const int np = scan ? a.P : n;
      for (int q = 0; q < np; ++q) {
        int p;
        if (scan) {
          p = q;
          if (a.tok[p] != t || !pair_ok(a, p)) continue;  // uniform across the CTA
        } else {
          p = pairs[q];
        }
        __syncthreads();  // the previous pair's values are no longer read
        if (threadIdx.x < a.R)
          sh[threadIdx.x] = __uint_as_float((uint32_t)shr[(long)p * a.R + threadIdx.x] << 16);
        __syncthreads();
        const float wp = a.w[p];
        const long brow = ((long)a.lora[t] * a.E + a.eid[p]) * F;
        const uint16_t *bw = a.b[s] + brow * a.R;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int f = f0 + (int)threadIdx.x + kExpandThreads * i;
          if (f < F) {
            const uint4 *br = reinterpret_cast<const uint4 *>(bw + (long)f * a.R);
            float v = 0.f;
            for (int c = 0; c < nv; ++c) {
              float bf[8];
              bf16x8_to_f32(__ldg(br + c), bf);
#pragma unroll
              for (int j = 0; j < 8; ++j) v = __fmaf_rn(bf[j], sh[8 * c + j], v);
            }
            acc[i] = __fadd_rn(acc[i], __fmul_rn(wp, v));
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int f = f0 + (int)threadIdx.x + kExpandThreads * i;
        if (f < F) yrow[f] = acc[i];
      }
    }
  }
  pdl_launch_dependents();
}

}  // namespace

size_t bgmv_workspace_bytes(int T, int contiguous_k) {
  return contiguous_k > 0 ? 0 : (size_t)T * (kSlots + 1) * sizeof(int32_t);
}

cudaError_t launch_bgmv(const BgmvPlan &p, const Launch &l) {
  BgmvArgs a;
  a.x = p.x;
  for (int s = 0; s < kBgmvMaxSlices; ++s) {
    a.a[s] = s < p.S ? p.a[s] : nullptr;
    a.b[s] = s < p.S ? p.b[s] : nullptr;
    a.f[s] = s < p.S ? p.f[s] : 0;
    a.off[s] = s < p.S ? p.off[s] : 0;
  }
  a.tok = p.tok;
  a.eid = p.eid;
  a.lora = p.lora;
  a.w = p.w;
  a.shrink = p.shrink;
  a.y = p.y;
  a.cnt = p.ws;
  a.idx = p.ws ? p.ws + p.T : nullptr;
  a.status = p.status;
  a.T = p.T;
  a.H = p.H;
  a.R = p.R;
  a.S = p.S;
  a.L = p.L;
  a.E = p.E;
  a.P = p.P;
  a.k = p.k;
  a.ld_y = p.ld_y;
  cudaError_t e;
  Launch first = l;  // the first kernel of the call waits for everything before it
  first.pdl = false;
  if (p.k == 0) {
    e = cudaMemsetAsync(p.ws, 0, (size_t)p.T * sizeof(int32_t), l.stream);
    if (e != cudaSuccess) return e;
    if (p.P > 0) {
      e = launch_kernel(bgmv_index_kernel, dim3((p.P + 255) / 256), dim3(256), 0, first, a);
      if (e != cudaSuccess) return e;
      first = l;
    }
  }
  if (p.P > 0) {
    e = launch_kernel(bgmv_shrink_kernel, dim3(p.P, p.S), dim3(kShrinkThreads), 0, first, a);
    if (e != cudaSuccess) return e;
    first = l;
  }
  return launch_kernel(bgmv_expand_kernel, dim3(p.T), dim3(kExpandThreads), 0, first, a);
}

}  // namespace moe
