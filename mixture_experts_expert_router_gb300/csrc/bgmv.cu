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
// Two pipelines compute exactly this.  The pair-grouped one groups the pairs
// by (LoRA, expert), ascending pair index inside a group, so each A and B
// block is read once per group instead of once per pair:
//   group    while groups x pairs <= kScanGroupingMax: one CTA per group scans
//            the pairs (bgmv_group_kernel); else, up to kBgmvSortMaxGroups
//            groups, key[p] = lora[t] * E + e (negative for an invalid pair,
//            whose shrink rows are zeroed) and the stable counting sort of the
//            routes (sort.cu);
//   gshrink  one CTA per (group, slice): tiles of 16 pairs times the group's
//            A block, H staged through shared memory 256 columns at a time
//            (cp.async, double-buffered) into m16n8k16 tensor-core MMAs with
//            fp32 accumulators, the eight warps' k-step sums added in warp
//            order;
//   gexpand  one CTA per (group, 256 output columns of a slice): the columns'
//            B rows staged once, tiles of 16 pairs' shrink values times them
//            (m16n8k16 MMAs, K = R), writing the fp32 partial
//            w_p * (B row . shrink_p) of every pair of the group;
// Per group the contraction is 16 or so pairs by R <= 64, far below the 64- and
// 128-row tiles of the single-thread-issued MMA, so the warp-level m16n8k16
// shape serves it; both kernels stay bound by the A and B bytes.
//   combine  one CTA per token adds its pairs' partials in ascending pair
//            index (the owner rule), so the output does not depend on the
//            grouping.
// The per-route pipeline below (one CTA per pair for the shrink, one per
// token for the expand) serves whatever neither grouping takes.
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

struct BgmvArgs;
__device__ __forceinline__ bool pair_ok(const BgmvArgs &a, int p);

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
  // grouped pipeline
  int32_t *keys;            // [P] (sorted grouping)
  const int32_t *g_indptr;  // [G + 1] pair rows of each (LoRA, expert) group (sorted grouping)
  int32_t *g_start, *g_cnt; // [G] each group's range of g_pairs (scanned grouping), else null
  int32_t *g_total;         // pairs placed so far (scanned grouping; zeroed before it)
  const int32_t *g_pairs;   // [P] pair numbers in group order, ascending inside a group
  float *partial;           // [P, ld_part] fp32 w_p * (B row . shrink_p)
  int ld_part;              // sum of feat_out
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

// ------------------------------------------------------------ grouped pipeline --
constexpr int kGroupTile = 16;  // pairs per tile: the M of the m16n8k16 tensor-core MMA

// Scanned grouping (few groups times pairs): after bgmv_key_kernel, one CTA
// per (LoRA, expert) group scans the keys, finds its pairs in ascending pair
// index and writes them to a range of g_pairs claimed with one atomic add.
// Where the range lands varies from run to run and does not matter: the
// shrink, expand and combine read each group's pairs in their order, wherever
// they sit.
constexpr int kGroupThreads = 512;

__global__ void __launch_bounds__(kGroupThreads) bgmv_group_kernel(const __grid_constant__ BgmvArgs a) {
  __shared__ int wsum[kGroupThreads / 32];
  __shared__ int base_s;
  pdl_wait();
  const int g = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int n = 0;
#pragma unroll 4
  for (int p = tid; p < a.P; p += kGroupThreads) n += __ldg(a.keys + p) == g;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  if (lane == 0) wsum[warp] = n;
  __syncthreads();
  if (tid == 0) {
    int tot = 0;
    for (int w = 0; w < kGroupThreads / 32; ++w) tot += wsum[w];
    const int off = tot > 0 ? atomicAdd(a.g_total, tot) : 0;
    a.g_start[g] = off;
    a.g_cnt[g] = tot;
    base_s = off;
  }
  __syncthreads();
  int run = base_s;
  for (int c = 0; c < a.P; c += kGroupThreads) {
    const int p = c + tid;
    const bool m = p < a.P && __ldg(a.keys + p) == g;
    const unsigned b = __ballot_sync(0xffffffffu, m);
    if (lane == 0) wsum[warp] = __popc(b);
    __syncthreads();
    int before = 0, tot = 0;
    for (int w = 0; w < kGroupThreads / 32; ++w) {
      const int x = wsum[w];
      before += w < warp ? x : 0;
      tot += x;
    }
    if (m) const_cast<int32_t *>(a.g_pairs)[run + before + __popc(b & ((1u << lane) - 1u))] = p;
    run += tot;
    __syncthreads();  // wsum is rewritten by the next round
  }
  pdl_launch_dependents();
}

// A group's range of g_pairs: from the scanned grouping, else the sort's offsets.
__device__ __forceinline__ void group_range(const BgmvArgs &a, int g, int &p0, int &p1) {
  if (a.g_start) {
    p0 = a.g_start[g];
    p1 = p0 + a.g_cnt[g];
  } else {
    p0 = a.g_indptr[g];
    p1 = a.g_indptr[g + 1];
  }
}

__global__ void __launch_bounds__(256) bgmv_key_kernel(const __grid_constant__ BgmvArgs a) {
  pdl_wait();
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p < a.P) {
    const bool ok = pair_ok(a, p);
    a.keys[p] = ok ? a.lora[a.tok[p]] * a.E + a.eid[p] : -1;  // no group takes -1
    if (!ok) {
      for (int s = 0; s < a.S; ++s)
        for (int r = 0; r < a.R; ++r) a.shrink[((long)s * a.P + p) * a.R + r] = 0;
      if (a.status) atomicOr(reinterpret_cast<unsigned int *>(a.status), MOE_DEV_BAD_EXPERT);
    }
  }
  pdl_launch_dependents();
}

// Shared-memory row pitch of the staged bf16 operands: a multiple of 16 bytes
// whose word stride is 4 mod 32, so the eight rows and four column pairs of an
// m16n8k16 fragment load fall in 32 distinct banks.
constexpr int kKC = 256;        // x / A columns per shrink stage
constexpr int kKP = kKC + 8;    // pitch (bf16) of a staged row

constexpr int kShrinkPass = 2 * kGroupTile;  // pairs per shrink pass: two m16 tiles share each A chunk
constexpr int kGsThreads = 512;               // 16 warps: 8 k-step lanes x 2 m-tiles

template <int R>
struct GShrinkSmem {
  static constexpr int NST = 3;  // ring depth (two CTAs per SM up to rank 32)
  static constexpr int STAGE = (R + kShrinkPass) * kKP;  // bf16: A rows, then the pass's x rows
  static constexpr size_t RING_BYTES = (size_t)NST * STAGE * 2;
  // the sixteen warps' sums [16][16][R] fp32 reuse the ring once a pass's k-loop is over
  static_assert((size_t)16 * kGroupTile * R * 4 <= RING_BYTES, "the warp sums fit in the ring");
  static constexpr size_t TOK_OFF = RING_BYTES;
  static constexpr size_t BYTES = TOK_OFF + kShrinkPass * 4;
};

__device__ __forceinline__ uint32_t lds32(const uint16_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

// One CTA per (group, slice): the group's pairs in passes of up to 32 (two
// 16-pair tiles, the M of the m16n8k16 MMA, sharing every A chunk), its A
// block [R, H] on N, H on K.  Each stage copies kKC columns of A and of the
// pass's x rows into shared memory (cp.async, one row per warp, a ring of NST
// stages with NST - 1 in flight).  Warp w works on tile w % 2 and takes the
// k-steps w / 2, w / 2 + 8 of every stage into its own accumulators; the eight
// warps' sums of a tile are added in k-step-lane order at the end of the pass.
template <int R>
__global__ void __launch_bounds__(kGsThreads) bgmv_gshrink_kernel(const __grid_constant__ BgmvArgs a) {
  using SM = GShrinkSmem<R>;
  extern __shared__ __align__(16) unsigned char gs_smem[];
  uint16_t *stage = reinterpret_cast<uint16_t *>(gs_smem);
  float *red = reinterpret_cast<float *>(gs_smem);  // [16 warps][16 pairs][R], over the ring
  int *tp = reinterpret_cast<int *>(gs_smem + SM::TOK_OFF);  // token of each pair of the pass
  pdl_wait();
  const int g = blockIdx.x, s = blockIdx.y;
  int p0, p1;
  group_range(a, g, p0, p1);
  if (p1 > p0) {
    const int l = g / a.E, e = g - l * a.E;
    const uint16_t *A = a.a[s] + ((long)l * a.E + e) * R * a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, c2 = 2 * (lane & 3);
    const int mt = warp & 1, kw = warp >> 1;  // this warp's tile and k-step lane
    const int nch = (a.H + kKC - 1) / kKC;
    const uint64_t pol_a = policy_evict_first();  // each A element is read by one pass of one CTA
    const uint64_t pol_x = policy_evict_normal();
    for (int q0 = p0; q0 < p1; q0 += kShrinkPass) {
      const int n = p1 - q0 < kShrinkPass ? p1 - q0 : kShrinkPass;
      __syncthreads();  // the previous pass no longer reads tp, red or the stages
      if (threadIdx.x < kShrinkPass) tp[threadIdx.x] = (int)threadIdx.x < n ? a.tok[a.g_pairs[q0 + threadIdx.x]] : -1;
      __syncthreads();
      auto load = [&](int ch) {  // row r of the stage by warp r % 16, 16 bytes a lane
        uint16_t *st = stage + (ch % SM::NST) * SM::STAGE;
        const int h0 = ch * kKC, hn = a.H - h0 < kKC ? a.H - h0 : kKC;  // hn % 8 == 0
        const bool in = 8 * lane < hn;
        for (int row = warp; row < R + kShrinkPass; row += kGsThreads / 32) {
          uint16_t *dst = st + row * kKP + 8 * lane;
          const uint16_t *src = nullptr;
          if (in) {
            if (row < R) src = A + (long)row * a.H + h0 + 8 * lane;
            else if (tp[row - R] >= 0) src = a.x + (long)tp[row - R] * a.H + h0 + 8 * lane;
          }
          if (src) cp_async_16(smem_u32(dst), src, row < R ? pol_a : pol_x);
          else *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        cp_async_commit();
      };
      const bool active = mt * kGroupTile < n;  // this warp's tile has pairs
      float d[R / 8][4];
#pragma unroll
      for (int nt = 0; nt < R / 8; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
      // one commit group per chunk (empty past the end), so that waiting for
      // all but the NST - 1 newest groups means chunk ch has landed
      for (int i = 0; i < SM::NST - 1; ++i) {
        if (i < nch) load(i);
        else cp_async_commit();
      }
      for (int ch = 0; ch < nch; ++ch) {
        // chunk ch + NST - 1 into the stage that chunk ch - 1 used, freed by
        // the barrier that ended ch - 1
        if (ch + SM::NST - 1 < nch) load(ch + SM::NST - 1);
        else cp_async_commit();
        cp_async_wait_pending<SM::NST - 1>();
        __syncthreads();  // stage ch has landed for every thread
        const uint16_t *As = stage + (ch % SM::NST) * SM::STAGE;
        const uint16_t *xs = As + (R + mt * kGroupTile) * kKP;
        const int hn = a.H - ch * kKC < kKC ? a.H - ch * kKC : kKC;
        if (active) {
          for (int ks = kw; ks < (hn + 15) / 16; ks += 8) {
            const int c = ks * 16 + c2;
            const uint32_t a0 = lds32(xs + gq * kKP + c), a1 = lds32(xs + (gq + 8) * kKP + c);
            const uint32_t a2 = lds32(xs + gq * kKP + c + 8), a3 = lds32(xs + (gq + 8) * kKP + c + 8);
#pragma unroll
            for (int nt = 0; nt < R / 8; ++nt) {
              const uint16_t *br = As + (nt * 8 + gq) * kKP + c;
              mma_bf16_16816(d[nt], a0, a1, a2, a3, lds32(br), lds32(br + 8));
            }
          }
        }
        __syncthreads();  // stage ch may be overwritten (by chunk ch + NST)
      }
      cp_async_wait_all();  // the empty trailing groups
#pragma unroll
      for (int nt = 0; nt < R / 8; ++nt) {
        float *r0 = red + (warp * kGroupTile + gq) * R + nt * 8 + c2;
        r0[0] = d[nt][0];
        r0[1] = d[nt][1];
        r0[8 * R] = d[nt][2];
        r0[8 * R + 1] = d[nt][3];
      }
      __syncthreads();
      for (int o = threadIdx.x; o < n * R; o += kGsThreads) {
        const int pr = o / R, col = o - pr * R, t = pr / kGroupTile, row = pr - t * kGroupTile;
        float v = red[(t * kGroupTile + row) * R + col];  // k-step lane 0 (warp t)
#pragma unroll
        for (int k = 1; k < 8; ++k) v = __fadd_rn(v, red[((2 * k + t) * kGroupTile + row) * R + col]);
        a.shrink[((long)s * a.P + a.g_pairs[q0 + pr]) * R + col] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      }
    }
  }
  pdl_launch_dependents();
}

// One CTA per (group, 256 output columns of a slice): the group's pairs in
// tiles of 16 (M), the columns' B rows [256, R] on N (staged once), R on K
// (zero-padded to 16).  Each warp owns 32 columns (four n-tiles) and writes
// w_p * (B row . shrink_p) of every pair of the tile.
template <int R>
__global__ void __launch_bounds__(256) bgmv_gexpand_kernel(const __grid_constant__ BgmvArgs a) {
  constexpr int RK = R < 16 ? 16 : R, RP = RK + 8;  // K and the row pitch (bf16)
  __shared__ __align__(16) uint16_t bs[256 * RP];
  __shared__ __align__(16) uint16_t sh[kGroupTile * RP];
  __shared__ float sw[kGroupTile];
  __shared__ int sp[kGroupTile];
  pdl_wait();
  const int g = blockIdx.x;
  int p0, p1;
  group_range(a, g, p0, p1);
  if (p1 > p0) {
    int s = 0, c = blockIdx.y;
    while (s < a.S && c >= (a.f[s] + 255) / 256) c -= (a.f[s++] + 255) / 256;
    const int F = a.f[s], f0 = c * 256, fn = F - f0 < 256 ? F - f0 : 256;  // fn % 8 == 0
    const int l = g / a.E, e = g - l * a.E;
    const uint16_t *B = a.b[s] + (((long)l * a.E + e) * F + f0) * R;
    const uint64_t pol_b = policy_evict_first();
    for (int i = threadIdx.x; i < 256 * (RK / 8); i += 256) {
      const int row = i / (RK / 8), v = i - row * (RK / 8);
      uint16_t *dst = bs + row * RP + 8 * v;
      if (row < fn && 8 * v < R) cp_async_16(smem_u32(dst), B + (long)row * R + 8 * v, pol_b);
      else *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    cp_async_commit();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, c2 = 2 * (lane & 3);
    const uint16_t *shr = a.shrink + (long)s * a.P * R;
    float *part = a.partial + a.off[s] + f0;
    for (int q0 = p0; q0 < p1; q0 += kGroupTile) {
      const int n = p1 - q0 < kGroupTile ? p1 - q0 : kGroupTile;
      __syncthreads();  // the previous tile no longer reads sh, sw, sp
      for (int i = threadIdx.x; i < kGroupTile * RK; i += 256) {
        const int pr = i / RK, rr = i - pr * RK;
        sh[pr * RP + rr] = pr < n && rr < R ? shr[(long)a.g_pairs[q0 + pr] * R + rr] : (uint16_t)0;
      }
      if (threadIdx.x < kGroupTile) {
        const int pr = threadIdx.x;
        sp[pr] = pr < n ? a.g_pairs[q0 + pr] : 0;
        sw[pr] = pr < n ? a.w[sp[pr]] : 0.f;
      }
      cp_async_wait_all();
      __syncthreads();
      uint32_t af[RK / 16][4];
#pragma unroll
      for (int ks = 0; ks < RK / 16; ++ks) {
        const int cc = ks * 16 + c2;
        af[ks][0] = lds32(sh + gq * RP + cc);
        af[ks][1] = lds32(sh + (gq + 8) * RP + cc);
        af[ks][2] = lds32(sh + gq * RP + cc + 8);
        af[ks][3] = lds32(sh + (gq + 8) * RP + cc + 8);
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int n0 = warp * 32 + nt * 8;
        if (n0 >= fn) break;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < RK / 16; ++ks) {
          const uint16_t *br = bs + (n0 + gq) * RP + ks * 16 + c2;
          mma_bf16_16816(d, af[ks][0], af[ks][1], af[ks][2], af[ks][3], lds32(br), lds32(br + 8));
        }
        if (gq < n)
          *reinterpret_cast<float2 *>(part + (long)sp[gq] * a.ld_part + n0 + c2) =
              make_float2(__fmul_rn(sw[gq], d[0]), __fmul_rn(sw[gq], d[1]));
        if (gq + 8 < n)
          *reinterpret_cast<float2 *>(part + (long)sp[gq + 8] * a.ld_part + n0 + c2) =
              make_float2(__fmul_rn(sw[gq + 8], d[2]), __fmul_rn(sw[gq + 8], d[3]));
      }
    }
  }
  pdl_launch_dependents();
}

// y[t] = sum of the partials of t's pairs in ascending pair index.  Token-major
// pairs are checked one per lane of the first warp; the columns go four at a
// time (the partial rows are 16-byte aligned: sum feat_out % 8 == 0).
__global__ void __launch_bounds__(256) bgmv_combine_kernel(const __grid_constant__ BgmvArgs a) {
  __shared__ int pairs[kSlots];
  __shared__ int n_pairs;
  pdl_wait();
  const int t = blockIdx.x;
  if (a.k > 0) {
    if (threadIdx.x < 32) {  // k <= MOE_MAX_TOP_K == kSlots <= 32
      const int lane = threadIdx.x, p = t * a.k + lane;
      bool mine = false, mismatch = false;
      if (lane < a.k && p < a.P) {
        if (a.tok[p] != t) mismatch = true;
        else mine = pair_ok(a, p);
      }
      const unsigned m = __ballot_sync(0xffffffffu, mine);
      if (mine) pairs[__popc(m & ((1u << lane) - 1u))] = p;
      if (__any_sync(0xffffffffu, mismatch) && lane == 0 && a.status)
        atomicOr(reinterpret_cast<unsigned int *>(a.status), MOE_DEV_BAD_EXPERT);
      if (lane == 0) n_pairs = __popc(m);
    }
  } else if (threadIdx.x == 0) {
    int n = a.cnt[t];
    if (n <= kSlots) {
      for (int i = 0; i < n; ++i) pairs[i] = a.idx[(long)t * kSlots + i];
      for (int i = 1; i < n; ++i) {
        const int v = pairs[i];
        int j = i - 1;
        while (j >= 0 && pairs[j] > v) {
          pairs[j + 1] = pairs[j];
          --j;
        }
        pairs[j + 1] = v;
      }
    } else {
      n = -1;  // more pairs than slots: walk all pairs in order
    }
    n_pairs = n;
  }
  __syncthreads();
  const int n = n_pairs;
  float *yrow = a.y + (long)t * a.ld_y;
  const bool vec_y = ((reinterpret_cast<uintptr_t>(yrow)) & 15u) == 0;
  for (int c = 4 * (int)threadIdx.x; c < a.ld_part; c += 4 * 256) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](int p) {
      const float4 v = __ldcs(reinterpret_cast<const float4 *>(a.partial + (long)p * a.ld_part + c));
      acc.x = __fadd_rn(acc.x, v.x);
      acc.y = __fadd_rn(acc.y, v.y);
      acc.z = __fadd_rn(acc.z, v.z);
      acc.w = __fadd_rn(acc.w, v.w);
    };
    if (n >= 0) {
      for (int q = 0; q < n; ++q) add(pairs[q]);
    } else {
      for (int p = 0; p < a.P; ++p)
        if (a.tok[p] == t && pair_ok(a, p)) add(p);
    }
    if (vec_y) {
      *reinterpret_cast<float4 *>(yrow + c) = acc;
    } else {
      yrow[c] = acc.x;
      yrow[c + 1] = acc.y;
      yrow[c + 2] = acc.z;
      yrow[c + 3] = acc.w;
    }
  }
  pdl_launch_dependents();
}

}  // namespace

static size_t bgmv_align(size_t v) { return (v + 255) / 256 * 256; }

template <int R>
static cudaError_t launch_gshrink(int G, int S, const Launch &l, const BgmvArgs &a) {
  constexpr size_t bytes = GShrinkSmem<R>::BYTES;
  static const cudaError_t attr =
      raise_smem_limit(bgmv_gshrink_kernel<R>, bytes);
  if (attr != cudaSuccess) return attr;
  return launch_kernel(bgmv_gshrink_kernel<R>, dim3(G, S), dim3(kGsThreads), bytes, l, a);
}

// Workspace: [route index (general order)] [grouped pipeline: keys, group
// offsets, pairs in group order, their inverse, the sort's table, partials].
struct BgmvLayout {
  size_t g_total, cnt, idx, keys, g_indptr, g_pairs, g_inv, sort_ws, g_start, g_cnt, partial, total;
  bool grouped;
};

// Group count times pairs up to which the grouping scans (one CTA per group
// reading every pair); above it the pairs are keyed and sorted (S2's sort).
constexpr long kScanGroupingMax = 1L << 22;

static bool bgmv_scan_grouping(int G, int P) { return G >= 1 && (long)G * P <= kScanGroupingMax; }

static BgmvLayout bgmv_layout(int T, int P, int k, int G, int total_f) {
  BgmvLayout o{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += bgmv_align(bytes > 0 ? bytes : 1);
    return at;
  };
  // g_total right before cnt: one memset clears both
  o.g_total = take(4);
  if (k == 0) {
    o.cnt = take((size_t)T * 4);
    o.idx = take((size_t)T * kSlots * 4);
  }
  o.grouped = bgmv_scan_grouping(G, P) || (G >= 1 && G <= kBgmvSortMaxGroups);
  if (o.grouped) {
    o.keys = take((size_t)P * 4);
    o.g_indptr = take((size_t)(G + 1) * 4);
    o.g_pairs = take((size_t)P * 4);
    o.g_inv = take((size_t)P * 4);
    o.sort_ws = take(sort_workspace_bytes(P, G));
    o.g_start = take((size_t)G * 4);
    o.g_cnt = take((size_t)G * 4);
    o.partial = take((size_t)P * total_f * 4);
  }
  o.total = off;
  return o;
}

size_t bgmv_workspace_bytes(int T, int P, int contiguous_k, int num_loras, int E, int total_f) {
  return bgmv_layout(T, P, contiguous_k, num_loras * E, total_f).total;
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
  const int G = p.L * p.E;
  int total_f = 0;
  for (int i = 0; i < p.S; ++i) total_f += p.f[i];
  const BgmvLayout lay = bgmv_layout(p.T, p.P, p.k, G, total_f);
  unsigned char *ws = reinterpret_cast<unsigned char *>(p.ws);
  a.cnt = p.k == 0 ? reinterpret_cast<int32_t *>(ws + lay.cnt) : nullptr;
  a.idx = p.k == 0 ? reinterpret_cast<int32_t *>(ws + lay.idx) : nullptr;
  a.status = p.status;
  a.keys = lay.grouped ? reinterpret_cast<int32_t *>(ws + lay.keys) : nullptr;
  a.g_indptr = lay.grouped ? reinterpret_cast<int32_t *>(ws + lay.g_indptr) : nullptr;
  a.g_pairs = lay.grouped ? reinterpret_cast<int32_t *>(ws + lay.g_pairs) : nullptr;
  const bool scan = bgmv_scan_grouping(G, p.P);
  a.g_start = scan ? reinterpret_cast<int32_t *>(ws + lay.g_start) : nullptr;
  a.g_cnt = scan ? reinterpret_cast<int32_t *>(ws + lay.g_cnt) : nullptr;
  a.g_total = reinterpret_cast<int32_t *>(ws + lay.g_total);
  a.partial = lay.grouped ? reinterpret_cast<float *>(ws + lay.partial) : nullptr;
  a.ld_part = total_f;
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
  // the scanned grouping's pair counter and the route index's counts start at 0
  if (p.k == 0 || scan) {
    const size_t bytes = p.k == 0 ? lay.cnt + (size_t)p.T * sizeof(int32_t) - lay.g_total : sizeof(int32_t);
    e = cudaMemsetAsync(a.g_total, 0, bytes, l.stream);
    if (e != cudaSuccess) return e;
  }
  if (p.k == 0) {
    if (p.P > 0) {
      e = launch_kernel(bgmv_index_kernel, dim3((p.P + 255) / 256), dim3(256), 0, first, a);
      if (e != cudaSuccess) return e;
      first = l;
    }
  }
  if (lay.grouped && p.P > 0) {
    e = launch_kernel(bgmv_key_kernel, dim3((p.P + 255) / 256), dim3(256), 0, first, a);
    if (e != cudaSuccess) return e;
    if (scan) {
      e = launch_kernel(bgmv_group_kernel, dim3(G), dim3(kGroupThreads), 0, l, a);
    } else {
      e = launch_sort(a.keys, p.P, G, 0, G, const_cast<int32_t *>(a.g_indptr), const_cast<int32_t *>(a.g_pairs),
                      reinterpret_cast<int32_t *>(ws + lay.g_inv), reinterpret_cast<int32_t *>(ws + lay.sort_ws),
                      p.status, l);
    }
    if (e != cudaSuccess) return e;
    switch (p.R) {
      case 8: e = launch_gshrink<8>(G, p.S, l, a); break;
      case 16: e = launch_gshrink<16>(G, p.S, l, a); break;
      case 32: e = launch_gshrink<32>(G, p.S, l, a); break;
      default: e = launch_gshrink<64>(G, p.S, l, a); break;
    }
    if (e != cudaSuccess) return e;
    int chunks = 0;
    for (int i = 0; i < p.S; ++i) chunks += (p.f[i] + 255) / 256;
    switch (p.R) {
      case 8: e = launch_kernel(bgmv_gexpand_kernel<8>, dim3(G, chunks), dim3(256), 0, l, a); break;
      case 16: e = launch_kernel(bgmv_gexpand_kernel<16>, dim3(G, chunks), dim3(256), 0, l, a); break;
      case 32: e = launch_kernel(bgmv_gexpand_kernel<32>, dim3(G, chunks), dim3(256), 0, l, a); break;
      default: e = launch_kernel(bgmv_gexpand_kernel<64>, dim3(G, chunks), dim3(256), 0, l, a); break;
    }
    if (e != cudaSuccess) return e;
    return launch_kernel(bgmv_combine_kernel, dim3(p.T), dim3(256), 0, l, a);
  }
  if (p.P > 0) {
    e = launch_kernel(bgmv_shrink_kernel, dim3(p.P, p.S), dim3(kShrinkThreads), 0, first, a);
    if (e != cudaSuccess) return e;
    first = l;
  }
  return launch_kernel(bgmv_expand_kernel, dim3(p.T), dim3(kExpandThreads), 0, first, a);
}

}  // namespace moe
