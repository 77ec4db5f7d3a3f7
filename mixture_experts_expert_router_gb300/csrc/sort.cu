// S2: deterministic stable counting sort of the routes by local expert.
//
// Group layout (Cake ragged BF16 grouped GEMM, operation table): the rows of
// expert i are the consecutive permuted rows [m_indptr[i], m_indptr[i+1]).
// Inside a group the rows keep ascending expanded index r = t*top_k + j, so
// the permutation is unique and every replay is bitwise identical.
//
// Small problems (routes <= kSortSingleMax) run in one CTA.  Larger ones run
// as three kernels with no grid-wide barrier: per-chunk histograms, one CTA
// that scans them into per-(chunk, expert) starting rows and m_indptr, and a
// scatter in which each chunk places its routes from those starting rows.
// Inside a chunk, routes are placed 1024 at a time: a warp's routes to the
// same expert are ranked with __match_any_sync, and warps are ordered by a
// per-(warp, expert) count table, so the order never depends on timing.
#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;  // 32 warps: the count table has one row per warp

struct ScatterSmem {
  uint16_t *warp_cnt;  // [32][L]
  int *cur;            // [L] next free permuted row of each expert
  int *tot;            // [L] routes of each expert in the current round
};

__device__ __forceinline__ ScatterSmem carve(unsigned char *base, int L) {
  ScatterSmem s;
  s.cur = reinterpret_cast<int *>(base);
  s.tot = s.cur + L;
  s.warp_cnt = reinterpret_cast<uint16_t *>(s.tot + L);
  return s;
}

__host__ __device__ inline size_t scatter_smem_bytes(int L) {
  return (size_t)L * 8 + (size_t)32 * L * 2;
}

// Place the routes r0 .. r0+1023 (those below r_end).
__device__ void scatter_round(const int32_t *__restrict__ ids, long r0, long r_end, int off, int L,
                              const ScatterSmem &s, int32_t *__restrict__ p2e,
                              int32_t *__restrict__ e2p) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long r = r0 + tid;
  const bool in_range = r < r_end;
  int e = -1;
  if (in_range) {
    const int g = ids[r];
    if (g >= off && g < off + L) e = g - off;  // off >= 0 and off + L <= E: local implies valid
  }
  uint32_t *cnt32 = reinterpret_cast<uint32_t *>(s.warp_cnt);
  for (int i = tid; i < 16 * L; i += kThreads) cnt32[i] = 0u;
  __syncthreads();
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && rank == 0) s.warp_cnt[warp * L + e] = (uint16_t)__popc(peers);
  __syncthreads();
  for (int x = tid; x < L; x += kThreads) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = s.warp_cnt[w * L + x];
      s.warp_cnt[w * L + x] = (uint16_t)run;
      run += c;
    }
    s.tot[x] = run;
  }
  __syncthreads();
  if (e >= 0) {
    const int p = s.cur[e] + s.warp_cnt[warp * L + e] + rank;
    p2e[p] = (int32_t)r;
    e2p[r] = p;
  } else if (in_range) {
    e2p[r] = -1;
  }
  __syncthreads();
  for (int x = tid; x < L; x += kThreads) s.cur[x] += s.tot[x];
  __syncthreads();
}

// Exclusive scan of v[0..n) (n <= 1024) in place; returns the total.  All
// kThreads threads must call it.
__device__ int block_exclusive_scan(int *v, int n, int *warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int x = tid < n ? v[tid] : 0;
  int inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int t = warp_tot[lane];
    int ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += y;
    }
    warp_tot[lane] = ti - t;  // exclusive prefix of warp totals
    if (lane == 31) warp_tot[32] = ti;
  }
  __syncthreads();
  if (tid < n) v[tid] = inc - x + warp_tot[warp];
  const int total = warp_tot[32];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kThreads, 1)
    sort_single_kernel(const int32_t *__restrict__ ids, int R, int E, int off, int L,
                       int32_t *__restrict__ m_indptr, int32_t *__restrict__ p2e,
                       int32_t *__restrict__ e2p, int32_t *status) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int warp_tot[33];
  __shared__ int bad;
  pdl_wait();
  const ScatterSmem s = carve(smem, L);
  const int tid = threadIdx.x;
  for (int x = tid; x < L; x += kThreads) s.cur[x] = 0;
  if (tid == 0) bad = 0;
  __syncthreads();
  for (int r = tid; r < R; r += kThreads) {
    const int g = ids[r];
    if (g < 0 || g >= E) bad = 1;
    else if (g >= off && g < off + L) atomicAdd(&s.cur[g - off], 1);
  }
  __syncthreads();
  const int total = block_exclusive_scan(s.cur, L, warp_tot);
  for (int x = tid; x < L; x += kThreads) m_indptr[x] = s.cur[x];
  if (tid == 0) {
    m_indptr[L] = total;
    if (bad && status) atomicOr(reinterpret_cast<unsigned int *>(status), MOE_DEV_BAD_EXPERT);
  }
  pdl_launch_dependents();
  for (int r0 = 0; r0 < R; r0 += kThreads) scatter_round(ids, r0, R, off, L, s, p2e, e2p);
}

__global__ void __launch_bounds__(kThreads, 1)
    sort_hist_kernel(const int32_t *__restrict__ ids, long R, int E, int off, int L,
                     int32_t *__restrict__ ws, int32_t *status) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int bad;
  pdl_wait();
  int *hist = reinterpret_cast<int *>(smem);
  const int tid = threadIdx.x;
  for (int x = tid; x < L; x += kThreads) hist[x] = 0;
  if (tid == 0) bad = 0;
  __syncthreads();
  const long r_begin = (long)blockIdx.x * kSortChunk;
  const long r_end = min(R, r_begin + kSortChunk);
  for (long r = r_begin + tid; r < r_end; r += kThreads) {
    const int g = ids[r];
    if (g < 0 || g >= E) bad = 1;
    else if (g >= off && g < off + L) atomicAdd(&hist[g - off], 1);
  }
  __syncthreads();
  for (int x = tid; x < L; x += kThreads) ws[(size_t)blockIdx.x * L + x] = hist[x];
  if (tid == 0 && bad && status) atomicOr(reinterpret_cast<unsigned int *>(status), MOE_DEV_BAD_EXPERT);
  pdl_launch_dependents();
}

// One CTA: ws[b][x] (chunk b's count of expert x) -> first permuted row of
// chunk b's routes to expert x; writes m_indptr.
__global__ void __launch_bounds__(kThreads, 1)
    sort_scan_kernel(int nblk, int L, int32_t *__restrict__ ws, int32_t *__restrict__ m_indptr) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int warp_tot[33];
  pdl_wait();
  int *base = reinterpret_cast<int *>(smem);
  const int tid = threadIdx.x;
  for (int x = tid; x < L; x += kThreads) {
    int t = 0;
    for (int b = 0; b < nblk; ++b) t += ws[(size_t)b * L + x];
    base[x] = t;
  }
  __syncthreads();
  const int total = block_exclusive_scan(base, L, warp_tot);
  for (int x = tid; x < L; x += kThreads) {
    m_indptr[x] = base[x];
    int run = base[x];
    for (int b = 0; b < nblk; ++b) {
      const int c = ws[(size_t)b * L + x];
      ws[(size_t)b * L + x] = run;
      run += c;
    }
  }
  if (tid == 0) m_indptr[L] = total;
  pdl_launch_dependents();
}

__global__ void __launch_bounds__(kThreads, 1)
    sort_scatter_kernel(const int32_t *__restrict__ ids, long R, int off, int L,
                        const int32_t *__restrict__ ws, int32_t *__restrict__ p2e,
                        int32_t *__restrict__ e2p) {
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_wait();
  const ScatterSmem s = carve(smem, L);
  for (int x = threadIdx.x; x < L; x += kThreads) s.cur[x] = ws[(size_t)blockIdx.x * L + x];
  __syncthreads();
  pdl_launch_dependents();
  const long r_begin = (long)blockIdx.x * kSortChunk;
  const long r_end = min(R, r_begin + kSortChunk);
  for (long r0 = r_begin; r0 < r_end; r0 += kThreads) scatter_round(ids, r0, r_end, off, L, s, p2e, e2p);
}

template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return raise_smem_limit(kernel, bytes);
}

}  // namespace

size_t sort_workspace_bytes(long routes, int L) {
  if (routes <= kSortSingleMax) return 0;
  const long nblk = (routes + kSortChunk - 1) / kSortChunk;
  return (size_t)nblk * (size_t)L * sizeof(int32_t);
}

cudaError_t launch_sort(const int32_t *ids, long routes, int E, int off, int L, int32_t *m_indptr,
                        int32_t *p2e, int32_t *e2p, int32_t *ws, int32_t *status,
                        const Launch &l) {
  const size_t sbytes = scatter_smem_bytes(L);
  cudaError_t err;
  if (routes <= kSortSingleMax) {
    if ((err = allow_smem(sort_single_kernel, sbytes)) != cudaSuccess) return err;
    return launch_kernel(sort_single_kernel, dim3(1), dim3(kThreads), sbytes, l, ids, (int)routes,
                         E, off, L, m_indptr, p2e, e2p, status);
  }
  const int nblk = (int)((routes + kSortChunk - 1) / kSortChunk);
  const size_t hbytes = (size_t)L * sizeof(int);
  if ((err = allow_smem(sort_scatter_kernel, sbytes)) != cudaSuccess) return err;
  if ((err = launch_kernel(sort_hist_kernel, dim3(nblk), dim3(kThreads), hbytes, l, ids, routes, E,
                           off, L, ws, status)) != cudaSuccess)
    return err;
  Launch chained = l;
  chained.pdl = true;
  if ((err = launch_kernel(sort_scan_kernel, dim3(1), dim3(kThreads), hbytes, chained, nblk, L, ws,
                           m_indptr)) != cudaSuccess)
    return err;
  return launch_kernel(sort_scatter_kernel, dim3(nblk), dim3(kThreads), sbytes, chained, ids,
                       routes, off, L, (const int32_t *)ws, p2e, e2p);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free sort for callers that cannot allocate device memory.
//
// The multi-CTA sort needs a per-(chunk, expert) table in device memory.
// moe_sort takes it from the caller's workspace; this variant keeps it in a
// fixed array in the library's own device memory instead, so the caller passes
// only inputs and outputs.  The array is kStaticSortScratchInts int32 (1 MiB)
// and exists on every device that loads the library until the process exits.
// Its address is looked up with the device current on every call outside
// stream capture (the first call on a device must come before any capture).
// Every call shares the array; the kernels write every entry they later read,
// so nothing has to be cleared between calls, but two calls whose kernels
// overlap on the GPU race on it.
#include <mutex>

namespace moe {
namespace {
constexpr long kStaticSortScratchInts = 1L << 18;
__device__ __align__(256) int32_t g_sort_scratch[kStaticSortScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
int32_t *g_scratch_addr[kMaxDevices] = {};
}  // namespace

long static_sort_scratch_ints() { return kStaticSortScratchInts; }

// Device address of the scratch array on the current device (host code must
// not pass the symbol itself: on the host it is only a stand-in).  Outside
// stream capture the address is looked up on every call, so a context that was
// destroyed and created again (cudaDeviceReset) never leaves a stale address
// behind; during capture, where a first lookup could load the module, the
// address of the last lookup on this device is used (the header asks for a
// first call before any capture).
cudaError_t static_sort_scratch(cudaStream_t stream, int32_t **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_sort_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<int32_t *>(p);
  } else if (!g_scratch_addr[dev]) {
    return cudaErrorStreamCaptureUnsupported;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace moe
