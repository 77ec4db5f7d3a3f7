// The C ABI (include/moe_gb300.h): argument checks, workspace layout, the
// prepared launch and the one-shot entry points.  Host code only; every step
// of the layer runs in the kernels of route.cu, sort.cu, rows.cu and gemm.cu.
#include <cstdlib>
#include <cstring>
#include <new>

#include "internal.h"
#include "moe_gb300.h"

namespace moe {

int device_sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
  }
  return n;
}

namespace {

// The kernels are built for sm_103a only.
int check_device() {
  static int cached = 1;  // 1 = unknown
  if (cached == 1) {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_DEVICE;
    }
    cached = (major == 10 && minor == 3) ? MOE_OK : MOE_ERR_DEVICE;
  }
  return cached;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct WsLayout {
  size_t ids, w, m_indptr, p2e, e2p, sort_ws, xp, h, y, comb, done1, sched, total;
};

// Claim counters of the two grouped GEMMs when the small-group kernel runs
// beside the CTA-pair kernel (four per GEMM), zeroed at the start of every launch.
constexpr int kSchedInts = 8;

WsLayout ws_layout(long T, int H, int I, int k, int L) {
  WsLayout o;
  const size_t R = (size_t)T * (size_t)k;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return at;
  };
  o.ids = take(R * 4);
  o.w = take(R * 4);
  o.m_indptr = take(((size_t)L + 1) * 4);
  o.p2e = take(R * 4);
  o.e2p = take(R * 4);
  o.sort_ws = take(sort_workspace_bytes((long)R, L));
  o.xp = take(R * (size_t)H * 2);
  o.h = take(R * (size_t)I * 2);
  o.y = take(R * (size_t)H * 4);
  o.comb = take(chain_comb_ints((int)T, H) * 4);
  o.done1 = take(((size_t)L + 1) * 4);
  o.sched = take(kSchedInts * 4);
  o.total = off;
  return o;
}

int check_layer_shape(int T, int H, int I, int E, int k, int off, int L) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || E > MOE_MAX_EXPERTS) return MOE_ERR_SHAPE;
  if (k < 1 || k > MOE_MAX_TOP_K || k > E) return MOE_ERR_SHAPE;
  if (off < 0 || L < 1 || (long)off + L > E) return MOE_ERR_SHAPE;
  if (H % 64 != 0 || I % 64 != 0) return MOE_ERR_SHAPE;
  if ((long)T * k > (1L << 30)) return MOE_ERR_SHAPE;
  return MOE_OK;
}

enum Stage { kRoute = 0, kSort, kGather, kFc1, kFc2, kFinalize, kNumStages };
const char *kStageNames[kNumStages] = {"route", "sort", "gather", "fc1_swiglu", "fc2", "finalize"};
constexpr int kTimingRing = 512;
// Token count up to which MOE_PATH_AUTO picks the weight-streaming decode path.
constexpr int kDecodeMaxTokens = 64;
// Small-group kernel beside the CTA-pair GEMMs: the CTAs it takes, and the
// routes per local expert up to which a plan uses it without a flag (above,
// groups of at most 64 rows are rare).  With 24 CTAs streaming weights at
// about 100 GB/s each, the small groups of the Zipf-routed 256-expert
// workload end about when the pair kernel's tiles do; claims at run time
// even out any other mix.
constexpr int kSmallGroupCtas = 24;
constexpr long kSmallGroupMeanRows = 512;

}  // namespace
}  // namespace moe

using namespace moe;

struct moe_plan {
  moe_forward_desc d;
  int path;
  bool logits_mode;
  long R;
  int32_t *ids;
  float *w;
  int32_t *m_indptr, *p2e, *e2p, *sort_ws;
  uint16_t *xp, *h;
  float *y;
  GemmPlan fc1, fc2;
  SwapPlan fc1d, fc2d;  // decode path, separate kernels
  ChainPlan chain;      // decode path: the chain (one launch or two kernels)
  bool use_chain;
  bool unreachable_wait;  // test hook MOE_PLAN_TEST_UNREACHABLE_WAIT
  bool fused_gather;    // grouped path: FC1 gathers its rows itself
  bool e4m3;            // E4M3 weight family (one-CTA kernels, quantising gather)
  int32_t *sched;       // grouped path beside the small-group kernel: claim counters (else null)
  bool timing;
  cudaEvent_t (*ev)[kNumStages + 1];
  long n_recorded;
};

extern "C" {

const char *moe_status_string(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "a required pointer is NULL";
    case MOE_ERR_SHAPE: return "a size is out of range or not a supported multiple";
    case MOE_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_MODE: return "give logits, or topk_ids with topk_w, not both or neither";
    case MOE_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case MOE_ERR_DEVICE: return "no CUDA device, or the device is not sm_103 (GB300/B300)";
    case MOE_ERR_TENSOR_MAP: return "the driver rejected a TMA tensor map";
    case MOE_ERR_STATE: return "call not valid for this plan";
    default: return "unknown status code";
  }
}

int moe_abi_version(void) { return 104; }

int moe_route(const float *logits, int T, int E, int top_k, int32_t *topk_ids, float *topk_w,
              void *stream) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || top_k < 1 || top_k > MOE_MAX_TOP_K || top_k > E)
    return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_NULL;
  if (int rc = check_device()) return rc;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_route(logits, T, E, top_k, topk_ids, topk_w, l));
}

size_t moe_sort_workspace_size(int T, int top_k, int num_local) {
  if (T < 0 || top_k < 1 || num_local < 1) return 0;
  return sort_workspace_bytes((long)T * top_k, num_local);
}

int moe_sort(const int32_t *topk_ids, int T, int top_k, int E, int local_offset, int num_local,
             int32_t *m_indptr, int32_t *perm_to_exp, int32_t *exp_to_perm, void *workspace,
             size_t workspace_bytes, int32_t *status, void *stream) {
  if (T < 0 || top_k < 1 || top_k > MOE_MAX_TOP_K || E < 1 || E > MOE_MAX_EXPERTS ||
      local_offset < 0 || num_local < 1 || (long)local_offset + num_local > E ||
      (long)T * top_k > (1L << 30))
    return MOE_ERR_SHAPE;
  if (!m_indptr) return MOE_ERR_NULL;
  if (int rc = check_device()) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  const long R = (long)T * top_k;
  if (R == 0) return cuda_rc(cudaMemsetAsync(m_indptr, 0, ((size_t)num_local + 1) * 4, s));
  if (!topk_ids || !perm_to_exp || !exp_to_perm) return MOE_ERR_NULL;
  const size_t need = sort_workspace_bytes(R, num_local);
  if (need > 0 && (!workspace || workspace_bytes < need)) return MOE_ERR_WORKSPACE;
  Launch l;
  l.stream = s;
  return cuda_rc(launch_sort(topk_ids, R, E, local_offset, num_local, m_indptr, perm_to_exp,
                             exp_to_perm, static_cast<int32_t *>(workspace), status, l));
}

int moe_sort_no_alloc(const int32_t *topk_ids, int T, int top_k, int E, int local_offset,
                      int num_local, int32_t *m_indptr, int32_t *perm_to_exp,
                      int32_t *exp_to_perm, int32_t *status, void *stream) {
  if (T < 0 || top_k < 1 || top_k > MOE_MAX_TOP_K || E < 1 || E > MOE_MAX_EXPERTS ||
      local_offset < 0 || num_local < 1 || (long)local_offset + num_local > E ||
      (long)T * top_k > (1L << 30))
    return MOE_ERR_SHAPE;
  const long R = (long)T * top_k;
  const size_t need = sort_workspace_bytes(R, num_local) / sizeof(int32_t);
  if ((long)need > static_sort_scratch_ints()) return MOE_ERR_WORKSPACE;
  if (!m_indptr) return MOE_ERR_NULL;
  if (R > 0 && (!topk_ids || !perm_to_exp || !exp_to_perm)) return MOE_ERR_NULL;
  if (int rc = check_device()) return rc;
  int32_t *scratch = nullptr;
  if (need > 0 && static_sort_scratch(static_cast<cudaStream_t>(stream), &scratch) != cudaSuccess)
    return MOE_ERR_CUDA;
  return moe_sort(topk_ids, T, top_k, E, local_offset, num_local, m_indptr, perm_to_exp,
                  exp_to_perm, scratch, need * sizeof(int32_t), status, stream);
}

int moe_gather(const moe_bf16 *x, const int32_t *perm_to_exp, const int32_t *m_indptr, int T,
               int H, int top_k, int num_local, moe_bf16 *xp, void *stream) {
  if (T < 0 || H <= 0 || H % 8 != 0 || top_k < 1 || top_k > MOE_MAX_TOP_K || num_local < 1)
    return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!x || !perm_to_exp || !m_indptr || !xp) return MOE_ERR_NULL;
  if (!aligned16(x) || !aligned16(xp)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_gather(x, perm_to_exp, m_indptr + num_local, H, top_k, (long)T * top_k, xp, l));
}

int moe_fc1_swiglu(const moe_bf16 *xp, const moe_bf16 *w1, const int32_t *m_indptr, int max_rows,
                   int H, int I, int num_local, moe_bf16 *h, void *stream) {
  if (max_rows < 0 || H <= 0 || I <= 0 || H % 64 || I % 64 || num_local < 1 ||
      num_local > MOE_MAX_EXPERTS)
    return MOE_ERR_SHAPE;
  if (max_rows == 0) return MOE_OK;
  if (!xp || !w1 || !m_indptr || !h) return MOE_ERR_NULL;
  if (!aligned16(xp) || !aligned16(w1) || !aligned16(h)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  GemmPlan p;
  if (int rc = gemm_prepare(p, Epi::kSwiGLU, xp, max_rows, w1, num_local, 2 * I, H, I,
                            m_indptr + 1, max_rows, h, nullptr))
    return rc;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_gemm(p, l));
}

int moe_fc1_swiglu_step(const moe_bf16 *xp, const moe_bf16 *w1, const float *clamp_limit,
                        const int32_t *m_indptr, int max_rows, int H, int I, int num_local, moe_bf16 *h,
                        void *stream) {
  if (max_rows < 0 || H <= 0 || I <= 0 || H % 64 || I % 64 || num_local < 1 ||
      num_local > MOE_MAX_EXPERTS)
    return MOE_ERR_SHAPE;
  if (max_rows == 0) return MOE_OK;
  if (!xp || !w1 || !clamp_limit || !m_indptr || !h) return MOE_ERR_NULL;
  if (!aligned16(xp) || !aligned16(w1) || !aligned16(h)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  GemmPlan p;
  if (int rc = gemm_prepare(p, Epi::kSwiGLU, xp, max_rows, w1, num_local, 2 * I, H, I,
                            m_indptr + 1, max_rows, h, nullptr))
    return rc;
  p.clamp = clamp_limit;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_gemm(p, l));
}

int moe_fc1_swiglu_e4m3(const uint8_t *xq, const uint8_t *w1q, const float *w1_scale, float x_scale,
                        float h_scale, const float *clamp_limit, const int32_t *m_indptr, int max_rows,
                        int H, int I, int num_local, uint8_t *hq, void *stream) {
  if (max_rows < 0 || H <= 0 || I <= 0 || H % 128 || I % 128 || num_local < 1 ||
      num_local > MOE_MAX_EXPERTS || !(x_scale > 0.f) || !(h_scale > 0.f))
    return MOE_ERR_SHAPE;
  if (max_rows == 0) return MOE_OK;
  if (!xq || !w1q || !w1_scale || !m_indptr || !hq) return MOE_ERR_NULL;
  if (!aligned16(xq) || !aligned16(w1q) || !aligned16(hq)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  GemmPlan p;
  if (int rc = gemm_prepare_e4m3(p, Epi::kSwiGLU, xq, max_rows, w1q, num_local, 2 * I, H, I, m_indptr + 1,
                                 max_rows, hq, nullptr))
    return rc;
  p.clamp = clamp_limit;
  p.wscale = w1_scale;
  p.ascale = x_scale;
  p.oscale = h_scale;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_gemm(p, l));
}

int moe_fc2_e4m3(const uint8_t *hq, const uint8_t *w2q, const float *w2_scale, float h_scale,
                 const int32_t *m_indptr, int max_rows, int H, int I, int num_local, float *y,
                 void *stream) {
  if (max_rows < 0 || H <= 0 || I <= 0 || H % 128 || I % 128 || num_local < 1 ||
      num_local > MOE_MAX_EXPERTS || !(h_scale > 0.f))
    return MOE_ERR_SHAPE;
  if (max_rows == 0) return MOE_OK;
  if (!hq || !w2q || !w2_scale || !m_indptr || !y) return MOE_ERR_NULL;
  if (!aligned16(hq) || !aligned16(w2q) || !aligned16(y)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  GemmPlan p;
  if (int rc = gemm_prepare_e4m3(p, Epi::kF32, hq, max_rows, w2q, num_local, H, I, H, m_indptr + 1,
                                 max_rows, y, nullptr))
    return rc;
  p.wscale = w2_scale;
  p.ascale = h_scale;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_gemm(p, l));
}

int moe_fc2(const moe_bf16 *h, const moe_bf16 *w2, const int32_t *m_indptr, int max_rows, int H,
            int I, int num_local, float *y, void *stream) {
  if (max_rows < 0 || H <= 0 || I <= 0 || H % 64 || I % 64 || num_local < 1 ||
      num_local > MOE_MAX_EXPERTS)
    return MOE_ERR_SHAPE;
  if (max_rows == 0) return MOE_OK;
  if (!h || !w2 || !m_indptr || !y) return MOE_ERR_NULL;
  if (!aligned16(h) || !aligned16(w2) || !aligned16(y)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  GemmPlan p;
  if (int rc = gemm_prepare(p, Epi::kF32, h, max_rows, w2, num_local, H, I, H, m_indptr + 1,
                            max_rows, y, nullptr))
    return rc;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_gemm(p, l));
}

int moe_fc1_swiglu_gathered(const moe_bf16 *x, const int32_t *perm_to_exp,
                            const int32_t *m_indptr, int T, int top_k, const moe_bf16 *w1, int H,
                            int I, int num_local, moe_bf16 *h, void *stream) {
  if (T < 0 || top_k < 1 || top_k > MOE_MAX_TOP_K || H <= 0 || H % 64 || I <= 0 || I % 128 ||
      num_local < 1 || num_local > MOE_MAX_EXPERTS)
    return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!x || !perm_to_exp || !m_indptr || !w1 || !h) return MOE_ERR_NULL;
  if (!aligned16(x) || !aligned16(w1) || !aligned16(h)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  GemmPlan p;
  const long R = (long)T * top_k;
  if (int rc = gemm_prepare_gather(p, x, T, perm_to_exp, top_k, w1, num_local, I, H, m_indptr + 1,
                                   R, h, nullptr))
    return rc;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_gemm(p, l));
}

int moe_fc1_swiglu_swapab(const moe_bf16 *xp, const moe_bf16 *w1, const int32_t *m_indptr,
                          int max_rows, int max_group_rows, int H, int I, int num_local,
                          moe_bf16 *h, void *stream) {
  if (max_rows < 0 || max_group_rows < 1 || H <= 0 || I <= 0 || H % 64 || I % 64 ||
      num_local < 1 || num_local > MOE_MAX_EXPERTS)
    return MOE_ERR_SHAPE;
  if (max_rows == 0) return MOE_OK;
  if (!xp || !w1 || !m_indptr || !h) return MOE_ERR_NULL;
  if (!aligned16(xp) || !aligned16(w1) || !aligned16(h)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  SwapPlan p;
  if (int rc = swap_prepare(p, true, w1, num_local, 2 * I, H, xp, max_rows, I, m_indptr + 1,
                            max_group_rows, h, nullptr, false))
    return rc;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_swap(p, l));
}

int moe_fc2_swapab(const moe_bf16 *h, const moe_bf16 *w2, const int32_t *m_indptr, int max_rows,
                   int max_group_rows, int H, int I, int num_local, float *y, void *stream) {
  if (max_rows < 0 || max_group_rows < 1 || H <= 0 || I <= 0 || H % 64 || I % 64 ||
      num_local < 1 || num_local > MOE_MAX_EXPERTS)
    return MOE_ERR_SHAPE;
  if (max_rows == 0) return MOE_OK;
  if (!h || !w2 || !m_indptr || !y) return MOE_ERR_NULL;
  if (!aligned16(h) || !aligned16(w2) || !aligned16(y)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  SwapPlan p;
  if (int rc = swap_prepare(p, false, w2, num_local, H, I, h, max_rows, H, m_indptr + 1,
                            max_group_rows, y, nullptr, false))
    return rc;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_swap(p, l));
}

int moe_finalize(const float *y, const int32_t *exp_to_perm, const float *topk_w, int T,
                 int top_k, int H, moe_bf16 *out, void *stream) {
  if (T < 0 || H <= 0 || H % 8 != 0 || top_k < 1 || top_k > MOE_MAX_TOP_K) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!y || !exp_to_perm || !topk_w || !out) return MOE_ERR_NULL;
  if (!aligned16(y) || !aligned16(out)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_finalize(y, exp_to_perm, topk_w, T, top_k, H, out, l));
}

int grouped_gemm_fwd_ex(const moe_bf16 *X, const moe_bf16 *W, const int32_t *offs, int sum_m, int E, int N,
                        int K, moe_bf16 *Y, int flags, int32_t *counters, void *stream) {
  if (sum_m < 0 || E < 1 || E > MOE_MAX_EXPERTS || N <= 0 || K <= 0 || N % 64 || K % 64)
    return MOE_ERR_SHAPE;
  if (sum_m == 0) return MOE_OK;
  if (!X || !W || !offs || !Y) return MOE_ERR_NULL;
  if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || !aligned16(counters)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  GemmPlan p;
  if (int rc = gemm_prepare(p, Epi::kBf16, X, sum_m, W, E, N, K, N, offs, sum_m, Y, nullptr))
    return rc;
  if (flags & MOE_PLAN_NO_TAIL_TILES) p.tail_max = 0;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  // The small-group kernel beside the pair kernel, on the caller's counters.
  if (counters && p.pair && p.tail_max >= small_gemm_max_rows()) {
    const int ctas = device_sm_count() >= 4 * kSmallGroupCtas ? kSmallGroupCtas : 2;
    if (int rc = gemm_attach_small(p, counters, ctas)) return rc;
    if (cudaMemsetAsync(counters, 0, MOE_GROUPED_GEMM_COUNTERS * sizeof(int32_t), l.stream) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return cuda_rc(launch_gemm(p, l));
}

int grouped_gemm_fwd_flags(const moe_bf16 *X, const moe_bf16 *W, const int32_t *offs, int sum_m, int E,
                           int N, int K, moe_bf16 *Y, int flags, void *stream) {
  return grouped_gemm_fwd_ex(X, W, offs, sum_m, E, N, K, Y, flags, nullptr, stream);
}

int grouped_gemm_fwd(const moe_bf16 *X, const moe_bf16 *W, const int32_t *offs, int sum_m, int E, int N,
                     int K, moe_bf16 *Y, void *stream) {
  return grouped_gemm_fwd_flags(X, W, offs, sum_m, E, N, K, Y, 0, stream);
}

int grouped_gemm_dgrad(const moe_bf16 *G, const moe_bf16 *W, const int32_t *offs, int sum_m, int E,
                       int N, int K, moe_bf16 *dX, void *stream) {
  if (sum_m < 0 || E < 1 || E > MOE_MAX_EXPERTS || N <= 0 || K <= 0 || N % 64 || K % 64)
    return MOE_ERR_SHAPE;
  if (sum_m == 0) return MOE_OK;
  if (!G || !W || !offs || !dX) return MOE_ERR_NULL;
  if (!aligned16(G) || !aligned16(W) || !aligned16(dX)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  BwdPlan p;
  if (int rc = bwd_prepare(p, false, false, G, W, offs, sum_m, E, N, K, dX, nullptr)) return rc;
  Launch l;
  l.stream = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_bwd(p, l));
}

int grouped_gemm_wgrad(const moe_bf16 *G, const moe_bf16 *X, const int32_t *offs, int sum_m, int E,
                       int N, int K, void *dW, int dw_fp32, void *stream) {
  if (sum_m < 0 || E < 1 || E > MOE_MAX_EXPERTS || N <= 0 || K <= 0 || N % 64 || K % 64)
    return MOE_ERR_SHAPE;
  if (!dW) return MOE_ERR_NULL;
  if (!aligned16(dW)) return MOE_ERR_ALIGN;
  if (int rc = check_device()) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (sum_m == 0)  // every group is empty: dW is exactly zero
    return cuda_rc(cudaMemsetAsync(dW, 0, (size_t)E * N * K * (dw_fp32 ? 4 : 2), s));
  if (!G || !X || !offs) return MOE_ERR_NULL;
  if (!aligned16(G) || !aligned16(X)) return MOE_ERR_ALIGN;
  BwdPlan p;
  if (int rc = bwd_prepare(p, true, dw_fp32 != 0, G, X, offs, sum_m, E, N, K, dW, nullptr)) return rc;
  Launch l;
  l.stream = s;
  return cuda_rc(launch_bwd(p, l));
}

size_t moe_bgmv_workspace_size(int T, int num_pairs, int contiguous_top_k, int num_loras, int E,
                               int total_feat_out) {
  if (T < 0 || num_pairs < 0 || contiguous_top_k < 0 || num_loras < 1 || E < 1 || total_feat_out < 0) return 0;
  return bgmv_workspace_bytes(T, num_pairs, contiguous_top_k, num_loras, E, total_feat_out);
}

int moe_bgmv(const moe_bf16 *x, int T, int H, const moe_bf16 *const *lora_a,
             const moe_bf16 *const *lora_b, int num_slices, const int *feat_out, int rank,
             int num_loras, int E, const int32_t *sorted_token_ids, const int32_t *expert_ids,
             const int32_t *lora_indices, const float *topk_weights, int num_pairs,
             int contiguous_top_k, moe_bf16 *shrink_out, float *y_accum, int ld_y,
             void *workspace, size_t workspace_bytes, int32_t *status, void *stream) {
  if (T < 0 || H <= 0 || H % 8 || num_slices < 1 || num_slices > kBgmvMaxSlices || num_loras < 1 ||
      E < 1 || num_pairs < 0 || contiguous_top_k < 0 || contiguous_top_k > MOE_MAX_TOP_K)
    return MOE_ERR_SHAPE;
  if (rank != 8 && rank != 16 && rank != 32 && rank != 64) return MOE_ERR_SHAPE;
  if (contiguous_top_k > 0 && (long)T * contiguous_top_k != num_pairs) return MOE_ERR_SHAPE;
  if (!lora_a || !lora_b || !feat_out) return MOE_ERR_NULL;
  long cols = 0;
  for (int s = 0; s < num_slices; ++s) {
    if (feat_out[s] <= 0 || feat_out[s] % 8) return MOE_ERR_SHAPE;
    cols += feat_out[s];
  }
  if (ld_y < cols) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!x || !y_accum || (num_pairs > 0 && (!sorted_token_ids || !expert_ids || !lora_indices ||
                                           !topk_weights || !shrink_out)))
    return MOE_ERR_NULL;
  for (int s = 0; s < num_slices; ++s) {
    if (!lora_a[s] || !lora_b[s]) return MOE_ERR_NULL;
    if (!aligned16(lora_a[s]) || !aligned16(lora_b[s])) return MOE_ERR_ALIGN;
  }
  if (!aligned16(x)) return MOE_ERR_ALIGN;
  const size_t need = bgmv_workspace_bytes(T, num_pairs, contiguous_top_k, num_loras, E, (int)cols);
  if (need > 0 && (!workspace || workspace_bytes < need)) return MOE_ERR_WORKSPACE;
  if (int rc = check_device()) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  BgmvPlan p;
  p.x = x;
  int off = 0;
  for (int i = 0; i < num_slices; ++i) {
    p.a[i] = lora_a[i];
    p.b[i] = lora_b[i];
    p.f[i] = feat_out[i];
    p.off[i] = off;
    off += feat_out[i];
  }
  p.tok = sorted_token_ids;
  p.eid = expert_ids;
  p.lora = lora_indices;
  p.w = topk_weights;
  p.shrink = shrink_out;
  p.y = y_accum;
  p.ws = static_cast<int32_t *>(workspace);
  p.status = status;
  p.T = T;
  p.H = H;
  p.R = rank;
  p.S = num_slices;
  p.L = num_loras;
  p.E = E;
  p.P = num_pairs;
  p.k = contiguous_top_k;
  p.ld_y = ld_y;
  Launch l;
  l.stream = s;
  l.pdl = true;
  return cuda_rc(launch_bgmv(p, l));
}

size_t moe_workspace_size(int T, int H, int I, int E, int top_k, int num_local) {
  if (check_layer_shape(T, H, I, E, top_k, 0, num_local) != MOE_OK) return 0;
  return ws_layout(T, H, I, top_k, num_local).total;
}

int moe_forward_prepare(const moe_forward_desc *desc, moe_plan **plan_out) {
  if (!desc || !plan_out) return MOE_ERR_NULL;
  *plan_out = nullptr;
  const moe_forward_desc &d = *desc;
  if (int rc = check_layer_shape(d.T, d.H, d.I, d.E, d.top_k, d.local_offset, d.num_local))
    return rc;
  const bool logits_mode = d.logits != nullptr;
  const bool routed_mode = d.topk_ids != nullptr || d.topk_w != nullptr;
  // With no tokens there is nothing to route (empty tensors may carry NULL).
  if (d.T > 0) {
    if (logits_mode == routed_mode) return MOE_ERR_MODE;
    if (routed_mode && (!d.topk_ids || !d.topk_w)) return MOE_ERR_MODE;
  }
  if (d.path < MOE_PATH_AUTO || d.path > MOE_PATH_DECODE) return MOE_ERR_SHAPE;
  if (d.weight_format != MOE_WEIGHTS_BF16 && d.weight_format != MOE_WEIGHTS_E4M3) return MOE_ERR_SHAPE;
  const bool e4m3 = d.weight_format == MOE_WEIGHTS_E4M3;
  if (e4m3) {
    if (d.H % 128 || d.I % 128 || d.path == MOE_PATH_DECODE) return MOE_ERR_SHAPE;
    if (!(d.x_scale > 0.f) || !(d.h_scale > 0.f)) return MOE_ERR_SHAPE;
    if (d.T > 0 && (!d.w1_scale || !d.w2_scale)) return MOE_ERR_NULL;
  }
  if (d.T > 0) {
    if (!d.x || !d.w1 || !d.w2 || !d.out) return MOE_ERR_NULL;
    if (!aligned16(d.x) || !aligned16(d.w1) || !aligned16(d.w2) || !aligned16(d.out))
      return MOE_ERR_ALIGN;
  }
  const WsLayout lay = ws_layout(d.T, d.H, d.I, d.top_k, d.num_local);
  if (d.T > 0) {
    if (!d.workspace || d.workspace_bytes < lay.total) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(d.workspace) & 255u) != 0) return MOE_ERR_ALIGN;
    if (int rc = check_device()) return rc;
  }
  moe_plan *p = new (std::nothrow) moe_plan();
  if (!p) return MOE_ERR_CUDA;
  p->d = d;
  p->logits_mode = logits_mode;
  // Few tokens: each expert gets at most a few rows, the layer streams weights.
  p->path = d.path != MOE_PATH_AUTO ? d.path : (d.T <= kDecodeMaxTokens ? MOE_PATH_DECODE : MOE_PATH_GROUPED);
  p->e4m3 = e4m3;
  if (e4m3) p->path = MOE_PATH_GROUPED;
  p->R = (long)d.T * d.top_k;
  unsigned char *ws = static_cast<unsigned char *>(d.workspace);
  if (d.T > 0) {
    p->ids = logits_mode ? reinterpret_cast<int32_t *>(ws + lay.ids) : const_cast<int32_t *>(d.topk_ids);
    p->w = logits_mode ? reinterpret_cast<float *>(ws + lay.w) : const_cast<float *>(d.topk_w);
    p->m_indptr = reinterpret_cast<int32_t *>(ws + lay.m_indptr);
    p->p2e = reinterpret_cast<int32_t *>(ws + lay.p2e);
    p->e2p = reinterpret_cast<int32_t *>(ws + lay.e2p);
    p->sort_ws = reinterpret_cast<int32_t *>(ws + lay.sort_ws);
    p->xp = reinterpret_cast<uint16_t *>(ws + lay.xp);
    p->h = reinterpret_cast<uint16_t *>(ws + lay.h);
    p->y = reinterpret_cast<float *>(ws + lay.y);
    int rc;
    // Decode: the chain saves launches but gathers its token rows and
    // combines inside the GEMM kernels; it is the faster form only for few
    // routes, so without a flag it runs, as one launch, up to kChainAutoRoutes
    // routes.  MOE_PLAN_DECODE_CHAIN alone asks for its two-kernel form.
    const bool force_chain = (d.flags & (MOE_PLAN_DECODE_CHAIN | MOE_PLAN_DECODE_ONE_LAUNCH)) != 0;
    const bool auto_chain = (d.flags & MOE_PLAN_DECODE_SEPARATE) == 0 && p->R <= kChainAutoRoutes &&
                            d.H % 64 == 0 && d.I % 64 == 0;
    p->use_chain = p->path == MOE_PATH_DECODE && p->R <= kChainMaxRoutes && (force_chain || auto_chain);
    if (p->use_chain) {
      ChainPlan &c = p->chain;
      c.x = d.x;
      c.w1 = d.w1;
      c.w2 = d.w2;
      c.ids = p->ids;
      c.w = p->w;
      c.h = p->h;
      c.y = p->y;
      c.out = d.out;
      c.comb = reinterpret_cast<int32_t *>(ws + lay.comb);
      c.done1 = reinterpret_cast<int32_t *>(ws + lay.done1);
      c.one_launch = (d.flags & MOE_PLAN_DECODE_ONE_LAUNCH) != 0 || !force_chain;
      c.m_indptr = p->m_indptr;
      c.p2e = p->p2e;
      c.e2p = p->e2p;
      c.status = d.status;
      c.T = d.T;
      c.k = d.top_k;
      c.E = d.E;
      c.off = d.local_offset;
      c.L = d.num_local;
      c.H = d.H;
      c.I = d.I;
      c.ids_early = !logits_mode;
      c.clamp = d.clamp_limit;
      rc = chain_prepare(c);
    } else if (p->path == MOE_PATH_DECODE) {
      rc = swap_prepare(p->fc1d, true, d.w1, d.num_local, 2 * d.I, d.H, p->xp, p->R, d.I,
                        p->m_indptr + 1, d.T, p->h, d.status, true);
      p->fc1d.clamp = d.clamp_limit;
      if (rc == MOE_OK)
        rc = swap_prepare(p->fc2d, false, d.w2, d.num_local, d.H, d.I, p->h, p->R, d.H,
                          p->m_indptr + 1, d.T, p->y, d.status, true);
    } else if (e4m3) {
      uint8_t *xq = reinterpret_cast<uint8_t *>(p->xp), *hq = reinterpret_cast<uint8_t *>(p->h);
      const bool pair = (d.flags & MOE_PLAN_ONE_CTA_GEMM) == 0;
      rc = gemm_prepare_e4m3(p->fc1, Epi::kSwiGLU, xq, p->R, static_cast<const uint8_t *>(static_cast<const void *>(d.w1)),
                             d.num_local, 2 * d.I, d.H, d.I, p->m_indptr + 1, p->R, hq, d.status, pair);
      p->fc1.clamp = d.clamp_limit;
      p->fc1.wscale = d.w1_scale;
      p->fc1.ascale = d.x_scale;
      p->fc1.oscale = d.h_scale;
      if (rc == MOE_OK) {
        rc = gemm_prepare_e4m3(p->fc2, Epi::kF32, hq, p->R, static_cast<const uint8_t *>(static_cast<const void *>(d.w2)),
                               d.num_local, d.H, d.I, d.H, p->m_indptr + 1, p->R, p->y, d.status, pair);
        p->fc2.wscale = d.w2_scale;
        p->fc2.ascale = d.h_scale;
      }
      if (d.flags & MOE_PLAN_NO_TAIL_TILES) p->fc1.tail_max = p->fc2.tail_max = 0;
    } else {
      const bool pair = (d.flags & MOE_PLAN_ONE_CTA_GEMM) == 0;
      // Either the gather kernel builds xp (one 128-row TMA box per k-block
      // feeds the tensor cores) or FC1's gather warps copy the rows from x.
      p->fused_gather = pair && (d.flags & MOE_PLAN_FUSED_GATHER) != 0 &&
                        pair_gemm_supported(Epi::kSwiGLU, d.I);
      if (p->fused_gather)
        rc = gemm_prepare_gather(p->fc1, d.x, d.T, p->p2e, d.top_k, d.w1, d.num_local, d.I, d.H,
                                 p->m_indptr + 1, p->R, p->h, d.status);
      else
        rc = gemm_prepare(p->fc1, Epi::kSwiGLU, p->xp, p->R, d.w1, d.num_local, 2 * d.I, d.H, d.I,
                          p->m_indptr + 1, p->R, p->h, d.status, pair);
      p->fc1.clamp = d.clamp_limit;
      if (rc == MOE_OK)
        rc = gemm_prepare(p->fc2, Epi::kF32, p->h, p->R, d.w2, d.num_local, d.H, d.I, d.H,
                          p->m_indptr + 1, p->R, p->y, d.status, pair);
      if (d.flags & MOE_PLAN_NO_TAIL_TILES) p->fc1.tail_max = p->fc2.tail_max = 0;
    }
    if (rc == MOE_OK && p->path == MOE_PATH_GROUPED && !p->fused_gather && p->fc1.pair &&
        p->fc2.pair && (d.flags & MOE_PLAN_NO_SMALL_GROUP_KERNEL) == 0 &&
        ((d.flags & MOE_PLAN_SMALL_GROUP_KERNEL) != 0 || p->R <= kSmallGroupMeanRows * d.num_local) &&
        p->fc1.tail_max >= small_gemm_max_rows()) {
      const int ctas = device_sm_count() >= 4 * kSmallGroupCtas ? kSmallGroupCtas : 2;
      int32_t *sched = reinterpret_cast<int32_t *>(ws + lay.sched);
      rc = gemm_attach_small(p->fc1, sched, ctas);
      if (rc == MOE_OK) rc = gemm_attach_small(p->fc2, sched + 4, ctas);
      if (rc == MOE_OK) p->sched = sched;
    }
    if (rc != MOE_OK) {
      delete p;
      return rc;
    }
  }
  p->unreachable_wait = (d.flags & MOE_PLAN_TEST_UNREACHABLE_WAIT) != 0;
  p->timing = (d.flags & MOE_PLAN_STAGE_TIMING) != 0 && d.T > 0;
  if (p->timing) {
    p->ev = new (std::nothrow) cudaEvent_t[kTimingRing][kNumStages + 1];
    if (!p->ev) {
      delete p;
      return MOE_ERR_CUDA;
    }
    for (int i = 0; i < kTimingRing; ++i)
      for (int s = 0; s <= kNumStages; ++s)
        if (cudaEventCreate(&p->ev[i][s]) != cudaSuccess) {
          // leave the plan consistent for destroy
          for (int j = 0; j <= i; ++j)
            for (int q = 0; q <= kNumStages; ++q)
              if (j < i || q < s) cudaEventDestroy(p->ev[j][q]);
          delete[] p->ev;
          delete p;
          return MOE_ERR_CUDA;
        }
  }
  *plan_out = p;
  return MOE_OK;
}

int moe_plan_launch(moe_plan *p, void *stream) {
  if (!p) return MOE_ERR_NULL;
  const moe_forward_desc &d = p->d;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The status word is cleared on the stream before any kernel of the launch
  // can OR a bit into it: by a memset, or, for the decode chain in one launch,
  // by the kernel that also zeroes the chain's counters (first of the launch).
  const bool chain_clear = p->use_chain && p->chain.one_launch && d.T > 0;
  if (d.status && !chain_clear && cudaMemsetAsync(d.status, 0, sizeof(int32_t), s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (d.T == 0) return MOE_OK;
  // The GEMMs' claim counters (the small-group kernel beside the pair kernel).
  if (p->sched && cudaMemsetAsync(p->sched, 0, kSchedInts * sizeof(int32_t), s) != cudaSuccess)
    return MOE_ERR_CUDA;
  Launch l;
  l.stream = s;
  l.pdl = !p->timing;
  if (chain_clear) {
    // The chain's counters live in the workspace, which other plans may
    // share: every launch zeroes them first.  The clearing kernel may start
    // under the stream's previous kernel (a previous launch's chain) and waits
    // for it before it clears; the chain behind it may start early too.
    if (launch_chain_clear(p->chain, p->unreachable_wait, l) != cudaSuccess) return MOE_ERR_CUDA;
  }
  cudaEvent_t *ev = p->timing ? p->ev[p->n_recorded % kTimingRing] : nullptr;
  auto mark = [&](int stage) -> bool {
    return !ev || cudaEventRecord(ev[stage], s) == cudaSuccess;
  };
  if (!mark(kRoute)) return MOE_ERR_CUDA;
  if (p->logits_mode) {
    if (launch_route(d.logits, d.T, d.E, d.top_k, p->ids, p->w, l) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (p->use_chain) {  // sort, gather and finalize run inside the GEMM kernels
    if (!mark(kSort) || !mark(kGather) || !mark(kFc1)) return MOE_ERR_CUDA;
    if (p->chain.one_launch) {
      if (launch_chain(p->chain, 0, l) != cudaSuccess) return MOE_ERR_CUDA;
      if (!mark(kFc2)) return MOE_ERR_CUDA;
    } else {
      if (launch_chain(p->chain, 1, l) != cudaSuccess) return MOE_ERR_CUDA;
      if (!mark(kFc2)) return MOE_ERR_CUDA;
      if (launch_chain(p->chain, 2, l) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (!mark(kFinalize) || !mark(kNumStages)) return MOE_ERR_CUDA;
    if (ev) ++p->n_recorded;
    return MOE_OK;
  }
  if (!mark(kSort)) return MOE_ERR_CUDA;
  if (launch_sort(p->ids, p->R, d.E, d.local_offset, d.num_local, p->m_indptr, p->p2e, p->e2p,
                  p->sort_ws, d.status, l) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!mark(kGather)) return MOE_ERR_CUDA;
  const bool dec = p->path == MOE_PATH_DECODE;
  // grouped path: one warp per token (x read once); decode path: one warp
  // per route (a handful of tokens would leave most of the GPU idle)
  if (p->e4m3) {
    if (launch_gather_tokens_q(d.x, p->e2p, d.T, d.H, d.top_k, d.x_scale, p->R,
                               reinterpret_cast<uint8_t *>(p->xp), l) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else if (!p->fused_gather &&
             (dec ? launch_gather(d.x, p->p2e, p->m_indptr + d.num_local, d.H, d.top_k, p->R, p->xp, l)
                  : launch_gather_tokens(d.x, p->e2p, d.T, d.H, d.top_k, p->R, p->xp, l)) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!mark(kFc1)) return MOE_ERR_CUDA;
  if ((dec ? launch_swap(p->fc1d, l) : launch_gemm(p->fc1, l)) != cudaSuccess) return MOE_ERR_CUDA;
  if (!mark(kFc2)) return MOE_ERR_CUDA;
  if ((dec ? launch_swap(p->fc2d, l) : launch_gemm(p->fc2, l)) != cudaSuccess) return MOE_ERR_CUDA;
  if (!mark(kFinalize)) return MOE_ERR_CUDA;
  if (launch_finalize(p->y, p->e2p, p->w, d.T, d.top_k, d.H, d.out, l) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!mark(kNumStages)) return MOE_ERR_CUDA;
  if (ev) ++p->n_recorded;
  return MOE_OK;
}

int moe_plan_buffers_get(const moe_plan *p, moe_plan_buffers *out) {
  if (!p || !out) return MOE_ERR_NULL;
  out->topk_ids = p->ids;
  out->topk_w = p->w;
  out->m_indptr = p->m_indptr;
  out->perm_to_exp = p->p2e;
  out->exp_to_perm = p->e2p;
  out->xp = p->xp;
  out->h = p->h;
  out->y = p->y;
  out->path = p->path;
  return MOE_OK;
}

int moe_plan_set_wait_limit(moe_plan *p, unsigned long long limit_ns) {
  if (!p) return MOE_ERR_NULL;
  if (limit_ns < MOE_WAIT_LIMIT_MIN_NS || limit_ns > MOE_WAIT_LIMIT_MAX_NS) return MOE_ERR_SHAPE;
  p->fc1.wait_ns = p->fc2.wait_ns = limit_ns;
  p->fc1d.wait_ns = p->fc2d.wait_ns = limit_ns;
  p->chain.wait_ns = limit_ns;
  return MOE_OK;
}

int moe_plan_stage_count(const moe_plan *p) { return p ? kNumStages : 0; }

const char *moe_plan_stage_name(const moe_plan *p, int stage) {
  if (!p || stage < 0 || stage >= kNumStages) return "";
  return kStageNames[stage];
}

int moe_plan_stage_times(moe_plan *p, float *ms, int max_stages, int *n_launches) {
  if (!p || !ms) return MOE_ERR_NULL;
  if (!p->timing) return MOE_ERR_STATE;
  const long n = p->n_recorded < kTimingRing ? p->n_recorded : kTimingRing;
  const int ns = max_stages < kNumStages ? max_stages : kNumStages;
  for (int s = 0; s < ns; ++s) ms[s] = 0.f;
  for (long i = 0; i < n; ++i) {
    const long slot = (p->n_recorded - 1 - i) % kTimingRing;
    if (cudaEventSynchronize(p->ev[slot][kNumStages]) != cudaSuccess) return MOE_ERR_CUDA;
    for (int s = 0; s < ns; ++s) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, p->ev[slot][s], p->ev[slot][s + 1]) != cudaSuccess)
        return MOE_ERR_CUDA;
      ms[s] += t;
    }
  }
  if (n_launches) *n_launches = (int)n;
  return MOE_OK;
}

int moe_plan_kernels_per_launch(const moe_plan *p) {
  if (!p || p->d.T == 0) return 0;
  if (p->use_chain) return (p->logits_mode ? 1 : 0) + (p->chain.one_launch ? 1 : 2);
  int n = p->logits_mode ? 1 : 0;                       // route
  n += p->R <= kSortSingleMax ? 1 : 3;                  // sort
  n += (p->fused_gather ? 0 : 1) + 1 + 1 + 1;           // gather, fc1, fc2, finalize
  if (p->sched) n += 2;                                  // small-group kernels beside fc1, fc2
  return n;
}

int moe_plan_stage_reset(moe_plan *p) {
  if (!p) return MOE_ERR_NULL;
  p->n_recorded = 0;
  return MOE_OK;
}

int moe_plan_destroy(moe_plan *p) {
  if (!p) return MOE_OK;
  if (p->timing && p->ev) {
    for (int i = 0; i < kTimingRing; ++i)
      for (int s = 0; s <= kNumStages; ++s) cudaEventDestroy(p->ev[i][s]);
    delete[] p->ev;
  }
  delete p;
  return MOE_OK;
}

int moe_forward(const moe_bf16 *x, const float *logits, const int32_t *topk_ids,
                const float *topk_w, const moe_bf16 *w1, const moe_bf16 *w2, int T, int H, int I,
                int E, int top_k, int local_offset, int num_local, moe_bf16 *out, void *workspace,
                size_t workspace_bytes, int32_t *status, void *stream) {
  moe_forward_desc d;
  std::memset(&d, 0, sizeof d);
  d.x = x;
  d.logits = logits;
  d.topk_ids = topk_ids;
  d.topk_w = topk_w;
  d.w1 = w1;
  d.w2 = w2;
  d.out = out;
  d.workspace = workspace;
  d.workspace_bytes = workspace_bytes;
  d.status = status;
  d.T = T;
  d.H = H;
  d.I = I;
  d.E = E;
  d.top_k = top_k;
  d.local_offset = local_offset;
  d.num_local = num_local;
  d.path = MOE_PATH_AUTO;
  moe_plan *p = nullptr;
  int rc = moe_forward_prepare(&d, &p);
  if (rc != MOE_OK) return rc;
  rc = moe_plan_launch(p, stream);
  moe_plan_destroy(p);
  return rc;
}

}  // extern "C"
