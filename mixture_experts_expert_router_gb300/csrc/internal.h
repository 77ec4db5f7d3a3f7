// Internal launchers shared by the C ABI (api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "moe_gb300.h"

namespace moe {

// Launch settings shared by every launcher: the stream and whether the kernel
// may start under programmatic dependent launch (its prologue overlapping the
// previous kernel's tail; it waits for the predecessor before reading).
struct Launch {
  cudaStream_t stream = nullptr;
  bool pdl = false;
};

int device_sm_count();

// Longest a single in-kernel wait may take before the kernel gives up, unless
// the plan sets another limit (moe_plan_set_wait_limit).
constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // 4 s

// S1 ---------------------------------------------------------------------------
cudaError_t launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                         const Launch &l);

// S2 ---------------------------------------------------------------------------
// Routes per CTA of the multi-CTA sort, and the largest route count the
// single-CTA sort handles (one chunk: below it the multi-CTA path would run
// three one-CTA kernels).
constexpr int kSortChunk = 4096;
constexpr int kSortSingleMax = kSortChunk;
size_t sort_workspace_bytes(long routes, int L);
cudaError_t launch_sort(const int32_t *ids, long routes, int E, int off, int L, int32_t *m_indptr,
                        int32_t *p2e, int32_t *e2p, int32_t *ws, int32_t *status,
                        const Launch &l);

// Library-owned scratch for the allocation-free sort (sort.cu).
long static_sort_scratch_ints();
cudaError_t static_sort_scratch(cudaStream_t stream, int32_t **out);

// S3 / S6 -----------------------------------------------------------------------
cudaError_t launch_gather(const uint16_t *x, const int32_t *p2e, const int32_t *m_total, int H,
                          int k, long max_rows, uint16_t *xp, const Launch &l);
// The same rows written token by token through exp_to_perm (x read once).
cudaError_t launch_gather_tokens(const uint16_t *x, const int32_t *e2p, int T, int H, int k,
                                 long max_rows, uint16_t *xp, const Launch &l);
cudaError_t launch_finalize(const float *y, const int32_t *e2p, const float *w, int T, int k,
                            int H, uint16_t *out, const Launch &l);
// Token-major copy with E4M3 quantisation: xq[p] = e4m3(x[t] / scale) (H % 16 == 0).
cudaError_t launch_gather_tokens_q(const uint16_t *x, const int32_t *e2p, int T, int H, int k,
                                   float scale, long max_rows, uint8_t *xq, const Launch &l);

// S4 / S5 / S8: persistent tcgen05 grouped GEMM --------------------------------
enum class Epi : int { kBf16 = 0, kSwiGLU = 1, kF32 = 2 };

struct GemmPlan {
  CUtensorMap map_a;            // A [rows, K] bf16, box {64, 128}
  CUtensorMap map_b;            // B [G * b_rows, K] bf16, box {64, box_b}
  CUtensorMap map_w64;          // pair kernel: B with box {64, 64} (FC1 tail tiles)
  CUtensorMap map_t[4];         // pair kernel: A with box {64, 8/16/32/64} (tail tiles)
  CUtensorMap map_y;            // pair kernel, fp32 output: TMA-store map
  const uint16_t *gather_x = nullptr;   // gather mode: rows of A are x[p2e[p] / k]
  const int32_t *gather_p2e = nullptr;
  long gather_rows = 0;
  int gather_k = 0;             // 0: A rows are given directly
  const int32_t *group_end;     // [G] cumulative group ends (device)
  int G = 0;                    // groups
  int K = 0;                    // reduction length
  int n_out = 0;                // output columns per row (N, or I for SwiGLU)
  int b_rows = 0;               // B rows per group (N, or 2I for SwiGLU)
  int bn = 0;                   // MMA N (total B rows per tile)
  int n_tiles = 0;              // output column tiles
  int m_major = 0;              // tile raster: m-tiles innermost (0) or n (1)
  long max_rows = 0;            // bound on total rows (grid sizing)
  void *out = nullptr;          // bf16 or fp32 output, row stride n_out
  Epi epi = Epi::kBf16;
  int pair = 0;                 // 1: CTA-pair kernel (gemm2sm.cu), 0: one-CTA kernel
  int grid = 0;
  size_t smem = 0;
  int32_t *status = nullptr;
  unsigned long long wait_ns = kWaitLimitNs;
  const float *clamp = nullptr;  // SwiGLU epilogue: [G] SwiGLUStep limits (device), or null
  // E4M3 operands (one-CTA kernel only): the accumulator is dequantised by
  // ascale * wscale[g]; the SwiGLU epilogue writes E4M3 h = e4m3(h / oscale)
  int q = 0;
  const float *wscale = nullptr;
  float ascale = 1.f, oscale = 1.f;
  // CTA-pair kernel: a group's last rows up to this many run as swap-AB tail
  // tiles (weights on the MMA's M side); 0 makes every remainder a main tile
  // whose rows past the group are computed and not stored
  int tail_max = 128;
  // CTA-pair kernel beside the small-group kernel (gemm_small.cu): side_ctas
  // CTAs of that kernel take the tiles of the groups of 1..small_max rows,
  // both kernels claim tiles through the four counters at sched (device,
  // zero before each launch).  side_ctas = 0: the pair kernel alone.
  int32_t *sched = nullptr;
  int side_ctas = 0;
  int small_max = 0;
};

// Encodes the tensor maps and picks tile shapes; host only.  allow_pair lets
// it choose the CTA-pair kernel when the shape allows.
int gemm_prepare(GemmPlan &p, Epi epi, const uint16_t *A, long a_rows, const uint16_t *B, int G,
                 int b_rows, int K, int n_out, const int32_t *group_end, long max_rows, void *out,
                 int32_t *status, bool allow_pair = true);
// The same for FC1 reading its rows straight from x through the permutation
// (row p of A = x[p2e[p] / k]); CTA-pair kernel only (MOE_ERR_SHAPE otherwise).
int gemm_prepare_gather(GemmPlan &p, const uint16_t *x, long x_rows, const int32_t *p2e, int k,
                        const uint16_t *W1, int G, int I, int H, const int32_t *group_end,
                        long max_rows, void *h, int32_t *status);
cudaError_t launch_gemm(const GemmPlan &p, const Launch &l);
// E4M3 operands A [a_rows, K], B [G * b_rows, K] (uint8 codes), SwiGLU (E4M3
// h out) or fp32 epilogue; K % 128 == 0.  The CTA-pair kernel where the shape
// allows it and allow_pair is set, else the one-CTA kernel.  Set wscale /
// ascale / oscale on the plan afterwards.
int gemm_prepare_e4m3(GemmPlan &p, Epi epi, const uint8_t *A, long a_rows, const uint8_t *B, int G,
                      int b_rows, int K, int n_out, const int32_t *group_end, long max_rows,
                      void *out, int32_t *status, bool allow_pair = true);

// CTA-pair form (gemm2sm.cu)
size_t pair_gemm_smem(Epi epi, int G);
int pair_gemm_encode_extra(GemmPlan &p, const uint16_t *A, long a_rows, const uint16_t *B,
                           long b_rows_total, int K);
// E4M3: all of the pair kernel's tensor maps from uint8 operands.
int pair_gemm_encode_u8(GemmPlan &p, const uint8_t *A, long a_rows, const uint8_t *B, long b_rows_total, int K);
bool pair_gemm_supported(Epi epi, int n_out);
cudaError_t pair_gemm_configure(Epi epi, size_t smem, int q = 0);
cudaError_t launch_pair_gemm(const GemmPlan &p, const Launch &l);

// Small-group kernel (gemm_small.cu), launched by launch_gemm ahead of the
// CTA-pair kernel when a plan has side_ctas > 0.
size_t small_gemm_smem(int G);
int small_gemm_max_rows();
cudaError_t small_gemm_configure(Epi epi, int q, size_t smem);
cudaError_t launch_small_gemm(const GemmPlan &p, const Launch &l);
// Gives a CTA-pair plan (any bf16 epilogue; SwiGLU or fp32 with E4M3) the small-group kernel:
// `ctas` CTAs (even), claim counters at sched (4 ints, zeroed before every
// launch).  MOE_ERR_SHAPE if the plan cannot take it.
int gemm_attach_small(GemmPlan &p, int32_t *sched, int ctas);

// Grouped GEMM backward (gemm_bwd.cu): dgrad dX = G . W[g] (W in place) and
// wgrad dW[g] = G^T . X over each group's rows, one-CTA tcgen05 kernels with
// MN-major operands.
struct BwdPlan {
  CUtensorMap map_a, map_b, map_o;
  const int32_t *group_end = nullptr;
  void *out = nullptr;
  int32_t *status = nullptr;
  unsigned long long wait_ns = kWaitLimitNs;
  long sum_m = 0;
  int E = 0, N = 0, K = 0, mode = 0, grid = 0;
  size_t smem = 0;
};
// G [sum_m, N]; B = W [E, N, K] (dgrad) or X [sum_m, K] (wgrad); out dX
// [sum_m, K] bf16, or dW [E, N, K] fp32 / bf16.  N % 64 == 0, K % 64 == 0.
int bwd_prepare(BwdPlan &p, bool wgrad, bool out_f32, const uint16_t *G, const uint16_t *B,
                const int32_t *offs, long sum_m, int E, int N, int K, void *out, int32_t *status);
cudaError_t launch_bwd(const BwdPlan &p, const Launch &l);

// BGMV LoRA-MoE shrink + expand (bgmv.cu) ----------------------------------------
constexpr int kBgmvMaxSlices = 8;
// (LoRA, expert) groups up to which the pair-grouped pipeline may group the
// pairs with the route sort (its scans take at most MOE_MAX_EXPERTS groups).
constexpr int kBgmvSortMaxGroups = MOE_MAX_EXPERTS;
struct BgmvPlan {
  const uint16_t *x = nullptr;
  const uint16_t *a[kBgmvMaxSlices] = {}, *b[kBgmvMaxSlices] = {};
  int f[kBgmvMaxSlices] = {}, off[kBgmvMaxSlices] = {};
  const int32_t *tok = nullptr, *eid = nullptr, *lora = nullptr;
  const float *w = nullptr;
  uint16_t *shrink = nullptr;
  float *y = nullptr;
  int32_t *ws = nullptr;      // general pair order: route index (bgmv_workspace_bytes)
  int32_t *status = nullptr;
  int T = 0, H = 0, R = 0, S = 0, L = 0, E = 0, P = 0, k = 0, ld_y = 0;
};
size_t bgmv_workspace_bytes(int T, int P, int contiguous_k, int num_loras, int E, int total_f);
cudaError_t launch_bgmv(const BgmvPlan &p, const Launch &l);

// S7: swap-AB weight-streaming GEMMs for few tokens per expert (decode.cu) ----
struct SwapPlan {
  CUtensorMap map_w;            // weights [G * w_rows, K], box {64, 64 | 128}
  CUtensorMap map_x;            // activations [max_rows, K], box {64, bnt}
  const int32_t *group_end = nullptr;
  void *out = nullptr;          // h (bf16) for FC1, y (fp32) for FC2
  int32_t *status = nullptr;
  long max_rows = 0;
  int G = 0, K = 0, n_out = 0, w_rows = 0, m_tiles = 0, bnt = 0, grid = 0;
  size_t smem = 0;
  bool swiglu = false;
  bool early = false;           // may read group_end and stream weights before the PDL wait
  unsigned long long wait_ns = kWaitLimitNs;
  const float *clamp = nullptr;  // FC1: [G] SwiGLUStep limits (device), or null
};

int swap_prepare(SwapPlan &p, bool swiglu, const uint16_t *W, int G, int w_rows, int K,
                 const uint16_t *X, long max_rows, int n_out, const int32_t *group_end,
                 long max_group_rows, void *out, int32_t *status, bool early);
cudaError_t launch_swap(const SwapPlan &p, const Launch &l);

// S7 as a chain with the sort, gather and finalize folded in (decode_chain.cu):
// two kernels, or both phases in one launch; for T * top_k <= kChainMaxRoutes.
constexpr int kChainMaxRoutes = 1024;
// Without a plan flag the decode path runs the chain in one launch up to this
// many routes.  Measured at H = 2048, I = 768, E = 128, top-8, pre-routed
// (one launch / two kernels / five kernels): T = 1: 28.2 / 28.7 / 31.1 us;
// T = 2: 41.2 / 47.1 us (one launch / two kernels); T = 4: 61.6 / 70.1 /
// 63.9 us; T = 8: 90.8 / 93.8 / 89.2 us.
constexpr int kChainAutoRoutes = 32;
struct ChainPlan {
  CUtensorMap map_w1, map_x, map_w2, map_h;
  const uint16_t *x = nullptr, *w1 = nullptr, *w2 = nullptr;
  const int32_t *ids = nullptr;
  const float *w = nullptr;
  uint16_t *h = nullptr, *out = nullptr;
  float *y = nullptr;
  int32_t *comb = nullptr, *m_indptr = nullptr, *p2e = nullptr, *e2p = nullptr, *status = nullptr;
  int32_t *done1 = nullptr;  // one launch: [L + 1] FC1 tile counts per expert (last unused)
  int T = 0, k = 0, E = 0, off = 0, L = 0, H = 0, I = 0, bnt = 0, grid1 = 0, grid2 = 0, grid_one = 0;
  bool ids_early = false;  // ids are layer inputs (pre-routed), not the routing kernel's output
  bool one_launch = false; // FC1 and FC2 in one kernel (CTAs wait for the FC1 tiles of an expert)
  size_t smem = 0;
  unsigned long long wait_ns = kWaitLimitNs;
  const float *clamp = nullptr;  // [L] SwiGLUStep limits (device), or null
};
size_t chain_comb_ints(int T, int H);
int chain_prepare(ChainPlan &p);
// part 1: FC1 kernel, 2: FC2 kernel, 0: both phases in one kernel
cudaError_t launch_chain(const ChainPlan &p, int part, const Launch &l);
// One launch keeps counters in the workspace; every launch first runs a
// one-CTA kernel that zeroes them and the status word (done1 follows comb in
// the workspace), and the chain kernel follows it by programmatic dependent
// launch.  unreachable: the test hook MOE_PLAN_TEST_UNREACHABLE_WAIT, which
// fills the per-expert FC1 counts with -1 instead, so that no FC2 wait can
// complete.
cudaError_t launch_chain_clear(const ChainPlan &p, bool unreachable, const Launch &l);

}  // namespace moe
