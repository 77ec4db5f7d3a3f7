"""Parity of the ragged grouped GEMM backward (grouped_gemm_dgrad and
grouped_gemm_wgrad, called through the C ABI) against the CPU oracle (Cake
ragged BF16 grouped GEMM, operation table: dgrad dX = G . W[e] with W in
place; wgrad dW[e] = G^T . X, fp32 or bf16, exact zeros for an empty group).

Outputs of the tensor-core kernels sum in another order than the oracle, so
dX and the bf16 dW use the strict output rule (check_bf16_close) and the fp32
dW the fp32 rule (check_f32_close); empty groups must give bitwise +0 and
replays must be bitwise identical."""
import numpy as np
import pytest
import torch

import mixture_experts_expert_router_gb300 as moe
import oracle
from mixture_experts_expert_router_gb300 import workloads as W
from tests.tolerances import check_bf16_close, check_f32_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mixture_experts_expert_router_gb300 import _build
    _build.build()
    moe.library()


# (sizes or Dirichlet draw, K, N): empty, one-row, non-multiple-of-tile groups,
# K not a multiple of the 256-column tile, N not a multiple of the 128-row dW tile
CASES = [
    (dict(sizes=[0, 1, 63, 64, 65, 130, 0, 255, 7, 300]), 192, 128),
    (dict(sum_m=700, E=9, alpha=0.3), 320, 192),
    (dict(sum_m=1000, E=1, alpha=1.0), 256, 256),
    (dict(sum_m=900, E=200, alpha=0.2), 128, 64),
]


def _make(case, K, N, seed):
    kw = dict(case)
    if "sizes" in kw:
        d = W.make_grouped_gemm(seed=seed, sizes=kw["sizes"], K=K, N=N, with_grad=True)
    else:
        d = W.make_grouped_gemm(seed=seed, K=K, N=N, with_grad=True, **kw)
    return d


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_dgrad_parity_and_rows_outside_untouched(ci):
    case, K, N = CASES[ci]
    d = _make(case, K, N, 20 + ci)
    G, Wt, offs = d["G"].to(DEV), d["W"].to(DEV), d["offs"].to(DEV)
    sum_m = d["sum_m"] + 5  # five rows past the last group must stay untouched
    Gp = torch.cat([G, torch.zeros((5, N), dtype=torch.bfloat16, device=DEV)])
    dX = torch.full((sum_m, K), 3.0, dtype=torch.bfloat16, device=DEV)
    moe.grouped_gemm_dgrad(Gp, Wt, offs, dX)
    torch.cuda.synchronize()
    want = oracle.grouped_gemm_dgrad_rows(W.bf16_bits(d["G"]), W.bf16_bits(d["W"]), d["offs"].numpy())
    got = W.bf16_bits(dX)
    check_bf16_close(got[:d["sum_m"]], want, f"dgrad case {ci}")
    assert torch.all(dX[d["sum_m"]:] == 3.0)
    again = moe.grouped_gemm_dgrad(Gp, Wt, offs)
    torch.cuda.synchronize()
    assert torch.equal(again[:d["sum_m"]], dX[:d["sum_m"]])  # replays bitwise identical


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("ci", range(len(CASES)))
def test_wgrad_parity_and_empty_groups_zero(ci, dtype):
    case, K, N = CASES[ci]
    d = _make(case, K, N, 40 + ci)
    G, X, offs = d["G"].to(DEV), d["X"].to(DEV), d["offs"].to(DEV)
    E = d["E"]
    dW = torch.full((E, N, K), 5.0, dtype=dtype, device=DEV)
    moe.grouped_gemm_wgrad(G, X, offs, out_dtype=dtype, dW=dW)
    torch.cuda.synchronize()
    sel_e = np.repeat(np.arange(E, dtype=np.int32), N)
    sel_n = np.tile(np.arange(N, dtype=np.int32), E)
    f32, b16 = oracle.grouped_gemm_wgrad_rows(W.bf16_bits(d["G"]), W.bf16_bits(d["X"]), d["offs"].numpy(),
                                              sel_e, sel_n)
    sizes = d["sizes"]
    if dtype == torch.float32:
        got = dW.cpu().numpy().reshape(E * N, K)
        nz = np.repeat(sizes > 0, N)
        check_f32_close(got[nz], f32[nz], f"wgrad fp32 case {ci}")
        assert np.all(got[~nz].view(np.uint32) == 0)  # exact +0 for empty groups
    else:
        got = W.bf16_bits(dW).reshape(E * N, K)
        check_bf16_close(got, b16, f"wgrad bf16 case {ci}")
        assert np.all(got[np.repeat(sizes == 0, N)] == 0)
    again = moe.grouped_gemm_wgrad(G, X, offs, out_dtype=dtype)
    torch.cuda.synchronize()
    assert torch.equal(again, dW)


def test_wgrad_without_rows_is_zero_and_dgrad_noop():
    E, N, K = 3, 64, 128
    offs = torch.zeros(E, dtype=torch.int32, device=DEV)
    dW = torch.full((E, N, K), 1.0, dtype=torch.float32, device=DEV)
    G = torch.zeros((0, N), dtype=torch.bfloat16, device=DEV)
    X = torch.zeros((0, K), dtype=torch.bfloat16, device=DEV)
    moe.grouped_gemm_wgrad(G, X, offs, dW=dW)
    moe.grouped_gemm_dgrad(G, torch.zeros((E, N, K), dtype=torch.bfloat16, device=DEV), offs)
    torch.cuda.synchronize()
    assert torch.all(dW == 0)


def _sample_rows(sizes, per_group, seed):
    rng = np.random.default_rng(seed)
    rows, start = [], 0
    for s in sizes:
        if s > 0:
            rows += [start, start + s - 1] + list(rng.integers(start, start + s, size=per_group))
        start += s
    return np.unique(np.asarray(rows, np.int32))


def test_backward_grouped_gemm_config_full_size_sampled():
    """sum_m = 16384 over 64 Dirichlet(0.3) groups, K = 4096, N = 1536 (the
    grouped GEMM workload): dgrad on rows covering every non-empty group, wgrad
    on two dW rows of every group (empty ones included), fp32 and bf16."""
    d = W.make_grouped_gemm(seed=0, device="cpu", weights_device=DEV, with_grad=True)
    G, X, Wt, offs = d["G"].to(DEV), d["X"].to(DEV), d["W"], d["offs"].to(DEV)
    E, N, K = Wt.shape
    dX = moe.grouped_gemm_dgrad(G, Wt, offs)
    dW32 = moe.grouped_gemm_wgrad(G, X, offs, out_dtype=torch.float32)
    dW16 = moe.grouped_gemm_wgrad(G, X, offs, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    G_h, X_h, W_h, offs_h = W.bf16_bits(d["G"]), W.bf16_bits(d["X"]), W.bf16_bits(Wt), d["offs"].numpy()
    rows = _sample_rows(d["sizes"], 2, 1)
    want = oracle.grouped_gemm_dgrad_rows(G_h, W_h, offs_h, rows)
    check_bf16_close(W.bf16_bits(dX)[rows], want, "dgrad full size")
    sel_e = np.repeat(np.arange(E, dtype=np.int32), 2)
    sel_n = np.random.default_rng(2).integers(0, N, size=2 * E).astype(np.int32)
    f32, b16 = oracle.grouped_gemm_wgrad_rows(G_h, X_h, offs_h, sel_e, sel_n)
    got32 = dW32.cpu().numpy()[sel_e, sel_n]
    nz = d["sizes"][sel_e] > 0
    check_f32_close(got32[nz], f32[nz], "wgrad fp32 full size")
    assert np.all(got32[~nz].view(np.uint32) == 0)
    check_bf16_close(W.bf16_bits(dW16)[sel_e, sel_n], b16, "wgrad bf16 full size")
