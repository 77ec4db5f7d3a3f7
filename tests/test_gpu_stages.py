"""Stage-by-stage parity of the CUDA kernels (through the C ABI) against the
CPU oracle.  Each stage is fed the oracle's own intermediate, so errors do not
compound: routing and sorting must match bit for bit, the GEMM stages within
the output acceptance rule."""
import numpy as np
import pytest
import torch

import mixture_experts_expert_router_gb300 as moe
import oracle
from mixture_experts_expert_router_gb300 import workloads as W
from tests.tolerances import WEIGHT_ATOL, check_bf16_close, check_f32_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mixture_experts_expert_router_gb300 import _build
    _build.build()
    moe.library()


# ------------------------------------------------------------------- route --

@pytest.mark.parametrize("T,E,k,ties", [
    (16, 4, 2, False), (1, 1, 1, False), (37, 8, 2, True), (300, 128, 8, False), (129, 256, 8, True),
    (64, 64, 16, True), (33, 1000, 16, False), (5, 33, 16, True), (2048, 160, 6, False)])
def test_route_parity(T, E, k, ties):
    rng = np.random.default_rng(T * 1000 + E)
    if ties:
        lg = (rng.integers(-3, 4, size=(T, E)) * 0.5).astype(np.float32)
    else:
        lg = rng.standard_normal((T, E)).astype(np.float32) * 2
    ids_o, w_o = oracle.route(lg, k)
    ids_g, w_g = moe.moe_route(torch.from_numpy(lg).to(DEV), k)
    torch.cuda.synchronize()
    assert np.array_equal(ids_g.cpu().numpy(), ids_o)
    assert np.max(np.abs(w_g.cpu().numpy() - w_o)) <= WEIGHT_ATOL


def test_route_zipf_full_size():
    wl = W.make_moe("prefill_many_fine", H=64, I=64)
    ids_o, w_o = oracle.route(wl.logits.numpy(), wl.top_k)
    ids_g, w_g = moe.moe_route(wl.logits.to(DEV), wl.top_k)
    assert np.array_equal(ids_g.cpu().numpy(), ids_o)
    assert np.max(np.abs(w_g.cpu().numpy() - w_o)) <= WEIGHT_ATOL


# -------------------------------------------------------------------- sort --

def _check_sort(ids, E, off, L):
    m_o, p2e_o, e2p_o, st_o = oracle.sort(ids, E, off, L)
    m, p2e, e2p, st = moe.moe_sort(torch.from_numpy(ids).to(DEV), E, off, L)
    torch.cuda.synchronize()
    M = int(m_o[-1])
    assert np.array_equal(m.cpu().numpy(), m_o)
    assert np.array_equal(p2e.cpu().numpy()[:M], p2e_o)
    assert np.array_equal(e2p.cpu().numpy(), e2p_o)
    assert int(st.item()) == st_o


@pytest.mark.parametrize("T,k,E,off,L", [
    (16, 2, 4, 0, 4), (1, 1, 1, 0, 1), (1024, 2, 8, 0, 8), (1025, 2, 8, 0, 8), (256, 8, 256, 0, 256),
    (2048, 2, 16, 0, 16), (2049, 2, 16, 0, 16),  # 4096 routes: one CTA; 4098: two chunks
    (8192, 8, 256, 0, 256), (4096, 2, 8, 2, 3), (25000, 8, 1000, 100, 900), (3000, 6, 64, 63, 1),
    (64, 8, 128, 0, 128)])
def test_sort_parity(T, k, E, off, L):
    rng = np.random.default_rng(T + k + E)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    _check_sort(ids, E, off, L)


@pytest.mark.parametrize("T,k", [(100, 4), (9000, 8)])
def test_sort_skewed_and_bad_ids(T, k):
    rng = np.random.default_rng(7)
    E = 32
    ids = np.where(rng.random((T, k)) < 0.7, 3, rng.integers(0, E, size=(T, k))).astype(np.int32)
    ids.flat[rng.integers(0, T * k, 9)] = rng.choice([-5, -1, E, 1 << 20], 9)
    _check_sort(ids, E, 0, E)
    _check_sort(ids, E, 2, 5)


def test_sort_zipf_routes():
    wl = W.make_moe("prefill_many_fine", H=64, I=64)
    ids, _ = oracle.route(wl.logits.numpy(), wl.top_k)
    _check_sort(ids, wl.E, 0, wl.E)


# ---------------------------------------------------- gather and finalize --

def test_gather_and_finalize_parity():
    wl = W.make_moe(T=300, H=192, I=64, E=9, top_k=3, mode="logits", seed=5)
    ids, w = oracle.route(wl.logits.numpy(), 3)
    m, p2e, e2p, _ = oracle.sort(ids, 9, 1, 7)
    x = wl.x.to(DEV)
    xp = moe.moe_gather(x, torch.from_numpy(np.pad(p2e, (0, 900 - len(p2e)))).to(DEV),
                        torch.from_numpy(m).to(DEV), 3)
    torch.cuda.synchronize()
    want = W.bf16_bits(wl.x)[p2e // 3]
    assert np.array_equal(W.bf16_bits(xp)[:len(p2e)], want)
    # finalize on a random fp32 y
    y = np.random.default_rng(1).standard_normal((900, 192)).astype(np.float32)
    out_o = oracle.finalize(y, e2p, w)
    out_g = moe.moe_finalize(torch.from_numpy(y).to(DEV), torch.from_numpy(e2p).to(DEV),
                             torch.from_numpy(w).to(DEV))
    assert np.array_equal(W.bf16_bits(out_g), out_o)  # same fp32 order, same rounding


# --------------------------------------------------------- GEMM stages -----

def _rows_sample(m_indptr, n_rand, seed):
    """Every group's first and last row plus random rows (all rows if few)."""
    M = int(m_indptr[-1])
    if M <= 2048:
        return np.arange(M, dtype=np.int32)
    rows = set()
    for i in range(len(m_indptr) - 1):
        if m_indptr[i + 1] > m_indptr[i]:
            rows.update([int(m_indptr[i]), int(m_indptr[i + 1]) - 1])
    rows.update(np.random.default_rng(seed).integers(0, M, n_rand).tolist())
    return np.array(sorted(rows), dtype=np.int32)


@pytest.mark.parametrize("T,H,I,E,k", [(16, 128, 128, 4, 2), (200, 256, 192, 5, 2), (700, 512, 256, 9, 3),
                                       (64, 128, 64, 128, 8), (900, 256, 384, 40, 4), (300, 512, 128, 3, 3)])
def test_fc1_fc2_stage_parity(T, H, I, E, k):
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", seed=T)
    x, w1, w2 = W.bf16_bits(wl.x), W.bf16_bits(wl.w1), W.bf16_bits(wl.w2)
    ids, w = oracle.route(wl.logits.numpy(), k)
    m, p2e, e2p, _ = oracle.sort(ids, E)
    R = T * k
    xp = np.zeros((R, H), np.uint16)
    xp[:len(p2e)] = x[p2e // k]
    m_d = torch.from_numpy(m).to(DEV)
    h_g = moe.moe_fc1_swiglu(W.from_bf16_bits(xp).to(DEV), wl.w1.to(DEV), m_d)
    rows = _rows_sample(m, 512, 0)
    h_o = oracle.fc1_swiglu_rows(xp, w1, m[1:], rows)
    check_bf16_close(W.bf16_bits(h_g)[rows], h_o, "h")
    # FC2 from the oracle's h rows (all rows of h computed by the oracle)
    all_rows = np.arange(len(p2e), dtype=np.int32)
    h_full = np.zeros((R, I), np.uint16)
    h_full[:len(p2e)] = oracle.fc1_swiglu_rows(xp, w1, m[1:], all_rows)
    y_g = moe.moe_fc2(W.from_bf16_bits(h_full).to(DEV), wl.w2.to(DEV), m_d)
    y_o = oracle.fc2_rows(h_full, w2, m[1:], rows)
    check_f32_close(y_g.cpu().numpy()[rows], y_o, "y")


@pytest.mark.parametrize("sizes,N,K", [
    ([0, 1, 127, 128, 129, 0, 300], 128, 128),
    ([5, 0, 0, 260, 1], 256, 256),
    ([130, 70, 1, 0, 64], 192, 64),
    ([1000, 3, 500], 64, 320),
    ([0, 0, 0, 7], 1536, 512),
    ([20, 33, 300, 0, 17, 100, 256, 512, 384, 129, 65], 512, 192),
    ([1, 16, 32, 64, 128, 200, 255, 257], 256, 128)])
def test_grouped_gemm_parity(sizes, N, K):
    d = W.make_grouped_gemm(seed=len(sizes), sizes=sizes, N=N, K=K)
    X, Wt, offs = d["X"].to(DEV), d["W"].to(DEV), d["offs"].to(DEV)
    sentinel = torch.full((d["sum_m"] + 3, N), -7.0, dtype=torch.bfloat16, device=DEV)
    Y = sentinel[:d["sum_m"]]
    moe.grouped_gemm_fwd(X, Wt, offs, Y)
    torch.cuda.synchronize()
    Yo = oracle.grouped_gemm_rows(W.bf16_bits(d["X"]), W.bf16_bits(d["W"]), d["offs"].numpy())
    check_bf16_close(W.bf16_bits(Y), Yo, "Y")
    assert torch.all(sentinel[d["sum_m"]:] == -7.0)  # nothing written past the last group


@pytest.mark.parametrize("sizes", [[0, 1, 129, 255, 256, 300, 0, 17], [1000, 3, 130, 64]])
def test_grouped_gemm_without_tail_tiles_parity(sizes):
    """MOE_PLAN_NO_TAIL_TILES: every remainder runs as a main tile whose rows
    past the group are computed and not stored."""
    d = W.make_grouped_gemm(seed=len(sizes) + 50, sizes=sizes, N=256, K=320)
    X, Wt, offs = d["X"].to(DEV), d["W"].to(DEV), d["offs"].to(DEV)
    sentinel = torch.full((d["sum_m"] + 3, 256), -7.0, dtype=torch.bfloat16, device=DEV)
    Y = sentinel[:d["sum_m"]]
    moe.grouped_gemm_fwd(X, Wt, offs, Y, no_tail_tiles=True)
    torch.cuda.synchronize()
    Yo = oracle.grouped_gemm_rows(W.bf16_bits(d["X"]), W.bf16_bits(d["W"]), d["offs"].numpy())
    check_bf16_close(W.bf16_bits(Y), Yo, "Y (no tail tiles)")
    assert torch.all(sentinel[d["sum_m"]:] == -7.0)


def test_grouped_gemm_many_small_groups_parity():
    """800 groups of 0..40 rows (nearly all of them tail tiles, the group
    tables filling a large part of shared memory); K = 192 is an odd number of
    64-wide k-blocks."""
    sizes = np.random.default_rng(800).integers(0, 41, 800).tolist()
    d = W.make_grouped_gemm(seed=800, sizes=sizes, N=256, K=192)
    X, Wt, offs = d["X"].to(DEV), d["W"].to(DEV), d["offs"].to(DEV)
    Y = moe.grouped_gemm_fwd(X, Wt, offs)
    torch.cuda.synchronize()
    Yo = oracle.grouped_gemm_rows(W.bf16_bits(d["X"]), W.bf16_bits(d["W"]), d["offs"].numpy())
    check_bf16_close(W.bf16_bits(Y), Yo, "Y")


def test_grouped_gemm_rows_beyond_offsets_untouched():
    d = W.make_grouped_gemm(seed=3, sizes=[40, 0, 90], N=128, K=128)
    X = torch.cat([d["X"], torch.ones(50, 128, dtype=torch.bfloat16)]).to(DEV)
    Y = torch.full((180, 128), 3.0, dtype=torch.bfloat16, device=DEV)
    moe.grouped_gemm_fwd(X, d["W"].to(DEV), d["offs"].to(DEV), Y)
    torch.cuda.synchronize()
    assert torch.all(Y[130:] == 3.0)


@pytest.mark.parametrize("T,H,I,E,k,max_group", [(1, 2048, 768, 128, 8, 1), (8, 256, 128, 16, 4, 8),
                                                 (64, 192, 320, 32, 8, 64), (40, 128, 64, 3, 2, 16),
                                                 (300, 128, 128, 5, 2, 32), (6, 64, 128, 4, 2, 16),
                                                 (64, 192, 320, 128, 8, 64)])
def test_swapab_fc1_fc2_stage_parity(T, H, I, E, k, max_group):
    """Decode-form kernels (weights on the MMA's M side) on the oracle's own
    intermediates; groups larger than the N tile run in several N tiles.  The
    k-blocks alternate between two accumulators: the shapes include one k-block
    (H = 64 for FC1, I = 64 for FC2) and odd counts (H = 192, I = 320), the
    last also with several tiles per CTA (hundreds of expert tiles)."""
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", seed=T + 11)
    x, w1, w2 = W.bf16_bits(wl.x), W.bf16_bits(wl.w1), W.bf16_bits(wl.w2)
    ids, w = oracle.route(wl.logits.numpy(), k)
    m, p2e, e2p, _ = oracle.sort(ids, E)
    R = T * k
    xp = np.zeros((R, H), np.uint16)
    xp[:len(p2e)] = x[p2e // k]
    m_d = torch.from_numpy(m).to(DEV)
    rows = np.arange(len(p2e), dtype=np.int32)
    h_g = moe.moe_fc1_swiglu_swapab(W.from_bf16_bits(xp).to(DEV), wl.w1.to(DEV), m_d, max_group)
    h_o = oracle.fc1_swiglu_rows(xp, w1, m[1:], rows)
    check_bf16_close(W.bf16_bits(h_g)[rows], h_o, "h (swap-AB)")
    h_full = np.zeros((R, I), np.uint16)
    h_full[:len(p2e)] = h_o
    y_g = moe.moe_fc2_swapab(W.from_bf16_bits(h_full).to(DEV), wl.w2.to(DEV), m_d, max_group)
    y_o = oracle.fc2_rows(h_full, w2, m[1:], rows)
    check_f32_close(y_g.cpu().numpy()[rows], y_o, "y (swap-AB)")
    # the decode-form and grouped FC2 read the same h: compare the two kernels too
    y_grouped = moe.moe_fc2(W.from_bf16_bits(h_full).to(DEV), wl.w2.to(DEV), m_d)
    check_f32_close(y_g.cpu().numpy()[rows], y_grouped.cpu().numpy()[rows], "y swap-AB vs grouped")


@pytest.mark.parametrize("T,H,I,E,k", [(16, 128, 128, 4, 2), (700, 512, 256, 9, 3), (900, 256, 384, 40, 4),
                                       (300, 192, 128, 3, 3), (5, 64, 128, 64, 8)])
def test_fc1_gathered_stage_parity(T, H, I, E, k):
    """FC1 taking its rows straight from x through the permutation (copied
    by the gather warps) against the oracle's FC1 on the gathered rows, and
    bitwise against FC1 on the gathered copy."""
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", seed=T + 3)
    x, w1 = W.bf16_bits(wl.x), W.bf16_bits(wl.w1)
    ids, _ = oracle.route(wl.logits.numpy(), k)
    m, p2e, e2p, _ = oracle.sort(ids, E)
    R = T * k
    p2e_full = np.zeros(R, np.int32)
    p2e_full[:len(p2e)] = p2e
    h_g = moe.moe_fc1_swiglu_gathered(wl.x.to(DEV), torch.from_numpy(p2e_full).to(DEV),
                                      torch.from_numpy(m).to(DEV), k, wl.w1.to(DEV))
    rows = np.arange(len(p2e), dtype=np.int32)
    xp = np.zeros((R, H), np.uint16)
    xp[:len(p2e)] = x[p2e // k]
    h_o = oracle.fc1_swiglu_rows(xp, w1, m[1:], rows)
    check_bf16_close(W.bf16_bits(h_g)[rows], h_o, "h (gathered rows)")
    h_c = moe.moe_fc1_swiglu(W.from_bf16_bits(xp).to(DEV), wl.w1.to(DEV), torch.from_numpy(m).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(W.bf16_bits(h_g)[rows], W.bf16_bits(h_c)[rows])
