"""End-to-end parity of the whole layer (moe_forward / prepared plans, called
through the C ABI) against the CPU oracle, at the five workload shapes and at
the edge cases; plus bitwise replay determinism."""
import numpy as np
import pytest
import torch

import mixture_experts_expert_router_gb300 as moe
import oracle
from mixture_experts_expert_router_gb300 import workloads as W
from tests import accum_model
from tests.tolerances import check_bf16_close, check_bf16_end_to_end, with_floor

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mixture_experts_expert_router_gb300 import _build
    _build.build()
    moe.library()


def _dev(wl):
    return {k: (getattr(wl, k).to(DEV) if getattr(wl, k) is not None else None)
            for k in ("x", "w1", "w2", "logits", "topk_ids", "topk_w")}


def _oracle_route(wl):
    if wl.mode == "logits":
        return oracle.route(wl.logits.cpu().numpy(), wl.top_k)
    return wl.topk_ids.cpu().numpy(), wl.topk_w.cpu().numpy()


def _oracle_out(wl, tokens=None, w1=None, w2=None, clamp_limit=None):
    """The oracle's output rows for the tokens, with the end-to-end floor (the
    tensor-core accumulation model's agreement with them) attached;
    clamp_limit [L] selects the SwiGLUStep(limit) epilogue."""
    ids, w = _oracle_route(wl)
    w1 = W.bf16_bits(wl.w1) if w1 is None else w1
    w2 = W.bf16_bits(wl.w2) if w2 is None else w2
    x = W.bf16_bits(wl.x)
    out, st = oracle.moe_tokens(x, ids, w, w1, w2, wl.E, tokens=tokens,
                                local_offset=wl.local_offset, num_local=wl.num_local, clamp_limit=clamp_limit)
    frac, n = accum_model.floor(x, ids, w, w1, w2, wl.E, out, tokens=tokens, local_offset=wl.local_offset,
                                num_local=wl.num_local, clamp_limit=clamp_limit)
    return with_floor(out, frac, n), st


def _forward(wl, d, path=moe.PATH_AUTO, status=None, one_cta_gemm=False, decode_chain=False,
             fused_gather=False, one_launch=False, no_tail_tiles=False, small_group_kernel=None):
    plan = moe.MoEPlan(d["x"], d["w1"], d["w2"], wl.E, wl.top_k, logits=d["logits"],
                       topk_ids=d["topk_ids"], topk_w=d["topk_w"], local_offset=wl.local_offset,
                       status=status, path=path, one_cta_gemm=one_cta_gemm, decode_chain=decode_chain,
                       fused_gather=fused_gather, decode_one_launch=one_launch, no_tail_tiles=no_tail_tiles,
                       small_group_kernel=small_group_kernel)
    out = plan.launch()
    torch.cuda.synchronize()
    return out, plan


PATHS = [moe.PATH_GROUPED, moe.PATH_DECODE, moe.PATH_AUTO]


@pytest.mark.parametrize("path", PATHS)
def test_tiny_both_routing_modes(path):
    wl = W.make_moe("tiny")
    d = _dev(wl)
    want, st = _oracle_out(wl)
    out = moe.moe_forward(d["x"], d["w1"], d["w2"], wl.E, wl.top_k, logits=d["logits"])
    torch.cuda.synchronize()
    check_bf16_close(W.bf16_bits(out), want, "tiny logits")
    out_p, _ = _forward(wl, d, path)
    check_bf16_close(W.bf16_bits(out_p), want, "tiny plan")
    ids, w = _oracle_route(wl)
    out_r = moe.moe_forward(d["x"], d["w1"], d["w2"], wl.E, wl.top_k,
                            topk_ids=torch.from_numpy(ids).to(DEV), topk_w=torch.from_numpy(w).to(DEV))
    torch.cuda.synchronize()
    check_bf16_close(W.bf16_bits(out_r), want, "tiny pre-routed")


ODD_SHAPES = [(1, 64, 64, 1, 1), (77, 192, 128, 6, 2), (300, 256, 320, 16, 4),
              (513, 128, 64, 3, 3), (40, 128, 128, 20, 8), (700, 512, 256, 5, 2)]


@pytest.mark.parametrize("one_cta", [False, True])
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T,H,I,E,k", ODD_SHAPES)
def test_odd_shapes(path, T, H, I, E, k, one_cta):
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", seed=T + E)
    out, _ = _forward(wl, _dev(wl), path, one_cta_gemm=one_cta)
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(out), want, f"T={T} H={H} I={I} E={E} k={k}")


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("T,H,I,E,k", [(700, 512, 256, 5, 2), (1500, 256, 256, 64, 6), (300, 256, 320, 16, 4)])
def test_without_tail_tiles(T, H, I, E, k, fused):
    """MOE_PLAN_NO_TAIL_TILES on the grouped path (gather kernel or fused
    gather): the oracle's output under the end-to-end rule."""
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", seed=T + E + 3)
    out, plan = _forward(wl, _dev(wl), moe.PATH_GROUPED, fused_gather=fused, no_tail_tiles=True)
    assert int(plan.status.item()) == 0
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(out), want, f"no tail tiles T={T} H={H} I={I} E={E} k={k}")


@pytest.mark.parametrize("T,H,I,E,k", ODD_SHAPES + [(2000, 320, 384, 7, 2), (1500, 256, 256, 64, 6)])
def test_fused_gather_matches_gather_kernel(T, H, I, E, k):
    """FC1 copying its rows from x (gather warps) runs the same MMAs on the
    same rows as FC1 on the gather kernel's copy: the outputs are bitwise
    equal, and equal the oracle within the acceptance rule."""
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", seed=T + E)
    d = _dev(wl)
    out_f, plan_f = _forward(wl, d, moe.PATH_GROUPED, fused_gather=True)
    out_f = out_f.clone()
    out_g, _ = _forward(wl, d, moe.PATH_GROUPED)
    assert int(plan_f.status.item()) == 0
    assert torch.equal(out_f, out_g), f"fused gather differs: T={T} H={H} I={I} E={E} k={k}"
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(out_f), want, f"fused gather T={T} H={H} I={I} E={E} k={k}")


def test_replays_bitwise_identical_and_graph_capture():
    wl = W.make_moe(T=600, H=256, I=192, E=12, top_k=3, mode="logits", seed=1)
    d = _dev(wl)
    plan = moe.MoEPlan(d["x"], d["w1"], d["w2"], wl.E, wl.top_k, logits=d["logits"])
    b = plan.buffers()
    R = wl.T * wl.top_k

    ws = plan.workspace

    def inter_bytes():
        """Raw bytes of the intermediates the launch left in the workspace."""
        parts = []
        for name, nbytes in (("topk_ids", R * 4), ("topk_w", R * 4), ("m_indptr", (wl.E + 1) * 4),
                             ("perm_to_exp", R * 4), ("exp_to_perm", R * 4), ("h", R * wl.I * 2),
                             ("y", R * wl.H * 4)):
            off = b[name] - ws.data_ptr()
            parts.append(ws[off:off + nbytes].clone())
        return parts

    ref = plan.launch().clone()
    torch.cuda.synchronize()
    ref_inter = inter_bytes()
    for _ in range(5):
        ws.fill_(0xAB)
        plan.launch()
        torch.cuda.synchronize()
        assert torch.equal(plan.out, ref)
        for a, c in zip(inter_bytes(), ref_inter):
            assert torch.equal(a, c)
    # the same plan captured in a CUDA graph
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        plan.launch()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    plan.out.zero_()
    with torch.cuda.graph(g):
        plan.launch()
    for _ in range(3):
        plan.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(plan.out, ref)
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(ref), want, "replay")


def test_prepared_launch_sees_new_values():
    wl = W.make_moe(T=100, H=128, I=128, E=5, top_k=2, mode="logits", seed=2)
    d = _dev(wl)
    plan = moe.MoEPlan(d["x"], d["w1"], d["w2"], wl.E, wl.top_k, logits=d["logits"])
    plan.launch()
    wl2 = W.make_moe(T=100, H=128, I=128, E=5, top_k=2, mode="logits", seed=3)
    d["x"].copy_(wl2.x.to(DEV))
    d["logits"].copy_(wl2.logits.to(DEV))
    wl2.w1, wl2.w2 = wl.w1, wl.w2
    out = plan.launch()
    torch.cuda.synchronize()
    want, _ = _oracle_out(wl2)
    check_bf16_end_to_end(W.bf16_bits(out), want, "rebound values")


@pytest.mark.parametrize("off,L", [(0, 3), (3, 4), (7, 1), (0, 8)])
def test_expert_parallel_shard(off, L):
    full = W.make_moe(T=64, H=128, I=128, E=8, top_k=3, mode="logits", seed=4)
    wl = W.make_moe(T=64, H=128, I=128, E=8, top_k=3, mode="logits", seed=4)
    wl.w1, wl.w2 = full.w1[off:off + L].contiguous(), full.w2[off:off + L].contiguous()
    wl.local_offset, wl.num_local = off, L
    out, _ = _forward(wl, _dev(wl))
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(out), want, f"shard {off}+{L}")


@pytest.mark.parametrize("T,path,chain", [(32, moe.PATH_AUTO, None), (8, moe.PATH_DECODE, None),
                                          (8, moe.PATH_DECODE, True), (200, moe.PATH_GROUPED, False)])
def test_shard_with_no_routed_tokens_is_zero(T, path, chain):
    """No route lands in the local shard: every form (five decode kernels,
    the chain in one launch or two kernels, the grouped path) writes zeros."""
    wl = W.make_moe(T=T, H=128, I=128, E=8, top_k=2, mode="prerouted", seed=5)
    wl.topk_ids = torch.zeros_like(wl.topk_ids)
    wl.topk_ids[:, 1] = 1
    wl.w1, wl.w2 = wl.w1[4:6].contiguous(), wl.w2[4:6].contiguous()
    wl.local_offset, wl.num_local = 4, 2
    d = _dev(wl)
    out, plan = _forward(wl, d, path, decode_chain=chain)
    assert torch.all(out == 0)
    plan.out.fill_(3.0)  # a second launch writes the zeros again (the chain's counters reset)
    plan.launch()
    torch.cuda.synchronize()
    assert torch.all(plan.out == 0)


def test_bad_expert_ids_flagged_and_dropped():
    wl = W.make_moe(T=50, H=128, I=64, E=6, top_k=2, mode="prerouted", seed=6)
    ids = wl.topk_ids.clone()
    ids[3, 0] = 6
    ids[10, 1] = -1
    wl.topk_ids = ids
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, _ = _forward(wl, _dev(wl), status=status)
    assert int(status.item()) & moe.DEV_BAD_EXPERT
    want, st = _oracle_out(wl)
    assert st == oracle.BAD_EXPERT
    check_bf16_end_to_end(W.bf16_bits(out), want, "bad ids")


def test_zero_tokens_is_noop():
    wl = W.make_moe(T=0, H=128, I=64, E=4, top_k=2, mode="logits", seed=1)
    out, _ = _forward(wl, _dev(wl))
    assert out.shape == (0, 128)


def test_all_tokens_on_one_expert():
    wl = W.make_moe(T=400, H=128, I=128, E=16, top_k=2, mode="prerouted", seed=8)
    ids = torch.full_like(wl.topk_ids, 5)
    ids[:, 1] = 9
    wl.topk_ids = ids
    out, _ = _forward(wl, _dev(wl))
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(out), want, "one expert")


# ---------------------------------------------------------- workload shapes --

@pytest.mark.parametrize("chain", [False, True, None, "one_launch"])
@pytest.mark.parametrize("name", ["decode_t1", "decode_t8", "decode_t64"])
@pytest.mark.parametrize("path", PATHS)
def test_decode_configs_full(name, path, chain):
    wl = W.make_moe(name)
    one = chain == "one_launch"
    out, _ = _forward(wl, _dev(wl), path, decode_chain=True if one else chain, one_launch=one)
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(out), want, name)


@pytest.mark.parametrize("T,kernels", [(1, 1), (4, 1), (8, 5)])
def test_decode_form_chosen_by_route_count(T, kernels):
    """Without a flag the decode path runs the chain as one launch for at
    most 32 routes (T <= 4 at top-8) and the five separate kernels above."""
    wl = W.make_moe(T=T, H=256, I=128, E=16, top_k=8, mode="prerouted", seed=T)
    out, plan = _forward(wl, _dev(wl), moe.PATH_AUTO, decode_chain=None)
    assert plan.kernels_per_launch() == kernels
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(out), want, f"T={T} automatic decode form")


@pytest.mark.parametrize("T,H,I,E,k,mode", [(3, 64, 192, 8, 2, "prerouted"), (5, 192, 64, 6, 3, "logits"),
                                             (40, 128, 320, 16, 4, "prerouted"),
                                             (20, 192, 320, 64, 8, "prerouted"), (64, 192, 320, 128, 8, "logits")])
@pytest.mark.parametrize("one", [False, True])
def test_decode_chain_small_shapes(T, H, I, E, k, mode, one):
    """The decode chain (two kernels, or one launch) at shapes with one
    k-block (FC1 at H = 64, FC2 at I = 64) and odd k-block counts (H = 192,
    I = 320, 192): the k-blocks alternate between two accumulators.  T = 20
    takes the 32-token tile form; the last two shapes give CTAs several
    tiles (in one launch, FC1 tiles and then FC2 tiles)."""
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode=mode, seed=T + H)
    out, _ = _forward(wl, _dev(wl), moe.PATH_DECODE, decode_chain=True, one_launch=one)
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(out), want, "decode chain")


def _sample_tokens(ids, T, n, seed):
    """n seeded random tokens plus, for every expert that receives routes, the
    first token routed to it (each output row depends only on its own token,
    so a subset check is exact for those rows)."""
    rng = np.random.default_rng(seed)
    chosen = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    flat = ids.reshape(T, -1)
    seen = set()
    for t in range(T):
        for e in flat[t]:
            if e not in seen:
                seen.add(int(e))
                chosen.add(t)
    return np.array(sorted(chosen), dtype=np.int32)


@pytest.mark.parametrize("form", ["pair", "pair_alone", "one_cta", "fused_gather"])
@pytest.mark.parametrize("name", ["prefill_few_large", "prefill_many_fine"])
def test_prefill_configs_sampled(name, form):
    """pair: the plan's default (at the many-fine-experts workload the
    small-group kernel beside the CTA-pair GEMMs); pair_alone: the CTA-pair
    GEMMs without it."""
    wl = W.make_moe(name, weights_device=DEV)
    d = _dev(wl)
    out, _ = _forward(wl, d, one_cta_gemm=form == "one_cta", fused_gather=form == "fused_gather",
                      small_group_kernel=False if form == "pair_alone" else None)
    ids, _ = _oracle_route(wl)
    tokens = _sample_tokens(ids, wl.T, 1024, 0)
    want, _ = _oracle_out(wl, tokens=tokens, w1=W.bf16_bits(wl.w1), w2=W.bf16_bits(wl.w2))
    check_bf16_end_to_end(W.bf16_bits(out)[tokens], want, f"{name} ({len(tokens)} sampled tokens)")


def test_grouped_gemm_config_full_size_sampled():
    d = W.make_grouped_gemm(seed=0, device="cpu", weights_device=DEV)
    X, Wt, offs = d["X"].to(DEV), d["W"], d["offs"].to(DEV)
    Y = moe.grouped_gemm_fwd(X, Wt, offs)
    torch.cuda.synchronize()
    ends = d["offs"].numpy()
    starts = np.concatenate([[0], ends[:-1]])
    rows = set(np.random.default_rng(0).integers(0, d["sum_m"], 1024).tolist())
    for s, e in zip(starts, ends):
        if e > s:
            rows.update([int(s), int(e) - 1])
    rows = np.array(sorted(rows), dtype=np.int32)
    Yo = oracle.grouped_gemm_rows(W.bf16_bits(d["X"]), W.bf16_bits(Wt), ends, rows)
    check_bf16_close(W.bf16_bits(Y)[rows], Yo, "grouped GEMM 16384x1536x4096")


# ----------------------------------------- stage chain at the workload shapes --

def _stage_chain(wl, tokens, swapab=False):
    """Full-size stage parity with the oracle's intermediates as inputs:
    GPU FC1+SwiGLU on the oracle's gathered rows against the oracle's h, and
    GPU FC2 + finalize on the oracle's h against the oracle's output; both
    under the strict rule (errors do not compound)."""
    ids, w = _oracle_route(wl)
    T, k, E = wl.T, wl.top_k, wl.E
    R = T * k
    want, h_o, _, st = oracle.moe_tokens(W.bf16_bits(wl.x), ids, w, W.bf16_bits(wl.w1), W.bf16_bits(wl.w2), E,
                                         tokens=tokens, want_intermediates=True)
    m_o, p2e_o, e2p_o, _ = oracle.sort(ids, E)
    w1, w2 = wl.w1.to(DEV), wl.w2.to(DEV)
    m_d = torch.from_numpy(m_o).to(DEV)
    # FC1: rows of the sampled routes only need to be right
    xp = np.zeros((R, wl.H), np.uint16)
    xp[:len(p2e_o)] = W.bf16_bits(wl.x)[p2e_o // k]
    if swapab:
        h_g = moe.moe_fc1_swiglu_swapab(W.from_bf16_bits(xp).to(DEV), w1, m_d, max(1, wl.T))
    else:
        h_g = moe.moe_fc1_swiglu(W.from_bf16_bits(xp).to(DEV), w1, m_d)
    slots = (tokens[:, None] * k + np.arange(k)[None, :]).ravel()
    rows = e2p_o[slots]
    check_bf16_close(W.bf16_bits(h_g)[rows], h_o, f"{wl.name}: h (FC1 on the oracle's rows)")
    # FC2 + finalize on the oracle's h
    h_in = np.zeros((R, wl.I), np.uint16)
    h_in[rows] = h_o
    if swapab:
        y = moe.moe_fc2_swapab(W.from_bf16_bits(h_in).to(DEV), w2, m_d, max(1, wl.T))
    else:
        y = moe.moe_fc2(W.from_bf16_bits(h_in).to(DEV), w2, m_d)
    out = moe.moe_finalize(y, torch.from_numpy(e2p_o).to(DEV), torch.from_numpy(w).to(DEV))
    torch.cuda.synchronize()
    check_bf16_close(W.bf16_bits(out)[tokens], want, f"{wl.name}: out (FC2 + finalize on the oracle's h)")


@pytest.mark.parametrize("swapab", [False, True])
@pytest.mark.parametrize("name", ["tiny", "decode_t1", "decode_t8", "decode_t64"])
def test_stage_chain_small_configs(name, swapab):
    wl = W.make_moe(name)
    _stage_chain(wl, np.arange(wl.T, dtype=np.int32), swapab)


@pytest.mark.parametrize("name", ["prefill_few_large", "prefill_many_fine"])
def test_stage_chain_prefill_configs(name):
    wl = W.make_moe(name, weights_device=DEV)
    ids, _ = _oracle_route(wl)
    _stage_chain(wl, _sample_tokens(ids, wl.T, 512, 1))


# ------------------------------------------------- decode chain (T * k <= 1024) --

@pytest.mark.parametrize("one", [False, True])
@pytest.mark.parametrize("name", ["decode_t1", "decode_t8", "decode_t64"])
def test_decode_chain_replays_bitwise_and_graph(name, one):
    """The decode chain combines each (token, column block) in the tile that
    arrives last; the sum order is fixed, so replays, in any arrival order,
    are bitwise identical.  In one launch this also checks that the
    per-expert counters start from zero again at every launch."""
    wl = W.make_moe(name)
    d = _dev(wl)
    plan = moe.MoEPlan(d["x"], d["w1"], d["w2"], wl.E, wl.top_k, topk_ids=d["topk_ids"], topk_w=d["topk_w"],
                       path=moe.PATH_DECODE, decode_chain=True, decode_one_launch=one)
    assert plan.kernels_per_launch() == (1 if one else 2)
    ref = plan.launch().clone()
    torch.cuda.synchronize()
    for _ in range(5):
        plan.out.fill_(1.0)
        plan.launch()
        torch.cuda.synchronize()
        assert torch.equal(plan.out, ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        plan.launch()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.launch()
    for _ in range(3):
        plan.out.fill_(2.0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(plan.out, ref)
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(ref), want, f"{name} chain")
    # the chain publishes its sort like the sort kernel would
    b = plan.buffers()
    ids = wl.topk_ids.numpy()
    m_o, p2e_o, e2p_o, _ = oracle.sort(ids, wl.E)
    ws = plan.workspace
    R = wl.T * wl.top_k

    def view(name, n):
        off = b[name] - ws.data_ptr()
        return ws[off:off + 4 * n].view(torch.int32).cpu().numpy()
    assert np.array_equal(view("m_indptr", wl.E + 1), m_o)
    assert np.array_equal(view("exp_to_perm", R), e2p_o)
    assert np.array_equal(view("perm_to_exp", len(p2e_o)), p2e_o)


@pytest.mark.parametrize("one", [False, True])
@pytest.mark.parametrize("T", [1, 3])
def test_decode_chain_repeated_ids(T, one):
    """Pre-routed ids may repeat an expert inside a token's routes: every
    route lands on expert 2, giving it 8 (T = 1) or 24 (T = 3, more than one
    16-row block) rows; the chain still matches the oracle."""
    wl = W.make_moe(T=T, H=256, I=192, E=16, top_k=8, mode="prerouted", seed=40 + T)
    wl.topk_ids = torch.full_like(wl.topk_ids, 2)
    out, _ = _forward(wl, _dev(wl), moe.PATH_DECODE, decode_chain=True, one_launch=one)
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(out), want, f"repeated ids T={T}")


def test_decode_one_launch_first_launch_captured():
    """A one-launch chain plan whose first launch is captured in a CUDA graph:
    the graph holds the zeroing of the kernel's counters (every launch zeroes
    them), and every replay gives the oracle's output."""
    wl = W.make_moe(T=2, H=256, I=192, E=16, top_k=4, mode="prerouted", seed=31)
    d = _dev(wl)
    plan = moe.MoEPlan(d["x"], d["w1"], d["w2"], wl.E, wl.top_k, topk_ids=d["topk_ids"], topk_w=d["topk_w"],
                       path=moe.PATH_DECODE, decode_one_launch=True)
    assert plan.kernels_per_launch() == 1
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.launch()
    want, _ = _oracle_out(wl)
    for _ in range(3):
        plan.out.fill_(5.0)
        g.replay()
        torch.cuda.synchronize()
        check_bf16_end_to_end(W.bf16_bits(plan.out), want, "captured first launch")
    plan.out.fill_(5.0)
    plan.launch()  # and a direct launch after the replays
    torch.cuda.synchronize()
    check_bf16_end_to_end(W.bf16_bits(plan.out), want, "launch after replays")


def test_plans_sharing_one_workspace_alternate():
    """A grouped-path plan and a one-launch decode plan bound to the same
    workspace, launched alternately: the grouped path's rows overwrite the
    bytes where the decode kernel keeps its counters, and every launch still
    gives the oracle's output with a clean status word."""
    wl_g = W.make_moe(T=600, H=256, I=192, E=12, top_k=3, mode="logits", seed=61)
    wl_d = W.make_moe(T=3, H=256, I=192, E=12, top_k=4, mode="prerouted", seed=62)
    need = max(moe.moe_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.top_k, wl.num_local) for wl in (wl_g, wl_d))
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    plans = []
    for wl, path, one in ((wl_g, moe.PATH_GROUPED, False), (wl_d, moe.PATH_DECODE, True)):
        d = _dev(wl)
        st = torch.full((1,), 0x40, dtype=torch.int32, device=DEV)
        p = moe.MoEPlan(d["x"], d["w1"], d["w2"], wl.E, wl.top_k, logits=d["logits"], topk_ids=d["topk_ids"],
                        topk_w=d["topk_w"], workspace=ws, status=st, path=path, decode_one_launch=one)
        plans.append((wl, p, _oracle_out(wl)[0]))
    assert plans[1][1].kernels_per_launch() == 1
    for rnd in range(3):
        for wl, p, want in (plans[1], plans[0]) if rnd % 2 == 0 else plans:
            p.out.fill_(3.0)
            p.launch()
            torch.cuda.synchronize()
            assert int(p.status.item()) == 0
            check_bf16_end_to_end(W.bf16_bits(p.out), want, f"shared workspace {wl.name} T={wl.T} round {rnd}")


def test_bounded_wait_runs_out_reports_and_the_next_launch_is_right():
    """A one-launch decode chain whose FC2 tiles wait for FC1 counts that can
    never complete (test hook: the counts start at -1) with a 2 ms wait limit:
    the launch returns, the status word carries MOE_DEV_TIMEOUT, and a normal
    plan on the same buffers and workspace then gives the oracle's output with
    a clean status word (the context stays usable)."""
    import time
    wl = W.make_moe(T=2, H=256, I=192, E=16, top_k=4, mode="prerouted", seed=71)
    d = _dev(wl)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    need = moe.moe_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.top_k, wl.num_local)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=DEV)
    kw = dict(topk_ids=d["topk_ids"], topk_w=d["topk_w"], out=out, workspace=ws, status=status,
              path=moe.PATH_DECODE, decode_one_launch=True)
    hooked = moe.MoEPlan(d["x"], d["w1"], d["w2"], wl.E, wl.top_k, test_unreachable_wait=True, **kw)
    hooked.set_wait_limit(2_000_000)
    assert hooked.kernels_per_launch() == 1
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    hooked.launch()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) & moe.DEV_TIMEOUT, f"status {int(status.item())}"
    assert dt < 2.0, f"the launch took {dt:.3f} s"
    normal = moe.MoEPlan(d["x"], d["w1"], d["w2"], wl.E, wl.top_k, **kw)
    want, _ = _oracle_out(wl)
    for _ in range(2):
        out.fill_(7.0)
        normal.launch()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        check_bf16_end_to_end(W.bf16_bits(out), want, "launch after a timed-out launch")


@pytest.mark.parametrize("one", [False, True])
def test_decode_chain_status_and_bad_ids(one):
    wl = W.make_moe(T=6, H=128, I=128, E=9, top_k=3, mode="prerouted", seed=12)
    ids = wl.topk_ids.clone()
    ids[2, 1] = 40
    wl.topk_ids = ids
    status = torch.full((1,), 0x40, dtype=torch.int32, device=DEV)  # stale bits are cleared
    out, plan = _forward(wl, _dev(wl), moe.PATH_DECODE, status=status, decode_chain=True, one_launch=one)
    assert plan.kernels_per_launch() == (1 if one else 2)
    assert int(status.item()) == moe.DEV_BAD_EXPERT
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(out), want, "chain bad ids")
    wl.topk_ids = wl.topk_ids.clamp(0, 8)
    d = _dev(wl)
    out2, _ = _forward(wl, d, moe.PATH_DECODE, status=status, decode_chain=True, one_launch=one)
    assert int(status.item()) == 0


@pytest.mark.parametrize("one", [False, True])
@pytest.mark.parametrize("off,L", [(0, 5), (5, 4), (2, 1)])
def test_decode_chain_expert_shard(off, L, one):
    full = W.make_moe(T=12, H=192, I=128, E=9, top_k=4, mode="logits", seed=21)
    wl = W.make_moe(T=12, H=192, I=128, E=9, top_k=4, mode="logits", seed=21)
    wl.w1, wl.w2 = full.w1[off:off + L].contiguous(), full.w2[off:off + L].contiguous()
    wl.local_offset, wl.num_local = off, L
    out, plan = _forward(wl, _dev(wl), moe.PATH_DECODE, decode_chain=True, one_launch=one)
    assert plan.kernels_per_launch() == (2 if one else 3)  # route + the chain kernel(s)
    want, _ = _oracle_out(wl)
    check_bf16_end_to_end(W.bf16_bits(out), want, f"chain shard {off}+{L}")


# ------------------------------------------------------- SwiGLUStep(limit) --

def _limits(L, seed):
    """Per-expert limits that bind on N(0,1) GEMM1 outputs (plus one +inf)."""
    lim = np.random.default_rng(seed).uniform(0.4, 2.5, size=L).astype(np.float32)
    lim[0] = np.inf
    return lim


@pytest.mark.parametrize("T,H,I,E,k", [(600, 256, 192, 12, 3), (40, 512, 256, 9, 4)])
def test_swiglu_step_stage_parity(T, H, I, E, k):
    """moe_fc1_swiglu with clamp limits on the oracle's gathered rows against
    the oracle's SwiGLUStep h (strict rule); limits of +inf give moe_fc1_swiglu
    bitwise."""
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", seed=T + 5)
    ids, _ = _oracle_route(wl)
    m_o, p2e_o, _, _ = oracle.sort(ids, E)
    xp = W.bf16_bits(wl.x)[p2e_o // k]
    lim = _limits(E, T)
    rows = np.arange(len(p2e_o), dtype=np.int32)
    want = oracle.fc1_swiglu_rows(xp, W.bf16_bits(wl.w1), m_o[1:], rows, clamp_limit=lim)
    xp_d, w1_d, m_d = W.from_bf16_bits(xp).to(DEV), wl.w1.to(DEV), torch.from_numpy(m_o).to(DEV)
    h = moe.moe_fc1_swiglu(xp_d, w1_d, m_d, clamp_limit=torch.from_numpy(lim).to(DEV))
    torch.cuda.synchronize()
    check_bf16_close(W.bf16_bits(h), want, f"SwiGLUStep h T={T} H={H} I={I}")
    plain = moe.moe_fc1_swiglu(xp_d, w1_d, m_d)
    inf = moe.moe_fc1_swiglu(xp_d, w1_d, m_d, clamp_limit=torch.full((E,), float("inf"), device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(plain, inf)
    assert not torch.equal(plain, h)  # the finite limits bind


@pytest.mark.parametrize("form", ["pair", "one_cta", "decode_separate", "decode_chain", "one_launch"])
def test_swiglu_step_layer_every_form(form):
    """The whole layer with per-expert SwiGLUStep limits on every kernel form
    against the oracle's SwiGLUStep layer."""
    decode = form.startswith("decode") or form == "one_launch"
    T = 3 if decode else 600
    wl = W.make_moe(T=T, H=256, I=192, E=12, top_k=3, mode="logits", seed=90 + T)
    d = _dev(wl)
    lim = _limits(wl.E, 7)
    plan = moe.MoEPlan(d["x"], d["w1"], d["w2"], wl.E, wl.top_k, logits=d["logits"],
                       path=moe.PATH_DECODE if decode else moe.PATH_GROUPED, one_cta_gemm=form == "one_cta",
                       decode_chain=True if form == "decode_chain" else (False if form == "decode_separate" else None),
                       decode_one_launch=form == "one_launch", clamp_limit=torch.from_numpy(lim).to(DEV))
    out = plan.launch()
    torch.cuda.synchronize()
    assert int(plan.status.item()) == 0
    want, _ = _oracle_out(wl, clamp_limit=lim)
    check_bf16_end_to_end(W.bf16_bits(out), want, f"SwiGLUStep layer ({form})")
    plain, _ = _oracle_out(wl)
    assert not np.array_equal(np.asarray(plain), np.asarray(want))  # the limits change the layer
