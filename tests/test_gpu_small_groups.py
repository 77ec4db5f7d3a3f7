"""The small-group kernel beside the CTA-pair GEMMs: on the grouped path the
groups of at most 64 rows run in a one-CTA swap-AB kernel on a few SMs while
the pair kernel takes the larger groups, both claiming tiles at run time
(MOE_PLAN_SMALL_GROUP_KERNEL forces it, MOE_PLAN_NO_SMALL_GROUP_KERNEL turns it
off, plans with at most 512 routes per local expert use it by default).

Checked against the CPU oracle through the C ABI: stage by stage on the plan's
own intermediates (FC1's h from the gathered rows, FC2 + finalize from h) under
the strict rule, and end to end under the accumulation model's floor.  The
layer output is also compared bit for bit with the pair kernel alone: each
tile is computed whole by one CTA, the K order of its sums does not depend on
the kernel, and tensor-core MMAs give an element the same value whatever the
instruction's shape, so which kernel claims a tile does not change a bit (the
property that keeps replays bitwise identical under run-time claims)."""
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


def _plan(wl, side, ids=None, w=None, clamp=None, local_offset=0, workspace=None):
    logits = None if ids is not None else wl.logits.to(DEV)
    tid = None if ids is None else torch.from_numpy(np.ascontiguousarray(ids, np.int32)).to(DEV)
    tw = None if w is None else torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(DEV)
    return moe.MoEPlan(wl.x.to(DEV), wl.w1.to(DEV), wl.w2.to(DEV), wl.E, wl.top_k, logits=logits, topk_ids=tid,
                       topk_w=tw, local_offset=local_offset, path=moe.PATH_GROUPED, small_group_kernel=side,
                       workspace=workspace,
                       clamp_limit=None if clamp is None else torch.from_numpy(clamp).to(DEV))


def _ws(plan, key, count, dtype):
    """count elements of a plan buffer (workspace bytes) as a numpy array."""
    b = plan.buffers()
    off = b[key] - plan.workspace.data_ptr()
    nbytes = count * np.dtype(dtype).itemsize
    return plan.workspace[off:off + nbytes].cpu().numpy().view(dtype)


def _routes(wl):
    if wl.mode == "logits":
        return oracle.route(wl.logits.numpy(), wl.top_k)
    return wl.topk_ids.numpy(), wl.topk_w.numpy()


def _ids_with_counts(counts, k, seed):
    """Pre-routed ids whose per-expert route counts are `counts` (each token
    k distinct experts; requires max(counts) <= sum(counts) / k)."""
    lst = np.repeat(np.arange(len(counts)), counts)
    T = len(lst) // k
    assert T * k == len(lst) and counts.max() <= T
    ids = np.empty((T, k), np.int32)
    for j, e in enumerate(lst):  # copy j of the list goes to token j % T: an expert's copies to distinct tokens
        ids[j % T, j // T] = e
    w = np.random.default_rng(seed).dirichlet(np.ones(k), size=T).astype(np.float32)
    return ids, w


def _end_to_end(wl, out, ids, w, clamp=None, local_offset=0, num_local=None, what=""):
    x, w1, w2 = W.bf16_bits(wl.x), W.bf16_bits(wl.w1), W.bf16_bits(wl.w2)
    want, st = oracle.moe_tokens(x, ids, w, w1, w2, wl.E, local_offset=local_offset, num_local=num_local,
                                 clamp_limit=clamp)
    frac, n = accum_model.floor(x, ids, w, w1, w2, wl.E, want, local_offset=local_offset, num_local=num_local,
                                clamp_limit=clamp)
    check_bf16_end_to_end(W.bf16_bits(out), with_floor(want, frac, n), what)


SHAPES = [  # T, H, I, E, top_k, routing bias
    (512, 512, 256, 64, 8, "zipf1.2"),
    (300, 256, 128, 32, 4, "zipf1.2"),
    (2048, 1024, 512, 128, 8, "zipf1.2"),
    (96, 384, 192, 48, 6, None),
]


@pytest.mark.parametrize("si", range(len(SHAPES)))
def test_stages_and_end_to_end(si):
    T, H, I, E, k, bias = SHAPES[si]
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", bias=bias, seed=90 + si)
    ids, w = _routes(wl)
    cnt = np.bincount(ids.ravel(), minlength=E)
    assert ((cnt > 0) & (cnt <= 64)).sum() > 0, "the shape must have small groups"
    plan = _plan(wl, True)
    out = plan.launch().clone()
    torch.cuda.synchronize()
    assert int(plan.status.item()) == 0
    m, p2e, e2p, _ = oracle.sort(ids, E)
    M = len(p2e)
    xp = _ws(plan, "xp", M * H, np.uint16).reshape(M, H)
    assert np.array_equal(xp, W.bf16_bits(wl.x)[p2e // k])
    rows = np.arange(M, dtype=np.int32)
    h = _ws(plan, "h", M * I, np.uint16).reshape(M, I)
    check_bf16_close(h, oracle.fc1_swiglu_rows(xp, W.bf16_bits(wl.w1), m[1:], rows), f"shape {si}: h")
    y_o = oracle.fc2_rows(h, W.bf16_bits(wl.w2), m[1:], rows)
    check_bf16_close(W.bf16_bits(out), oracle.finalize(y_o, e2p, w), f"shape {si}: FC2 + finalize on the plan's h")
    _end_to_end(wl, out, ids, w, what=f"shape {si} end to end")


@pytest.mark.parametrize("si", [0, 2])
def test_bitwise_same_as_pair_kernel_alone_and_replays(si):
    T, H, I, E, k, bias = SHAPES[si]
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", bias=bias, seed=90 + si)
    outs = {}
    for side in (True, False):
        plan = _plan(wl, side)
        ref = plan.launch().clone()
        torch.cuda.synchronize()
        for _ in range(5):
            plan.out.fill_(0)
            plan.launch()
            torch.cuda.synchronize()
            assert torch.equal(plan.out, ref)
        outs[side] = ref
    assert torch.equal(outs[True], outs[False])
    # replays of a captured graph, with the claim counters cleared inside it
    plan = _plan(wl, True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.launch(s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            plan.launch(s)
    for _ in range(3):
        plan.out.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(plan.out, outs[True])
    assert int(plan.status.item()) == 0


def test_group_size_boundaries():
    """Groups of 1, 15-17, 31-33, 63-65, 128, 129, 300 rows and empty ones:
    the token-box heights (16, 32, 64) and the kernel's 64-row limit."""
    counts = np.array([1, 15, 16, 17, 0, 31, 32, 33, 63, 64, 65, 128, 129, 300, 0, 4], np.int64)
    ids, w = _ids_with_counts(counts, 2, seed=5)
    T = ids.shape[0]
    wl = W.make_moe(T=T, H=320, I=192, E=len(counts), top_k=2, mode="prerouted", seed=7)
    outs = {}
    for side in (True, False):
        plan = _plan(wl, side, ids, w)
        outs[side] = plan.launch().clone()
        torch.cuda.synchronize()
        assert int(plan.status.item()) == 0
    assert torch.equal(outs[True], outs[False])
    _end_to_end(wl, outs[True], ids, w, what="group size boundaries")


def test_forced_without_small_groups_and_only_small_groups():
    # every group above 64 rows: the small-group kernel finds no tiles
    wl = W.make_moe(T=1024, H=256, I=256, E=8, top_k=2, mode="prerouted", seed=11)
    ids, w = _routes(wl)
    assert np.bincount(ids.ravel(), minlength=8).min() > 64
    outs = [_plan(wl, side, ids, w).launch().clone() for side in (True, False)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    _end_to_end(wl, outs[0], ids, w, what="no small groups, kernel forced")
    # every group at most 64 rows (and the default choice takes the kernel)
    wl = W.make_moe(T=128, H=256, I=128, E=64, top_k=4, mode="prerouted", seed=12)
    ids, w = _routes(wl)
    assert np.bincount(ids.ravel(), minlength=64).max() <= 64
    plan = _plan(wl, None, ids, w)
    assert plan.kernels_per_launch() == _plan(wl, False, ids, w).kernels_per_launch() + 2
    out = plan.launch().clone()
    torch.cuda.synchronize()
    _end_to_end(wl, out, ids, w, what="only small groups")


def test_clamp_and_local_expert_range():
    wl = W.make_moe(T=512, H=256, I=256, E=64, top_k=8, mode="logits", bias="zipf1.2", seed=21,
                    local_offset=16, num_local=32)
    ids, w = _routes(wl)
    clamp = np.random.default_rng(3).uniform(0.3, 2.0, size=32).astype(np.float32)
    clamp[0] = np.inf
    outs = {side: _plan(wl, side, clamp=clamp, local_offset=16).launch().clone() for side in (True, False)}
    torch.cuda.synchronize()
    assert torch.equal(outs[True], outs[False])
    _end_to_end(wl, outs[True], ids, w, clamp=clamp, local_offset=16, num_local=32, what="clamp, experts 16..47")


def test_plans_sharing_a_workspace():
    """Two plans on one workspace, launched in turn: the claim counters live
    in the workspace and every launch clears them first."""
    wa = W.make_moe(T=512, H=256, I=128, E=64, top_k=8, mode="logits", bias="zipf1.2", seed=31)
    wb = W.make_moe(T=256, H=256, I=128, E=16, top_k=2, mode="logits", seed=32)
    need = max(moe.moe_workspace_size(512, 256, 128, 64, 8), moe.moe_workspace_size(256, 256, 128, 16, 2))
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    pa, pb = _plan(wa, True, workspace=ws), _plan(wb, None, workspace=ws)
    ref_a, ref_b = pa.launch().clone(), pb.launch().clone()
    for _ in range(3):
        assert torch.equal(pa.launch(), ref_a)
        assert torch.equal(pb.launch(), ref_b)
    torch.cuda.synchronize()
    ids, w = _routes(wa)
    _end_to_end(wa, ref_a, ids, w, what="shared workspace, plan A")


def test_e4m3_family_with_small_groups():
    T, H, I, E, k = 512, 512, 256, 64, 8
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", bias="zipf1.2", seed=41)
    fw = W.make_fp8_weights(E, H, I, seed=41)
    ids, w = _routes(wl)
    e4 = dict(w1_scale=fw.s1.to(DEV), w2_scale=fw.s2.to(DEV), x_scale=fw.a1, h_scale=fw.a2)
    outs = {}
    for side in (True, False):
        plan = moe.MoEPlan(wl.x.to(DEV), fw.w1q.to(DEV), fw.w2q.to(DEV), E, k, logits=wl.logits.to(DEV), e4m3=e4,
                           small_group_kernel=side)
        outs[side] = plan.launch().clone()
        torch.cuda.synchronize()
        assert int(plan.status.item()) == 0
    assert torch.equal(outs[True], outs[False])
    x = W.bf16_bits(wl.x)
    args = (x, ids, w, fw.w1q.numpy(), fw.w2q.numpy(), fw.s1.numpy(), fw.s2.numpy(), fw.a1, fw.a2, E)
    want, st = oracle.moe_tokens_fp8(*args)
    frac, n = accum_model.floor_e4m3(*args, want)
    from tests.tolerances import RMS_FRAC_E4M3
    check_bf16_end_to_end(W.bf16_bits(outs[True]), with_floor(want, frac, n), "E4M3 with small groups",
                          rms_frac=RMS_FRAC_E4M3)


@pytest.mark.parametrize("sizes,N,K", [
    ([1, 16, 17, 64, 65, 128, 300, 0, 33], 256, 320),
    ([0, 0, 0, 7], 1536, 512),
    (np.random.default_rng(7).integers(0, 90, 200).tolist(), 512, 192)])
def test_grouped_gemm_fwd_with_small_groups(sizes, N, K):
    """The ragged grouped GEMM forward with the small-group kernel (caller's
    counters): bitwise the same as the pair kernel alone, and the oracle's Y;
    rows past the last group untouched."""
    d = W.make_grouped_gemm(seed=len(sizes) + 900, sizes=sizes, N=N, K=K)
    X, Wt, offs = d["X"].to(DEV), d["W"].to(DEV), d["offs"].to(DEV)
    counters = torch.full((moe.GROUPED_GEMM_COUNTERS,), 12345, dtype=torch.int32, device=DEV)
    sentinel = torch.full((d["sum_m"] + 3, N), -7.0, dtype=torch.bfloat16, device=DEV)
    Y = sentinel[:d["sum_m"]]
    moe.grouped_gemm_fwd(X, Wt, offs, Y, small_group_kernel=True, counters=counters)
    Y_off = moe.grouped_gemm_fwd(X, Wt, offs, small_group_kernel=False)
    moe.grouped_gemm_fwd(X, Wt, offs, Y, small_group_kernel=True, counters=counters)  # counters reused
    torch.cuda.synchronize()
    assert torch.equal(Y, Y_off)
    assert torch.all(sentinel[d["sum_m"]:] == -7.0)
    Yo = oracle.grouped_gemm_rows(W.bf16_bits(d["X"]), W.bf16_bits(d["W"]), d["offs"].numpy())
    check_bf16_close(W.bf16_bits(Y), Yo, "Y with the small-group kernel")


def test_grouped_gemm_fwd_full_size_with_small_groups():
    """The grouped-GEMM workload (sum_m = 16384, E = 64, K = 4096, N = 1536;
    22 groups of at most 64 rows): bitwise the same with and without the
    small-group kernel, and sampled rows of every group against the oracle."""
    d = W.make_grouped_gemm(seed=0, device="cpu", weights_device=DEV)
    X, Wt, offs = d["X"].to(DEV), d["W"], d["offs"].to(DEV)
    sizes = d["sizes"]
    assert ((sizes > 0) & (sizes <= 64)).sum() > 10
    Y_on = moe.grouped_gemm_fwd(X, Wt, offs, small_group_kernel=True)
    Y_off = moe.grouped_gemm_fwd(X, Wt, offs, small_group_kernel=False)
    torch.cuda.synchronize()
    assert torch.equal(Y_on, Y_off)
    ends = d["offs"].numpy()
    rows = set()
    for e in range(len(ends)):
        s0 = 0 if e == 0 else int(ends[e - 1])
        if ends[e] > s0:
            rows.update([s0, int(ends[e]) - 1, (s0 + int(ends[e])) // 2])
    rows = np.array(sorted(rows), dtype=np.int32)
    Yo = oracle.grouped_gemm_rows(W.bf16_bits(d["X"]), W.bf16_bits(Wt.cpu()), ends, rows)
    check_bf16_close(W.bf16_bits(Y_on)[rows], Yo, "grouped GEMM workload with the small-group kernel")
