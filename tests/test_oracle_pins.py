"""Pins for the CPU oracle against facts fixed outside the oracle itself.

Each test checks the oracle against something it does not compute the same
way: hand-worked cases, brute force over all subsets, an fp64 evaluation of
the layer written as a dense masked sum over every (token, expert) pair, a
library routine (numpy stable argsort, torch fp32 matmul, torch's bf16
rounding), or an invariant of the mathematics (sum of weights, identical
experts, token permutation, expert-range partition).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_expert_router_gb300 import workloads as W
from tests.tolerances import bf16_to_f64, check_bf16_close, ulp_distance

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def torch_bf16_bits(a64: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 with torch (a library rounding, RNE)."""
    t = torch.from_numpy(np.ascontiguousarray(a64, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- rounding --

def test_bf16_rounding_matches_torch():
    lib = oracle.load()
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(4000).astype(np.float32) * 10.0 ** rng.integers(-40, 38, 4000))
    # exact ties, values just around them, extremes
    for hi in (0x3F80, 0x3F81, 0xBF80, 0x0001, 0x7F7F, 0x0080):
        for lo in (0x7FFF, 0x8000, 0x8001):
            vals.append(np.array([(hi << 16) | lo], np.uint32).view(np.float32)[0])
    vals += [0.0, -0.0, np.float32(np.inf), np.float32(-np.inf), np.float32(3.4e38), np.float32(1e-45)]
    vals = np.array(vals, np.float32)
    got = np.array([lib.oracle_float_to_bf16(float(v)) for v in vals], np.uint16)
    want = torch_bf16_bits(vals)
    assert np.array_equal(got, want)


# ----------------------------------------------------------------- routing --

def test_route_hand_worked():
    cases = json.load(open(GOLDEN))["route"]
    for c in cases:
        lg = np.array([c["logits"]], np.float32)
        ids, w = oracle.route(lg, c["top_k"])
        assert ids[0].tolist() == c["ids"], c
        want = [eval(s, {"exp": math.exp}) for s in c["weights_closed_form"]]
        assert np.allclose(w[0], want, atol=1e-6, rtol=0), (w[0], want)


def _total_order_first_k(row, k):
    """Brute force: the k-subset S such that every member precedes every
    non-member under (logit desc, id asc); found by trying all subsets."""
    E = len(row)
    before = lambda a, b: row[a] > row[b] or (row[a] == row[b] and a < b)
    hits = []
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if all(before(a, b) for a in S for b in rest):
            hits.append(S)
    assert len(hits) == 1
    S = list(hits[0])
    # order inside S by the same total order (insertion, no sort call)
    ordered = []
    for a in S:
        pos = 0
        while pos < len(ordered) and before(ordered[pos], a):
            pos += 1
        ordered.insert(pos, a)
    return ordered


@pytest.mark.parametrize("E", [1, 2, 3, 5, 8])
def test_route_bruteforce_with_ties(E):
    rng = np.random.default_rng(E)
    T = 60
    lg = rng.integers(-2, 3, size=(T, E)).astype(np.float32) * np.float32(0.75)  # many ties
    for k in range(1, E + 1):
        ids, _ = oracle.route(lg, k)
        for t in range(T):
            assert ids[t].tolist() == _total_order_first_k(lg[t], k)


@pytest.mark.parametrize("E,k", [(4, 2), (8, 2), (128, 8), (256, 8), (64, 16)])
def test_route_weights_vs_fp64_softmax_topk_renorm(E, k):
    rng = np.random.default_rng(E * 100 + k)
    lg = (rng.standard_normal((200, E)) * 3).astype(np.float32)
    ids, w = oracle.route(lg, k)
    # an independent formulation: full softmax over all E in fp64, pick the
    # chosen ids, renormalise
    l64 = lg.astype(np.float64)
    p = np.exp(l64 - l64.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    ref = sel / sel.sum(axis=1, keepdims=True)
    assert np.max(np.abs(w - ref)) <= 1e-6
    assert np.max(np.abs(w.astype(np.float64).sum(axis=1) - 1.0)) <= 1e-6
    assert np.all(np.diff(w, axis=1) <= 0)  # descending weight order


def test_route_zipf_config_histogram():
    """The Zipf-biased configuration must contain empty and one-row groups."""
    wl = W.make_moe("prefill_many_fine", H=64, I=64)
    ids, _ = oracle.route(wl.logits.numpy(), wl.top_k)
    cnt = np.bincount(ids.ravel(), minlength=wl.E)
    assert (cnt == 0).sum() >= 1 and (cnt == 1).sum() >= 1
    assert cnt.sum() == wl.T * wl.top_k


# ----------------------------------------------------------------- sorting --

def test_sort_hand_worked():
    for c in json.load(open(GOLDEN))["sort"]:
        ids = np.array(c["ids"], np.int32)
        m, p2e, e2p, st = oracle.sort(ids, c["num_experts"], c["local_offset"], c["num_local"])
        assert m.tolist() == c["m_indptr"]
        assert p2e.tolist() == c["perm_to_exp"]
        assert e2p.tolist() == c["exp_to_perm"]
        assert st == c["status"]


@pytest.mark.parametrize("T,k,E,off,L,bad", [
    (1, 1, 1, 0, 1, False), (37, 2, 8, 0, 8, False), (100, 8, 256, 0, 256, False),
    (64, 8, 128, 32, 40, False), (50, 4, 16, 15, 1, True), (513, 3, 7, 2, 3, True),
    (300, 6, 64, 0, 64, True)])
def test_sort_vs_stable_argsort(T, k, E, off, L, bad):
    rng = np.random.default_rng(T * 7 + k)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    if bad:
        ids.flat[rng.integers(0, T * k, 5)] = rng.choice([-3, -1, E, E + 5], 5)
    m, p2e, e2p, st = oracle.sort(ids, E, off, L)
    flat = ids.ravel()
    local = (flat >= off) & (flat < off + L)
    # histogram and offsets
    hist = np.bincount(flat[local] - off, minlength=L)
    assert m.tolist() == [0] + np.cumsum(hist).tolist()
    # stable sort (a library routine) of the local routes by expert
    r_local = np.nonzero(local)[0]
    order = r_local[np.argsort(flat[r_local], kind="stable")]
    assert p2e.tolist() == order.tolist()
    # bijection and inverse
    assert len(set(p2e.tolist())) == len(p2e)
    assert np.array_equal(e2p[p2e], np.arange(len(p2e)))
    assert np.all(e2p[~local] == -1)
    assert st == (1 if bad else 0)


def test_sort_all_on_one_expert_and_empty():
    ids = np.full((33, 2), 3, np.int32)
    m, p2e, e2p, st = oracle.sort(ids, 5)
    assert m.tolist() == [0, 0, 0, 0, 66, 66]
    assert p2e.tolist() == list(range(66))
    ids0 = np.zeros((0, 2), np.int32)
    m, p2e, e2p, st = oracle.sort(ids0, 5)
    assert m.tolist() == [0] * 6 and p2e.size == 0


# --------------------------------------------------------- expert layer -----

def _dense_masked_fp64(x, ids, w, w1, w2, E):
    """Reference written as a dense sum over all (token, expert) pairs with a
    gate matrix G[t, e] (zero for experts a token did not choose), in fp64.
    Returns u, g (fp64) for every (t, e)."""
    x64 = bf16_to_f64(x)
    w1_64 = bf16_to_f64(w1)
    I = w1.shape[1] // 2
    G = np.zeros((x.shape[0], E))
    for t in range(ids.shape[0]):
        for j in range(ids.shape[1]):
            G[t, ids[t, j]] += w[t, j]
    u = np.einsum("th,enh->ten", x64, w1_64[:, :I, :])
    g = np.einsum("th,enh->ten", x64, w1_64[:, I:, :])
    return G, u, g


def test_layer_bruteforce_fp64_tiny():
    wl = W.make_moe("tiny")
    x = W.bf16_bits(wl.x)
    w1 = W.bf16_bits(wl.w1)
    w2 = W.bf16_bits(wl.w2)
    ids, w = oracle.route(wl.logits.numpy(), wl.top_k)
    out, h, y, st = oracle.moe_tokens(x, ids, w, w1, w2, wl.E, want_intermediates=True)
    assert st == 0
    G, u, g = _dense_masked_fp64(x, ids, w, w1, w2, wl.E)
    T, k, I, H = wl.T, wl.top_k, wl.I, wl.H
    x64, w1_64, w2_64 = bf16_to_f64(x), bf16_to_f64(w1), bf16_to_f64(w2)
    # step 1: h = bf16(silu(g) * u), each (token, slot).  The fp32 sums can
    # move a value that sits next to a bf16 rounding boundary across it, so
    # one ulp is allowed, and nearly all elements must agree exactly.
    n_exact = 0
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            h64 = (g[t, e] / (1.0 + np.exp(-g[t, e]))) * u[t, e]
            ulp = ulp_distance(h[t * k + j], torch_bf16_bits(h64))
            assert np.all(ulp <= 1)
            n_exact += int(np.sum(ulp == 0))
    assert n_exact >= 0.99 * T * k * I
    # step 2: y = h . W2^T from the oracle's own h, fp64 with an fp32 bound
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            hv = bf16_to_f64(h[t * k + j])
            y64 = w2_64[e] @ hv
            bound = I * 2.0 ** -23 * (np.abs(w2_64[e]) @ np.abs(hv)) + 1e-30
            assert np.all(np.abs(y[t * k + j] - y64) <= bound)
    # step 3: out = bf16(sum_j w * y) against the dense masked combine in fp64
    Y = np.zeros((T, wl.E, H))
    for t in range(T):
        for j in range(k):
            Y[t, ids[t, j]] = y[t * k + j]
    out64 = np.einsum("te,teh->th", G, Y)
    want = torch_bf16_bits(out64)
    assert np.all(ulp_distance(out, want) <= 1)
    assert np.mean(ulp_distance(out, want) == 0) >= 0.99


def _dense_swiglu_mlp_torch(x_bits, w1_bits, w2_bits):
    """Dense SwiGLU MLP with torch fp32 matmuls and a bf16 round of h."""
    xt = torch.from_numpy(bf16_to_f64(x_bits).astype(np.float32))
    w1t = torch.from_numpy(bf16_to_f64(w1_bits).astype(np.float32))
    w2t = torch.from_numpy(bf16_to_f64(w2_bits).astype(np.float32))
    I = w1t.shape[0] // 2
    u = xt @ w1t[:I].T
    g = xt @ w1t[I:].T
    h = (torch.nn.functional.silu(g) * u).to(torch.bfloat16).float()
    y = h @ w2t.T
    return y.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("T,H,I", [(9, 64, 64), (33, 128, 192), (4, 256, 64)])
def test_e1_k1_equals_dense_swiglu_mlp(T, H, I):
    wl = W.make_moe(T=T, H=H, I=I, E=1, top_k=1, mode="logits", seed=3)
    x, w1, w2 = W.bf16_bits(wl.x), W.bf16_bits(wl.w1), W.bf16_bits(wl.w2)
    ids, w = oracle.route(wl.logits.numpy(), 1)
    assert np.all(ids == 0) and np.all(w == 1.0)  # e/e == 1 exactly in IEEE
    out, st = oracle.moe_tokens(x, ids, w, w1, w2, 1)
    want = _dense_swiglu_mlp_torch(x, w1[0], w2[0])
    check_bf16_close(out, want, "E=1,k=1 vs dense MLP")


def test_identical_experts_independent_of_routing():
    T, H, I, E, k = 24, 64, 64, 6, 3
    base = W.make_moe(T=T, H=H, I=I, E=1, top_k=1, mode="logits", seed=5)
    x = W.bf16_bits(base.x)
    w1 = np.repeat(W.bf16_bits(base.w1), E, axis=0)
    w2 = np.repeat(W.bf16_bits(base.w2), E, axis=0)
    ref, _ = oracle.moe_tokens(x, np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32),
                               W.bf16_bits(base.w1), W.bf16_bits(base.w2), 1)
    for seed in range(3):
        lg = np.random.default_rng(seed).standard_normal((T, E)).astype(np.float32)
        ids, w = oracle.route(lg, k)
        out, _ = oracle.moe_tokens(x, ids, w, w1, w2, E)
        # sum_j w_j * y = (sum_j w_j) * y with sum w = 1 up to fp32 rounding
        assert np.all(ulp_distance(out, ref) <= 1)


def test_token_permutation_equivariance():
    wl = W.make_moe(T=20, H=64, I=64, E=5, top_k=2, mode="logits", seed=9)
    x, w1, w2 = W.bf16_bits(wl.x), W.bf16_bits(wl.w1), W.bf16_bits(wl.w2)
    lg = wl.logits.numpy()
    ids, w = oracle.route(lg, 2)
    out, _ = oracle.moe_tokens(x, ids, w, w1, w2, 5)
    perm = np.random.default_rng(0).permutation(20)
    ids_p, w_p = oracle.route(lg[perm], 2)
    out_p, _ = oracle.moe_tokens(x[perm], ids_p, w_p, w1, w2, 5)
    assert np.array_equal(out_p, out[perm])


def test_expert_parallel_partition_sums_to_full():
    """Routes outside the shard contribute zero: the fp32 partial combines of
    disjoint expert ranges add up to the full layer."""
    wl = W.make_moe(T=16, H=64, I=64, E=8, top_k=3, mode="logits", seed=11)
    x, w1, w2 = W.bf16_bits(wl.x), W.bf16_bits(wl.w1), W.bf16_bits(wl.w2)
    ids, w = oracle.route(wl.logits.numpy(), 3)
    full, st = oracle.moe_tokens(x, ids, w, w1, w2, 8)
    parts = np.zeros((16, 64))
    bound = np.zeros((16, 64))
    for off, L in ((0, 3), (3, 4), (7, 1)):
        part, st = oracle.moe_tokens(x, ids, w, w1[off:off + L], w2[off:off + L], 8,
                                     local_offset=off, num_local=L)
        assert st == 0
        pv = bf16_to_f64(part)
        parts += pv
        bound += np.abs(pv) * 2.0 ** -8 + 1e-6   # half a bf16 ulp per rounded partial
    fv = bf16_to_f64(full)
    bound += np.abs(fv) * 2.0 ** -8 + 1e-6
    assert np.all(np.abs(parts - fv) <= bound)
    # a shard holding none of the chosen experts gives exact zeros
    none_ids = np.zeros_like(ids)
    zero, _ = oracle.moe_tokens(x, none_ids, w, w1[4:6], w2[4:6], 8, local_offset=4, num_local=2)
    assert np.all(bf16_to_f64(zero) == 0)


def test_bad_expert_ids_are_dropped_and_flagged():
    wl = W.make_moe(T=4, H=64, I=64, E=4, top_k=2, mode="prerouted", seed=2)
    x, w1, w2 = W.bf16_bits(wl.x), W.bf16_bits(wl.w1), W.bf16_bits(wl.w2)
    ids = wl.topk_ids.numpy().copy()
    w = wl.topk_w.numpy()
    ref_ids = ids.copy()
    ids[1, 1] = 9
    out, st = oracle.moe_tokens(x, ids, w, w1, w2, 4)
    assert st == oracle.BAD_EXPERT
    ok, _ = oracle.moe_tokens(x, ref_ids, w, w1, w2, 4)
    assert np.array_equal(out[[0, 2, 3]], ok[[0, 2, 3]])
    # token 1 keeps only its first route
    one_ids = ref_ids.copy()
    w_one = w.copy()
    w_one[1, 1] = 0.0
    alt, _ = oracle.moe_tokens(x, one_ids, w_one, w1, w2, 4)
    assert np.array_equal(out[1], alt[1])


def test_stage_functions_compose_to_layer():
    """The stage-by-stage oracle (route, sort, gather, FC1, FC2, combine)
    equals the per-token layer bitwise."""
    wl = W.make_moe(T=30, H=128, I=64, E=6, top_k=2, mode="logits", seed=4)
    x, w1, w2 = W.bf16_bits(wl.x), W.bf16_bits(wl.w1), W.bf16_bits(wl.w2)
    ids, w = oracle.route(wl.logits.numpy(), 2)
    m, p2e, e2p, st = oracle.sort(ids, 6)
    xp = x[p2e // 2]
    rows = np.arange(len(p2e), dtype=np.int32)
    h = oracle.fc1_swiglu_rows(xp, w1, m[1:], rows)
    y = oracle.fc2_rows(h, w2, m[1:], rows)
    out = oracle.finalize(y, e2p, w)
    ref, _ = oracle.moe_tokens(x, ids, w, w1, w2, 6)
    assert np.array_equal(out, ref)


# ------------------------------------------------------- SwiGLUStep(limit) --
# Reading of "SwiGLUStep(limit) with a per-expert clamp limit"
# (flashinfer.experimental.cake_stepfun_moe, opening paragraph; Unified MoE API
# opt-in, gemm1_clamp_limit): GEMM1's gate output is clamped from above at the
# expert's limit and its up output to [-limit, limit] before silu(g) * u.

def _bits_exact(vals):
    a = np.asarray(vals, np.float32).view(np.uint32)
    assert np.all(a & 0xFFFF == 0)
    return (a >> 16).astype(np.uint16)


def test_swiglu_step_hand_worked():
    """x = e_0 and W1's column 0 carry (u, g) pairs exactly; W2 = identity
    passes h through to the output (one route of weight 1)."""
    H = I = 64
    gs = [-9.0, -2.0, 0.0, 3.0, 6.5, 7.0, 8.0, 20.0]
    us = [-100.0, -7.5, -1.0, 0.5, 6.5, 7.0, 7.5, 100.0]
    pairs = [(g, u) for g in gs for u in us][:I]
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = _bits_exact([1.0])[0]
    w1 = np.zeros((1, 2 * I, H), np.uint16)
    w1[0, :I, 0] = _bits_exact([u for _, u in pairs])
    w1[0, I:, 0] = _bits_exact([g for g, _ in pairs])
    w2 = np.zeros((1, H, I), np.uint16)
    w2[0, np.arange(H), np.arange(I)] = _bits_exact([1.0])[0]
    ids = np.zeros((1, 1), np.int32)
    w = np.ones((1, 1), np.float32)
    for limit in (7.0, 0.75):
        out, st = oracle.moe_tokens(x, ids, w, w1, w2, 1, clamp_limit=np.array([limit], np.float32))
        assert st == 0
        want = []
        for g, u in pairs:
            gc = min(g, limit)
            uc = min(max(u, -limit), limit)
            want.append(gc / (1.0 + math.exp(-gc)) * uc)
        # the oracle's fp32 silu may differ from fp64 by an fp32 rounding: the
        # bf16 results agree within one ulp and almost always exactly
        ulp = ulp_distance(out[0], torch_bf16_bits(np.array(want)))
        assert np.all(ulp <= 1) and np.mean(ulp == 0) >= 0.95, (limit, ulp)
        # the clamp binds: g = 20 gives silu(limit) * u, not silu(20) * u
        i = pairs.index((20.0, 0.5))
        want_i = limit / (1 + math.exp(-limit)) * min(0.5, limit)
        assert abs(bf16_to_f64(out[0, i:i + 1])[0] - want_i) < 0.01 * want_i


def test_swiglu_step_fp64_bruteforce_tiny():
    """The whole layer with per-expert limits against an fp64 dense masked
    evaluation (h and out within one bf16 ulp, nearly all exact)."""
    wl = W.make_moe("tiny")
    x, w1, w2 = W.bf16_bits(wl.x), W.bf16_bits(wl.w1), W.bf16_bits(wl.w2)
    ids, w = oracle.route(wl.logits.numpy(), wl.top_k)
    limits = np.array([0.25, 0.6, 1.0, 50.0], np.float32)
    out, h, y, st = oracle.moe_tokens(x, ids, w, w1, w2, wl.E, want_intermediates=True, clamp_limit=limits)
    assert st == 0
    G, u, g = _dense_masked_fp64(x, ids, w, w1, w2, wl.E)
    T, k, H = wl.T, wl.top_k, wl.H
    w2_64 = bf16_to_f64(w2)
    n_exact, Y = 0, np.zeros((T, wl.E, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            lim = float(limits[e])
            gc = np.minimum(g[t, e], lim)
            uc = np.clip(u[t, e], -lim, lim)
            ulp = ulp_distance(h[t * k + j], torch_bf16_bits(gc / (1.0 + np.exp(-gc)) * uc))
            assert np.all(ulp <= 1)
            n_exact += int(np.sum(ulp == 0))
            Y[t, e] = w2_64[e] @ bf16_to_f64(h[t * k + j])
    assert n_exact >= 0.99 * T * k * wl.I
    want = torch_bf16_bits(np.einsum("te,teh->th", G, Y))
    assert np.all(ulp_distance(out, want) <= 1) and np.mean(ulp_distance(out, want) == 0) >= 0.99


def test_swiglu_step_infinite_limit_is_plain_swiglu_and_limits_are_per_local_expert():
    wl = W.make_moe(T=40, H=64, I=64, E=5, top_k=1, mode="logits", seed=8)
    x, w1, w2 = W.bf16_bits(wl.x), W.bf16_bits(wl.w1), W.bf16_bits(wl.w2)
    ids, w = oracle.route(wl.logits.numpy(), 1)
    plain, _ = oracle.moe_tokens(x, ids, w, w1, w2, 5)
    inf, _ = oracle.moe_tokens(x, ids, w, w1, w2, 5, clamp_limit=np.full(5, np.inf, np.float32))
    assert np.array_equal(plain, inf)
    # shard of local experts 2..4 with limits (0.3, 1.5, inf): a token's row
    # equals the row computed with its own expert's limit everywhere
    off, L = 2, 3
    lims = np.array([0.3, 1.5, np.inf], np.float32)
    sl = slice(off, off + L)
    out, _ = oracle.moe_tokens(x, ids, w, w1[sl], w2[sl], 5, local_offset=off, num_local=L, clamp_limit=lims)
    changed = 0
    for i in range(L):
        ref, _ = oracle.moe_tokens(x, ids, w, w1[sl], w2[sl], 5, local_offset=off, num_local=L,
                                   clamp_limit=np.full(L, lims[i], np.float32))
        rows = ids[:, 0] == off + i
        assert np.array_equal(out[rows], ref[rows])
        changed += int(not np.array_equal(out[rows], plain[rows]))
    assert changed >= 2  # the two finite limits bind on these inputs


# ------------------------------------------------------------ grouped GEMM --

def test_grouped_gemm_vs_torch_per_group():
    d = W.make_grouped_gemm(seed=1, sum_m=300, E=7, K=128, N=64, alpha=0.3)
    X, Wt, offs = W.bf16_bits(d["X"]), W.bf16_bits(d["W"]), d["offs"].numpy()
    assert (d["sizes"] == 0).any()
    Y = oracle.grouped_gemm_rows(X, Wt, offs)
    start = 0
    for e in range(d["E"]):
        end = int(offs[e])
        if end > start:
            xs = torch.from_numpy(bf16_to_f64(X[start:end]).astype(np.float32))
            ws = torch.from_numpy(bf16_to_f64(Wt[e]).astype(np.float32))
            ref = (xs @ ws.T).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            check_bf16_close(Y[start:end], ref, f"group {e}")
        start = end


# ------------------------------------------------- grouped GEMM backward --
# Cake ragged BF16 grouped GEMM (experimental), operation table: dgrad
# dX = G . W[e] (W in place, bf16), wgrad dW[e] = G^T . X (fp32 or bf16, exact
# zeros for an empty group).

def _gg_bwd(seed, **kw):
    d = W.make_grouped_gemm(seed=seed, with_grad=True, **kw)
    return (W.bf16_bits(d["X"]), W.bf16_bits(d["W"]), W.bf16_bits(d["G"]), d["offs"].numpy(), d["sizes"])


def test_grouped_gemm_dgrad_vs_torch_per_group():
    X, Wt, G, offs, sizes = _gg_bwd(2, sum_m=300, E=7, K=128, N=64, alpha=0.3)
    assert (sizes == 0).any()
    dX = oracle.grouped_gemm_dgrad_rows(G, Wt, offs)
    start = 0
    for e, end in enumerate(offs):
        if end > start:
            ge = torch.from_numpy(bf16_to_f64(G[start:end]).astype(np.float32))
            we = torch.from_numpy(bf16_to_f64(Wt[e]).astype(np.float32))
            check_bf16_close(dX[start:end], torch_bf16_bits((ge @ we).numpy()), f"dgrad group {e}")
        start = end


def test_grouped_gemm_wgrad_vs_torch_per_group_and_empty_groups_zero():
    X, Wt, G, offs, sizes = _gg_bwd(3, sum_m=300, E=7, K=128, N=64, alpha=0.3)
    E, N, K = Wt.shape
    assert (sizes == 0).any() and (sizes > 0).any()
    sel_e = np.repeat(np.arange(E, dtype=np.int32), N)
    sel_n = np.tile(np.arange(N, dtype=np.int32), E)
    f32, b16 = oracle.grouped_gemm_wgrad_rows(G, X, offs, sel_e, sel_n)
    f32, b16 = f32.reshape(E, N, K), b16.reshape(E, N, K)
    assert np.array_equal(b16, torch_bf16_bits(f32))  # the bf16 output is one rounding of the fp32 sum
    start = 0
    for e, end in enumerate(offs):
        if end == start:
            assert np.all(f32[e].view(np.uint32) == 0) and np.all(b16[e] == 0)  # exact +0
        else:
            ge = torch.from_numpy(bf16_to_f64(G[start:end]).astype(np.float32))
            xe = torch.from_numpy(bf16_to_f64(X[start:end]).astype(np.float32))
            want = (ge.T @ xe).numpy().astype(np.float64)
            rms = np.sqrt(np.mean(want ** 2))
            assert np.max(np.abs(f32[e] - want)) <= 1e-5 * rms * max(1, end - start) ** 0.5, e
        start = end


def test_grouped_gemm_adjoint_identity():
    """sum(G * (X W^T)) = sum(dX * X) = sum(dW * W) over all groups (the
    three operations of the operation table are adjoint), fp64 sums of the
    oracle's results against the fp64 forward."""
    X, Wt, G, offs, sizes = _gg_bwd(4, sum_m=500, E=6, K=192, N=128, alpha=0.5)
    E, N, K = Wt.shape
    x64, w64, g64 = bf16_to_f64(X), bf16_to_f64(Wt), bf16_to_f64(G)
    fwd, start = 0.0, 0
    for e, end in enumerate(offs):
        fwd += float(np.sum(g64[start:end] * (x64[start:end] @ w64[e].T)))
        start = end
    dX = bf16_to_f64(oracle.grouped_gemm_dgrad_rows(G, Wt, offs))
    sel_e = np.repeat(np.arange(E, dtype=np.int32), N)
    sel_n = np.tile(np.arange(N, dtype=np.int32), E)
    dW = oracle.grouped_gemm_wgrad_rows(G, X, offs, sel_e, sel_n)[0].astype(np.float64).reshape(E, N, K)
    by_dx = float(np.sum(dX * x64[:dX.shape[0]]))
    by_dw = float(np.sum(dW * w64))
    scale = float(np.sqrt(np.sum(g64 ** 2) * np.sum(x64 ** 2)))
    assert abs(by_dw - fwd) <= 1e-5 * scale, (by_dw, fwd)
    assert abs(by_dx - fwd) <= 2e-3 * scale, (by_dx, fwd)   # dX carries one bf16 rounding


# ----------------------------------------------------- BGMV LoRA-MoE --------
# flashinfer.fused_moe.prepare_bgmv_moe: shrink s = bf16(A[l,e] x[t]) per pair,
# expand y[t] = sum over the token's pairs (ascending) of w * (B[l,e] s), fp32.

def _bgmv_bits(wl):
    return (W.bf16_bits(wl.x), [W.bf16_bits(a) for a in wl.lora_a], [W.bf16_bits(b) for b in wl.lora_b],
            wl.tok.numpy(), wl.eid.numpy(), wl.lora.numpy(), wl.w.numpy())


@pytest.mark.parametrize("contiguous", [True, False])
def test_bgmv_vs_torch_per_pair(contiguous):
    wl = W.make_bgmv(T=40, H=64, R=16, E=6, num_loras=3, top_k=2, feat_out=[64, 32], contiguous=contiguous,
                     seed=5)
    x, A, B, tok, eid, lora, w = _bgmv_bits(wl)
    shrink, y, st = oracle.bgmv(x, A, B, tok, eid, lora, w)
    assert st == 0
    xf = torch.from_numpy(bf16_to_f64(x).astype(np.float32))
    want_y = torch.zeros((wl.T, y.shape[1]), dtype=torch.float64)
    col = 0
    for s in range(2):
        Af = torch.from_numpy(bf16_to_f64(A[s]).astype(np.float32))
        Bf = torch.from_numpy(bf16_to_f64(B[s]).astype(np.float32))
        la, ea = torch.from_numpy(lora[tok].astype(np.int64)), torch.from_numpy(eid.astype(np.int64))
        sh = torch.bmm(Af[la, ea], xf[torch.from_numpy(tok.astype(np.int64))].unsqueeze(2)).squeeze(2)
        check_bf16_close(shrink[s], torch_bf16_bits(sh.numpy()), f"shrink slice {s}")
        sp = torch.from_numpy(bf16_to_f64(shrink[s]).astype(np.float32))          # the oracle's own s
        v = torch.bmm(Bf[la, ea], sp.unsqueeze(2)).squeeze(2) * torch.from_numpy(w).unsqueeze(1)
        F = Bf.shape[2]
        want_y[:, col:col + F].index_add_(0, torch.from_numpy(tok.astype(np.int64)), v.double())
        col += F
    from tests.tolerances import check_f32_close
    check_f32_close(y, want_y.numpy(), "bgmv y")


def test_bgmv_rank_padding_linearity_and_zero_b():
    wl = W.make_bgmv(T=30, H=64, R=8, E=4, num_loras=2, top_k=3, seed=6)
    x, A, B, tok, eid, lora, w = _bgmv_bits(wl)
    _, y, _ = oracle.bgmv(x, A, B, tok, eid, lora, w)
    # zero-padding the rank from 8 to 16 adds exact zero terms: y is bitwise equal
    A2 = np.zeros(A[0].shape[:2] + (16, 64), np.uint16)
    A2[:, :, :8] = A[0]
    B2 = np.zeros(B[0].shape[:3] + (16,), np.uint16)
    B2[..., :8] = B[0]
    _, y2, _ = oracle.bgmv(x, [A2], [B2], tok, eid, lora, w)
    assert np.array_equal(y, y2)
    # doubling every routing weight doubles y exactly (a power-of-two scale)
    _, y3, _ = oracle.bgmv(x, A, B, tok, eid, lora, 2 * w)
    assert np.array_equal(2 * y, y3)
    # B = 0 gives y = 0
    _, y4, _ = oracle.bgmv(x, A, [np.zeros_like(B[0])], tok, eid, lora, w)
    assert not np.any(y4)


def test_bgmv_out_of_range_pairs_are_dropped_and_flagged():
    wl = W.make_bgmv(T=20, H=64, R=8, E=4, num_loras=2, top_k=2, seed=7)
    x, A, B, tok, eid, lora, w = _bgmv_bits(wl)
    _, y_ok, st = oracle.bgmv(x, A, B, tok, eid, lora, w)
    assert st == 0
    keep = np.ones(len(tok), bool)
    keep[[3, 10]] = False
    eid_bad = eid.copy()
    eid_bad[3] = 9            # expert out of range
    lora_bad = lora.copy()
    lora_bad[tok[10]] = 5     # LoRA of token tok[10] out of range: all its pairs drop
    keep[tok == tok[10]] = False
    shrink, y_bad, st = oracle.bgmv(x, A, B, tok, eid_bad, lora_bad, w)
    assert st == oracle.BAD_EXPERT
    assert not np.any(shrink[0][~keep])
    _, y_ref, _ = oracle.bgmv(x, A, B, tok[keep], eid[keep], lora, w[keep])
    assert np.array_equal(y_bad, y_ref)


# ------------------------------------------------- FP8 per-tensor family --
# flashinfer.experimental.cake_stepfun_moe, opening paragraph ("fp8
# (per-tensor)").  E4M3 as the OCP 8-bit format defines it; reading of the
# family: xq = e4m3(x / a1), u, g dequantised by a1 * s1[e], hq = e4m3(h / a2),
# y dequantised by a2 * s2[e].

def _torch_e4m3_decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).float().numpy()


def _torch_e4m3_encode(vals):
    return torch.from_numpy(np.ascontiguousarray(vals, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_codes_exhaustive_against_torch():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue  # NaN codes
        v = oracle.e4m3_decode(c)
        assert v == float(_torch_e4m3_decode(np.array([c]))[0]), c
        assert oracle.e4m3_encode(v) == c, c
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_rounding_ties_and_saturation():
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0)]).astype(np.float32)
    vals = vals[np.abs(vals) < 440]
    got = np.array([oracle.e4m3_encode(v) for v in vals], np.uint8)
    assert np.array_equal(got, _torch_e4m3_encode(vals))  # a library rounding, nearest even
    # exact midpoints between neighbouring codes go to the even code
    for c in range(0, 0x7D):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = np.float32((lo + hi) / 2)
        assert oracle.e4m3_encode(mid) == (c if c % 2 == 0 else c + 1), c
        assert oracle.e4m3_encode(-mid) == 0x80 | (c if c % 2 == 0 else c + 1), c
    # above the largest finite magnitude: saturate
    for v in (448.0, 449.0, 470.0, 1e6):
        assert oracle.e4m3_encode(v) == 0x7E and oracle.e4m3_encode(-v) == 0xFE


def _fp8_case(seed=11, T=20, H=64, I=64, E=5, k=2):
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", seed=seed)
    fw = W.make_fp8_weights(E, H, I, seed=seed)
    x = W.bf16_bits(wl.x)
    ids, w = oracle.route(wl.logits.numpy(), k)
    return wl, fw, x, ids, w


def test_fp8_layer_fp64_tiny():
    """Dense fp64 evaluation from torch's E4M3 decoding of the same codes:
    xq exact, hq within one code (fp32 sums may straddle a rounding boundary),
    out within one bf16 ulp of the fp64 combine of the oracle's own y."""
    wl, fw, x, ids, w = _fp8_case()
    w1q, w2q, s1, s2 = fw.w1q.numpy(), fw.w2q.numpy(), fw.s1.numpy(), fw.s2.numpy()
    out, hq, y, st = oracle.moe_tokens_fp8(x, ids, w, w1q, w2q, s1, s2, fw.a1, fw.a2, wl.E, want_intermediates=True)
    assert st == 0
    xq = oracle.quantize_e4m3(x, fw.a1)
    v = bf16_to_f64(x).astype(np.float32) / np.float32(fw.a1)
    inr = np.abs(v) < 448  # torch's cast gives NaN above 448 where this family saturates
    assert np.array_equal(xq[inr], _torch_e4m3_encode(v[inr]))
    assert np.all(xq[~inr] & 0x7F == 0x7E)
    xq64 = _torch_e4m3_decode(xq).astype(np.float64)
    I = wl.I
    near = 0
    for t in range(wl.T):
        for j in range(wl.top_k):
            e = ids[t, j]
            w1 = _torch_e4m3_decode(w1q[e]).astype(np.float64)
            sc = float(np.float32(fw.a1) * np.float32(s1[e]))
            u, g = (w1[:I] @ xq64[t]) * sc, (w1[I:] @ xq64[t]) * sc
            h64 = g / (1 + np.exp(-g)) * u / fw.a2
            want = _torch_e4m3_encode(np.clip(h64, -448, 448))
            d = np.abs(_torch_e4m3_decode(hq[t * wl.top_k + j]).astype(np.float64) - _torch_e4m3_decode(want))
            step = np.maximum(np.abs(_torch_e4m3_decode(want)) * 2.0 ** -3, 2.0 ** -9)
            assert np.all(d <= step + 1e-12)
            near += int(np.sum(d == 0))
            w2 = _torch_e4m3_decode(w2q[e]).astype(np.float64)
            y64 = (w2 @ _torch_e4m3_decode(hq[t * wl.top_k + j]).astype(np.float64)) * float(np.float32(fw.a2) * np.float32(s2[e]))
            assert np.all(np.abs(y[t * wl.top_k + j] - y64) <= 1e-5 * (np.abs(y64).max() + 1e-6))
    assert near >= 0.99 * wl.T * wl.top_k * I
    comb = np.zeros((wl.T, wl.H))
    for t in range(wl.T):
        for j in range(wl.top_k):
            comb[t] += w[t, j] * y[t * wl.top_k + j]
    assert np.all(ulp_distance(out, torch_bf16_bits(comb)) <= 1)


def test_fp8_stages_compose_to_layer():
    wl, fw, x, ids, w = _fp8_case(seed=12, T=30, H=128, I=64, E=6, k=2)
    w1q, w2q, s1, s2 = fw.w1q.numpy(), fw.w2q.numpy(), fw.s1.numpy(), fw.s2.numpy()
    m, p2e, e2p, _ = oracle.sort(ids, wl.E)
    xq = oracle.quantize_e4m3(x, fw.a1)[p2e // 2]
    rows = np.arange(len(p2e), dtype=np.int32)
    hq = oracle.fc1_fp8_rows(xq, w1q, s1, fw.a1, fw.a2, m[1:], rows)
    y = oracle.fc2_fp8_rows(hq, w2q, s2, fw.a2, m[1:], rows)
    out = oracle.finalize(y, e2p, w)
    ref, _ = oracle.moe_tokens_fp8(x, ids, w, w1q, w2q, s1, s2, fw.a1, fw.a2, wl.E)
    assert np.array_equal(out, ref)


def test_workload_generator_is_seeded():
    a = W.make_moe("tiny", seed=0)
    b = W.make_moe("tiny", seed=0)
    c = W.make_moe("tiny", seed=1)
    assert torch.equal(a.x, b.x) and torch.equal(a.w1, b.w1) and torch.equal(a.logits, b.logits)
    assert not torch.equal(a.x, c.x)
    d = W.make_moe("decode_t8")
    assert torch.allclose(d.topk_w.double().sum(1), torch.ones(8, dtype=torch.float64), atol=1e-6)
    ids = d.topk_ids.numpy()
    assert all(len(set(r)) == 8 for r in ids)
    s = W.grouped_sizes(16384, 64, 0.3, 0)
    assert s.sum() == 16384 and (s == 0).any() and ((s % 128) != 0).any()
