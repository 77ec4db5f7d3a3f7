"""Pins of the end-to-end acceptance floor (CPU only).

The acceptance rule asks, end to end, for at least 99.9% of the outputs within
2 bf16 ulp of the oracle.  The layer rounds h to bf16 between the two GEMMs, so any
fp32 difference that moves an h value across a rounding boundary shows up
again in every output that h value feeds, and outputs near zero have tiny
ulps.  These tests pin, on the CPU and without the GPU path:

  * the accumulation model of tests/accum_model.c on hand-worked cases (its
    fp32 blocked mode rounds to nearest even; its tensor-core mode truncates
    toward zero after aligning each block of 16 products with two guard bits);
  * the model's error growth against exact (fp64) dot products: truncation
    errors add up, so its relative error grows with K while a round-to-nearest
    fp32 sum's does not;
  * the end-to-end agreement with the oracle of (a) a correct fp32 evaluation
    that differs only in summation order, which already misses 99.9% at both
    prefill shapes, and (b) the tensor-core model, whose agreement is the floor
    the GPU parity tests use.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_expert_router_gb300 import workloads as W
from tests import accum_model as AM
from tests.tolerances import ulp_distance

ONE = 0x3F80  # bf16 1.0


def _bits(vals):
    """bf16 bits of values that bf16 represents exactly."""
    a = np.asarray(vals, np.float32)
    b = a.view(np.uint32)
    assert np.all(b & 0xFFFF == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def test_exact_sums_are_exact_in_both_modes():
    a = _bits([1, 2, 3, 4, -5, 6, 7, 8] * 4)
    b = _bits([1, -1, 2, 0.5, 1, 1, -2, 0.25] * 4)
    want = float(np.sum(np.asarray([1, 2, 3, 4, -5, 6, 7, 8] * 4, np.float64) *
                        np.asarray([1, -1, 2, 0.5, 1, 1, -2, 0.25] * 4, np.float64)))
    for mode in (AM.BLOCKED_FP32, AM.TENSOR_CORE):
        assert AM.dot(a, b, mode) == want


def test_tensor_core_mode_truncates_where_fp32_rounds_to_nearest():
    # block 1 leaves 1 + 2^-23; block 2 adds -2^-25: exact 1 + 0.75 ulp(1)
    a = np.zeros(32, np.uint16)
    b = np.full(32, ONE, np.uint16)
    a[0], a[1], a[16] = ONE, _bits([2.0 ** -23])[0], _bits([-(2.0 ** -25)])[0]
    assert AM.dot(a, b, AM.BLOCKED_FP32) == 1.0 + 2.0 ** -23   # nearest
    assert AM.dot(a, b, AM.TENSOR_CORE) == 1.0                 # toward zero
    # the same with every sign flipped: truncation is symmetric
    a_neg = a ^ np.uint16(0x8000) * (a != 0)
    assert AM.dot(a_neg, b, AM.BLOCKED_FP32) == -(1.0 + 2.0 ** -23)
    assert AM.dot(a_neg, b, AM.TENSOR_CORE) == -1.0


def test_tensor_core_mode_keeps_two_guard_bits():
    # acc = 1.0, then 16 products of 0.75 * 2^-25 each: each is below the cut
    # (2^-25 = ulp(1) / 4) and vanishes; exact and fp32 give 1 + 3 * 2^-23
    a = np.zeros(32, np.uint16)
    b = np.full(32, ONE, np.uint16)
    a[0] = ONE
    a[16:32] = _bits([0.75 * 2.0 ** -25])[0]
    assert AM.dot(a, b, AM.BLOCKED_FP32) == 1.0 + 3 * 2.0 ** -23
    assert AM.dot(a, b, AM.TENSOR_CORE) == 1.0
    # one guard-bit quantum (2^-25) per product is kept: 16 of them = 4 ulp
    a[16:32] = _bits([2.0 ** -25])[0]
    assert AM.dot(a, b, AM.TENSOR_CORE) == 1.0 + 4 * 2.0 ** -23


def test_tensor_core_mode_error_grows_with_k():
    """Mean |error| / sum|terms| against exact fp64 dot products of
    N(0,1) x N(0,1/K) bf16 vectors: the truncating model's grows about like
    sqrt(K) and is several times the round-to-nearest fp32 sum's at K=14336."""
    rng = np.random.default_rng(5)
    err = {}
    for K in (1024, 14336):
        a32 = rng.standard_normal((8, K)).astype(np.float32)
        b32 = (rng.standard_normal((32, K)) / np.sqrt(K)).astype(np.float32)
        A = W.bf16_bits(torch.from_numpy(a32).to(torch.bfloat16))
        B = W.bf16_bits(torch.from_numpy(b32).to(torch.bfloat16))
        a64 = (A.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        b64 = (B.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        exact = a64 @ b64.T
        scale = np.abs(a64) @ np.abs(b64).T
        for mode in (AM.BLOCKED_FP32, AM.TENSOR_CORE):
            err[K, mode] = float(np.mean(np.abs(AM.dots(A, B, mode) - exact) / scale))
    print({f"K={k} mode={m}": f"{v:.3e}" for (k, m), v in err.items()})
    assert err[14336, AM.TENSOR_CORE] > 2.5 * err[1024, AM.TENSOR_CORE]
    assert err[14336, AM.BLOCKED_FP32] < 2.0 * err[1024, AM.BLOCKED_FP32]
    assert err[14336, AM.TENSOR_CORE] > 5.0 * err[14336, AM.BLOCKED_FP32]


# (H, I, E, top_k) at the two prefill workloads' reduction lengths; the
# fraction depends on H, I and top_k, not on how many experts exist
PREFILL_SHAPES = {"few_large": (4096, 14336, 2, 2), "many_fine": (7168, 2048, 8, 8)}


@pytest.mark.parametrize("shape", sorted(PREFILL_SHAPES))
def test_end_to_end_floors_at_prefill_shapes(shape):
    H, I, E, k = PREFILL_SHAPES[shape]
    n_tok = 24
    wl = W.make_moe(T=n_tok, H=H, I=I, E=E, top_k=k, mode="logits", seed=9)
    x, w1, w2 = W.bf16_bits(wl.x), W.bf16_bits(wl.w1), W.bf16_bits(wl.w2)
    ids, w = oracle.route(wl.logits.numpy(), k)
    ref, st = oracle.moe_tokens(x, ids, w, w1, w2, E)
    assert st == 0
    frac = {}
    for mode in (AM.BLOCKED_FP32, AM.TENSOR_CORE):
        out = AM.moe_tokens(x, ids, w, w1, w2, E, mode)
        frac[mode] = float(np.mean(ulp_distance(out, ref) <= 2))
    print(f"{shape}: blocked fp32 {frac[AM.BLOCKED_FP32]:.5f}, tensor-core model {frac[AM.TENSOR_CORE]:.5f}")
    # a correct fp32 evaluation in another summation order misses 99.9% ...
    assert 0.995 <= frac[AM.BLOCKED_FP32] < 0.999
    # ... and tensor-core accumulation lands near 99%
    assert 0.980 <= frac[AM.TENSOR_CORE] < frac[AM.BLOCKED_FP32]
