"""Parity of the fp8 per-tensor weight family (MOE_WEIGHTS_E4M3; reading of
flashinfer.experimental.cake_stepfun_moe, opening paragraph) against the CPU
oracle, called through the C ABI.

Stage rules: the quantised activations xq = e4m3(x / x_scale) are bit-exact
(both sides divide in fp32 and round the same value to nearest even); FC1's
requantised h (E4M3 codes) may differ where the fp32 sums straddle a rounding
boundary of the 3-bit mantissa, so at least 99.9% of the codes must be equal
and every code within one E4M3 step; FC2 + finalize fed the oracle's hq give
outputs under the strict bf16 rule.  End to end: the accumulation model's
floor on the 2-ulp fraction, as for the bf16 family, and the per-element max
bound of the E4M3 family (RMS_FRAC_E4M3: one requantisation flip of h moves an
output 32 times further than a bf16 flip does)."""
import numpy as np
import pytest
import torch

import mixture_experts_expert_router_gb300 as moe
import oracle
from mixture_experts_expert_router_gb300 import workloads as W
from tests import accum_model
from tests.tolerances import RMS_FRAC_E4M3, check_bf16_close, check_bf16_end_to_end, with_floor

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mixture_experts_expert_router_gb300 import _build
    _build.build()
    moe.library()


SHAPES = [(300, 256, 128, 8, 2), (40, 512, 256, 16, 4), (1500, 1024, 512, 32, 4), (7, 128, 128, 3, 2)]


def _case(T, H, I, E, k, seed):
    wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", seed=seed)
    fw = W.make_fp8_weights(E, H, I, seed=seed)
    ids, w = oracle.route(wl.logits.numpy(), k)
    return wl, fw, ids, w


def _e4m3_value(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def check_e4m3_close(got, want, what):
    """E4M3 codes: >= 99.9% equal, every one within one E4M3 step of the other."""
    got, want = np.asarray(got, np.uint8), np.asarray(want, np.uint8)
    assert got.shape == want.shape
    if want.size == 0:
        return
    g, r = _e4m3_value(got), _e4m3_value(want)
    step = np.maximum(np.maximum(np.abs(g), np.abs(r)) * 2.0 ** -3, 2.0 ** -9)
    assert np.all(np.abs(g - r) <= step + 1e-12), f"{what}: a code differs by more than one step"
    frac = float(np.mean(got == want))
    assert frac >= 0.999, f"{what}: only {frac:.5f} of the codes equal"


def _plan(wl, fw, clamp=None, one_cta=False):
    d = dict(x=wl.x.to(DEV), logits=wl.logits.to(DEV))
    e4 = dict(w1_scale=fw.s1.to(DEV), w2_scale=fw.s2.to(DEV), x_scale=fw.a1, h_scale=fw.a2)
    return moe.MoEPlan(d["x"], fw.w1q.to(DEV), fw.w2q.to(DEV), wl.E, wl.top_k, logits=d["logits"], e4m3=e4,
                       clamp_limit=None if clamp is None else torch.from_numpy(clamp).to(DEV),
                       one_cta_gemm=one_cta)


@pytest.mark.parametrize("si", range(len(SHAPES)))
def test_e4m3_gather_and_stages(si):
    T, H, I, E, k = SHAPES[si]
    wl, fw, ids, w = _case(T, H, I, E, k, 50 + si)
    plan = _plan(wl, fw)
    plan.launch()
    torch.cuda.synchronize()
    assert int(plan.status.item()) == 0
    m, p2e, e2p, _ = oracle.sort(ids, E)
    M = len(p2e)
    # quantised gather: bit-exact
    b = plan.buffers()
    off = b["xp"] - plan.workspace.data_ptr()
    xq_gpu = plan.workspace[off:off + M * H].view(M, H).cpu().numpy()
    xq = oracle.quantize_e4m3(W.bf16_bits(wl.x), fw.a1)[p2e // k]
    assert np.array_equal(xq_gpu, xq)
    # FC1 + requantisation on the oracle's rows
    w1q, w2q, s1, s2 = fw.w1q.numpy(), fw.w2q.numpy(), fw.s1.numpy(), fw.s2.numpy()
    rows = np.arange(M, dtype=np.int32)
    hq_o = oracle.fc1_fp8_rows(xq, w1q, s1, fw.a1, fw.a2, m[1:], rows)
    m_d = torch.from_numpy(m).to(DEV)
    hq = moe.moe_fc1_swiglu_e4m3(torch.from_numpy(xq).to(DEV), fw.w1q.to(DEV), fw.s1.to(DEV), fw.a1, fw.a2, m_d)
    torch.cuda.synchronize()
    check_e4m3_close(hq.cpu().numpy(), hq_o, f"E4M3 h shape {si}")
    # FC2 + finalize on the oracle's hq
    y = moe.moe_fc2_e4m3(torch.from_numpy(hq_o).to(DEV), fw.w2q.to(DEV), fw.s2.to(DEV), fw.a2, m_d)
    out = moe.moe_finalize(y, torch.from_numpy(e2p).to(DEV), torch.from_numpy(w).to(DEV))
    torch.cuda.synchronize()
    y_o = oracle.fc2_fp8_rows(hq_o, w2q, s2, fw.a2, m[1:], rows)
    want = oracle.finalize(y_o, e2p, w)
    check_bf16_close(W.bf16_bits(out), want, f"E4M3 FC2 + finalize shape {si}")


@pytest.mark.parametrize("one_cta", [False, True])
@pytest.mark.parametrize("clamped", [False, True])
@pytest.mark.parametrize("si", range(len(SHAPES)))
def test_e4m3_layer_end_to_end(si, clamped, one_cta):
    """CTA-pair GEMMs where the shape allows them (the default), and the one-CTA kernel."""
    T, H, I, E, k = SHAPES[si]
    wl, fw, ids, w = _case(T, H, I, E, k, 70 + si)
    clamp = None
    if clamped:
        clamp = np.random.default_rng(si).uniform(0.3, 2.0, size=E).astype(np.float32)
        clamp[0] = np.inf
    plan = _plan(wl, fw, clamp, one_cta)
    out = plan.launch().clone()
    torch.cuda.synchronize()
    assert int(plan.status.item()) == 0
    x = W.bf16_bits(wl.x)
    args = (x, ids, w, fw.w1q.numpy(), fw.w2q.numpy(), fw.s1.numpy(), fw.s2.numpy(), fw.a1, fw.a2, E)
    want, st = oracle.moe_tokens_fp8(*args, clamp_limit=clamp)
    assert st == 0
    frac, n = accum_model.floor_e4m3(*args, want, clamp_limit=clamp)
    check_bf16_end_to_end(W.bf16_bits(out), with_floor(want, frac, n), f"E4M3 layer shape {si} clamp {clamped}",
                          rms_frac=RMS_FRAC_E4M3)
    again = plan.launch()
    torch.cuda.synchronize()
    assert torch.equal(again, out)
