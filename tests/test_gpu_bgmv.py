"""Parity of the BGMV LoRA-MoE shrink + expand (moe_bgmv, called through the C
ABI) against the CPU oracle (flashinfer.fused_moe.prepare_bgmv_moe: shrink
bf16(A[l,e] . x[t]) per routed pair, expand summed per token in ascending pair
order in fp32, one owner per output), on the pair-grouped pipeline (grouped by
a scan while groups x pairs <= 2^22, else by keys and the route sort up to 1024
(LoRA, expert) groups) and on the per-route one beyond.  The shrink values use
the strict bf16 rule, y the fp32 rule; replays are bitwise identical."""
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


def _dev(wl):
    return dict(x=wl.x.to(DEV), a=[a.to(DEV) for a in wl.lora_a], b=[b.to(DEV) for b in wl.lora_b],
                tok=wl.tok.to(DEV), eid=wl.eid.to(DEV), lora=wl.lora.to(DEV), w=wl.w.to(DEV))


def _oracle(wl, tok=None, eid=None, lora=None):
    return oracle.bgmv(W.bf16_bits(wl.x), [W.bf16_bits(a) for a in wl.lora_a], [W.bf16_bits(b) for b in wl.lora_b],
                       wl.tok.numpy() if tok is None else tok, wl.eid.numpy() if eid is None else eid,
                       wl.lora.numpy() if lora is None else lora, wl.w.numpy())


SHAPES = [  # T, H, R, E, L, k, feat_out
    (37, 64, 8, 5, 2, 2, None), (200, 256, 16, 16, 3, 2, [256, 64]), (64, 3072, 32, 64, 4, 2, None),
    (50, 512, 64, 8, 1, 6, [128]), (300, 128, 32, 32, 5, 4, [96, 128, 32]),
    (60, 64, 8, 1024, 3, 2, None),  # 3072 (LoRA, expert) groups x 120 pairs: scanned grouping
    (2100, 128, 16, 256, 4, 2, None),  # 1024 groups x 4200 pairs: keyed and sorted grouping
    (700, 64, 8, 1024, 3, 2, None),  # 3072 groups x 1400 pairs: the per-route pipeline
]


@pytest.mark.parametrize("contiguous", [True, False])
@pytest.mark.parametrize("si", range(len(SHAPES)))
def test_bgmv_parity_and_replays(si, contiguous):
    T, H, R, E, L, k, F = SHAPES[si]
    wl = W.make_bgmv(T=T, H=H, R=R, E=E, num_loras=L, top_k=k, feat_out=F, contiguous=contiguous, seed=si)
    d = _dev(wl)
    status = torch.full((1,), 9, dtype=torch.int32, device=DEV)
    y, sh = moe.bgmv(d["x"], d["a"], d["b"], d["tok"], d["eid"], d["lora"], d["w"],
                     contiguous_top_k=k if contiguous else 0, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sh_o, y_o, st = _oracle(wl)
    assert st == 0
    check_bf16_close(W.bf16_bits(sh), sh_o, f"bgmv shrink shape {si}")
    check_f32_close(y.cpu().numpy(), y_o, f"bgmv y shape {si}")
    y2, sh2 = moe.bgmv(d["x"], d["a"], d["b"], d["tok"], d["eid"], d["lora"], d["w"],
                       contiguous_top_k=k if contiguous else 0)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(sh, sh2)


def test_bgmv_token_with_more_pairs_than_slots_and_column_slice():
    """General order with one token owning 20 pairs (more than the route
    index keeps: the exact in-order scan) and y written into a column slice of
    a wider buffer."""
    wl = W.make_bgmv(T=24, H=128, R=16, E=32, num_loras=2, top_k=2, contiguous=False, seed=9)
    tok = wl.tok.numpy().copy()
    tok[:20] = 5  # 20 pairs on token 5, in pair order
    d = _dev(wl)
    d["tok"] = torch.from_numpy(tok).to(DEV)
    wide = torch.full((wl.T, 128 + 40), 4.0, dtype=torch.float32, device=DEV)
    y, sh = moe.bgmv(d["x"], d["a"], d["b"], d["tok"], d["eid"], d["lora"], d["w"], y_accum=wide[:, 8:136])
    torch.cuda.synchronize()
    sh_o, y_o, _ = _oracle(wl, tok=tok)
    check_bf16_close(W.bf16_bits(sh), sh_o, "bgmv shrink (overflow)")
    check_f32_close(wide[:, 8:136].cpu().numpy(), y_o, "bgmv y (overflow)")
    assert torch.all(wide[:, :8] == 4.0) and torch.all(wide[:, 136:] == 4.0)


def test_bgmv_bad_indices_flagged_and_dropped():
    wl = W.make_bgmv(T=30, H=64, R=8, E=4, num_loras=2, top_k=2, contiguous=True, seed=3)
    eid = wl.eid.numpy().copy()
    eid[7] = 11
    lora = wl.lora.numpy().copy()
    lora[4] = -1
    d = _dev(wl)
    d["eid"], d["lora"] = torch.from_numpy(eid).to(DEV), torch.from_numpy(lora).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, sh = moe.bgmv(d["x"], d["a"], d["b"], d["tok"], d["eid"], d["lora"], d["w"], contiguous_top_k=2,
                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == moe.DEV_BAD_EXPERT
    sh_o, y_o, st = _oracle(wl, eid=eid, lora=lora)
    assert st == oracle.BAD_EXPERT
    check_bf16_close(W.bf16_bits(sh), sh_o, "bgmv shrink (bad ids)")
    check_f32_close(y.cpu().numpy(), y_o, "bgmv y (bad ids)")
