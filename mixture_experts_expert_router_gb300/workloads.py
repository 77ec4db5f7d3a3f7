"""Seeded synthetic inputs for the MoE expert layer and the ragged grouped GEMM.

This module only draws random numbers and lays them out; it holds none of the
layer's arithmetic (no routing, sorting, matmul or activation).  Tests, the
benchmark and the CPU oracle all read the exact tensors it returns.

Distributions (one independent stream per tensor, derived from ``seed``):
  x        ~ N(0, 1)                       bf16 [T, H]
  W1       ~ N(0, 1/H)  ([up | gate] rows) bf16 [L, 2I, H]
  W2       ~ N(0, 1/I)                     bf16 [L, H, I]
  logits   ~ N(0, 1) (+ optional per-expert bias)        fp32 [T, E]
  pre-routed ids: a uniform random k-subset of the E experts per token (the
           same law as the top-k of i.i.d. N(0,1) logits), weights a flat
           Dirichlet draw (positive, summing to 1), both per token.
  grouped GEMM sizes: Dirichlet(alpha * 1_E) proportions of sum_m, floored,
           the remainder handed to the largest fractional parts.
  grouped GEMM upstream gradient G ~ N(0, 1)  bf16 [sum_m, N] (backward).
  FP8 per-tensor family: W1q, W2q E4M3 codes of N(0, 1) draws (torch's
           float8_e4m3fn cast), per-expert scales s1 = u / sqrt(H), s2 = u / sqrt(I)
           with u ~ U(0.5, 1.5), static activation scales a1 = 4/448, a2 = 2/448.
  BGMV LoRA-MoE: x ~ N(0,1) [T, H]; per slice A ~ N(0, 1/H) [L, E, R, H] and
           B ~ N(0, 1/R) [L, E, F, R]; each token a uniform LoRA index and a
           uniform k-subset of the experts, weights a flat Dirichlet draw; pairs
           laid out token-major (p = t*k + j) or sorted by expert (stable).

Small tensors are drawn on the host with numpy's PCG64 generator (the same
stream on every platform) and converted to bf16 by round-to-nearest-even.
Large weight banks may be drawn directly on a CUDA device with torch's
generator (``weights_device="cuda"``); the values then differ from the host
draw but are equally seeded, and every comparison reads back the same bytes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream])


def _normal_bf16(shape, std: float, seed: int, stream: int, device="cpu") -> torch.Tensor:
    dev = torch.device(device)
    if dev.type == "cuda":
        g = torch.Generator(device=dev)
        g.manual_seed(seed * 1_000_003 + stream)
        out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        # fill in slabs so the fp32 temporary stays small
        flat = out.view(-1)
        slab = 1 << 28
        for s in range(0, flat.numel(), slab):
            n = min(slab, flat.numel() - s)
            flat[s:s + n].copy_(torch.randn(n, generator=g, device=dev, dtype=torch.float32).mul_(std))
        return out
    a = _rng(seed, stream).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return torch.from_numpy(a).to(torch.bfloat16)


@dataclass
class MoEWorkload:
    """One MoE expert-layer problem (all tensors on the devices requested)."""
    name: str
    T: int
    H: int
    I: int
    E: int
    top_k: int
    local_offset: int
    num_local: int
    mode: str                      # "logits" or "prerouted"
    x: torch.Tensor                # [T, H] bf16
    w1: torch.Tensor               # [L, 2I, H] bf16, rows [up | gate]
    w2: torch.Tensor               # [L, H, I] bf16
    logits: torch.Tensor | None = None     # [T, E] fp32
    topk_ids: torch.Tensor | None = None   # [T, k] int32
    topk_w: torch.Tensor | None = None     # [T, k] fp32
    meta: dict = field(default_factory=dict)


# name -> (T, H, I, E, k, mode, bias)
MOE_CONFIGS = {
    "tiny": dict(T=16, H=128, I=128, E=4, top_k=2, mode="logits", bias=None),
    "prefill_few_large": dict(T=4096, H=4096, I=14336, E=8, top_k=2, mode="logits", bias=None),
    "prefill_many_fine": dict(T=8192, H=7168, I=2048, E=256, top_k=8, mode="logits", bias="zipf1.2"),
    "decode_t1": dict(T=1, H=2048, I=768, E=128, top_k=8, mode="prerouted", bias=None),
    "decode_t8": dict(T=8, H=2048, I=768, E=128, top_k=8, mode="prerouted", bias=None),
    "decode_t64": dict(T=64, H=2048, I=768, E=128, top_k=8, mode="prerouted", bias=None),
}

GROUPED_GEMM_CONFIG = dict(sum_m=16384, E=64, K=4096, N=1536, alpha=0.3)


def zipf_bias(E: int, s: float, seed: int) -> np.ndarray:
    """Per-expert logit bias ln(p_e), p_e proportional to rank_e^-s, with the
    ranks 1..E assigned to experts by a seeded permutation."""
    rank = _rng(seed, 7).permutation(E).astype(np.float64) + 1.0
    p = rank ** (-s)
    p /= p.sum()
    return np.log(p).astype(np.float32)


def make_moe(name: str | None = None, *, seed: int = 0, device="cpu", weights_device=None,
             T=None, H=None, I=None, E=None, top_k=None, mode=None, bias=None,
             local_offset: int = 0, num_local: int | None = None) -> MoEWorkload:
    """Build a named configuration (``MOE_CONFIGS``) or a custom one.

    ``weights_device`` (default ``device``) is where W1/W2 are drawn; drawing
    them on "cuda" is much faster for the multi-GB banks."""
    cfg = dict(MOE_CONFIGS[name]) if name is not None else dict(T=T, H=H, I=I, E=E, top_k=top_k,
                                                               mode=mode or "logits", bias=bias)
    for key, val in (("T", T), ("H", H), ("I", I), ("E", E), ("top_k", top_k), ("mode", mode), ("bias", bias)):
        if val is not None:
            cfg[key] = val
    T_, H_, I_, E_, k_ = cfg["T"], cfg["H"], cfg["I"], cfg["E"], cfg["top_k"]
    L = E_ if num_local is None else num_local
    wdev = device if weights_device is None else weights_device
    x = _normal_bf16((T_, H_), 1.0, seed, 1).to(device)
    w1 = _normal_bf16((L, 2 * I_, H_), 1.0 / np.sqrt(H_), seed, 2, wdev)
    w2 = _normal_bf16((L, H_, I_), 1.0 / np.sqrt(I_), seed, 3, wdev)
    wl = MoEWorkload(name=name or "custom", T=T_, H=H_, I=I_, E=E_, top_k=k_, local_offset=local_offset,
                     num_local=L, mode=cfg["mode"], x=x, w1=w1, w2=w2)
    if cfg["mode"] == "logits":
        lg = _rng(seed, 4).standard_normal(size=(T_, E_), dtype=np.float32)
        b = cfg.get("bias")
        if b is not None:
            if isinstance(b, str) and b.startswith("zipf"):
                lg += zipf_bias(E_, float(b[4:]), seed)[None, :]
            else:
                lg += np.asarray(b, np.float32)[None, :]
        wl.logits = torch.from_numpy(lg).to(device)
    else:
        r = _rng(seed, 5)
        ids = np.argsort(r.random((T_, E_)), axis=1)[:, :k_].astype(np.int32)
        w = r.dirichlet(np.ones(k_), size=T_).astype(np.float32)
        wl.topk_ids = torch.from_numpy(ids).to(device)
        wl.topk_w = torch.from_numpy(w).to(device)
    return wl


def grouped_sizes(sum_m: int, E: int, alpha: float, seed: int) -> np.ndarray:
    """Group row counts: floor(p * sum_m), p ~ Dirichlet(alpha), remainder to
    the largest fractional parts (ties to the lower group)."""
    p = _rng(seed, 11).dirichlet(np.full(E, alpha))
    raw = p * sum_m
    sizes = np.floor(raw).astype(np.int64)
    rem = sum_m - int(sizes.sum())
    frac = raw - sizes
    order = np.lexsort((np.arange(E), -frac))
    sizes[order[:rem]] += 1
    return sizes.astype(np.int32)


def make_grouped_gemm(*, seed: int = 0, device="cpu", weights_device=None, sum_m=None, E=None, K=None,
                      N=None, alpha=None, sizes=None, with_grad: bool = False) -> dict:
    """Inputs of the ragged grouped GEMM: X [sum_m, K], W [E, N, K], offs [E]
    (cumulative group ends, int32); with_grad adds the upstream gradient
    G [sum_m, N] of the backward (dgrad, wgrad)."""
    cfg = dict(GROUPED_GEMM_CONFIG)
    for key, val in (("sum_m", sum_m), ("E", E), ("K", K), ("N", N), ("alpha", alpha)):
        if val is not None:
            cfg[key] = val
    if sizes is None:
        sizes = grouped_sizes(cfg["sum_m"], cfg["E"], cfg["alpha"], seed)
    sizes = np.asarray(sizes, np.int32)
    cfg["E"] = int(sizes.shape[0])
    cfg["sum_m"] = int(sizes.sum())
    wdev = device if weights_device is None else weights_device
    X = _normal_bf16((cfg["sum_m"], cfg["K"]), 1.0, seed, 12).to(device)
    W = _normal_bf16((cfg["E"], cfg["N"], cfg["K"]), 1.0 / np.sqrt(cfg["K"]), seed, 13, wdev)
    offs = torch.from_numpy(np.cumsum(sizes).astype(np.int32)).to(device)
    out = dict(X=X, W=W, offs=offs, sizes=sizes, **cfg)
    if with_grad:
        out["G"] = _normal_bf16((cfg["sum_m"], cfg["N"]), 1.0, seed, 14).to(device)
    return out


@dataclass
class BgmvWorkload:
    """BGMV LoRA-MoE inputs (prepare_bgmv_moe's tensors)."""
    T: int
    H: int
    R: int
    E: int
    num_loras: int
    top_k: int
    x: torch.Tensor                 # [T, H] bf16
    lora_a: list                    # per slice [L, E, R, H] bf16
    lora_b: list                    # per slice [L, E, F_s, R] bf16
    tok: torch.Tensor               # [P] int32 (sorted_token_ids)
    eid: torch.Tensor               # [P] int32 (expert_ids)
    lora: torch.Tensor              # [T] int32 (lora_indices)
    w: torch.Tensor                 # [P] fp32 (topk_weights)
    contiguous: bool                # pairs laid out p = t*k + j


def make_bgmv(*, T: int, H: int, R: int, E: int, num_loras: int, top_k: int, feat_out=None, slices: int = 1,
              contiguous: bool = True, seed: int = 0, device="cpu", weights_device=None) -> BgmvWorkload:
    wdev = device if weights_device is None else weights_device
    F = list(feat_out) if feat_out is not None else [H] * slices
    x = _normal_bf16((T, H), 1.0, seed, 21).to(device)
    A = [_normal_bf16((num_loras, E, R, H), 1.0 / np.sqrt(H), seed, 22 + 2 * s, wdev) for s in range(len(F))]
    B = [_normal_bf16((num_loras, E, F[s], R), 1.0 / np.sqrt(R), seed, 23 + 2 * s, wdev) for s in range(len(F))]
    r = _rng(seed, 24)
    lora = r.integers(0, num_loras, size=T).astype(np.int32)
    ex = np.argsort(r.random((T, E)), axis=1)[:, :top_k].astype(np.int32)
    wt = r.dirichlet(np.ones(top_k), size=T).astype(np.float32)
    tok = np.repeat(np.arange(T, dtype=np.int32), top_k)
    eid, w = ex.ravel(), wt.ravel()
    if not contiguous:  # expert-sorted dispatch order (stable)
        order = np.argsort(eid, kind="stable")
        tok, eid, w = tok[order], eid[order], w[order]
    return BgmvWorkload(T=T, H=H, R=R, E=E, num_loras=num_loras, top_k=top_k, x=x, lora_a=A, lora_b=B,
                        tok=torch.from_numpy(np.ascontiguousarray(tok)).to(device),
                        eid=torch.from_numpy(np.ascontiguousarray(eid)).to(device),
                        lora=torch.from_numpy(lora).to(device),
                        w=torch.from_numpy(np.ascontiguousarray(w)).to(device), contiguous=contiguous)


@dataclass
class Fp8Weights:
    """E4M3 expert banks (uint8 codes) with their scales."""
    w1q: torch.Tensor   # [L, 2I, H] uint8 codes, rows [up | gate]
    w2q: torch.Tensor   # [L, H, I] uint8 codes
    s1: torch.Tensor    # [L] fp32
    s2: torch.Tensor    # [L] fp32
    a1: float           # x scale
    a2: float           # h scale (requantisation)


def _e4m3_codes(shape, seed: int, stream: int, device="cpu") -> torch.Tensor:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed * 1_000_003 + stream)
    out = torch.empty(shape, dtype=torch.uint8, device=dev)
    flat = out.view(-1)
    slab = 1 << 28
    for s in range(0, flat.numel(), slab):
        n = min(slab, flat.numel() - s)
        flat[s:s + n].copy_(torch.randn(n, generator=g, device=dev).to(torch.float8_e4m3fn).view(torch.uint8))
    return out


def make_fp8_weights(L: int, H: int, I: int, *, seed: int = 0, device="cpu") -> Fp8Weights:
    r = _rng(seed, 31)
    s1 = (r.uniform(0.5, 1.5, size=L) / np.sqrt(H)).astype(np.float32)
    s2 = (r.uniform(0.5, 1.5, size=L) / np.sqrt(I)).astype(np.float32)
    return Fp8Weights(w1q=_e4m3_codes((L, 2 * I, H), seed, 32, device), w2q=_e4m3_codes((L, H, I), seed, 33, device),
                      s1=torch.from_numpy(s1).to(device), s2=torch.from_numpy(s2).to(device),
                      a1=4.0 / 448.0, a2=2.0 / 448.0)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy uint16 view of a bf16 tensor's bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bf16_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16)
