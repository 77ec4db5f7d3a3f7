"""CPU oracle for the routed MoE expert-layer forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the CUDA library and its Python binding) never imports, loads or calls it,
and the two share no code.

The arithmetic lives in ``moe_oracle.c`` (plain sequential fp32 loops, built
with ``-ffp-contract=off``); this module only marshals numpy arrays into it.
Every function cites the documentation passage it follows in the C source.
All bf16 tensors are carried as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

BAD_EXPERT = 1

_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with gcc (OpenMP if available) into ``out``."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    tmp = out + ".tmp"
    try:
        subprocess.run(base + ["-fopenmp", src, "-o", tmp, "-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [src, "-o", tmp, "-lm"], check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        build()
        _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


def _declare(lib):
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_route.argtypes = [P, i, i, i, P, P, i]
    lib.oracle_route.restype = None
    lib.oracle_sort.argtypes = [P, i, i, i, i, i, P, P, P]
    lib.oracle_sort.restype = i
    lib.oracle_moe_tokens.argtypes = [P, P, P, P, P, i, i, i, i, i, i, i, P, i, P, P, P, i, P]
    lib.oracle_moe_tokens.restype = i
    lib.oracle_fc1_swiglu_rows.argtypes = [P, P, P, i, i, i, P, i, P, i, P]
    lib.oracle_fc1_swiglu_rows.restype = None
    lib.oracle_fc2_rows.argtypes = [P, P, P, i, i, i, P, i, P, i]
    lib.oracle_fc2_rows.restype = None
    lib.oracle_finalize.argtypes = [P, P, P, i, i, i, P, i]
    lib.oracle_finalize.restype = None
    lib.oracle_grouped_gemm_rows.argtypes = [P, P, P, i, i, i, P, i, P, i]
    lib.oracle_grouped_gemm_rows.restype = None
    lib.oracle_grouped_gemm_dgrad_rows.argtypes = [P, P, P, i, i, i, P, i, P, i]
    lib.oracle_grouped_gemm_dgrad_rows.restype = None
    lib.oracle_grouped_gemm_wgrad_rows.argtypes = [P, P, P, i, i, i, P, P, i, P, P, i]
    lib.oracle_grouped_gemm_wgrad_rows.restype = None
    lib.oracle_bgmv.argtypes = [P, i, i, P, P, i, P, i, i, i, P, P, P, P, i, P, P, i, i]
    lib.oracle_bgmv.restype = i
    f = ctypes.c_float
    lib.oracle_float_to_e4m3.argtypes = [f]
    lib.oracle_float_to_e4m3.restype = ctypes.c_uint8
    lib.oracle_e4m3_to_float.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_float.restype = f
    lib.oracle_quantize_e4m3.argtypes = [P, ctypes.c_long, f, P]
    lib.oracle_quantize_e4m3.restype = None
    lib.oracle_moe_tokens_fp8.argtypes = [P, P, P, P, P, P, P, f, f, i, i, i, i, i, i, i, P, i, P, P, P, i, P]
    lib.oracle_moe_tokens_fp8.restype = i
    lib.oracle_fc1_fp8_rows.argtypes = [P, P, P, f, f, P, i, i, i, P, i, P, i, P]
    lib.oracle_fc1_fp8_rows.restype = None
    lib.oracle_fc2_fp8_rows.argtypes = [P, P, P, f, P, i, i, i, P, i, P, i]
    lib.oracle_fc2_fp8_rows.restype = None
    lib.oracle_float_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_float_to_bf16.restype = ctypes.c_uint16
    lib.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_float.restype = ctypes.c_float
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i
    return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads(lib=None) -> int:
    return (lib or load()).oracle_max_threads()


def route(logits: np.ndarray, top_k: int, nthreads: int = 0, lib=None):
    """Renormalised top-k routing of fp32 logits [T, E] -> (ids [T,k] int32, w [T,k] fp32)."""
    lib = lib or load()
    logits = _c(logits, np.float32)
    T, E = logits.shape
    if not (1 <= top_k <= min(E, 64)):
        raise ValueError("top_k out of range")
    ids = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float32)
    lib.oracle_route(_p(logits), T, E, top_k, _p(ids), _p(w), nthreads)
    return ids, w


def sort(ids: np.ndarray, num_experts: int, local_offset: int = 0, num_local: int | None = None, lib=None):
    """Stable sort of routes by local expert.

    Returns (m_indptr [L+1], perm_to_exp [M], exp_to_perm [T*k], status)."""
    lib = lib or load()
    ids = _c(ids, np.int32)
    T, k = ids.shape
    L = num_experts if num_local is None else num_local
    m_indptr = np.empty(L + 1, np.int32)
    p2e = np.full(T * k, -7, np.int32)
    e2p = np.empty(T * k, np.int32)
    st = lib.oracle_sort(_p(ids), T, k, num_experts, local_offset, L, _p(m_indptr), _p(p2e), _p(e2p))
    M = int(m_indptr[-1])
    return m_indptr, p2e[:M].copy(), e2p, st


def moe_tokens(x, ids, w, w1, w2, num_experts, tokens=None, local_offset=0, num_local=None,
               want_intermediates=False, nthreads=0, lib=None, clamp_limit=None):
    """Full layer for the selected tokens.

    x [T,H] u16(bf16); ids/w [T,k]; w1 [L,2I,H] u16; w2 [L,H,I] u16;
    clamp_limit [L] fp32 per local expert (SwiGLUStep) or None (SwiGLU).
    Returns out [n_tok, H] u16 (and h [n_tok*k, I] u16, y [n_tok*k, H] f32 when asked), status."""
    lib = lib or load()
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    w1 = _c(w1, np.uint16)
    w2 = _c(w2, np.uint16)
    T, H = x.shape
    k = ids.shape[1]
    L = w1.shape[0] if num_local is None else num_local
    I = w1.shape[1] // 2
    assert w1.shape == (L, 2 * I, H) and w2.shape == (L, H, I)
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    tokens = _c(tokens, np.int32)
    n = tokens.shape[0]
    out = np.empty((n, H), np.uint16)
    h = y = None
    if want_intermediates:
        h = np.zeros((n * k, I), np.uint16)
        y = np.zeros((n * k, H), np.float32)
    clamp = None if clamp_limit is None else _c(clamp_limit, np.float32)
    assert clamp is None or clamp.shape == (L,)
    st = lib.oracle_moe_tokens(_p(x), _p(ids), _p(w), _p(w1), _p(w2), T, H, I, num_experts, k,
                               local_offset, L, _p(tokens), n, _p(out), _p(h), _p(y), nthreads, _p(clamp))
    if want_intermediates:
        return out, h, y, st
    return out, st


def fc1_swiglu_rows(xp, w1, group_end, rows, nthreads=0, lib=None, clamp_limit=None):
    """h rows (bf16 bits) of FC1 + SwiGLU (SwiGLUStep with clamp_limit [L])."""
    lib = lib or load()
    xp = _c(xp, np.uint16)
    w1 = _c(w1, np.uint16)
    ge = _c(group_end, np.int32)
    rows = _c(rows, np.int32)
    L, twoI, H = w1.shape
    I = twoI // 2
    out = np.empty((rows.shape[0], I), np.uint16)
    clamp = None if clamp_limit is None else _c(clamp_limit, np.float32)
    assert clamp is None or clamp.shape == (L,)
    lib.oracle_fc1_swiglu_rows(_p(xp), _p(w1), _p(ge), L, H, I, _p(rows), rows.shape[0], _p(out), nthreads,
                               _p(clamp))
    return out


def fc2_rows(h, w2, group_end, rows, nthreads=0, lib=None):
    lib = lib or load()
    h = _c(h, np.uint16)
    w2 = _c(w2, np.uint16)
    ge = _c(group_end, np.int32)
    rows = _c(rows, np.int32)
    L, H, I = w2.shape
    out = np.empty((rows.shape[0], H), np.float32)
    lib.oracle_fc2_rows(_p(h), _p(w2), _p(ge), L, H, I, _p(rows), rows.shape[0], _p(out), nthreads)
    return out


def finalize(y, exp_to_perm, w, nthreads=0, lib=None):
    lib = lib or load()
    y = _c(y, np.float32)
    e2p = _c(exp_to_perm, np.int32)
    w = _c(w, np.float32)
    T, k = w.shape
    H = y.shape[1]
    out = np.empty((T, H), np.uint16)
    lib.oracle_finalize(_p(y), _p(e2p), _p(w), T, k, H, _p(out), nthreads)
    return out


def grouped_gemm_rows(X, W, offs, rows=None, nthreads=0, lib=None):
    """Y rows of the ragged grouped GEMM forward (bf16 bits)."""
    lib = lib or load()
    X = _c(X, np.uint16)
    W = _c(W, np.uint16)
    offs = _c(offs, np.int32)
    E, N, K = W.shape
    if rows is None:
        rows = np.arange(int(offs[-1]) if E else 0, dtype=np.int32)
    rows = _c(rows, np.int32)
    out = np.empty((rows.shape[0], N), np.uint16)
    lib.oracle_grouped_gemm_rows(_p(X), _p(W), _p(offs), E, N, K, _p(rows), rows.shape[0], _p(out), nthreads)
    return out


def grouped_gemm_dgrad_rows(G, W, offs, rows=None, nthreads=0, lib=None):
    """dX rows (bf16 bits) of the grouped GEMM's data gradient dX = G . W[e]
    for G [sum_m, N], W [E, N, K] (W used in place)."""
    lib = lib or load()
    G = _c(G, np.uint16)
    W = _c(W, np.uint16)
    offs = _c(offs, np.int32)
    E, N, K = W.shape
    assert G.shape[1] == N
    if rows is None:
        rows = np.arange(int(offs[-1]) if E else 0, dtype=np.int32)
    rows = _c(rows, np.int32)
    out = np.empty((rows.shape[0], K), np.uint16)
    lib.oracle_grouped_gemm_dgrad_rows(_p(G), _p(W), _p(offs), E, N, K, _p(rows), rows.shape[0], _p(out), nthreads)
    return out


def grouped_gemm_wgrad_rows(G, X, offs, sel_e, sel_n, K=None, nthreads=0, lib=None):
    """Rows (e, n) of the grouped GEMM's weight gradient dW[e] = G_e^T . X_e:
    returns (fp32 [n_sel, K], bf16 bits [n_sel, K])."""
    lib = lib or load()
    G = _c(G, np.uint16)
    X = _c(X, np.uint16)
    offs = _c(offs, np.int32)
    sel_e = _c(sel_e, np.int32)
    sel_n = _c(sel_n, np.int32)
    N = G.shape[1]
    K = X.shape[1]
    n = sel_e.shape[0]
    f32 = np.empty((n, K), np.float32)
    b16 = np.empty((n, K), np.uint16)
    lib.oracle_grouped_gemm_wgrad_rows(_p(G), _p(X), _p(offs), offs.shape[0], N, K, _p(sel_e), _p(sel_n), n,
                                       _p(f32), _p(b16), nthreads)
    return f32, b16


def bgmv(x, lora_a, lora_b, tok, eid, lora, w, nthreads=0, lib=None):
    """BGMV LoRA-MoE shrink + expand (prepare_bgmv_moe).

    x [T, H] u16; lora_a / lora_b lists (one entry per slice) of
    [num_loras, E, R, H] / [num_loras, E, F_s, R] u16; tok, eid [P] int32 per
    routed pair; lora [T] int32 per token; w [P] fp32.
    Returns (shrink [S, P, R] u16, y [T, sum F_s] fp32, status)."""
    lib = lib or load()
    x = _c(x, np.uint16)
    T, H = x.shape
    A = [_c(a, np.uint16) for a in lora_a]
    B = [_c(b, np.uint16) for b in lora_b]
    S = len(A)
    L, E, R, H2 = A[0].shape
    assert H2 == H and all(a.shape == (L, E, R, H) for a in A)
    F = [b.shape[2] for b in B]
    assert all(b.shape == (L, E, f, R) for b, f in zip(B, F))
    tok, eid, lora, w = _c(tok, np.int32), _c(eid, np.int32), _c(lora, np.int32), _c(w, np.float32)
    P = tok.shape[0]
    shrink = np.empty((S, P, R), np.uint16)
    y = np.empty((T, sum(F)), np.float32)
    a_ptrs = (ctypes.c_void_p * S)(*[a.ctypes.data for a in A])
    b_ptrs = (ctypes.c_void_p * S)(*[b.ctypes.data for b in B])
    f_arr = (ctypes.c_int * S)(*F)
    st = lib.oracle_bgmv(_p(x), T, H, ctypes.cast(a_ptrs, ctypes.c_void_p), ctypes.cast(b_ptrs, ctypes.c_void_p),
                         S, ctypes.cast(f_arr, ctypes.c_void_p), L, E, R, _p(tok), _p(eid), _p(lora), _p(w), P,
                         _p(shrink), _p(y), sum(F), nthreads)
    return shrink, y, st


def e4m3_encode(v: float, lib=None) -> int:
    return int((lib or load()).oracle_float_to_e4m3(float(v)))


def e4m3_decode(code: int, lib=None) -> float:
    return float((lib or load()).oracle_e4m3_to_float(int(code)))


def quantize_e4m3(x_bits, a1, lib=None):
    """E4M3 codes of x / a1 (x as bf16 bits), any shape."""
    lib = lib or load()
    x = _c(x_bits, np.uint16)
    out = np.empty(x.shape, np.uint8)
    lib.oracle_quantize_e4m3(_p(x), x.size, float(a1), _p(out))
    return out


def moe_tokens_fp8(x, ids, w, w1q, w2q, s1, s2, a1, a2, num_experts, tokens=None, local_offset=0,
                   num_local=None, want_intermediates=False, nthreads=0, lib=None, clamp_limit=None):
    """The layer with E4M3 weights (codes w1q [L,2I,H], w2q [L,H,I], per-expert
    scales s1, s2 [L]) and per-tensor activation scales a1 (x) and a2 (h).
    Returns out [n_tok, H] u16 (and hq [n_tok*k, I] u8, y [n_tok*k, H] f32), status."""
    lib = lib or load()
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    w1q = _c(w1q, np.uint8)
    w2q = _c(w2q, np.uint8)
    T, H = x.shape
    k = ids.shape[1]
    L = w1q.shape[0] if num_local is None else num_local
    I = w1q.shape[1] // 2
    assert w1q.shape == (L, 2 * I, H) and w2q.shape == (L, H, I)
    s1, s2 = _c(s1, np.float32), _c(s2, np.float32)
    tokens = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
    n = tokens.shape[0]
    out = np.empty((n, H), np.uint16)
    hq = y = None
    if want_intermediates:
        hq = np.zeros((n * k, I), np.uint8)
        y = np.zeros((n * k, H), np.float32)
    clamp = None if clamp_limit is None else _c(clamp_limit, np.float32)
    st = lib.oracle_moe_tokens_fp8(_p(x), _p(ids), _p(w), _p(w1q), _p(w2q), _p(s1), _p(s2), float(a1), float(a2),
                                   T, H, I, num_experts, k, local_offset, L, _p(tokens), n, _p(out), _p(hq), _p(y),
                                   nthreads, _p(clamp))
    if want_intermediates:
        return out, hq, y, st
    return out, st


def fc1_fp8_rows(xq, w1q, s1, a1, a2, group_end, rows, nthreads=0, lib=None, clamp_limit=None):
    lib = lib or load()
    xq, w1q = _c(xq, np.uint8), _c(w1q, np.uint8)
    ge, rows, s1 = _c(group_end, np.int32), _c(rows, np.int32), _c(s1, np.float32)
    L, twoI, H = w1q.shape
    I = twoI // 2
    out = np.empty((rows.shape[0], I), np.uint8)
    clamp = None if clamp_limit is None else _c(clamp_limit, np.float32)
    lib.oracle_fc1_fp8_rows(_p(xq), _p(w1q), _p(s1), float(a1), float(a2), _p(ge), L, H, I, _p(rows), rows.shape[0],
                            _p(out), nthreads, _p(clamp))
    return out


def fc2_fp8_rows(hq, w2q, s2, a2, group_end, rows, nthreads=0, lib=None):
    lib = lib or load()
    hq, w2q = _c(hq, np.uint8), _c(w2q, np.uint8)
    ge, rows, s2 = _c(group_end, np.int32), _c(rows, np.int32), _c(s2, np.float32)
    L, H, I = w2q.shape
    out = np.empty((rows.shape[0], H), np.float32)
    lib.oracle_fc2_fp8_rows(_p(hq), _p(w2q), _p(s2), float(a2), _p(ge), L, H, I, _p(rows), rows.shape[0], _p(out),
                            nthreads)
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)
