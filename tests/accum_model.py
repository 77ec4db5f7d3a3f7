"""Python access to accum_model.c: the layer evaluated with two other fp32
accumulation orders, used to derive the end-to-end acceptance floor.

TEST INFRASTRUCTURE ONLY (imported by tests/ alone).  It shares no code with
the oracle or the CUDA path.

BLOCKED_FP32 (mode 0): a correct fp32 evaluation that sums each dot product in
blocks of 16 (block sums added to the running sum), i.e. the oracle's formula
in another summation order.
TENSOR_CORE (mode 1): blocks of 16 exact products added to the fp32
accumulator together, aligned to the largest magnitude, cut toward zero with
two guard bits (a fixed-point block accumulation of the kind Fasi et al. 2021
describe for tensor cores).

floor() evaluates the tensor-core model on (a bounded subset of) a test's
tokens and returns the fraction of its outputs within 2 bf16 ulp of the
oracle's, the end-to-end floor of the parity tests.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "accum_model.c")
_LIB = os.path.join(_HERE, "libaccum_model.so")

BLOCKED_FP32 = 0
TENSOR_CORE = 1

_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    tmp = _LIB + f".{os.getpid()}.tmp"
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True, capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P, i = ctypes.c_void_p, ctypes.c_int
        lib.am_dot.argtypes = [P, P, i, i]
        lib.am_dot.restype = ctypes.c_double
        lib.am_dots.argtypes = [P, P, i, i, i, i, P]
        lib.am_dots.restype = None
        f = ctypes.c_float
        lib.am_moe_tokens_e4m3.argtypes = [P, P, P, P, P, P, P, f, f, i, i, i, i, i, i, i, P, i, P, i, i, P]
        lib.am_moe_tokens_e4m3.restype = i
        lib.am_moe_tokens.argtypes = [P, P, P, P, P, i, i, i, i, i, i, i, P, i, P, P, i, i, P]
        lib.am_moe_tokens.restype = i
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def dot(a_bits: np.ndarray, b_bits: np.ndarray, mode: int) -> float:
    a = np.ascontiguousarray(a_bits, np.uint16)
    b = np.ascontiguousarray(b_bits, np.uint16)
    assert a.shape == b.shape and a.ndim == 1
    return float(load().am_dot(_p(a), _p(b), a.shape[0], mode))


def dots(A_bits: np.ndarray, B_bits: np.ndarray, mode: int) -> np.ndarray:
    """[M, N] float64 array of the fp32 results a_m . b_n for A [M, K], B [N, K]."""
    A = np.ascontiguousarray(A_bits, np.uint16)
    B = np.ascontiguousarray(B_bits, np.uint16)
    M, K = A.shape
    N = B.shape[0]
    out = np.empty((M, N), np.float64)
    load().am_dots(_p(A), _p(B), M, N, K, mode, _p(out))
    return out


def moe_tokens(x, ids, w, w1, w2, num_experts, mode, tokens=None, local_offset=0, num_local=None,
               want_h=False, nthreads=0, clamp_limit=None):
    """out [n_tok, H] bf16 bits (and h [n_tok*k, I] when asked) for the tokens."""
    x = np.ascontiguousarray(x, np.uint16)
    ids = np.ascontiguousarray(ids, np.int32)
    w = np.ascontiguousarray(w, np.float32)
    w1 = np.ascontiguousarray(w1, np.uint16)
    w2 = np.ascontiguousarray(w2, np.uint16)
    T, H = x.shape
    k = ids.shape[1]
    L = w1.shape[0] if num_local is None else num_local
    I = w1.shape[1] // 2
    assert w1.shape == (L, 2 * I, H) and w2.shape == (L, H, I) and k <= 16
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, np.int32)
    n = tokens.shape[0]
    out = np.empty((n, H), np.uint16)
    h = np.zeros((n * k, I), np.uint16) if want_h else None
    clamp = None if clamp_limit is None else np.ascontiguousarray(clamp_limit, np.float32)
    assert clamp is None or clamp.shape == (L,)
    rc = load().am_moe_tokens(_p(x), _p(ids), _p(w), _p(w1), _p(w2), T, H, I, num_experts, k, local_offset, L,
                              _p(tokens), n, _p(out), _p(h), mode, nthreads, _p(clamp))
    assert rc & 2 == 0, "host memory ran out"
    return (out, h) if want_h else out


def floor(x, ids, w, w1, w2, num_experts, want_bits, tokens=None, local_offset=0, num_local=None,
          max_macs=1.5e10, clamp_limit=None):
    """(fraction within 2 bf16 ulp of want_bits, elements compared) for the
    tensor-core model on the first tokens of `tokens` (all T when None) whose
    multiply-adds stay within max_macs; want_bits holds the oracle's output
    rows for `tokens` in order."""
    from tests.tolerances import ulp_distance
    x = np.ascontiguousarray(x, np.uint16)
    T, H = x.shape
    k = ids.shape[1]
    I = w1.shape[1] // 2
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    per_token = max(1.0, k * 3.0 * H * I)
    n = int(min(len(tokens), max(1, max_macs // per_token)))
    if n == 0:
        return 1.0, 0
    sub = tokens[:n]
    out = moe_tokens(x, ids, w, w1, w2, num_experts, TENSOR_CORE, tokens=sub, local_offset=local_offset,
                     num_local=num_local, clamp_limit=clamp_limit)
    ref = np.asarray(want_bits)[:n]
    return float(np.mean(ulp_distance(out, ref) <= 2)), int(out.size)


def floor_e4m3(x, ids, w, w1q, w2q, s1, s2, a1, a2, num_experts, want_bits, tokens=None, local_offset=0,
               num_local=None, max_macs=1.5e10, clamp_limit=None):
    """The floor of the fp8 per-tensor family: the tensor-core model of the
    E4M3 layer on (a subset of) the tokens against the oracle's rows."""
    from tests.tolerances import ulp_distance
    x = np.ascontiguousarray(x, np.uint16)
    T, H = x.shape
    ids = np.ascontiguousarray(ids, np.int32)
    k = ids.shape[1]
    w1q = np.ascontiguousarray(w1q, np.uint8)
    w2q = np.ascontiguousarray(w2q, np.uint8)
    L = w1q.shape[0] if num_local is None else num_local
    I = w1q.shape[1] // 2
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    n = int(min(len(tokens), max(1, max_macs // max(1.0, k * 3.0 * H * I))))
    sub = np.ascontiguousarray(tokens[:n])
    out = np.empty((n, H), np.uint16)
    clamp = None if clamp_limit is None else np.ascontiguousarray(clamp_limit, np.float32)
    rc = load().am_moe_tokens_e4m3(_p(x), _p(ids), _p(np.ascontiguousarray(w, np.float32)), _p(w1q), _p(w2q),
                                   _p(np.ascontiguousarray(s1, np.float32)), _p(np.ascontiguousarray(s2, np.float32)),
                                   float(a1), float(a2), T, H, I, num_experts, k, local_offset, L, _p(sub), n,
                                   _p(out), TENSOR_CORE, 0, _p(clamp))
    assert rc & 2 == 0
    ref = np.asarray(want_bits)[:n]
    return float(np.mean(ulp_distance(out, ref) <= 2)), int(out.size)
