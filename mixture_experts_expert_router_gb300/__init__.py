"""GB300-native (sm_103a) routed mixture-of-experts expert layer.

Python binding of the C ABI declared in ``include/moe_gb300.h``.  The
functions here carry the ABI's names and only marshal arguments: they check
dtypes, devices and contiguity, allocate outputs with torch when the caller
does not pass them, and hand raw device pointers plus the current CUDA stream
to ``libmoe_gb300.so``.  Every step of the layer runs in that library's CUDA
kernels; there is no Python or CPU fallback, and a missing library raises.

    out = moe_forward(x, w1, w2, num_experts=E, top_k=k, logits=logits)

Shapes: x [T, H] bf16; w1 [L, 2I, H] bf16 with the I "up" rows of each expert
followed by its I "gate" rows; w2 [L, H, I] bf16; logits [T, E] fp32, or
topk_ids [T, k] int32 with topk_w [T, k] fp32 (weights normalised by the
caller).  out [T, H] bf16.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "MoEError", "library", "library_path", "moe_status_string", "moe_route", "moe_sort", "moe_sort_no_alloc",
    "moe_sort_workspace_size", "moe_gather", "moe_fc1_swiglu", "moe_fc2", "moe_finalize",
    "moe_fc1_swiglu_swapab", "moe_fc2_swapab", "moe_fc1_swiglu_gathered",
    "grouped_gemm_fwd", "grouped_gemm_dgrad", "grouped_gemm_wgrad", "bgmv", "moe_workspace_size", "moe_forward", "MoEPlan", "ABI_SYMBOLS",
    "PATH_AUTO", "PATH_GROUPED", "PATH_DECODE", "DEV_BAD_EXPERT", "DEV_TIMEOUT",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

PATH_AUTO, PATH_GROUPED, PATH_DECODE = 0, 1, 2
PLAN_STAGE_TIMING = 1
PLAN_ONE_CTA_GEMM = 2
PLAN_DECODE_CHAIN = 4
PLAN_DECODE_SEPARATE = 8
PLAN_FUSED_GATHER = 16
PLAN_DECODE_ONE_LAUNCH = 32
PLAN_TEST_UNREACHABLE_WAIT = 64
PLAN_NO_TAIL_TILES = 128
PLAN_NO_SMALL_GROUP_KERNEL = 256
PLAN_SMALL_GROUP_KERNEL = 512
WEIGHTS_BF16, WEIGHTS_E4M3 = 0, 1
WAIT_LIMIT_MIN_NS, WAIT_LIMIT_MAX_NS = 1000, 600_000_000_000
DEV_BAD_EXPERT, DEV_TIMEOUT = 1, 2
MAX_EXPERTS, MAX_TOP_K = 1024, 16

# Every function include/moe_gb300.h declares.
ABI_SYMBOLS = [
    "moe_status_string", "moe_abi_version", "moe_route", "moe_sort_workspace_size", "moe_sort",
    "moe_gather", "moe_fc1_swiglu", "moe_fc2", "moe_finalize", "grouped_gemm_fwd",
    "moe_workspace_size", "moe_forward", "moe_forward_prepare", "moe_plan_launch",
    "moe_plan_buffers_get", "moe_plan_stage_count", "moe_plan_stage_name", "moe_plan_stage_times",
    "moe_plan_stage_reset", "moe_plan_kernels_per_launch", "moe_plan_destroy", "moe_sort_no_alloc",
    "moe_fc1_swiglu_swapab", "moe_fc2_swapab", "moe_fc1_swiglu_gathered", "moe_plan_set_wait_limit",
    "moe_fc1_swiglu_step", "grouped_gemm_dgrad", "grouped_gemm_wgrad", "moe_bgmv_workspace_size", "moe_bgmv",
    "moe_fc1_swiglu_e4m3", "moe_fc2_e4m3", "grouped_gemm_fwd_flags", "grouped_gemm_fwd_ex",
]


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {moe_status_string(code)} (code {code})")
        self.code = code


class _Desc(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p), ("logits", ctypes.c_void_p), ("topk_ids", ctypes.c_void_p),
        ("topk_w", ctypes.c_void_p), ("w1", ctypes.c_void_p), ("w2", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("status", ctypes.c_void_p), ("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
        ("E", ctypes.c_int), ("top_k", ctypes.c_int), ("local_offset", ctypes.c_int),
        ("num_local", ctypes.c_int), ("path", ctypes.c_int), ("flags", ctypes.c_int),
        ("clamp_limit", ctypes.c_void_p), ("weight_format", ctypes.c_int), ("w1_scale", ctypes.c_void_p),
        ("w2_scale", ctypes.c_void_p), ("x_scale", ctypes.c_float), ("h_scale", ctypes.c_float),
    ]


class _Buffers(ctypes.Structure):
    _fields_ = [
        ("topk_ids", ctypes.c_void_p), ("topk_w", ctypes.c_void_p), ("m_indptr", ctypes.c_void_p),
        ("perm_to_exp", ctypes.c_void_p), ("exp_to_perm", ctypes.c_void_p), ("xp", ctypes.c_void_p),
        ("h", ctypes.c_void_p), ("y", ctypes.c_void_p), ("path", ctypes.c_int),
    ]


_lib = None


def library_path() -> str:
    return _LIB_PATH


def library():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        sig = {
            "moe_status_string": ([I], ctypes.c_char_p),
            "moe_abi_version": ([], I),
            "moe_route": ([P, I, I, I, P, P, P], I),
            "moe_sort_workspace_size": ([I, I, I], Z),
            "moe_sort": ([P, I, I, I, I, I, P, P, P, P, Z, P, P], I),
            "moe_sort_no_alloc": ([P, I, I, I, I, I, P, P, P, P, P], I),
            "moe_gather": ([P, P, P, I, I, I, I, P, P], I),
            "moe_fc1_swiglu": ([P, P, P, I, I, I, I, P, P], I),
            "moe_fc1_swiglu_step": ([P, P, P, P, I, I, I, I, P, P], I),
            "moe_fc1_swiglu_e4m3": ([P, P, P, ctypes.c_float, ctypes.c_float, P, P, I, I, I, I, P, P], I),
            "moe_fc2_e4m3": ([P, P, P, ctypes.c_float, P, I, I, I, I, P, P], I),
            "moe_fc2": ([P, P, P, I, I, I, I, P, P], I),
            "moe_fc1_swiglu_swapab": ([P, P, P, I, I, I, I, I, P, P], I),
            "moe_fc1_swiglu_gathered": ([P, P, P, I, I, P, I, I, I, P, P], I),
            "moe_fc2_swapab": ([P, P, P, I, I, I, I, I, P, P], I),
            "moe_finalize": ([P, P, P, I, I, I, P, P], I),
            "grouped_gemm_fwd": ([P, P, P, I, I, I, I, P, P], I),
            "grouped_gemm_fwd_flags": ([P, P, P, I, I, I, I, P, I, P], I),
            "grouped_gemm_fwd_ex": ([P, P, P, I, I, I, I, P, I, P, P], I),
            "grouped_gemm_dgrad": ([P, P, P, I, I, I, I, P, P], I),
            "moe_bgmv_workspace_size": ([I, I, I, I, I, I], Z),
            "moe_bgmv": ([P, I, I, P, P, I, P, I, I, I, P, P, P, P, I, I, P, P, I, P, Z, P, P], I),
            "grouped_gemm_wgrad": ([P, P, P, I, I, I, I, P, I, P], I),
            "moe_workspace_size": ([I, I, I, I, I, I], Z),
            "moe_forward": ([P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, Z, P, P], I),
            "moe_forward_prepare": ([ctypes.POINTER(_Desc), ctypes.POINTER(P)], I),
            "moe_plan_launch": ([P, P], I),
            "moe_plan_buffers_get": ([P, ctypes.POINTER(_Buffers)], I),
            "moe_plan_stage_count": ([P], I),
            "moe_plan_stage_name": ([P, I], ctypes.c_char_p),
            "moe_plan_stage_times": ([P, ctypes.POINTER(ctypes.c_float), I, ctypes.POINTER(I)], I),
            "moe_plan_stage_reset": ([P], I),
            "moe_plan_set_wait_limit": ([P, ctypes.c_ulonglong], I),
            "moe_plan_kernels_per_launch": ([P], I),
            "moe_plan_destroy": ([P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def moe_status_string(code: int) -> str:
    return library().moe_status_string(int(code)).decode()


def _check(rc: int, where: str):
    if rc != 0:
        raise MoEError(rc, where)


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, dtype, name: str, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


# ----------------------------------------------------------------- stages --

def moe_route(logits: torch.Tensor, top_k: int, topk_ids=None, topk_w=None):
    """Renormalised top-k routing: (ids [T,k] int32, weights [T,k] fp32)."""
    _need(logits, torch.float32, "logits")
    T, E = logits.shape
    dev = logits.device
    topk_ids = torch.empty((T, top_k), dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
    topk_w = torch.empty((T, top_k), dtype=torch.float32, device=dev) if topk_w is None else topk_w
    _need(topk_ids, torch.int32, "topk_ids", (T, top_k), dev)
    _need(topk_w, torch.float32, "topk_w", (T, top_k), dev)
    _check(library().moe_route(_ptr(logits), T, E, top_k, _ptr(topk_ids), _ptr(topk_w), _stream(dev)),
           "moe_route")
    return topk_ids, topk_w


def moe_sort_workspace_size(T: int, top_k: int, num_local: int) -> int:
    return int(library().moe_sort_workspace_size(T, top_k, num_local))


def moe_sort(topk_ids: torch.Tensor, num_experts: int, local_offset: int = 0, num_local=None,
             m_indptr=None, perm_to_exp=None, exp_to_perm=None, workspace=None, status=None):
    """Stable sort of routes by local expert.

    Returns (m_indptr [L+1], perm_to_exp [T*k], exp_to_perm [T*k], status [1])."""
    _need(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    dev = topk_ids.device
    L = num_experts if num_local is None else num_local
    R = T * k
    m_indptr = torch.empty(L + 1, dtype=torch.int32, device=dev) if m_indptr is None else m_indptr
    perm_to_exp = torch.empty(max(R, 1), dtype=torch.int32, device=dev) if perm_to_exp is None else perm_to_exp
    exp_to_perm = torch.empty(max(R, 1), dtype=torch.int32, device=dev) if exp_to_perm is None else exp_to_perm
    status = torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status
    need = moe_sort_workspace_size(T, k, L)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(library().moe_sort(_ptr(topk_ids), T, k, num_experts, local_offset, L, _ptr(m_indptr),
                              _ptr(perm_to_exp), _ptr(exp_to_perm), _ptr(workspace), wbytes,
                              _ptr(status), _stream(dev)), "moe_sort")
    return m_indptr, perm_to_exp[:R], exp_to_perm[:R], status


def moe_sort_no_alloc(topk_ids: torch.Tensor, num_experts: int, local_offset: int = 0, num_local=None,
                      m_indptr=None, perm_to_exp=None, exp_to_perm=None, status=None):
    """moe_sort without a workspace, for callers that cannot allocate device
    memory (a plugin that only receives its input and output buffers, or a
    runtime that forbids allocating after start-up): the library keeps the
    sort's scratch table in its own fixed device array (see the C header for
    the size limit and for why overlapping calls race).  This wrapper still
    creates missing output tensors with torch for convenience; pass them in
    to allocate nothing."""
    _need(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    dev = topk_ids.device
    L = num_experts if num_local is None else num_local
    R = T * k
    m_indptr = torch.empty(L + 1, dtype=torch.int32, device=dev) if m_indptr is None else m_indptr
    perm_to_exp = torch.empty(max(R, 1), dtype=torch.int32, device=dev) if perm_to_exp is None else perm_to_exp
    exp_to_perm = torch.empty(max(R, 1), dtype=torch.int32, device=dev) if exp_to_perm is None else exp_to_perm
    status = torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status
    _check(library().moe_sort_no_alloc(_ptr(topk_ids), T, k, num_experts, local_offset, L, _ptr(m_indptr),
                                       _ptr(perm_to_exp), _ptr(exp_to_perm), _ptr(status), _stream(dev)),
           "moe_sort_no_alloc")
    return m_indptr, perm_to_exp[:R], exp_to_perm[:R], status


def moe_gather(x: torch.Tensor, perm_to_exp: torch.Tensor, m_indptr: torch.Tensor, top_k: int, xp=None):
    _need(x, torch.bfloat16, "x")
    T, H = x.shape
    dev = x.device
    L = m_indptr.numel() - 1
    xp = torch.empty((T * top_k, H), dtype=torch.bfloat16, device=dev) if xp is None else xp
    _need(xp, torch.bfloat16, "xp", device=dev)
    _check(library().moe_gather(_ptr(x), _ptr(perm_to_exp), _ptr(m_indptr), T, H, top_k, L, _ptr(xp),
                                _stream(dev)), "moe_gather")
    return xp


def moe_fc1_swiglu(xp: torch.Tensor, w1: torch.Tensor, m_indptr: torch.Tensor, h=None, clamp_limit=None):
    """FC1 + SwiGLU; with clamp_limit [L] fp32 the SwiGLUStep(limit) epilogue."""
    _need(xp, torch.bfloat16, "xp")
    _need(w1, torch.bfloat16, "w1")
    _need(m_indptr, torch.int32, "m_indptr")
    rows, H = xp.shape
    L, twoI, H2 = w1.shape
    if H2 != H or twoI % 2:
        raise ValueError("w1 must be [L, 2I, H]")
    I = twoI // 2
    h = torch.empty((rows, I), dtype=torch.bfloat16, device=xp.device) if h is None else h
    _need(h, torch.bfloat16, "h", (rows, I), xp.device)
    if clamp_limit is not None:
        _need(clamp_limit, torch.float32, "clamp_limit", (L,), xp.device)
        _check(library().moe_fc1_swiglu_step(_ptr(xp), _ptr(w1), _ptr(clamp_limit), _ptr(m_indptr), rows, H, I,
                                             L, _ptr(h), _stream(xp.device)), "moe_fc1_swiglu_step")
        return h
    _check(library().moe_fc1_swiglu(_ptr(xp), _ptr(w1), _ptr(m_indptr), rows, H, I, L, _ptr(h),
                                    _stream(xp.device)), "moe_fc1_swiglu")
    return h


def moe_fc1_swiglu_e4m3(xq, w1q, w1_scale, x_scale: float, h_scale: float, m_indptr, hq=None, clamp_limit=None):
    """FC1 + SwiGLU(Step) on E4M3 rows: hq = e4m3(swiglu(dequantised u, g) / h_scale)."""
    _need(xq, torch.uint8, "xq")
    _need(w1q, torch.uint8, "w1q")
    rows, H = xq.shape
    L, twoI, _ = w1q.shape
    I = twoI // 2
    _need(w1_scale, torch.float32, "w1_scale", (L,), xq.device)
    hq = torch.empty((rows, I), dtype=torch.uint8, device=xq.device) if hq is None else hq
    _check(library().moe_fc1_swiglu_e4m3(_ptr(xq), _ptr(w1q), _ptr(w1_scale), float(x_scale), float(h_scale),
                                         _ptr(clamp_limit), _ptr(m_indptr), rows, H, I, L, _ptr(hq),
                                         _stream(xq.device)), "moe_fc1_swiglu_e4m3")
    return hq


def moe_fc2_e4m3(hq, w2q, w2_scale, h_scale: float, m_indptr, y=None):
    """FC2 on E4M3 rows: y = (hq . W2q^T) * h_scale * w2_scale[e], fp32."""
    _need(hq, torch.uint8, "hq")
    _need(w2q, torch.uint8, "w2q")
    rows, I = hq.shape
    L, H, _ = w2q.shape
    _need(w2_scale, torch.float32, "w2_scale", (L,), hq.device)
    y = torch.empty((rows, H), dtype=torch.float32, device=hq.device) if y is None else y
    _check(library().moe_fc2_e4m3(_ptr(hq), _ptr(w2q), _ptr(w2_scale), float(h_scale), _ptr(m_indptr), rows, H, I,
                                  L, _ptr(y), _stream(hq.device)), "moe_fc2_e4m3")
    return y


def moe_fc2(h: torch.Tensor, w2: torch.Tensor, m_indptr: torch.Tensor, y=None):
    _need(h, torch.bfloat16, "h")
    _need(w2, torch.bfloat16, "w2")
    _need(m_indptr, torch.int32, "m_indptr")
    rows, I = h.shape
    L, H, I2 = w2.shape
    if I2 != I:
        raise ValueError("w2 must be [L, H, I]")
    y = torch.empty((rows, H), dtype=torch.float32, device=h.device) if y is None else y
    _need(y, torch.float32, "y", (rows, H), h.device)
    _check(library().moe_fc2(_ptr(h), _ptr(w2), _ptr(m_indptr), rows, H, I, L, _ptr(y),
                             _stream(h.device)), "moe_fc2")
    return y


def moe_fc1_swiglu_gathered(x: torch.Tensor, perm_to_exp: torch.Tensor, m_indptr: torch.Tensor, top_k: int,
                            w1: torch.Tensor, h=None):
    """FC1 + SwiGLU with the rows taken straight from x through the permutation."""
    _need(x, torch.bfloat16, "x")
    _need(perm_to_exp, torch.int32, "perm_to_exp")
    _need(m_indptr, torch.int32, "m_indptr")
    _need(w1, torch.bfloat16, "w1")
    T, H = x.shape
    L, twoI, H2 = w1.shape
    if H2 != H or twoI % 2:
        raise ValueError("w1 must be [L, 2I, H]")
    I = twoI // 2
    h = torch.empty((T * top_k, I), dtype=torch.bfloat16, device=x.device) if h is None else h
    _need(h, torch.bfloat16, "h", (T * top_k, I), x.device)
    _check(library().moe_fc1_swiglu_gathered(_ptr(x), _ptr(perm_to_exp), _ptr(m_indptr), T, top_k, _ptr(w1),
                                             H, I, L, _ptr(h), _stream(x.device)), "moe_fc1_swiglu_gathered")
    return h


def moe_fc1_swiglu_swapab(xp: torch.Tensor, w1: torch.Tensor, m_indptr: torch.Tensor, max_group_rows: int,
                          h=None):
    """Decode-form FC1 + SwiGLU (weights on the MMA's M side)."""
    _need(xp, torch.bfloat16, "xp")
    _need(w1, torch.bfloat16, "w1")
    _need(m_indptr, torch.int32, "m_indptr")
    rows, H = xp.shape
    L, twoI, H2 = w1.shape
    if H2 != H or twoI % 2:
        raise ValueError("w1 must be [L, 2I, H]")
    I = twoI // 2
    h = torch.empty((rows, I), dtype=torch.bfloat16, device=xp.device) if h is None else h
    _need(h, torch.bfloat16, "h", (rows, I), xp.device)
    _check(library().moe_fc1_swiglu_swapab(_ptr(xp), _ptr(w1), _ptr(m_indptr), rows, max_group_rows, H, I, L,
                                           _ptr(h), _stream(xp.device)), "moe_fc1_swiglu_swapab")
    return h


def moe_fc2_swapab(h: torch.Tensor, w2: torch.Tensor, m_indptr: torch.Tensor, max_group_rows: int, y=None):
    """Decode-form FC2 (weights on the MMA's M side), fp32 out."""
    _need(h, torch.bfloat16, "h")
    _need(w2, torch.bfloat16, "w2")
    _need(m_indptr, torch.int32, "m_indptr")
    rows, I = h.shape
    L, H, I2 = w2.shape
    if I2 != I:
        raise ValueError("w2 must be [L, H, I]")
    y = torch.empty((rows, H), dtype=torch.float32, device=h.device) if y is None else y
    _need(y, torch.float32, "y", (rows, H), h.device)
    _check(library().moe_fc2_swapab(_ptr(h), _ptr(w2), _ptr(m_indptr), rows, max_group_rows, H, I, L, _ptr(y),
                                    _stream(h.device)), "moe_fc2_swapab")
    return y


def moe_finalize(y: torch.Tensor, exp_to_perm: torch.Tensor, topk_w: torch.Tensor, out=None):
    _need(y, torch.float32, "y")
    _need(exp_to_perm, torch.int32, "exp_to_perm")
    _need(topk_w, torch.float32, "topk_w")
    T, k = topk_w.shape
    H = y.shape[1]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device) if out is None else out
    _need(out, torch.bfloat16, "out", (T, H), y.device)
    _check(library().moe_finalize(_ptr(y), _ptr(exp_to_perm), _ptr(topk_w), T, k, H, _ptr(out),
                                  _stream(y.device)), "moe_finalize")
    return out


GROUPED_GEMM_COUNTERS = 4


def grouped_gemm_fwd(X: torch.Tensor, W: torch.Tensor, offs: torch.Tensor, Y=None, no_tail_tiles: bool = False,
                     small_group_kernel: bool | None = None, counters=None):
    """Ragged grouped GEMM forward: Y[group e] = X[group e] @ W[e].T (bf16).

    small_group_kernel=True runs the groups of at most 64 rows in the
    small-group kernel beside the CTA-pair kernel (grouped_gemm_fwd_ex); it
    pays where the GEMM is tensor-bound (active groups averaging well over
    about 280 rows) with some small groups, and not where weight streaming
    bounds it (off by default).  counters: the call's int32
    [GROUPED_GEMM_COUNTERS] claim counters (allocated when None)."""
    _need(X, torch.bfloat16, "X")
    _need(W, torch.bfloat16, "W")
    _need(offs, torch.int32, "offs")
    sum_m, K = X.shape
    E, N, K2 = W.shape
    if K2 != K or offs.numel() != E:
        raise ValueError("shapes: X [sum_m, K], W [E, N, K], offs [E]")
    Y = torch.empty((sum_m, N), dtype=torch.bfloat16, device=X.device) if Y is None else Y
    _need(Y, torch.bfloat16, "Y", (sum_m, N), X.device)
    flags = PLAN_NO_TAIL_TILES if no_tail_tiles else 0
    if small_group_kernel:
        if counters is None:
            counters = torch.empty(GROUPED_GEMM_COUNTERS, dtype=torch.int32, device=X.device)
        _need(counters, torch.int32, "counters", (GROUPED_GEMM_COUNTERS,), X.device)
        _check(library().grouped_gemm_fwd_ex(_ptr(X), _ptr(W), _ptr(offs), sum_m, E, N, K, _ptr(Y), flags,
                                             _ptr(counters), _stream(X.device)), "grouped_gemm_fwd")
        return Y
    _check(library().grouped_gemm_fwd_flags(_ptr(X), _ptr(W), _ptr(offs), sum_m, E, N, K, _ptr(Y),
                                            flags, _stream(X.device)),
           "grouped_gemm_fwd")
    return Y


def grouped_gemm_dgrad(G: torch.Tensor, W: torch.Tensor, offs: torch.Tensor, dX=None):
    """Data gradient of the ragged grouped GEMM: dX[group e] = G[group e] @ W[e]
    (W [E, N, K] used in place, bf16)."""
    _need(G, torch.bfloat16, "G")
    _need(W, torch.bfloat16, "W")
    _need(offs, torch.int32, "offs")
    sum_m, N = G.shape
    E, N2, K = W.shape
    if N2 != N or offs.numel() != E:
        raise ValueError("shapes: G [sum_m, N], W [E, N, K], offs [E]")
    dX = torch.empty((sum_m, K), dtype=torch.bfloat16, device=G.device) if dX is None else dX
    _need(dX, torch.bfloat16, "dX", (sum_m, K), G.device)
    _check(library().grouped_gemm_dgrad(_ptr(G), _ptr(W), _ptr(offs), sum_m, E, N, K, _ptr(dX),
                                        _stream(G.device)), "grouped_gemm_dgrad")
    return dX


def grouped_gemm_wgrad(G: torch.Tensor, X: torch.Tensor, offs: torch.Tensor, out_dtype=torch.float32, dW=None):
    """Weight gradient of the ragged grouped GEMM: dW[e] = G[group e].T @ X[group e]
    ([E, N, K], fp32 or bf16; exactly zero for an empty group)."""
    _need(G, torch.bfloat16, "G")
    _need(X, torch.bfloat16, "X")
    _need(offs, torch.int32, "offs")
    sum_m, N = G.shape
    sum_m2, K = X.shape
    E = offs.numel()
    if sum_m2 != sum_m or out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("shapes: G [sum_m, N], X [sum_m, K], offs [E]; out_dtype fp32 or bf16")
    dW = torch.empty((E, N, K), dtype=out_dtype, device=G.device) if dW is None else dW
    _need(dW, out_dtype, "dW", (E, N, K), G.device)
    _check(library().grouped_gemm_wgrad(_ptr(G), _ptr(X), _ptr(offs), sum_m, E, N, K, _ptr(dW),
                                        1 if out_dtype == torch.float32 else 0, _stream(G.device)),
           "grouped_gemm_wgrad")
    return dW


def bgmv(x, lora_a, lora_b, sorted_token_ids, expert_ids, lora_indices, topk_weights, contiguous_top_k=0,
         shrink_out=None, y_accum=None, workspace=None, status=None):
    """BGMV LoRA-MoE shrink + expand (moe_bgmv): returns (y_accum [T, sum F]
    fp32, shrink_out [S, P, R] bf16).  lora_a / lora_b are lists with one
    tensor per slice ([L, E, R, H] / [L, E, F_s, R] bf16)."""
    _need(x, torch.bfloat16, "x")
    T, H = x.shape
    S = len(lora_a)
    if S < 1 or len(lora_b) != S:
        raise ValueError("lora_a and lora_b need one tensor per slice")
    L, E, R, H2 = lora_a[0].shape
    if H2 != H:
        raise ValueError("lora_a must be [num_loras, E, rank, H]")
    F = []
    for a_s, b_s in zip(lora_a, lora_b):
        _need(a_s, torch.bfloat16, "lora_a", (L, E, R, H), x.device)
        _need(b_s, torch.bfloat16, "lora_b", None, x.device)
        if tuple(b_s.shape[:2]) != (L, E) or b_s.shape[3] != R:
            raise ValueError("lora_b must be [num_loras, E, feat_out, rank]")
        F.append(int(b_s.shape[2]))
    P = sorted_token_ids.numel()
    for t_, n_, dt in ((sorted_token_ids, "sorted_token_ids", torch.int32), (expert_ids, "expert_ids", torch.int32),
                       (topk_weights, "topk_weights", torch.float32)):
        _need(t_, dt, n_, (P,), x.device)
    _need(lora_indices, torch.int32, "lora_indices", (T,), x.device)
    dev = x.device
    shrink_out = torch.empty((S, P, R), dtype=torch.bfloat16, device=dev) if shrink_out is None else shrink_out
    _need(shrink_out, torch.bfloat16, "shrink_out", (S, P, R), dev)
    if y_accum is None:
        y_accum = torch.empty((T, sum(F)), dtype=torch.float32, device=dev)
    if y_accum.dtype != torch.float32 or not y_accum.is_cuda or y_accum.shape[0] != T or y_accum.stride(1) != 1:
        raise ValueError("y_accum must be a CUDA fp32 [T, >= sum(feat_out)] tensor with unit column stride")
    need = int(library().moe_bgmv_workspace_size(T, P, contiguous_top_k, L, E, sum(F)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    a_ptrs = (ctypes.c_void_p * S)(*[a_s.data_ptr() for a_s in lora_a])
    b_ptrs = (ctypes.c_void_p * S)(*[b_s.data_ptr() for b_s in lora_b])
    f_arr = (ctypes.c_int * S)(*F)
    _check(library().moe_bgmv(_ptr(x), T, H, ctypes.cast(a_ptrs, ctypes.c_void_p), ctypes.cast(b_ptrs, ctypes.c_void_p),
                              S, ctypes.cast(f_arr, ctypes.c_void_p), R, L, E, _ptr(sorted_token_ids),
                              _ptr(expert_ids), _ptr(lora_indices), _ptr(topk_weights), P, contiguous_top_k,
                              _ptr(shrink_out), _ptr(y_accum), y_accum.stride(0), _ptr(workspace),
                              workspace.numel(), _ptr(status), _stream(dev)), "moe_bgmv")
    return y_accum, shrink_out


# ------------------------------------------------------------ whole layer --

def moe_workspace_size(T: int, H: int, I: int, E: int, top_k: int, num_local: int | None = None) -> int:
    return int(library().moe_workspace_size(T, H, I, E, top_k, E if num_local is None else num_local))


def _layer_args(x, w1, w2, num_experts, top_k, logits, topk_ids, topk_w, local_offset, out, wdtype=torch.bfloat16):
    _need(x, torch.bfloat16, "x")
    dev = x.device
    T, H = x.shape
    _need(w1, wdtype, "w1", device=dev)
    _need(w2, wdtype, "w2", device=dev)
    L, twoI, H1 = w1.shape
    I = twoI // 2
    if H1 != H or tuple(w2.shape) != (L, H, I):
        raise ValueError("w1 must be [L, 2I, H] and w2 [L, H, I]")
    if logits is not None:
        _need(logits, torch.float32, "logits", (T, num_experts), dev)
    if topk_ids is not None:
        _need(topk_ids, torch.int32, "topk_ids", (T, top_k), dev)
    if topk_w is not None:
        _need(topk_w, torch.float32, "topk_w", (T, top_k), dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if out is None else out
    _need(out, torch.bfloat16, "out", (T, H), dev)
    return T, H, I, L, out


def moe_forward(x, w1, w2, num_experts: int, top_k: int, logits=None, topk_ids=None, topk_w=None,
                local_offset: int = 0, out=None, workspace=None, status=None):
    """One-shot layer forward (route or pre-routed -> sort -> FC1 -> FC2 -> finalize)."""
    T, H, I, L, out = _layer_args(x, w1, w2, num_experts, top_k, logits, topk_ids, topk_w,
                                  local_offset, out)
    dev = x.device
    need = moe_workspace_size(T, H, I, num_experts, top_k, L)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(library().moe_forward(_ptr(x), _ptr(logits), _ptr(topk_ids), _ptr(topk_w), _ptr(w1), _ptr(w2),
                                 T, H, I, num_experts, top_k, local_offset, L, _ptr(out), _ptr(workspace),
                                 workspace.numel(), _ptr(status), _stream(dev)), "moe_forward")
    return out


class MoEPlan:
    """Prepared launch: validate and lay out once, then ``launch()`` only
    enqueues kernels (no allocation, no host synchronisation; capturable in a
    CUDA graph).  The plan binds the given tensors; write new values into them
    between launches."""

    def __init__(self, x, w1, w2, num_experts: int, top_k: int, logits=None, topk_ids=None, topk_w=None,
                 local_offset: int = 0, out=None, workspace=None, status=None, path: int = PATH_AUTO,
                 stage_timing: bool = False, one_cta_gemm: bool = False, decode_chain: bool | None = None,
                 fused_gather: bool = False, decode_one_launch: bool = False,
                 test_unreachable_wait: bool = False, clamp_limit=None, e4m3=None, no_tail_tiles: bool = False,
                 small_group_kernel: bool | None = None):
        """decode_chain: None lets the library choose the decode form (the
        chain in one launch for few routes, else five kernels), True forces
        the chain as two kernels, False the five separate kernels.
        decode_one_launch: always the chain in one launch.  fused_gather: on the grouped path FC1 copies
        its token rows straight from x instead of a gather kernel.
        test_unreachable_wait: test hook (MOE_PLAN_TEST_UNREACHABLE_WAIT) that
        makes the one-launch decode chain's FC2 waits run out.
        clamp_limit: [L] fp32 device tensor of per-expert SwiGLUStep limits
        (None: plain SwiGLU).
        e4m3: the fp8 per-tensor weight family: w1 / w2 are uint8 E4M3 codes and
        e4m3 = dict(w1_scale=[L] fp32, w2_scale=[L] fp32, x_scale=float,
        h_scale=float).
        small_group_kernel: None lets the library decide whether the groups of
        at most 64 rows run in their own kernel beside the CTA-pair GEMMs, True
        forces it, False keeps every group in the pair kernel."""
        T, H, I, L, out = _layer_args(x, w1, w2, num_experts, top_k, logits, topk_ids, topk_w,
                                      local_offset, out, torch.uint8 if e4m3 is not None else torch.bfloat16)
        dev = x.device
        need = moe_workspace_size(T, H, I, num_experts, top_k, L)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        if status is None:
            status = torch.zeros(1, dtype=torch.int32, device=dev)
        q = dict(weight_format=WEIGHTS_BF16)
        if e4m3 is not None:
            _need(e4m3["w1_scale"], torch.float32, "w1_scale", (L,), dev)
            _need(e4m3["w2_scale"], torch.float32, "w2_scale", (L,), dev)
            q = dict(weight_format=WEIGHTS_E4M3, w1_scale=_ptr(e4m3["w1_scale"]), w2_scale=_ptr(e4m3["w2_scale"]),
                     x_scale=float(e4m3["x_scale"]), h_scale=float(e4m3["h_scale"]))
        if clamp_limit is not None:
            _need(clamp_limit, torch.float32, "clamp_limit", (L,), dev)
        self._keep = (x, w1, w2, logits, topk_ids, topk_w, out, workspace, status, clamp_limit, e4m3)
        self.x, self.w1, self.w2, self.logits, self.topk_ids, self.topk_w = x, w1, w2, logits, topk_ids, topk_w
        self.out, self.workspace, self.status = out, workspace, status
        self.T, self.H, self.I, self.E, self.top_k, self.L = T, H, I, num_experts, top_k, L
        self.device = dev
        d = _Desc(x=_ptr(x), logits=_ptr(logits), topk_ids=_ptr(topk_ids), topk_w=_ptr(topk_w),
                  w1=_ptr(w1), w2=_ptr(w2), out=_ptr(out), workspace=_ptr(workspace),
                  workspace_bytes=workspace.numel(), status=_ptr(status), T=T, H=H, I=I, E=num_experts,
                  top_k=top_k, local_offset=local_offset, num_local=L, path=path,
                  flags=(PLAN_STAGE_TIMING if stage_timing else 0) | (PLAN_ONE_CTA_GEMM if one_cta_gemm else 0)
                  | (PLAN_DECODE_CHAIN if decode_chain is True else 0)
                  | (PLAN_DECODE_SEPARATE if decode_chain is False else 0)
                  | (PLAN_FUSED_GATHER if fused_gather else 0)
                  | (PLAN_DECODE_ONE_LAUNCH if decode_one_launch else 0)
                  | (PLAN_TEST_UNREACHABLE_WAIT if test_unreachable_wait else 0)
                  | (PLAN_NO_TAIL_TILES if no_tail_tiles else 0)
                  | (PLAN_SMALL_GROUP_KERNEL if small_group_kernel is True else 0)
                  | (PLAN_NO_SMALL_GROUP_KERNEL if small_group_kernel is False else 0),
                  clamp_limit=_ptr(clamp_limit), **q)
        handle = ctypes.c_void_p()
        _check(library().moe_forward_prepare(ctypes.byref(d), ctypes.byref(handle)), "moe_forward_prepare")
        self._h = handle

    def launch(self, stream=None):
        s = _stream(self.device) if stream is None else (stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)
        _check(library().moe_plan_launch(self._h, s), "moe_plan_launch")
        return self.out

    def buffers(self) -> dict:
        b = _Buffers()
        _check(library().moe_plan_buffers_get(self._h, ctypes.byref(b)), "moe_plan_buffers_get")
        return {name: getattr(b, name) for name, _ in _Buffers._fields_}

    def stage_names(self):
        lib = library()
        return [lib.moe_plan_stage_name(self._h, i).decode() for i in range(lib.moe_plan_stage_count(self._h))]

    def stage_times(self):
        """(per-stage summed ms, launches counted) since the last reset."""
        names = self.stage_names()
        arr = (ctypes.c_float * len(names))()
        n = ctypes.c_int(0)
        _check(library().moe_plan_stage_times(self._h, arr, len(names), ctypes.byref(n)), "moe_plan_stage_times")
        return dict(zip(names, list(arr))), n.value

    def kernels_per_launch(self) -> int:
        return int(library().moe_plan_kernels_per_launch(self._h))

    def set_wait_limit(self, limit_ns: int):
        """Longest one in-kernel wait of this plan may take (default 4 s)."""
        _check(library().moe_plan_set_wait_limit(self._h, int(limit_ns)), "moe_plan_set_wait_limit")

    def stage_reset(self):
        _check(library().moe_plan_stage_reset(self._h), "moe_plan_stage_reset")

    def close(self):
        if getattr(self, "_h", None):
            library().moe_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
