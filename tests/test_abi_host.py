"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/moe_gb300.h declares, and rejects bad arguments with
the documented codes before touching the device."""
import ctypes
import os
import re

import pytest

import mixture_experts_expert_router_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_expert_router_gb300 import _build
    _build.build()
    return moe.library()


def header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^MOE_API\s+[^;(]*?\b([A-Za-z_][A-Za-z0-9_]*)\s*\(", text, re.M)))


def test_header_lists_functions():
    names = header_functions()
    assert "moe_forward" in names and "grouped_gemm_fwd" in names and len(names) >= 20
    assert sorted(moe.ABI_SYMBOLS) == names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    raw = ctypes.CDLL(moe.library_path())
    for name in header_functions():
        getattr(raw, name)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, -9):
        s = moe.moe_status_string(code)
        assert s and s != "unknown status code"
    assert moe.moe_status_string(-99) == "unknown status code"
    assert lib.moe_abi_version() == 104


def test_argument_errors_before_device(lib):
    # shape errors are reported before any CUDA call
    assert lib.moe_route(None, 4, 8, 9, None, None, None) == -2          # top_k > E
    assert lib.moe_route(None, 4, 8, 17, None, None, None) == -2         # top_k > 16
    assert lib.moe_route(None, 0, 8, 2, None, None, None) == 0           # T == 0: no-op
    assert lib.moe_route(None, 3, 8, 2, None, None, None) == -1          # null pointers
    assert lib.moe_sort(None, 4, 2, 8, 6, 4, None, None, None, None, 0, None, None) == -2  # shard past E
    assert lib.grouped_gemm_fwd(None, None, None, 16, 4, 100, 64, None, None) == -2      # N % 64
    assert lib.grouped_gemm_fwd(None, None, None, 0, 4, 128, 64, None, None) == 0        # empty
    # the claim counters of the small-group kernel: 16-byte aligned, checked before the device
    assert lib.grouped_gemm_fwd_ex(None, None, None, 16, 4, 100, 64, None, 0, None, None) == -2  # N % 64
    assert lib.grouped_gemm_fwd_ex(None, None, None, 0, 4, 256, 64, None, 0, None, None) == 0   # empty
    assert lib.grouped_gemm_fwd_ex(256, 256, 256, 16, 4, 256, 64, 256, 0, 8, None) == -3     # counters
    assert lib.moe_fc1_swiglu(None, None, None, 8, 96, 64, 2, None, None) == -2          # H % 64
    assert lib.moe_finalize(None, None, None, 4, 2, 12, None, None) == -2                # H % 8


def test_workspace_size_and_prepare_errors(lib):
    assert moe.moe_workspace_size(16, 128, 128, 4, 2) > 0
    assert moe.moe_workspace_size(16, 100, 128, 4, 2) == 0      # H % 64 != 0
    # more rows need more workspace
    assert moe.moe_workspace_size(64, 128, 128, 4, 2) > moe.moe_workspace_size(16, 128, 128, 4, 2)
    h = ctypes.c_void_p()
    d0 = moe._Desc(T=0, H=128, I=128, E=4, top_k=2, local_offset=0, num_local=4)
    assert lib.moe_forward_prepare(ctypes.byref(d0), ctypes.byref(h)) == 0   # T == 0: empty plan
    assert lib.moe_plan_kernels_per_launch(h) == 0
    # the bounded-wait limit is range-checked on the host
    assert lib.moe_plan_set_wait_limit(h, moe.WAIT_LIMIT_MIN_NS - 1) == -2
    assert lib.moe_plan_set_wait_limit(h, moe.WAIT_LIMIT_MAX_NS + 1) == -2
    assert lib.moe_plan_set_wait_limit(h, 2_000_000) == 0
    assert lib.moe_plan_set_wait_limit(None, 2_000_000) == -1
    assert lib.moe_plan_destroy(h) == 0
    d = moe._Desc(T=4, H=128, I=128, E=4, top_k=2, local_offset=0, num_local=4)
    assert lib.moe_forward_prepare(ctypes.byref(d), ctypes.byref(h)) == -5   # no routing input
    d.logits = 16
    d.topk_ids = 16
    d.topk_w = 16
    assert lib.moe_forward_prepare(ctypes.byref(d), ctypes.byref(h)) == -5   # both modes
    d.topk_ids = None
    d.topk_w = None
    assert lib.moe_forward_prepare(ctypes.byref(d), ctypes.byref(h)) == -1   # null tensors
    d.x = d.w1 = d.w2 = d.out = 256
    d.workspace = None
    assert lib.moe_forward_prepare(ctypes.byref(d), ctypes.byref(h)) == -4   # no workspace
    d.x = 8
    assert lib.moe_forward_prepare(ctypes.byref(d), ctypes.byref(h)) == -3   # misaligned
    d.top_k = 5
    assert lib.moe_forward_prepare(ctypes.byref(d), ctypes.byref(h)) == -2   # top_k > E
    assert lib.moe_plan_launch(None, None) == -1
    assert lib.moe_plan_destroy(None) == 0


def test_binding_constants_match_header():
    """The Python binding's path, plan-flag and device-status constants carry
    the values include/moe_gb300.h defines."""
    text = open(HEADER).read()
    defines = {m.group(1): int(m.group(2)) for m in re.finditer(r"^#define\s+(MOE_\w+)\s+(-?\d+)", text, re.M)}
    pairs = {"MOE_PATH_AUTO": moe.PATH_AUTO, "MOE_PATH_GROUPED": moe.PATH_GROUPED,
             "MOE_PATH_DECODE": moe.PATH_DECODE, "MOE_PLAN_STAGE_TIMING": moe.PLAN_STAGE_TIMING,
             "MOE_PLAN_ONE_CTA_GEMM": moe.PLAN_ONE_CTA_GEMM, "MOE_PLAN_DECODE_CHAIN": moe.PLAN_DECODE_CHAIN,
             "MOE_PLAN_DECODE_SEPARATE": moe.PLAN_DECODE_SEPARATE, "MOE_PLAN_FUSED_GATHER": moe.PLAN_FUSED_GATHER,
             "MOE_PLAN_DECODE_ONE_LAUNCH": moe.PLAN_DECODE_ONE_LAUNCH,
             "MOE_PLAN_TEST_UNREACHABLE_WAIT": moe.PLAN_TEST_UNREACHABLE_WAIT,
             "MOE_PLAN_NO_TAIL_TILES": moe.PLAN_NO_TAIL_TILES,
             "MOE_PLAN_NO_SMALL_GROUP_KERNEL": moe.PLAN_NO_SMALL_GROUP_KERNEL,
             "MOE_PLAN_SMALL_GROUP_KERNEL": moe.PLAN_SMALL_GROUP_KERNEL,
             "MOE_GROUPED_GEMM_COUNTERS": moe.GROUPED_GEMM_COUNTERS,
             "MOE_WEIGHTS_BF16": moe.WEIGHTS_BF16, "MOE_WEIGHTS_E4M3": moe.WEIGHTS_E4M3,
             "MOE_WAIT_LIMIT_MIN_NS": moe.WAIT_LIMIT_MIN_NS, "MOE_WAIT_LIMIT_MAX_NS": moe.WAIT_LIMIT_MAX_NS,
             "MOE_DEV_BAD_EXPERT": moe.DEV_BAD_EXPERT, "MOE_DEV_TIMEOUT": moe.DEV_TIMEOUT}
    for name, value in pairs.items():
        assert defines.get(name) == value, name
    plan_flags = {k: v for k, v in defines.items() if k.startswith("MOE_PLAN_")}
    assert "MOE_WEIGHTS_E4M3" not in plan_flags
    assert len(set(plan_flags.values())) == len(plan_flags)  # distinct bits
    assert all(v & (v - 1) == 0 for v in plan_flags.values())
