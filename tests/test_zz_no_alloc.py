"""The allocation-free sort entry point (moe_sort_no_alloc).

Some callers cannot allocate device memory: a plugin whose host framework
hands it only its input and output buffers, or a runtime that plans all device
memory at start-up and forbids allocating later.  moe_sort_no_alloc serves
them by keeping the sort's scratch table in a fixed array inside the library.
These tests call it through the C ABI and check that it gives exactly what
moe_sort (the workspace-taking entry point) gives, and exactly what the CPU
oracle's sort gives, on two calls in a row, so that the shared array carries
nothing over from one call to the next.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import mixture_experts_expert_router_gb300 as moe
import oracle


def _ids(seed, T, k, E, skew):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    if skew:
        ids[rng.random((T, k)) < 0.5] = 3
    return torch.from_numpy(ids)


def _no_alloc_outputs(ids, E, off, L, dev):
    """Call the C entry point with caller-made buffers (nothing allocated inside)."""
    T, k = ids.shape
    R = T * k
    m = torch.full((L + 1,), -9, dtype=torch.int32, device=dev)
    p2e = torch.full((R,), -9, dtype=torch.int32, device=dev)
    e2p = torch.full((R,), -9, dtype=torch.int32, device=dev)
    st = torch.full((1,), 77, dtype=torch.int32, device=dev)
    d_ids = ids.to(dev)
    rc = moe.library().moe_sort_no_alloc(d_ids.data_ptr(), T, k, E, off, L, m.data_ptr(), p2e.data_ptr(),
                                         e2p.data_ptr(), st.data_ptr(), torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0, moe.moe_status_string(rc)
    torch.cuda.synchronize()
    return m.cpu(), p2e.cpu(), e2p.cpu(), st.cpu()


@pytest.mark.gpu
def test_no_alloc_sort_matches_workspace_sort_twice_in_a_row():
    from mixture_experts_expert_router_gb300 import _build
    _build.build()
    dev = torch.device("cuda:0")
    # two different problems back to back, both large enough to use the table
    cases = [(_ids(1, 8192, 8, 256, False), 256, 0, 256),
             (_ids(2, 3000, 6, 64, True), 64, 5, 40)]
    for ids, E, off, L in cases:
        m_w, p2e_w, e2p_w, st_w = moe.moe_sort(ids.to(dev), E, off, L)
        torch.cuda.synchronize()
        m_n, p2e_n, e2p_n, st_n = _no_alloc_outputs(ids, E, off, L, dev)
        M = int(m_w[-1].item())
        assert torch.equal(m_n, m_w.cpu())
        assert torch.equal(p2e_n[:M], p2e_w.cpu()[:M])
        assert torch.equal(e2p_n, e2p_w.cpu())
        assert int(st_n.item()) == int(st_w.item()) == 0
        # and bit-exact against the oracle's stable counting sort
        m_o, p2e_o, e2p_o, st_o = oracle.sort(ids.numpy(), E, off, L)
        assert np.array_equal(m_n.numpy(), m_o)
        assert np.array_equal(p2e_n[:M].numpy(), p2e_o)
        assert np.array_equal(e2p_n.numpy(), e2p_o)
        assert st_o == 0


def test_no_alloc_sort_rejects_problems_beyond_its_table():
    from mixture_experts_expert_router_gb300 import _build
    _build.build()
    lib = moe.library()
    # ceil(2^20 * 16 / 4096) * 1024 = 4 Mi entries > 256 Ki: refused before any device call
    rc = lib.moe_sort_no_alloc(None, 1 << 20, 16, 1024, 0, 1024, None, None, None, None, None)
    assert rc == -4, moe.moe_status_string(rc)
