"""mok_plan_static: the plan for callers that cannot provide device scratch.

Such callers (device memory owned by another allocator, or code paths that
must not allocate) get the plan's histogram scratch from a fixed array inside
libmok.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a
fresh process.  Each case calls the new entry point twice in a row through
the C ABI, on different inputs, and requires the same bytes as mok_plan
(plan outputs are integers: bit-exact); further cases sit exactly at the
array's size limit and at zero tokens.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import mok

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _topk(T, E, K, seed, skew=0.0):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g) - skew * torch.log(torch.arange(1, E + 1, dtype=torch.float32))
    return torch.topk(logits, K, dim=1).indices.to(torch.int32).to(DEV)


def _outputs(T, E, K):
    R = T * K
    return (torch.full((E,), -7, dtype=torch.int32, device=DEV),
            torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
            torch.full((R, 3), -7, dtype=torch.int32, device=DEV),
            torch.full((R,), -7, dtype=torch.int32, device=DEV))


def _plan_with_ws(m, topk, E):
    T, K = topk.shape
    outs = _outputs(T, E, K)
    shape = m.make_shape(T=T, D=256, I=128, E=E, K=K)
    ws = torch.empty(m.workspace_bytes(shape, m.OP_PLAN), dtype=torch.uint8, device=DEV)
    m.plan(topk, E, *outs, ws)
    return outs


def _plan_static_cabi(m, topk, E):
    """Direct C-ABI call of mok_plan_static."""
    T, K = topk.shape
    counts, offsets, table, route_dst = _outputs(T, E, K)
    lib = m._lib_handle()
    st = lib.mok_plan_static(ctypes.c_void_p(topk.data_ptr()), T, E, K, ctypes.c_void_p(counts.data_ptr()),
                             ctypes.c_void_p(offsets.data_ptr()), ctypes.c_void_p(table.data_ptr()),
                             ctypes.c_void_p(route_dst.data_ptr()),
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == m.MOK_OK, m.status_string(st)
    return counts, offsets, table, route_dst


@pytest.mark.parametrize("first,second", [((7168, 256, 8, 0.0), (700, 16, 4, 2.0)),
                                          ((16384, 128, 8, 2.0), (256, 8, 2, 0.0))])
def test_plan_static_matches_plan_twice(first, second):
    m = mok()
    for i, (T, E, K, skew) in enumerate((first, second)):
        topk = _topk(T, E, K, seed=10 + i, skew=skew)
        want = _plan_with_ws(m, topk, E)
        got = _plan_static_cabi(m, topk, E)
        torch.cuda.synchronize()
        assert m.get_error() == m.MOK_OK
        for w, g in zip(want, got):
            assert torch.equal(w, g)
        counts = got[0].cpu().numpy()
        assert counts.sum() == T * K and np.all(counts >= 0)


def test_plan_static_rejects_oversize():
    m = mok()
    lib = m._lib_handle()
    # ceil(R / 1024) * E = 300 * 1024 > 262144: refused before any launch
    st = lib.mok_plan_static(None, 300 * 1024 // 8, 1024, 8, None, None, None, None, None)
    assert st == m.MOK_ERR_WORKSPACE


def test_plan_static_at_the_exact_limit():
    """ceil(T*K / 1024) * E == 262144 (E 256, T*K = 1,048,576) is accepted and
    gives mok_plan's bytes; one more route is refused."""
    m = mok()
    T, E, K = 131072, 256, 8
    topk = _topk(T, E, K, seed=21)
    want = _plan_with_ws(m, topk, E)
    got = _plan_static_cabi(m, topk, E)
    torch.cuda.synchronize()
    assert m.get_error() == m.MOK_OK
    for w, g in zip(want, got):
        assert torch.equal(w, g)
    lib = m._lib_handle()
    st = lib.mok_plan_static(None, T + 1, E, K, None, None, None, None, None)
    assert st == m.MOK_ERR_WORKSPACE


def test_plan_static_zero_tokens():
    """T = 0: every count and offset is zero and nothing else is written."""
    m = mok()
    E, K = 64, 4
    counts, offsets, table, route_dst = _outputs(0, E, K)
    lib = m._lib_handle()
    for _ in range(2):
        counts.fill_(-7)
        offsets.fill_(-7)
        st = lib.mok_plan_static(None, 0, E, K, ctypes.c_void_p(counts.data_ptr()),
                                 ctypes.c_void_p(offsets.data_ptr()), None, None,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == m.MOK_OK, m.status_string(st)
        torch.cuda.synchronize()
        assert m.get_error() == m.MOK_OK
        assert torch.all(counts == 0) and torch.all(offsets == 0)
