"""Host-side checks of libmok.so: it builds for sm_103a, loads without a GPU,
exports every entry point include/mok.h declares, and rejects bad arguments
before touching the device."""
import ctypes

import pytest

from helpers import mok


@pytest.fixture(scope="module")
def m():
    return mok()


def test_exports_every_header_symbol(m):
    lib = ctypes.CDLL(m.LIB_PATH)
    syms = m.header_symbols()
    assert len(syms) >= 12
    for name in syms:
        assert hasattr(lib, name), name


def test_status_strings(m):
    for st in range(7):
        assert m.status_string(st)


def test_workspace_bytes_host_only(m):
    good = m.make_shape(T=7168, D=7168, I=2048, E=256, K=8, I_shared=2048)
    fwd = m.workspace_bytes(good, m.OP_FWD)
    R = 7168 * 8
    assert fwd >= R * 7168 * 2 * 2 + R * 2048 * 2
    assert m.workspace_bytes(good, m.OP_PLAN) > 0
    # the ring: 4 chunks of 2048 rows (+ 128 mirrored rows) and 2 counters per chunk
    assert m.workspace_bytes(good, m.OP_RING) >= (4 * 2048 + 128) * 7168 * 2 + 2 * 28 * 4
    ring = m.make_shape(T=7168, D=7168, I=2048, E=256, K=8, I_shared=2048, chunk_rows=512)
    assert m.workspace_bytes(ring, m.OP_FWD) < fwd  # the ring replaces the R x D gathered copy
    assert m.workspace_bytes(m.make_shape(T=16, D=256, I=128, E=8, K=2, chunk_rows=100), m.OP_RING) == 0
    # chunk_rows 0 chooses the ring (b = 2048) for 512 or more routed rows per
    # expert: no R x D copy, as chunk_rows 2048; -1 keeps the whole-batch copy
    skew = dict(T=16384, D=4096, I=1536, E=128, K=8)
    auto = m.workspace_bytes(m.make_shape(**skew), m.OP_FWD)
    assert auto == m.workspace_bytes(m.make_shape(**skew, chunk_rows=2048), m.OP_FWD)
    whole = m.workspace_bytes(m.make_shape(**skew, chunk_rows=-1), m.OP_FWD)
    assert whole - auto > 16384 * 8 * 4096 * 2 // 2
    assert m.workspace_bytes(m.make_shape(**skew, chunk_rows=-2), m.OP_FWD) == 0
    assert m.workspace_bytes(m.make_shape(T=16, D=200, I=128, E=8, K=2), m.OP_FWD) == 0
    assert m.workspace_bytes(m.make_shape(T=16, D=256, I=128, E=8, K=9), m.OP_FWD) == 0


def test_bad_arguments_rejected_on_host(m):
    lib = m._lib_handle()
    assert lib.mok_route(None, 16, 8, 9, None, None, None) == m.MOK_ERR_INVALID_ARG
    assert lib.mok_route(None, 16, 8, 2, None, None, None) == m.MOK_ERR_INVALID_ARG
    assert lib.mok_plan(None, 16, 8, 2, None, None, None, None, None, 0, None) == m.MOK_ERR_INVALID_ARG
    sh = m.make_shape(T=16, D=256, I=128, E=8, K=2)
    assert lib.mok_moe_fwd(ctypes.byref(sh), ctypes.byref(m.Weights()), None, None, None, None, None, 0,
                           None) == m.MOK_ERR_INVALID_ARG
    assert lib.mok_quantize_mxfp8(None, 4, 33, None, None, None) == m.MOK_ERR_INVALID_ARG


def test_mxfp8_scale_bytes(m):
    lib = m._lib_handle()
    # plain layout: rows rounded up to 128, one word per row and 128 columns
    assert lib.mok_mxfp8_scale_bytes(301, 512, 0) == 4 * 384 * 4
    assert lib.mok_mxfp8_scale_bytes(128, 128, 0) == 128 * 4
    assert lib.mok_mxfp8_scale_bytes(0, 128, 0) == 0
    # grouped layout: room for every expert to start a new 128-row block
    R, D, E = 7168 * 8, 7168, 256
    assert lib.mok_mxfp8_scale_bytes(R, D, E) == (D // 128) * 128 * (R // 128 + E) * 4
    assert lib.mok_mxfp8_scale_bytes(301, 256, 5) == 2 * 128 * (3 + 5) * 4
    for bad in ((10, 100, 0), (-1, 128, 0), (10, 128, -1), (10, 0, 0)):
        assert lib.mok_mxfp8_scale_bytes(*bad) == 0
    assert m.mx_scale_words(301, 512) == 4 * 384


def test_dispatch_argument_checks(m):
    lib = m._lib_handle()
    sh = m.make_shape(T=16, D=256, I=128, E=8, K=2, dtype=m.MOK_MXFP8)
    fake = ctypes.c_void_p(256)  # never dereferenced: each call is rejected first
    # MXFP8 needs offsets, the table and the scale output
    assert lib.mok_dispatch(ctypes.byref(sh), fake, fake, fake, None, fake, fake, None) == m.MOK_ERR_INVALID_ARG
    assert lib.mok_dispatch(ctypes.byref(sh), fake, None, fake, fake, fake, fake, None) == m.MOK_ERR_INVALID_ARG
    assert lib.mok_dispatch(ctypes.byref(sh), fake, fake, fake, fake, fake, None, None) == m.MOK_ERR_INVALID_ARG
    # every dtype needs route_dst
    sb = m.make_shape(T=16, D=256, I=128, E=8, K=2)
    assert lib.mok_dispatch(ctypes.byref(sb), fake, fake, None, fake, fake, None, None) == m.MOK_ERR_INVALID_ARG


def test_plan_ranks_host_checks(m):
    lib = m._lib_handle()
    assert m.plan_ranks_workspace_bytes(256, 8, 2, 4) > m.plan_ranks_workspace_bytes(256, 8, 2, 1)
    assert m.plan_ranks_workspace_bytes(250, 8, 2, 4) == 0  # ranks must divide T
    assert lib.mok_plan_ranks(None, 250, 8, 2, 4, None, None, None, None, None, 0, None) == m.MOK_ERR_INVALID_ARG
    assert lib.mok_plan_ranks(None, 256, 8, 2, 0, None, None, None, None, None, 0, None) == m.MOK_ERR_INVALID_ARG


def test_mxfp8_backward_argument_checks(m):
    lib = m._lib_handle()
    fake = ctypes.c_void_p(256)  # never dereferenced: each call is rejected first
    names = ("w_gate", "w_up", "w_down", "q_gate", "q_up", "q_down", "sc_gate", "sc_up", "sc_down",
             "qt_down", "sct_down", "qt_gu", "sct_gu")
    w = m.Weights(**{n: 256 for n in names})
    pb = m.PlanBuf(*([256] * 6))
    args = lambda sh, ww: (ctypes.byref(sh), ctypes.byref(ww), fake, fake, ctypes.byref(pb), fake, fake, fake,
                           fake, fake, fake, fake, fake, fake, fake, fake, 0, None)
    # the t and dX products run on 256-column tiles: I = 128 is unsupported
    sh = m.make_shape(T=16, D=256, I=128, E=8, K=2, dtype=m.MOK_MXFP8)
    assert lib.mok_moe_bwd(*args(sh, w)) == m.MOK_ERR_UNSUPPORTED
    # the backward's weight copies are required
    sh = m.make_shape(T=16, D=256, I=256, E=8, K=2, dtype=m.MOK_MXFP8)
    w2 = m.Weights(**{n: 256 for n in names[:9]})
    assert lib.mok_moe_bwd(*args(sh, w2)) == m.MOK_ERR_INVALID_ARG
    # the weight-copy quantiser wants D and I multiples of 128
    bad = m.make_shape(T=16, D=192, I=256, E=8, K=2)
    assert lib.mok_quantize_mxfp8_bwd_weights(ctypes.byref(bad), ctypes.byref(w), fake, fake, fake, fake,
                                              None) == m.MOK_ERR_INVALID_ARG
