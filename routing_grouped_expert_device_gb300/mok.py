"""ctypes binding of libmok (include/mok.h).

Argument marshalling only: every function takes torch tensors (or None),
passes their device pointers, sizes and the current CUDA stream to the C ABI,
and raises MokError on any status other than MOK_OK.  There is no fallback:
if libmok.so is missing the import of the library raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Dict, Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmok.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "mok.h")

MOK_OK, MOK_ERR_INVALID_ARG, MOK_ERR_UNSUPPORTED, MOK_ERR_WORKSPACE, MOK_ERR_CUDA, \
    MOK_ERR_TIMEOUT, MOK_ERR_BAD_ROUTE = range(7)
MOK_BF16, MOK_MXFP8 = 0, 1
OP_PLAN, OP_EXPERT_FFN, OP_SHARED_FFN, OP_FWD, OP_BWD, OP_RING = range(6)


class MokError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib_handle().mok_status_string(status).decode() if _LIB is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "D", "I", "E", "K", "I_shared", "dtype", "chunk_rows", "producer_sms", "bwd_shared_sms")]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_gate", "w_up", "w_down", "q_gate", "q_up", "q_down",
                 "sc_gate", "sc_up", "sc_down", "ws_gate", "ws_up", "ws_down",
                 "qt_down", "sct_down", "qt_gu", "sct_gu", "sc_gu_pair")]


class PlanBuf(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_void_p) for n in ("topk_idx", "g", "counts", "offsets", "table", "route_dst", "act")]
                + [("act_rows", ctypes.c_int64), ("act_shared", ctypes.c_void_p)])


_LIB: Optional[ctypes.CDLL] = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

_SIGS = {
    "mok_workspace_bytes": (_SZ, [ctypes.POINTER(Shape), ctypes.c_int]),
    "mok_workspace_offset": (_SZ, [ctypes.POINTER(Shape), ctypes.c_int]),
    "mok_bwd_shared_sms": (ctypes.c_int32, [ctypes.POINTER(Shape)]),
    "mok_route": (ctypes.c_int, [_P, _I32, _I32, _I32, _P, _P, _P]),
    "mok_plan": (ctypes.c_int, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "mok_plan_static": (ctypes.c_int, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "mok_dispatch": (ctypes.c_int, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, _P, _P]),
    "mok_expert_ffn": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(Weights), _P, _P, _P, _P, _P,
                                      _P, _SZ, _P]),
    "mok_expert_upgate": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(Weights), _P, _P, _P, _P, _P, _P, _P,
                                         _P]),
    "mok_expert_upgate_ring": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(Weights), _P, _P, _P, _P, _P,
                                               ctypes.c_size_t, _P]),
    "mok_expert_down": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(Weights), _P, _P, _P, _P, _P, _P, _P]),
    "mok_shared_ffn": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(Weights), _P, _P, _P, _SZ, _P]),
    "mok_combine": (ctypes.c_int, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, _P]),
    "mok_moe_fwd": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(Weights), _P, _P, _P,
                                   ctypes.POINTER(PlanBuf), _P, _SZ, _P]),
    "mok_moe_bwd": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(Weights), _P, _P,
                                   ctypes.POINTER(PlanBuf), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _P, _SZ, _P]),
    "mok_quantize_mxfp8": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P]),
    "mok_quantize_mxfp8_bwd_weights": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(Weights), _P, _P, _P,
                                                      _P, _P]),
    "mok_mxfp8_scale_bytes": (ctypes.c_size_t, [_I64, _I64, ctypes.c_int32]),
    "mok_mxfp8_pair_scales": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(Weights), _P, _P]),
    "mok_check_wait_timeout": (ctypes.c_int, [_P]),
    "mok_router": (ctypes.c_int, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, _P]),
    "mok_plan_ranks_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int32] * 4),
    "mok_plan_ranks": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "mok_get_error": (ctypes.c_int, [_P]),
    "mok_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}


def _lib_handle() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libmok.so not built ({LIB_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def header_symbols():
    """Every entry point declared in include/mok.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(mok_[a-z0-9_]+)\s*\(", text)))


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(status: int, where: str):
    if status != MOK_OK:
        raise MokError(status, where)


def make_shape(T, D, I, E, K, I_shared=0, dtype=MOK_BF16, chunk_rows=0, producer_sms=0, bwd_shared_sms=0) -> Shape:
    return Shape(T, D, I, E, K, I_shared, dtype, chunk_rows, producer_sms, bwd_shared_sms)


def shape_of(cfg, dtype=None, chunk_rows=0, producer_sms=0, bwd_shared_sms=0) -> Shape:
    dt = MOK_MXFP8 if (dtype or cfg.dtype) == "mxfp8" else MOK_BF16
    return make_shape(cfg.T, cfg.D, cfg.I, cfg.E, cfg.K, cfg.I_shared, dt, chunk_rows, producer_sms, bwd_shared_sms)


def make_weights(t: Dict[str, object]) -> Weights:
    w = Weights()
    for name in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down",
                 "q_gate", "q_up", "q_down", "sc_gate", "sc_up", "sc_down",
                 "qt_down", "sct_down", "qt_gu", "sct_gu", "sc_gu_pair"):
        if t.get(name) is not None:
            setattr(w, name, _ptr(t[name]))
    return w


def make_plan_buf(t: Dict[str, object]) -> PlanBuf:
    """The forward's saved state; optional "act" (fp32 [rows][2I]) keeps h, u
    of the experts whose rows lie below its row count for the backward, and
    optional "act_shared" (fp32 [T][2 I_shared]) the shared expert's."""
    act = t.get("act")
    rows = int(act.shape[0]) if act is not None else 0
    return PlanBuf(*(_ptr(t[n]) for n in ("topk_idx", "g", "counts", "offsets", "table", "route_dst")),
                   _ptr(act), rows, _ptr(t.get("act_shared")))


def workspace_bytes(shape: Shape, op: int) -> int:
    return int(_lib_handle().mok_workspace_bytes(ctypes.byref(shape), op))


WS_BWD_DH, WS_BWD_DU, WS_BWD_AG = 1, 2, 3


def bwd_shared_sms(shape: Shape) -> int:
    """SMs mok_moe_bwd gives the shared expert's backward on its side stream (0: none)."""
    n = int(_lib_handle().mok_bwd_shared_sms(ctypes.byref(shape)))
    if n < 0:
        raise ValueError("invalid shape")
    return n


def workspace_offset(shape: Shape, region: int) -> int:
    """Byte offset of a backward intermediate (WS_BWD_*) in the MOK_OP_BWD workspace."""
    off = int(_lib_handle().mok_workspace_offset(ctypes.byref(shape), region))
    if off == ctypes.c_size_t(-1).value:
        raise ValueError("invalid shape or region")
    return off


def route(s, K, topk_idx, g, stream=None):
    T, E = s.shape
    _check(_lib_handle().mok_route(_ptr(s), T, E, K, _ptr(topk_idx), _ptr(g), _stream(stream)), "mok_route")


def plan(topk_idx, E, counts, offsets, table, route_dst, ws, stream=None):
    T, K = topk_idx.shape
    _check(_lib_handle().mok_plan(_ptr(topk_idx), T, E, K, _ptr(counts), _ptr(offsets), _ptr(table),
                                  _ptr(route_dst), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)), "mok_plan")


def plan_static(topk_idx, E, counts, offsets, table, route_dst, stream=None):
    """mok_plan with the library's own fixed scratch (no workspace argument)."""
    T, K = topk_idx.shape
    _check(_lib_handle().mok_plan_static(_ptr(topk_idx), T, E, K, _ptr(counts), _ptr(offsets), _ptr(table),
                                         _ptr(route_dst), _stream(stream)), "mok_plan_static")


def dispatch(shape: Shape, x, table, route_dst, xg, xg_scale=None, offsets=None, stream=None):
    """Rows of x to expert order (each token read once, stored at its
    route_dst positions); for MXFP8 also quantise, which needs the plan's
    table and offsets."""
    _check(_lib_handle().mok_dispatch(ctypes.byref(shape), _ptr(x), _ptr(table), _ptr(route_dst), _ptr(offsets),
                                      _ptr(xg), _ptr(xg_scale), _stream(stream)), "mok_dispatch")


def expert_ffn(shape: Shape, weights: Weights, xg, offsets, yg, a_out=None, ws=None, xg_scale=None, stream=None):
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(_lib_handle().mok_expert_ffn(ctypes.byref(shape), ctypes.byref(weights), _ptr(xg), _ptr(xg_scale),
                                        _ptr(offsets), _ptr(a_out), _ptr(yg), _ptr(ws), nbytes,
                                        _stream(stream)), "mok_expert_ffn")


def expert_upgate(shape: Shape, weights: Weights, xg, offsets, a, xg_scale=None, a_scale=None,
                  x_shared=None, a_shared=None, stream=None):
    """Grouped up/gate + SwiGLU; with x_shared / a_shared the shared expert's
    up/gate runs in the same launch."""
    _check(_lib_handle().mok_expert_upgate(ctypes.byref(shape), ctypes.byref(weights), _ptr(xg), _ptr(xg_scale),
                                           _ptr(offsets), _ptr(a), _ptr(a_scale), _ptr(x_shared), _ptr(a_shared),
                                           _stream(stream)), "mok_expert_upgate")


def expert_upgate_ring(shape: Shape, weights: Weights, x, table, offsets, a, ws, stream=None):
    """Up/gate with the dispatch fused in as a ring of shape.chunk_rows-row chunks."""
    _check(_lib_handle().mok_expert_upgate_ring(ctypes.byref(shape), ctypes.byref(weights), _ptr(x), _ptr(table),
                                                _ptr(offsets), _ptr(a), _ptr(ws), ws.numel() * ws.element_size(),
                                                _stream(stream)), "mok_expert_upgate_ring")


def expert_down(shape: Shape, weights: Weights, a, offsets, yg, a_scale=None, a_shared=None, ys=None, stream=None):
    """Grouped down projection; with a_shared / ys the shared expert's down
    projection runs in the same launch."""
    _check(_lib_handle().mok_expert_down(ctypes.byref(shape), ctypes.byref(weights), _ptr(a), _ptr(a_scale),
                                         _ptr(offsets), _ptr(yg), _ptr(a_shared), _ptr(ys), _stream(stream)),
           "mok_expert_down")


def shared_ffn(shape: Shape, weights: Weights, x, ys, ws, stream=None):
    _check(_lib_handle().mok_shared_ffn(ctypes.byref(shape), ctypes.byref(weights), _ptr(x), _ptr(ys), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(stream)), "mok_shared_ffn")


def combine(shape: Shape, yg, ys, g, route_dst, out, stream=None):
    _check(_lib_handle().mok_combine(ctypes.byref(shape), _ptr(yg), _ptr(ys), _ptr(g), _ptr(route_dst),
                                     _ptr(out), _stream(stream)), "mok_combine")


def moe_fwd(shape: Shape, weights: Weights, x, s, out, ws, saved: Optional[PlanBuf] = None, stream=None):
    _check(_lib_handle().mok_moe_fwd(ctypes.byref(shape), ctypes.byref(weights), _ptr(x), _ptr(s), _ptr(out),
                                     ctypes.byref(saved) if saved is not None else None, _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)), "mok_moe_fwd")


def moe_bwd(shape: Shape, weights: Weights, x, s, saved: PlanBuf, dy, dx, dw_gate, dw_up, dw_down,
            dws_gate, dws_up, dws_down, ds, dg, ws, stream=None):
    _check(_lib_handle().mok_moe_bwd(ctypes.byref(shape), ctypes.byref(weights), _ptr(x), _ptr(s),
                                     ctypes.byref(saved), _ptr(dy), _ptr(dx), _ptr(dw_gate), _ptr(dw_up),
                                     _ptr(dw_down), _ptr(dws_gate), _ptr(dws_up), _ptr(dws_down), _ptr(ds),
                                     _ptr(dg), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "mok_moe_bwd")


def quantize_mxfp8(src, q, scale, stream=None):
    rows, cols = src.shape
    _check(_lib_handle().mok_quantize_mxfp8(_ptr(src), rows, cols, _ptr(q), _ptr(scale), _stream(stream)),
           "mok_quantize_mxfp8")


def quantize_mxfp8_bwd_weights(shape: Shape, weights: Weights, qt_down, sct_down, qt_gu, sct_gu, stream=None):
    """The backward's MXFP8 weight copies (W_down^T along D; [W_gate^T | W_up^T]
    along 2I) from the bf16 weights in `weights`."""
    _check(_lib_handle().mok_quantize_mxfp8_bwd_weights(ctypes.byref(shape), ctypes.byref(weights), _ptr(qt_down),
                                                        _ptr(sct_down), _ptr(qt_gu), _ptr(sct_gu),
                                                        _stream(stream)), "mok_quantize_mxfp8_bwd_weights")


def mxfp8_pair_scales(shape: Shape, weights: Weights, sc_gu_pair, stream=None):
    """The paired W_up / W_gate scale blocks of the MXFP8 up/gate with the
    routed rows as N (mok_mxfp8_pair_scales), from weights' sc_gate, sc_up."""
    _check(_lib_handle().mok_mxfp8_pair_scales(ctypes.byref(shape), ctypes.byref(weights), _ptr(sc_gu_pair),
                                               _stream(stream)), "mok_mxfp8_pair_scales")


def mx_scale_words(rows: int, cols: int, groups: int = 0) -> int:
    """32-bit scale words of a [rows][cols] MXFP8 tensor: plain layout
    (groups = 0) or grouped over `groups` experts (mok_mxfp8_scale_bytes)."""
    n = int(_lib_handle().mok_mxfp8_scale_bytes(rows, cols, groups))
    if n == 0 and rows > 0:
        raise MokError(MOK_ERR_INVALID_ARG, f"mok_mxfp8_scale_bytes({rows}, {cols}, {groups})")
    return n // 4


def plan_ranks(topk_idx, E: int, ranks: int, counts, offsets, table, route_dst, ws, stream=None):
    """mok_plan with `ranks` virtual source ranks (round-robin order within each expert)."""
    T, K = topk_idx.shape
    _check(_lib_handle().mok_plan_ranks(_ptr(topk_idx), T, E, K, ranks, _ptr(counts), _ptr(offsets), _ptr(table),
                                        _ptr(route_dst), _ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(stream)), "mok_plan_ranks")


def plan_ranks_workspace_bytes(T: int, E: int, K: int, ranks: int) -> int:
    return int(_lib_handle().mok_plan_ranks_workspace_bytes(T, E, K, ranks))


def router(shape: Shape, x, w_router, s, topk_idx, g, stream=None):
    """s = softmax(x W_r^T), then top-K and g on it."""
    _check(_lib_handle().mok_router(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(s), _ptr(topk_idx), _ptr(g),
                                    _stream(stream)), "mok_router")


def check_wait_timeout(stream=None):
    """Enqueue the bounded-wait check (two waits that run out); read the
    result with get_error()."""
    _check(_lib_handle().mok_check_wait_timeout(_stream(stream)), "mok_check_wait_timeout")


def get_error(stream=None) -> int:
    return int(_lib_handle().mok_get_error(_stream(stream)))


def check_device_status(stream=None):
    st = get_error(stream)
    _check(st, "device status")


def status_string(status: int) -> str:
    return _lib_handle().mok_status_string(status).decode()
