"""Shared test plumbing: library loading, host copies, tolerances."""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

BF16_TOL = 2e-2   # |gpu - oracle| <= BF16_TOL * max(1, |oracle|)
MXFP8_TOL = 6e-2


def mok():
    """The binding, with libmok.so built first if it is missing."""
    from routing_grouped_expert_device_gb300 import build, mok as m
    if not os.path.exists(m.LIB_PATH):
        build.build()
    m._lib_handle()
    return m


def host(inp):
    """Host numpy copies: bf16 -> uint16 bits, fp32 -> float32."""
    import torch
    from routing_grouped_expert_device_gb300 import workloads as W
    out = {}
    for k, v in inp.items():
        if v is None:
            continue
        out[k] = W.bf16_bits(v) if v.dtype == torch.bfloat16 else W.f32_host(v)
    return out


def bf16_tensor_to_f32(t):
    return t.float().cpu().numpy()


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.abs(got - ref) / np.maximum(1.0, np.abs(ref))


def assert_close(got, ref, tol=BF16_TOL, what="", slack=None):
    """|got - ref| <= tol * max(1, |ref|) (+ slack: the oracle's bound for
    bf16 rounding decisions that fp32 summation order does not fix)."""
    got64 = np.asarray(got, dtype=np.float64)
    ref64 = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got64)), f"{what}: non-finite values"
    if slack is not None:
        excess = np.abs(got64 - ref64) - np.asarray(slack, dtype=np.float64)
        e = np.maximum(excess, 0.0) / np.maximum(1.0, np.abs(ref64))
    else:
        e = rel_err(got, ref)
    if e.max() > tol:
        idx = np.unravel_index(np.argmax(e), e.shape)
        raise AssertionError(f"{what}: max err {e.max():.3e} at {idx}: got {np.asarray(got)[idx]} "
                             f"want {np.asarray(ref)[idx]}; {np.mean(e > tol) * 100:.3f}% over tol")


def alloc_plan(cfg, dev):
    import torch
    R = cfg.T * cfg.K
    return dict(topk_idx=torch.empty(cfg.T, cfg.K, dtype=torch.int32, device=dev),
                g=torch.empty(cfg.T, cfg.K, dtype=torch.float32, device=dev),
                counts=torch.empty(cfg.E, dtype=torch.int32, device=dev),
                offsets=torch.empty(cfg.E + 1, dtype=torch.int32, device=dev),
                table=torch.empty(max(R, 1), 3, dtype=torch.int32, device=dev),
                route_dst=torch.empty(max(R, 1), dtype=torch.int32, device=dev))


def device_weights_fetch(d):
    """Per-expert host copies of device weights, for the sampled oracle."""
    from routing_grouped_expert_device_gb300 import workloads as W
    import oracle as O

    def fetch(e):
        return W.bf16_bits(d["w_gate"][e]), W.bf16_bits(d["w_up"][e]), W.bf16_bits(d["w_down"][e])

    sh = None
    if d.get("ws_gate") is not None:
        sh = (W.bf16_bits(d["ws_gate"]), W.bf16_bits(d["ws_up"]), W.bf16_bits(d["ws_down"]))
    return O.HostWeights(fetch, sh)
