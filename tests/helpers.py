"""Shared test plumbing: library loading, host copies, tolerances."""
from __future__ import annotations

import os
import re
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


# Largest |got - ref| / (tol * max(1, |ref|)) seen by each named check of
# this process (conftest prints the table when MOK_PARITY_REPORT is set).
PARITY_RATIOS = {}


def assert_close(got, ref, tol=BF16_TOL, what=""):
    """|got - ref| <= tol * max(1, |ref|) for every element."""
    got64 = np.asarray(got, dtype=np.float64)
    ref64 = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got64)), f"{what}: non-finite values"
    e = rel_err(got, ref)
    worst = float(e.max()) if e.size else 0.0
    key = re.sub(r"(expert|row) \d+", r"\1", what).strip()
    PARITY_RATIOS[key] = max(PARITY_RATIOS.get(key, 0.0), worst / tol)
    if worst > tol:
        idx = np.unravel_index(np.argmax(e), e.shape)
        raise AssertionError(f"{what}: max err {worst:.3e} at {idx}: got {np.asarray(got)[idx]} "
                             f"want {np.asarray(ref)[idx]}; {np.mean(e > tol) * 100:.3f}% over tol")


# Elements of one weight-gradient check that may need an admissible
# alternative.  A weight gradient sums its bf16 dh / du / a_g operands over
# an expert's rows (the shared expert: all T tokens, g = 1); at the flip rate
# the intermediates test measures (about 1 % of the points the arithmetic
# leaves open), a sum over 4096 rows collects tens of flips and ~0.6 % of
# the elements land beyond the bare tolerance.  On the grid inputs (exact
# products) every output is held to the bare tolerance instead.
RANGED_MAX_FRAC = 1e-2


def assert_close_ranged(got, ref, shift, tol=BF16_TOL, what=""):
    """A weight gradient, element by element: |got - ref| <= tol * max(1, |ref|),
    except that an element may instead be within that tolerance of the
    oracle's admissible range [ref + lo_shift, ref + hi_shift] (shift, from
    oracle.sum_range: the dh / du / a_g points whose bf16 rounding the
    arithmetic does not fix, rounded the other way).  At most
    RANGED_MAX_FRAC of the elements (and at least one) may need it; the
    count is recorded with the plain ratio."""
    got64 = np.asarray(got, dtype=np.float64)
    ref64 = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got64)), f"{what}: non-finite values"
    scale = tol * np.maximum(1.0, np.abs(ref64))
    plain = np.abs(got64 - ref64) / scale
    over = plain > 1.0
    key = re.sub(r"(expert|row) \d+", r"\1", what).strip()
    PARITY_RATIOS[key] = max(PARITY_RATIOS.get(key, 0.0), float(plain.max()) if plain.size else 0.0)
    if not over.any():
        return
    lo = ref64 + np.asarray(shift[0], dtype=np.float64)
    hi = ref64 + np.asarray(shift[1], dtype=np.float64)
    dist = np.maximum(np.maximum(lo - got64, got64 - hi), 0.0) / scale
    n = int(over.sum())
    PARITY_RATIOS[key + " (elements on an admissible alternative)"] = (
        PARITY_RATIOS.get(key + " (elements on an admissible alternative)", 0) + n)
    worst = float(dist[over].max())
    if worst > 1.0:
        idx = np.unravel_index(np.argmax(np.where(over, dist, 0)), dist.shape)
        raise AssertionError(f"{what}: {got64[idx]} vs {ref64[idx]} is outside the admissible range "
                             f"[{lo[idx]}, {hi[idx]}] by {worst:.3f} x tol")
    assert n <= max(1, RANGED_MAX_FRAC * got64.size), f"{what}: {n} elements need an admissible alternative"


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


def sample_tokens(T, n, seed):
    """n seeded token indices (sorted, distinct), always with the first and last."""
    rng = np.random.default_rng(seed)
    if n >= T:
        return np.arange(T)
    pick = set(rng.choice(T, n, replace=False).tolist())
    pick.discard(0)
    pick.discard(T - 1)
    rest = sorted(pick)[: n - 2]
    return np.array(sorted([0, T - 1] + rest), dtype=np.int64)


def sample_experts(counts, n, seed):
    """n distinct experts: the fullest, the emptiest (an empty one if any) and
    seeded others."""
    counts = np.asarray(counts)
    picks = [int(np.argmax(counts)), int(np.argmin(counts))]
    rng = np.random.default_rng(seed)
    for e in rng.permutation(len(counts)):
        if len(set(picks)) >= n:
            break
        picks.append(int(e))
    return sorted(set(picks))
