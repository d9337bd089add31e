"""Pins of the oracle's backward pass.

Central finite differences of L = <dY, MoE(x, s)> in the fp64 shadow (no
rounding points) for dX, every weight gradient and ds; the identity
sum_{j in topk} s_j ds_j = 0 (g is invariant to scaling the selected scores);
the weight gradients as dense matmuls over each expert's rows.
"""
import numpy as np
import pytest

import oracle as O

NUM = O.FP64_SHADOW


def _problem(seed=0, T=6, D=24, I=16, E=4, K=2, Is=8):
    rng = np.random.default_rng(seed)
    inp = dict(
        x=rng.standard_normal((T, D)),
        w_gate=rng.standard_normal((E, I, D)) / np.sqrt(D),
        w_up=rng.standard_normal((E, I, D)) / np.sqrt(D),
        w_down=rng.standard_normal((E, D, I)) / np.sqrt(I),
    )
    if Is:
        inp.update(ws_gate=rng.standard_normal((Is, D)) / np.sqrt(D),
                   ws_up=rng.standard_normal((Is, D)) / np.sqrt(D),
                   ws_down=rng.standard_normal((D, Is)) / np.sqrt(Is))
    logits = rng.standard_normal((T, E))
    s = np.exp(logits) / np.exp(logits).sum(1, keepdims=True)
    inp["s"] = s
    dy = rng.standard_normal((T, D))
    return inp, dy, K


def _loss(inp, dy, K):
    return float(np.sum(O.moe_forward(inp, K, NUM)["out"] * dy))


def _fd(inp, dy, K, key, index, eps=1e-6):
    p = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in inp.items()}
    p[key][index] += eps
    lp = _loss(p, dy, K)
    p[key][index] -= 2 * eps
    lm = _loss(p, dy, K)
    return (lp - lm) / (2 * eps)


@pytest.mark.parametrize("seed", [0, 1])
def test_backward_matches_finite_differences(seed):
    inp, dy, K = _problem(seed)
    g = O.moe_backward(inp, dy, K, NUM)
    rng = np.random.default_rng(100 + seed)
    names = {"x": "dX", "w_gate": "dW_gate", "w_up": "dW_up", "w_down": "dW_down",
             "ws_gate": "dWs_gate", "ws_up": "dWs_up", "ws_down": "dWs_down", "s": "ds"}
    for key, gname in names.items():
        arr = inp[key]
        picks = [tuple(rng.integers(0, n) for n in arr.shape) for _ in range(12)]
        if key.startswith("w_"):
            # make sure used experts are probed
            used = np.unique(O.route(inp["s"], K, NUM)[0])
            picks += [(int(used[0]),) + tuple(rng.integers(0, n) for n in arr.shape[1:]) for _ in range(6)]
        if key == "s":
            idx = O.route(inp["s"], K, NUM)[0]
            picks += [(t, int(idx[t, k])) for t in range(3) for k in range(K)]
        for ix in picks:
            fd = _fd(inp, dy, K, key, ix)
            an = g[gname][ix]
            assert abs(fd - an) <= 1e-6 * (1 + abs(an)), (key, ix, fd, an)


def test_router_grad_scale_invariance_identity():
    inp, dy, K = _problem(3, T=20, E=8, K=3)
    for num in (NUM, O.FP32):
        res = O.moe_backward(inp, dy, K, num)
        ds = res["ds"]
        s = inp["s"]
        idx = O.route(s, K, num)[0]
        sel = np.take_along_axis(s, idx.astype(np.int64), 1)
        dsel = np.take_along_axis(ds, idx.astype(np.int64), 1)
        tol = 1e-12 if num is NUM else 1e-5
        assert np.all(np.abs((sel * dsel).sum(1)) <= tol * (1 + np.abs(dsel).sum(1)))
        mask = np.ones_like(ds, dtype=bool)
        np.put_along_axis(mask, idx.astype(np.int64), False, 1)
        assert np.all(ds[mask] == 0)


def test_weight_grads_are_dense_matmuls():
    inp, dy, K = _problem(4, T=30, E=3, K=2)
    fwd = O.moe_forward(inp, K, NUM)
    res = O.moe_backward(inp, dy, K, NUM, fwd=dict(fwd))
    for e in range(3):
        p0, p1 = fwd["offsets"][e], fwd["offsets"][e + 1]
        toks = fwd["table"][p0:p1, 0] // K
        ks = fwd["table"][p0:p1, 0] % K
        gr = fwd["g"][toks, ks]
        # dW_down[e] = sum over the expert's routes of g * dY (outer) a
        want = np.einsum("p,pd,pi->di", gr, dy[toks], fwd["a"][p0:p1])
        assert np.allclose(res["dW_down"][e], want, rtol=1e-10, atol=1e-12)


def test_fp32_backward_close_to_fp64():
    inp, dy, K = _problem(5, T=16, D=64, I=32, E=4, K=2, Is=32)
    r64 = O.moe_backward(inp, dy, K, NUM)
    inp32 = {k: O.round_bf16(v.astype(np.float32)) if k != "s" else v.astype(np.float32) for k, v in inp.items()}
    r32 = O.moe_backward(inp32, O.round_bf16(dy.astype(np.float32)), K, O.FP32)
    for k in ("dX", "dW_gate", "dW_up", "dW_down", "ds"):
        err = np.abs(r32[k] - r64[k]) / np.maximum(1.0, np.abs(r64[k]))
        assert err.max() < 0.05, k


def test_fp32_and_fp64_roundings_agree_within_slack():
    """Two correct evaluations (fp32 and fp64 sums, same bf16 rounding
    points) may round ambiguous dh/du/a_g/a/dx the other way; they must agree
    within 2e-2 * max(1, |ref|) plus the oracle's ambiguity slack."""
    import sys, os
    sys.path.insert(0, os.path.dirname(__file__))
    from helpers import assert_close, host
    from routing_grouped_expert_device_gb300 import workloads as W
    cfg = W.MoEConfig("r", T=300, D=512, I=256, E=5, K=3, I_shared=128)
    h = host(W.make_inputs(cfg, "cpu", with_dy=True))
    a = O.moe_backward(h, h["dy"], cfg.K, with_slack=True)
    b = O.moe_backward(h, h["dy"], cfg.K, O.Numerics(np.float64, True))
    for k in ["dX", "dW_gate", "dW_up", "dW_down", "dWs_gate", "dWs_up", "dWs_down", "dg", "ds"]:
        assert_close(b[k], a[k], 2e-2, k, a["slack"][k])
    # the ambiguous rounding decisions are a small fraction of all of them
    x = O.bf16_to_f32(h["x"])
    r = O.route_backward_rows(x[:200], O.bf16_to_f32(h["dy"])[:200], np.full(200, 0.3, np.float32),
                              h["w_gate"][0], h["w_up"][0], h["w_down"][0])
    for f in ("flip_dh", "flip_du", "flip_ag"):
        assert np.mean(r[f] > 0) < 0.05, f
