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


def test_fp32_and_fp64_roundings_agree_at_the_bare_tolerance():
    """Two correct evaluations of the same rounding points (fp32 sums in
    numpy's order, and fp64 sums) may round a bf16 point the other way where
    the sum lands next to a midpoint; the parity tolerance must absorb that
    by itself: every output within 2e-2 * max(1, |ref|), with room to spare
    (the worst seen is under 0.8 of it on these shapes)."""
    import sys, os
    sys.path.insert(0, os.path.dirname(__file__))
    from helpers import host, rel_err
    from routing_grouped_expert_device_gb300 import workloads as W
    for cfg in (W.MoEConfig("r", T=300, D=512, I=256, E=5, K=3, I_shared=128),
                W.MoEConfig("s", T=700, D=512, I=256, E=32, K=4, I_shared=256, skew=2.0)):
        h = host(W.make_inputs(cfg, "cpu", with_dy=True))
        a = O.moe_backward(h, h["dy"], cfg.K)
        b = O.moe_backward(h, h["dy"], cfg.K, O.Numerics(np.float64, True))
        for k in ["dX", "dW_gate", "dW_up", "dW_down", "dWs_gate", "dWs_up", "dWs_down", "dg", "ds"]:
            assert rel_err(b[k], a[k]).max() <= 0.9 * 2e-2, (cfg.name, k)


def test_sampled_token_backward_matches_full_backward():
    """moe_backward_tokens (routes grouped by expert over a token sample)
    gives the whole layer's dX rows, dg and ds of those tokens."""
    import sys, os
    sys.path.insert(0, os.path.dirname(__file__))
    from helpers import host
    from routing_grouped_expert_device_gb300 import workloads as W
    cfg = W.MoEConfig("r", T=300, D=512, I=256, E=5, K=3, I_shared=128)
    h = host(W.make_inputs(cfg, "cpu", with_dy=True))
    full = O.moe_backward(h, h["dy"], cfg.K)
    toks = np.array([0, 3, 150, 299])
    part = O.moe_backward_tokens(h["x"][toks], h["dy"][toks], h["s"][toks], O.HostWeights.from_arrays(h), cfg.K)
    # the per-route products run in other row batches (another matmul
    # blocking, so a bf16 point may round the other way): a tenth of the
    # parity tolerance
    from helpers import rel_err
    for k in ("dX", "dg", "ds"):
        assert rel_err(part[k], full[k][toks]).max() <= 2e-3, k
    assert np.array_equal(part["ds"] == 0, full["ds"][toks] == 0)


def test_rounding_ranges_cover_another_evaluation_and_stay_tight():
    """rounding_ranges marks the bf16 points of dh, du, a, a_g whose decision
    another correct evaluation could take the other way.  An fp64 evaluation
    with the same rounding points (closer to exact than fp32) must land in
    the range at every point; unmarked points are the oracle's value; and
    most points are unmarked."""
    import sys, os
    sys.path.insert(0, os.path.dirname(__file__))
    from helpers import host
    from routing_grouped_expert_device_gb300 import workloads as W
    cfg = W.MoEConfig("r", T=300, D=512, I=256, E=5, K=3, I_shared=0)
    h = host(W.make_inputs(cfg, "cpu", with_dy=True))
    idx, g, _ = O.route(h["s"], cfg.K)
    F64R = O.Numerics(np.float64, True)
    marked = total = 0
    for e in range(cfg.E):
        rows, ks = np.nonzero(idx == e)
        if len(rows) == 0:
            continue
        args = (h["x"][rows], h["dy"][rows], g[rows, ks], h["w_gate"][e], h["w_up"][e], h["w_down"][e])
        b = O.route_backward_rows(*args, ranges=True)
        c = O.route_backward_rows(*args, num=F64R)
        for k in ("dh", "du", "a", "a_g"):
            lo, hi = b["ranges"][k]
            assert np.all(lo <= b[k]) and np.all(b[k] <= hi), k
            other = np.asarray(c[k], dtype=np.float32)
            assert np.all(lo <= other) and np.all(other <= hi), k
            fixed = lo == hi
            assert np.array_equal(lo[fixed], b[k][fixed])
            marked += int(np.count_nonzero(~fixed))
            total += fixed.size
    # the bounds are worst cases (about 5x the largest accumulation error
    # measured on the GPU): some 7 % of the points are marked on this shape
    assert 0 < marked < 0.15 * total


def test_sum_range_is_the_extreme_choice_brute_force():
    """sum_range's shifts are the least and greatest fp32-exact sums over
    every choice of the marked values (2^n combinations, n small)."""
    rng = np.random.default_rng(9)
    v = O.round_bf16(rng.standard_normal((6, 2)).astype(np.float32))
    lo, hi = v.copy(), v.copy()
    ulp = np.abs(O.round_bf16(v * (1 + 2.0 ** -7)) - v)
    pick = [(0, 0), (2, 0), (5, 0), (1, 1), (3, 1)]
    for i, (p, c) in enumerate(pick):
        if i % 2:
            hi[p, c] += ulp[p, c]
        else:
            lo[p, c] -= ulp[p, c]
    other = rng.standard_normal((6, 3))
    slo, shi = O.sum_range(v, (lo, hi), other)
    base = v.T.astype(np.float64) @ other
    import itertools
    for c in range(2):
        marks = [p for (p, cc) in pick if cc == c]
        sums = []
        for choice in itertools.product([0, 1], repeat=len(marks)):
            w = v[:, c].astype(np.float64).copy()
            for p, ch in zip(marks, choice):
                if ch:
                    w[p] = lo[p, c] if lo[p, c] != v[p, c] else hi[p, c]
            sums.append(w @ other)
        sums = np.array(sums)
        assert np.allclose(slo[c], sums.min(0) - base[c]) and np.allclose(shi[c], sums.max(0) - base[c])
