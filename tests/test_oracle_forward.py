"""Pins of the oracle's forward pass.

* E = K = 1, no shared expert: the layer is one dense SwiGLU FFN, checked
  against torch fp64 matmuls with torch's bf16 casts at the same points.
* Identity weights and one-hot tokens: each output is a hand-computed scalar
  that names which experts and which g were used.
* W_up = 0 reduces the layer to the shared expert exactly.
* Doubling W_down doubles every expert output exactly.
* Relabelling experts and permuting tokens leave the outputs unchanged.
* K = E: every expert is used and g = s / sum(s).
* The fp32 oracle against an fp64 evaluation with the same rounding points.
"""
import numpy as np
import pytest
import torch

import oracle as O
from routing_grouped_expert_device_gb300 import workloads as W


def _np_inputs(cfg, seed=0):
    t = W.make_inputs(cfg, "cpu", seed)
    out = {}
    for k, v in t.items():
        out[k] = W.bf16_bits(v) if v.dtype == torch.bfloat16 else W.f32_host(v)
    return out


def _bits(a):
    return O.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def test_single_expert_is_dense_ffn():
    for D, I in [(64, 32), (48, 48)]:
        cfg = W.MoEConfig("t", T=40, D=D, I=I, E=1, K=1, I_shared=0)
        inp = _np_inputs(cfg, seed=7)
        res = O.moe_forward(inp, 1)
        x = torch.from_numpy(O.bf16_to_f32(inp["x"])).double()
        Wg = torch.from_numpy(O.bf16_to_f32(inp["w_gate"][0])).double()
        Wu = torch.from_numpy(O.bf16_to_f32(inp["w_up"][0])).double()
        Wd = torch.from_numpy(O.bf16_to_f32(inp["w_down"][0])).double()
        h, u = x @ Wg.T, x @ Wu.T
        a = (torch.nn.functional.silu(h) * u).to(torch.bfloat16).double()
        y = (a @ Wd.T).to(torch.bfloat16).double().numpy()
        assert np.all(res["g"] == 1.0)
        err = np.abs(res["out"] - y)
        # fp32 vs fp64 sums may flip a bf16 rounding: one bf16 ulp of slack
        assert np.all(err <= 2.0 ** -7 * np.maximum(np.abs(y), 2.0 ** -6) * 2)
        assert np.mean(err == 0) > 0.9


def test_identity_weights_one_hot_tokens_hand_computed():
    D = I = 16
    E, K, T = 4, 2, 8
    eye = np.eye(D, dtype=np.float32)
    w_gate = np.stack([_bits(eye)] * E)
    w_up = np.stack([_bits(eye)] * E)
    w_down = np.stack([_bits((e + 1) * eye) for e in range(E)])
    x = np.zeros((T, D), dtype=np.float32)
    vals = [0.5, -1.25, 2.0, 3.0, -0.75, 1.5, 0.25, -2.5]
    cols = [3, 0, 15, 7, 7, 1, 9, 4]
    # scores chosen so g is exact: top two are 0.375 and 0.125 -> g = 0.75, 0.25
    s = np.full((T, E), 0.03125, dtype=np.float32)
    top = [(2, 0), (1, 3), (3, 2), (0, 1), (2, 3), (3, 0), (1, 2), (0, 3)]
    for t in range(T):
        x[t, cols[t]] = vals[t]
        s[t, top[t][0]] = 0.375
        s[t, top[t][1]] = 0.125
    inp = dict(x=_bits(x), s=s, w_gate=w_gate, w_up=w_up, w_down=w_down)
    res = O.moe_forward(inp, K)
    assert res["topk_idx"].tolist() == [list(p) for p in top]
    assert np.all(res["g"] == np.array([0.75, 0.25], dtype=np.float32))

    def bf(v):
        return float(torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).float())

    for t in range(T):
        v = vals[t]
        a = bf(np.float32(v / (1.0 + np.exp(-v))) * np.float32(v))
        y0 = bf((top[t][0] + 1) * a)
        y1 = bf((top[t][1] + 1) * a)
        want = bf(np.float32(0.75) * np.float32(y0) + np.float32(0.25) * np.float32(y1))
        row = res["out"][t]
        assert abs(row[cols[t]] - want) <= 2.0 ** -8 * abs(want), (t, row[cols[t]], want)
        assert np.count_nonzero(row) == 1


def test_zero_up_projection_gives_shared_expert_exactly():
    cfg = W.CONFIGS["tiny"]
    inp = _np_inputs(cfg)
    inp["w_up"] = np.zeros_like(inp["w_up"])
    res = O.moe_forward(inp, cfg.K)
    assert np.all(res["y"] == 0)
    assert np.array_equal(res["out"], res["ys"])
    ys = O.shared_ffn(O.bf16_to_f32(inp["x"]), inp["ws_gate"], inp["ws_up"], inp["ws_down"])
    assert np.array_equal(res["out"], ys)


def test_doubling_down_projection_doubles_expert_outputs():
    cfg = W.CONFIGS["tiny"]
    inp = _np_inputs(cfg)
    r1 = O.moe_forward(inp, cfg.K)
    inp2 = dict(inp)
    inp2["w_down"] = _bits(2.0 * O.bf16_to_f32(inp["w_down"]))
    r2 = O.moe_forward(inp2, cfg.K)
    assert np.array_equal(r2["y"], 2.0 * r1["y"])
    assert np.array_equal(r2["a"], r1["a"])


def _close_bf16(a, b, ulps=2):
    return np.all(np.abs(a - b) <= ulps * 2.0 ** -8 * np.maximum(np.abs(b), 2.0 ** -4))


def test_expert_relabelling_invariance():
    cfg = W.CONFIGS["tiny"]
    inp = _np_inputs(cfg)
    r1 = O.moe_forward(inp, cfg.K)
    perm = np.random.default_rng(9).permutation(cfg.E)  # new label j holds old expert perm[j]
    inp2 = dict(inp)
    inp2["s"] = np.ascontiguousarray(inp["s"][:, perm])
    for k in ("w_gate", "w_up", "w_down"):
        inp2[k] = np.ascontiguousarray(inp[k][perm])
    r2 = O.moe_forward(inp2, cfg.K)
    assert np.array_equal(perm[r2["topk_idx"]], r1["topk_idx"])
    assert np.array_equal(r2["g"], r1["g"])
    assert _close_bf16(r2["out"], r1["out"])


def test_token_permutation_invariance():
    cfg = W.CONFIGS["tiny"]
    inp = _np_inputs(cfg)
    r1 = O.moe_forward(inp, cfg.K)
    perm = np.random.default_rng(10).permutation(cfg.T)
    inp2 = dict(inp)
    inp2["x"] = np.ascontiguousarray(inp["x"][perm])
    inp2["s"] = np.ascontiguousarray(inp["s"][perm])
    r2 = O.moe_forward(inp2, cfg.K)
    assert np.array_equal(r2["topk_idx"], r1["topk_idx"][perm])
    assert np.array_equal(r2["counts"], r1["counts"])
    assert _close_bf16(r2["out"], r1["out"][perm])


def test_all_experts_selected_weights_are_normalised_scores():
    cfg = W.MoEConfig("t", T=32, D=32, I=32, E=4, K=4, I_shared=0)
    inp = _np_inputs(cfg, seed=3)
    res = O.moe_forward(inp, 4)
    s = inp["s"].astype(np.float64)
    assert np.array_equal(np.sort(res["topk_idx"], axis=1), np.tile(np.arange(4), (32, 1)))
    g_want = np.take_along_axis(s, res["topk_idx"].astype(np.int64), 1) / s.sum(1, keepdims=True)
    assert np.allclose(res["g"], g_want, rtol=4 * 2.0 ** -23, atol=0)


def test_fp32_oracle_vs_fp64_evaluation():
    """The fp32 oracle's own error (summation order, fp32 products) is far
    below the 2e-2 parity tolerance: compare against fp64 arithmetic with the
    same bf16 rounding points."""
    cfg = W.CONFIGS["tiny"]
    inp = _np_inputs(cfg)
    r32 = O.moe_forward(inp, cfg.K, O.FP32)
    r64 = O.moe_forward(inp, cfg.K, O.Numerics(np.float64, True))
    assert np.array_equal(r32["topk_idx"], r64["topk_idx"])
    err = np.abs(r32["out"] - r64["out"]) / np.maximum(1.0, np.abs(r64["out"]))
    assert err.max() <= 2e-2 / 4
    exact = O.moe_forward(inp, cfg.K, O.FP64_SHADOW)
    err2 = np.abs(r32["out"] - exact["out"]) / np.maximum(1.0, np.abs(exact["out"]))
    assert err2.max() <= 2e-2


def test_sampled_token_forward_matches_full_forward():
    cfg = W.CONFIGS["tiny"]
    inp = _np_inputs(cfg)
    full = O.moe_forward(inp, cfg.K)
    toks = [0, 5, 77, 255]
    part = O.moe_forward_tokens(toks, inp["x"][toks], inp["s"][toks], O.HostWeights.from_arrays(inp), cfg.K)
    assert np.array_equal(part["topk_idx"], full["topk_idx"][toks])
    rd = full["route_dst"].reshape(cfg.T, cfg.K)
    for j, t in enumerate(toks):
        for k in range(cfg.K):
            assert _close_bf16(part["y"][j, k], full["y"][rd[t, k]], 1)
    assert _close_bf16(part["out"], full["out"][toks], 2)


def test_mxfp8_forward_close_to_bf16_forward():
    cfg = W.CONFIGS["tiny"]
    inp = _np_inputs(cfg)
    rb = O.moe_forward(inp, cfg.K)
    rq = O.moe_forward_mxfp8(inp, cfg.K)
    assert np.array_equal(rq["table"], rb["table"])
    assert np.array_equal(rq["ys"], rb["ys"])
    rel = np.abs(rq["out"] - rb["out"]) / np.maximum(1.0, np.abs(rb["out"]))
    assert rel.max() < 0.25 and rel.mean() < 0.03
    # quantised a round-trips within E4M3 precision
    d = O.mxfp8_dequantize(rq["aq"], rq["asc"])
    assert np.all(np.abs(d - rq["a"]) <= 2.0 ** -4 * np.abs(rq["a"]) + 2.0 ** -10 * 2.0 ** (
        np.repeat(rq["asc"].astype(np.int64) - 127, 32, axis=1)))


def test_mxfp8_rows_function_matches_layer_function():
    cfg = W.CONFIGS["tiny"]
    inp = _np_inputs(cfg)
    rq = O.moe_forward_mxfp8(inp, cfg.K)
    e = 3
    p0, p1 = rq["offsets"][e], rq["offsets"][e + 1]
    rows = inp["x"][rq["table"][p0:p1, 0] // cfg.K]
    r = O.expert_ffn_rows_mxfp8(rows, inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e])
    assert np.array_equal(r["y"], rq["y"][p0:p1])
    assert np.array_equal(r["aq"], rq["aq"][p0:p1])
