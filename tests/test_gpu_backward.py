"""GPU parity of the backward (mok_moe_bwd through the C ABI) against the oracle.

Small shapes: every output element by element (dX, dW_gate/up/down, the
shared expert's weight gradients, ds, dg).  The DSV3-shaped fwd+bwd workload
(T 4096): sampled tokens for dX / ds / dg, whole weight gradients of sampled
experts (the fullest, the emptiest, a middle one), and a 128-wide slice of
the shared expert's weight gradients, each computed by the oracle from its
own routing.  Two runs must agree bitwise.
"""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import BF16_TOL, alloc_plan, assert_close, host, mok
from routing_grouped_expert_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")

SMALL = {
    "tiny": W.CONFIGS["tiny"],
    "ragged": W.MoEConfig("ragged", T=300, D=512, I=256, E=5, K=3, I_shared=128),
    "skew_small": W.MoEConfig("skew_small", T=700, D=256, I=128, E=16, K=4, I_shared=0, skew=2.0),
    "one_expert": W.MoEConfig("one_expert", T=200, D=256, I=128, E=1, K=1, I_shared=0),
    # D and I multiples of 256 (256-column weight-gradient tiles throughout),
    # with empty experts and ragged expert ends
    "skew_256": W.MoEConfig("skew_256", T=700, D=512, I=256, E=32, K=4, I_shared=256, skew=2.0),
    # degenerate shapes: one token; every expert chosen by every token; the
    # largest E and K the boundary accepts (most experts empty)
    "one_token": W.MoEConfig("one_token", T=1, D=256, I=128, E=8, K=2, I_shared=128),
    "k_equals_e": W.MoEConfig("k_equals_e", T=65, D=256, I=128, E=8, K=8, I_shared=128),
    "max_e_k": W.MoEConfig("max_e_k", T=40, D=256, I=128, E=1024, K=32, I_shared=0),
}


@pytest.fixture(scope="module")
def m():
    return mok()


def _fwd_bwd(m, cfg, d):
    shape = m.shape_of(cfg)
    ws = torch.empty(max(m.workspace_bytes(shape, m.OP_FWD), m.workspace_bytes(shape, m.OP_BWD)),
                     dtype=torch.uint8, device=DEV)
    out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    saved = alloc_plan(cfg, DEV)
    pb = m.make_plan_buf(saved)
    w = m.make_weights(d)
    m.moe_fwd(shape, w, d["x"], d["s"], out, ws, pb)
    bf = torch.bfloat16
    T, D, I, E, K, Is = cfg.T, cfg.D, cfg.I, cfg.E, cfg.K, cfg.I_shared
    g = dict(dx=torch.empty(T, D, dtype=bf, device=DEV),
             dw_gate=torch.empty(E, I, D, dtype=bf, device=DEV),
             dw_up=torch.empty(E, I, D, dtype=bf, device=DEV),
             dw_down=torch.empty(E, D, I, dtype=bf, device=DEV),
             dws_gate=torch.empty(Is, D, dtype=bf, device=DEV) if Is else None,
             dws_up=torch.empty(Is, D, dtype=bf, device=DEV) if Is else None,
             dws_down=torch.empty(D, Is, dtype=bf, device=DEV) if Is else None,
             ds=torch.empty(T, E, dtype=torch.float32, device=DEV),
             dg=torch.empty(T, K, dtype=torch.float32, device=DEV))
    # poison outputs so unwritten elements show up
    for v in g.values():
        if v is not None:
            v.fill_(float("nan"))
    m.moe_bwd(shape, w, d["x"], d["s"], pb, d["dy"], g["dx"], g["dw_gate"], g["dw_up"], g["dw_down"],
              g["dws_gate"], g["dws_up"], g["dws_down"], g["ds"], g["dg"], ws)
    m.check_device_status()
    return g, saved


def _f(t):
    return t.float().cpu().numpy()


@pytest.mark.parametrize("name", list(SMALL))
def test_backward_elementwise_and_deterministic(m, name):
    cfg = SMALL[name]
    inp = W.make_inputs(cfg, "cpu", with_dy=True)
    h = host(inp)
    d = {k: v.to(DEV) for k, v in inp.items()}
    got, _ = _fwd_bwd(m, cfg, d)
    ref = O.moe_backward(h, h["dy"], cfg.K, with_slack=True)
    sl = ref["slack"]
    assert_close(_f(got["dx"]), ref["dX"], BF16_TOL, "dX", sl["dX"])
    assert_close(_f(got["dw_gate"]), ref["dW_gate"], BF16_TOL, "dW_gate", sl["dW_gate"])
    assert_close(_f(got["dw_up"]), ref["dW_up"], BF16_TOL, "dW_up", sl["dW_up"])
    assert_close(_f(got["dw_down"]), ref["dW_down"], BF16_TOL, "dW_down", sl["dW_down"])
    if cfg.I_shared:
        assert_close(_f(got["dws_gate"]), ref["dWs_gate"], BF16_TOL, "dWs_gate", sl["dWs_gate"])
        assert_close(_f(got["dws_up"]), ref["dWs_up"], BF16_TOL, "dWs_up", sl["dWs_up"])
        assert_close(_f(got["dws_down"]), ref["dWs_down"], BF16_TOL, "dWs_down", sl["dWs_down"])
    assert_close(_f(got["dg"]), ref["dg"], BF16_TOL, "dg", sl["dg"])
    assert_close(_f(got["ds"]), ref["ds"], BF16_TOL, "ds", sl["ds"])
    if name in ("skew_small", "skew_256"):
        empty = np.flatnonzero(np.bincount(O.route(h["s"], cfg.K)[0].reshape(-1), minlength=cfg.E) == 0)
        assert len(empty) > 0 and torch.all(got["dw_down"][torch.from_numpy(empty).to(DEV)] == 0)
    again, _ = _fwd_bwd(m, cfg, d)
    for k, v in got.items():
        if v is not None:
            assert torch.equal(v.view(torch.int16) if v.dtype == torch.bfloat16 else v.view(torch.int32),
                               again[k].view(torch.int16) if v.dtype == torch.bfloat16 else again[k].view(torch.int32)), k


def test_backward_full_size_sampled(m):
    cfg = W.CONFIGS["dsv3_bf16_fwdbwd"]
    d = W.make_inputs(cfg, DEV)
    got, saved = _fwd_bwd(m, cfg, d)
    s_host = d["s"].cpu().numpy()
    idx, g, den = O.route(s_host, cfg.K)
    counts, offsets, table, route_dst = O.plan(idx, cfg.E)
    assert np.array_equal(saved["table"].cpu().numpy(), table)
    Wsh = (W.bf16_bits(d["ws_gate"]), W.bf16_bits(d["ws_up"]), W.bf16_bits(d["ws_down"]))

    def ew(e):
        return W.bf16_bits(d["w_gate"][e]), W.bf16_bits(d["w_up"][e]), W.bf16_bits(d["w_down"][e])

    # sampled tokens: dX rows, dg, ds
    rng = np.random.default_rng(1)
    toks = sorted(set([0, cfg.T - 1] + list(rng.choice(cfg.T, 3, replace=False))))
    for t in toks:
        xr = W.bf16_bits(d["x"][t:t + 1])
        dyr = W.bf16_bits(d["dy"][t:t + 1])
        bs = O.route_backward_rows(xr, dyr, np.ones(1, np.float32), *Wsh)
        acc = bs["dx"][0].copy()
        sl_dx = bs["flip_dx"][0].copy()
        dg_t = np.zeros(cfg.K, np.float32)
        sl_dg = np.zeros(cfg.K)
        for k in range(cfg.K):
            b = O.route_backward_rows(xr, dyr, g[t:t + 1, k], *ew(int(idx[t, k])))
            acc = acc + b["dx"][0]
            sl_dx += b["flip_dx"][0]
            dg_t[k] = b["dg"][0]
            sl_dg[k] = b["flip_dg"][0]
        dx_ref = O.round_bf16(acc)
        assert_close(_f(got["dx"][t]), dx_ref, BF16_TOL, f"dX[{t}]", sl_dx + O.bf16_flip_ulp(acc))
        assert_close(_f(got["dg"][t]), dg_t, BF16_TOL, f"dg[{t}]", sl_dg)
        ds_ref = O.router_grad(dg_t[None], g[t:t + 1], den[t:t + 1], idx[t:t + 1], cfg.E)[0]
        sl_ds = O.router_grad_slack(sl_dg[None], g[t:t + 1], den[t:t + 1], idx[t:t + 1], cfg.E)[0]
        assert_close(_f(got["ds"][t]), ds_ref, BF16_TOL, f"ds[{t}]", sl_ds)
    # sampled experts: whole weight gradients
    picks = {int(np.argmax(counts)), int(np.argmin(counts)), cfg.E // 2}
    x_all = W.bf16_bits(d["x"])
    dy_all = W.bf16_bits(d["dy"])
    for e in sorted(picks):
        p0, p1 = int(offsets[e]), int(offsets[e + 1])
        if p0 == p1:
            assert torch.all(got["dw_down"][e] == 0) and torch.all(got["dw_gate"][e] == 0)
            continue
        toks_e = table[p0:p1, 0] // cfg.K
        gr = g[toks_e, table[p0:p1, 0] % cfg.K]
        b = O.route_backward_rows(x_all[toks_e], dy_all[toks_e], gr, *ew(e))
        X = O.bf16_to_f32(x_all[toks_e])
        dY = O.bf16_to_f32(dy_all[toks_e])
        aX, adY = np.abs(X).astype(np.float64), np.abs(dY).astype(np.float64)
        assert_close(_f(got["dw_down"][e]), O.round_bf16(dY.T @ b["a_g"]), BF16_TOL, f"dW_down[{e}]",
                     adY.T @ b["flip_ag"])
        assert_close(_f(got["dw_gate"][e]), O.round_bf16(b["dh"].T @ X), BF16_TOL, f"dW_gate[{e}]",
                     b["flip_dh"].T @ aX)
        assert_close(_f(got["dw_up"][e]), O.round_bf16(b["du"].T @ X), BF16_TOL, f"dW_up[{e}]",
                     b["flip_du"].T @ aX)
    # shared expert: a 128-wide slice of I_shared, every token
    i0, i1 = 640, 768
    bs = O.route_backward_rows(x_all, dy_all, np.ones(cfg.T, np.float32), Wsh[0][i0:i1], Wsh[1][i0:i1],
                               np.ascontiguousarray(Wsh[2][:, i0:i1]))
    X = O.bf16_to_f32(x_all)
    dY = O.bf16_to_f32(dy_all)
    aX, adY = np.abs(X).astype(np.float64), np.abs(dY).astype(np.float64)
    assert_close(_f(got["dws_gate"][i0:i1]), O.round_bf16(bs["dh"].T @ X), BF16_TOL, "dWs_gate slice",
                 bs["flip_dh"].T @ aX)
    assert_close(_f(got["dws_up"][i0:i1]), O.round_bf16(bs["du"].T @ X), BF16_TOL, "dWs_up slice",
                 bs["flip_du"].T @ aX)
    assert_close(_f(got["dws_down"][:, i0:i1]), O.round_bf16(dY.T @ bs["a_g"]), BF16_TOL, "dWs_down slice",
                 adY.T @ bs["flip_ag"])
