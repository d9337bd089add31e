"""GPU parity of the backward (mok_moe_bwd through the C ABI) against the oracle.

Every float output at 2e-2 * max(1, |oracle|) per element, with no other
allowance.  Small shapes: every output element by element (dX,
dW_gate/up/down, the shared expert's weight gradients, ds, dg).  The
DSV3-shaped fwd+bwd workload (T 4096): dX, dg and ds of 512 seeded tokens,
whole weight gradients of four experts (the fullest, the emptiest and two
seeded ones), and a 128-wide slice of the shared expert's weight gradients,
each computed by the oracle from its own routing.  Two runs must agree
bitwise.
"""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import (BF16_TOL, PARITY_RATIOS, alloc_plan, assert_close, assert_close_ranged, device_weights_fetch, host, mok,
                     sample_experts, sample_tokens)
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
    # experts of 512 or more routed rows on average: the routed dX on the
    # 128-row single-CTA tiles instead of the CTA pairs
    "big_experts": W.MoEConfig("big_experts", T=1100, D=256, I=256, E=2, K=1, I_shared=128),
}


@pytest.fixture(scope="module")
def m():
    return mok()


def weight_grads(b, x_bits, dy_bits):
    """The oracle's weight gradients of one expert's rows from its
    route_backward_rows(..., ranges=True) result: name -> (dW, (lo_shift,
    hi_shift)) with dW_down [D][I], dW_gate / dW_up [I][D]."""
    X = O.bf16_to_f32(x_bits)
    dY = O.bf16_to_f32(dy_bits)
    rg = b["ranges"]
    lo, hi = O.sum_range(b["a_g"], rg["a_g"], dY)
    return {"dW_down": (O.round_bf16(dY.T @ b["a_g"]), (lo.T, hi.T)),
            "dW_gate": (O.round_bf16(b["dh"].T @ X), O.sum_range(b["dh"], rg["dh"], X)),
            "dW_up": (O.round_bf16(b["du"].T @ X), O.sum_range(b["du"], rg["du"], X))}


def _fwd_bwd(m, cfg, d, act_rows=None, bwd_shared_sms=0, act_shared=False):
    """Forward + backward through the C ABI.  act_rows: rows of the kept
    h, u store (None: no store, the backward replays every expert);
    act_shared: also keep the shared expert's h, u; bwd_shared_sms:
    shape.bwd_shared_sms."""
    shape = m.shape_of(cfg, bwd_shared_sms=bwd_shared_sms)
    ws = torch.empty(max(m.workspace_bytes(shape, m.OP_FWD), m.workspace_bytes(shape, m.OP_BWD)),
                     dtype=torch.uint8, device=DEV)
    out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    saved = alloc_plan(cfg, DEV)
    if act_rows is not None:
        saved["act"] = torch.full((act_rows, 2 * cfg.I), float("nan"), dtype=torch.float32, device=DEV)
    if act_shared and cfg.I_shared:
        saved["act_shared"] = torch.full((cfg.T, 2 * cfg.I_shared), float("nan"), dtype=torch.float32, device=DEV)
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
    ref = O.moe_backward(h, h["dy"], cfg.K, ranges=True)
    for k, r in (("dx", "dX"), ("dg", "dg"), ("ds", "ds")):
        assert_close(_f(got[k]), ref[r], BF16_TOL, f"bf16 bwd {r} [{name}]")
    pairs = [("dw_gate", "dW_gate"), ("dw_up", "dW_up"), ("dw_down", "dW_down")]
    if cfg.I_shared:
        pairs += [("dws_gate", "dWs_gate"), ("dws_up", "dWs_up"), ("dws_down", "dWs_down")]
    for k, r in pairs:
        assert_close_ranged(_f(got[k]), ref[r], ref["range"][r], BF16_TOL, f"bf16 bwd {r} [{name}]")
    if name in ("skew_small", "skew_256"):
        empty = np.flatnonzero(np.bincount(O.route(h["s"], cfg.K)[0].reshape(-1), minlength=cfg.E) == 0)
        assert len(empty) > 0 and torch.all(got["dw_down"][torch.from_numpy(empty).to(DEV)] == 0)
    again, _ = _fwd_bwd(m, cfg, d)
    for k, v in got.items():
        if v is not None:
            assert torch.equal(v.view(torch.int16) if v.dtype == torch.bfloat16 else v.view(torch.int32),
                               again[k].view(torch.int16) if v.dtype == torch.bfloat16 else again[k].view(torch.int32)), k


def test_backward_full_size_sampled(m):
    """The DSV3 fwd+bwd layer as bench.py runs it (every expert's h, u kept
    by the forward, no replay), equal bit for bit to the all-replay path."""
    from concurrent.futures import ThreadPoolExecutor
    cfg = W.CONFIGS["dsv3_bf16_fwdbwd"]
    d = W.make_inputs(cfg, DEV)
    got, saved = _fwd_bwd(m, cfg, d, act_rows=cfg.R)
    replayed, _ = _fwd_bwd(m, cfg, d)
    for k, v in got.items():
        if v is not None:
            assert torch.equal(_bits(v), _bits(replayed[k])), k
    del replayed
    s_host = d["s"].cpu().numpy()
    idx, g, den = O.route(s_host, cfg.K)
    counts, offsets, table, route_dst = O.plan(idx, cfg.E)
    assert np.array_equal(saved["table"].cpu().numpy(), table)
    hw = device_weights_fetch(d)
    toks = sample_tokens(cfg.T, 512, seed=1)
    x_all = W.bf16_bits(d["x"])
    dy_all = W.bf16_bits(d["dy"])
    with ThreadPoolExecutor(max_workers=16) as pool:
        # 512 seeded tokens: dX rows, dg, ds
        ref = O.moe_backward_tokens(x_all[toks], dy_all[toks], s_host[toks], hw, cfg.K, map_fn=pool.map)
        assert_close(_f(got["dx"][torch.from_numpy(toks).to(DEV)]), ref["dX"], BF16_TOL, "bf16 bwd dX [full]")
        assert_close(_f(got["dg"][torch.from_numpy(toks).to(DEV)]), ref["dg"], BF16_TOL, "bf16 bwd dg [full]")
        assert_close(_f(got["ds"][torch.from_numpy(toks).to(DEV)]), ref["ds"], BF16_TOL, "bf16 bwd ds [full]")
        # four experts: whole weight gradients
        experts = sample_experts(counts, 4, seed=2)

        def expert_grads(e):
            p0, p1 = int(offsets[e]), int(offsets[e + 1])
            if p0 == p1:
                return None
            toks_e = table[p0:p1, 0] // cfg.K
            gr = g[toks_e, table[p0:p1, 0] % cfg.K]
            return weight_grads(O.route_backward_rows(x_all[toks_e], dy_all[toks_e], gr, *hw.fetch(e), ranges=True),
                                x_all[toks_e], dy_all[toks_e])

        for e, res in zip(experts, pool.map(expert_grads, experts)):
            if counts[e] == 0:
                assert torch.all(got["dw_down"][e] == 0) and torch.all(got["dw_gate"][e] == 0)
                assert torch.all(got["dw_up"][e] == 0)
                continue
            for k, r in (("dw_down", "dW_down"), ("dw_gate", "dW_gate"), ("dw_up", "dW_up")):
                assert_close_ranged(_f(got[k][e]), res[r][0], res[r][1], BF16_TOL, f"bf16 bwd {r} [full, expert {e}]")
    # shared expert: a 128-wide slice of I_shared, every token
    Wsh = hw.shared
    i0, i1 = 640, 768
    bs = O.route_backward_rows(x_all, dy_all, np.ones(cfg.T, np.float32), Wsh[0][i0:i1], Wsh[1][i0:i1],
                               np.ascontiguousarray(Wsh[2][:, i0:i1]), ranges=True)
    res = weight_grads(bs, x_all, dy_all)
    assert_close_ranged(_f(got["dws_gate"][i0:i1]), *res["dW_gate"], BF16_TOL, "bf16 bwd dWs_gate [full]")
    assert_close_ranged(_f(got["dws_up"][i0:i1]), *res["dW_up"], BF16_TOL, "bf16 bwd dWs_up [full]")
    assert_close_ranged(_f(got["dws_down"][:, i0:i1]), *res["dW_down"], BF16_TOL, "bf16 bwd dWs_down [full]")


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("name", ["tiny", "ragged", "skew_256", "max_e_k"])
def test_backward_kept_activations(m, name):
    """The forward keeps h, u (fp32) for every expert that fits in the store;
    the backward reads them there and replays only the other experts.  With
    the store holding every row, half the rows, or one row less than the
    first expert, and with or without the shared expert's own store, the
    gradients equal the all-replay path bit for bit (the kept h, u are the
    same tensor-core sums the replay forms) and the oracle at the bare
    tolerance."""
    cfg = SMALL[name]
    inp = W.make_inputs(cfg, "cpu", with_dy=True)
    h = host(inp)
    d = {k: v.to(DEV) for k, v in inp.items()}
    base, saved = _fwd_bwd(m, cfg, d)
    offsets = saved["offsets"].cpu().numpy()
    first = int(offsets[np.flatnonzero(np.diff(offsets) > 0)[0] + 1])  # end of the first non-empty expert
    ref = O.moe_backward(h, h["dy"], cfg.K)
    for rows, keep_shared in ((cfg.R, True), (cfg.R, False), (cfg.R // 2, True), (max(first - 1, 1), False)):
        got, sv = _fwd_bwd(m, cfg, d, act_rows=rows, act_shared=keep_shared)
        for k, v in base.items():
            if v is not None:
                assert torch.equal(_bits(v), _bits(got[k])), (rows, k)
        assert_close(_f(got["dx"]), ref["dX"], BF16_TOL, f"bf16 bwd kept dX [{name}]")
        assert_close(_f(got["ds"]), ref["ds"], BF16_TOL, f"bf16 bwd kept ds [{name}]")
        # the store holds exactly the kept experts' rows; the rest is untouched
        act = sv["act"].cpu().numpy()
        kept_end = int(offsets[np.searchsorted(offsets, rows, side="right") - 1])
        assert np.all(np.isfinite(act[:kept_end])) and np.all(np.isnan(act[kept_end:]))
        if keep_shared and cfg.I_shared:  # the shared expert's h, u: every token's row written
            assert torch.isfinite(sv["act_shared"]).all()


@pytest.mark.parametrize("name", ["ragged", "skew_256", "tiny"])
def test_backward_intermediates_are_admissible(m, name):
    """The GPU's bf16 dh, du and a_g (read from the backward's workspace)
    equal the oracle's at every rounding point whose decision the arithmetic
    fixes, and at the others are one of the admissible neighbours
    (oracle.rounding_ranges): their differences from the oracle are single
    rounding flips at marked points, nothing else."""
    cfg = SMALL[name]
    inp = W.make_inputs(cfg, "cpu", with_dy=True)
    h = host(inp)
    d = {k: v.to(DEV) for k, v in inp.items()}
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
    g = [torch.empty(T, D, dtype=bf, device=DEV), torch.empty(E, I, D, dtype=bf, device=DEV),
         torch.empty(E, I, D, dtype=bf, device=DEV), torch.empty(E, D, I, dtype=bf, device=DEV),
         torch.empty(max(Is, 1), D, dtype=bf, device=DEV), torch.empty(max(Is, 1), D, dtype=bf, device=DEV),
         torch.empty(D, max(Is, 1), dtype=bf, device=DEV), torch.empty(T, E, device=DEV), torch.empty(T, K, device=DEV)]
    m.moe_bwd(shape, w, d["x"], d["s"], pb, d["dy"], *g, ws)
    m.check_device_status()
    R = cfg.R
    inter = {}
    for key, reg in (("dh", m.WS_BWD_DH), ("du", m.WS_BWD_DU), ("a_g", m.WS_BWD_AG)):
        off = m.workspace_offset(shape, reg)
        inter[key] = ws[off:off + R * I * 2].view(bf).view(R, I).float().cpu().numpy()
    idx, gg, _ = O.route(h["s"], K)
    _, offsets, table, _ = O.plan(idx, E)
    flips = marked = total = 0
    for e in range(E):
        p0, p1 = int(offsets[e]), int(offsets[e + 1])
        if p0 == p1:
            continue
        toks = table[p0:p1, 0] // K
        b = O.route_backward_rows(h["x"][toks], h["dy"][toks], gg[toks, table[p0:p1, 0] % K],
                                  h["w_gate"][e], h["w_up"][e], h["w_down"][e], ranges=True)
        for key in ("dh", "du", "a_g"):
            got = inter[key][p0:p1]
            lo, hi = b["ranges"][key]
            fixed = lo == hi
            assert np.array_equal(got[fixed], b[key][fixed]), (e, key)
            assert np.all((got >= lo) & (got <= hi)), (e, key)
            flips += int(np.count_nonzero(got != b[key]))
            marked += int(np.count_nonzero(~fixed))
            total += got.size
    PARITY_RATIOS[f"bf16 bwd intermediates [{name}]: flipped / marked / points"] = f"{flips} / {marked} / {total}"


GRID = {
    "tiny": W.CONFIGS["tiny"].replace(values="grid"),
    "ragged": SMALL["ragged"].replace(values="grid"),
    "skew_256": SMALL["skew_256"].replace(values="grid"),
}


@pytest.mark.parametrize("name", list(GRID))
def test_backward_grid_inputs_bare_tolerance(m, name):
    """Grid inputs (small integers times powers of two): every product sum
    over D or I is exact in fp32 in any order, so the GPU and the oracle take
    the same bf16 rounding decisions (up to the exponential's last bits) and
    every output, weight gradients included, must be within
    2e-2 * max(1, |oracle|) with no other allowance, on both the replay and
    the kept-activation paths."""
    cfg = GRID[name]
    inp = W.make_inputs(cfg, "cpu", with_dy=True)
    h = host(inp)
    d = {k: v.to(DEV) for k, v in inp.items()}
    ref = O.moe_backward(h, h["dy"], cfg.K)
    pairs = [("dx", "dX"), ("dg", "dg"), ("ds", "ds"), ("dw_gate", "dW_gate"), ("dw_up", "dW_up"),
             ("dw_down", "dW_down")]
    if cfg.I_shared:
        pairs += [("dws_gate", "dWs_gate"), ("dws_up", "dWs_up"), ("dws_down", "dWs_down")]
    for act_rows in (None, cfg.R):
        got, _ = _fwd_bwd(m, cfg, d, act_rows=act_rows)
        for k, r in pairs:
            assert_close(_f(got[k]), ref[r], BF16_TOL, f"bf16 bwd grid {r} [{name}]")


def test_backward_grid_inputs_full_size(m):
    """The DSV3 fwd+bwd shapes (T 4096, 256 experts) on grid inputs: dX, dg,
    ds of 512 seeded tokens, whole weight gradients of four experts and a
    128-wide slice of the shared expert's (sums over all 4096 tokens), every
    one at the bare tolerance."""
    from concurrent.futures import ThreadPoolExecutor
    cfg = W.CONFIGS["dsv3_bf16_fwdbwd"].replace(values="grid")
    d = W.make_inputs(cfg, DEV)
    got, saved = _fwd_bwd(m, cfg, d, act_rows=cfg.R)
    s_host = d["s"].cpu().numpy()
    idx, g, den = O.route(s_host, cfg.K)
    counts, offsets, table, _ = O.plan(idx, cfg.E)
    hw = device_weights_fetch(d)
    toks = sample_tokens(cfg.T, 512, seed=5)
    x_all = W.bf16_bits(d["x"])
    dy_all = W.bf16_bits(d["dy"])
    sel = torch.from_numpy(toks).to(DEV)
    with ThreadPoolExecutor(max_workers=16) as pool:
        ref = O.moe_backward_tokens(x_all[toks], dy_all[toks], s_host[toks], hw, cfg.K, map_fn=pool.map)
        for k, r in (("dx", "dX"), ("dg", "dg"), ("ds", "ds")):
            assert_close(_f(got[k][sel]), ref[r], BF16_TOL, f"bf16 bwd grid {r} [full]")

        def expert_grads(e):
            p0, p1 = int(offsets[e]), int(offsets[e + 1])
            if p0 == p1:
                return None
            toks_e = table[p0:p1, 0] // cfg.K
            gr = g[toks_e, table[p0:p1, 0] % cfg.K]
            return weight_grads(O.route_backward_rows(x_all[toks_e], dy_all[toks_e], gr, *hw.fetch(e), ranges=True),
                                x_all[toks_e], dy_all[toks_e])

        experts = sample_experts(counts, 4, seed=6)
        for e, res in zip(experts, pool.map(expert_grads, experts)):
            if res is None:
                assert torch.all(got["dw_down"][e] == 0)
                continue
            for k, r in (("dw_down", "dW_down"), ("dw_gate", "dW_gate"), ("dw_up", "dW_up")):
                assert_close(_f(got[k][e]), res[r][0], BF16_TOL, f"bf16 bwd grid {r} [full, expert {e}]")
    Wsh = hw.shared
    i0, i1 = 640, 768
    bs = O.route_backward_rows(x_all, dy_all, np.ones(cfg.T, np.float32), Wsh[0][i0:i1], Wsh[1][i0:i1],
                               np.ascontiguousarray(Wsh[2][:, i0:i1]), ranges=True)
    res = weight_grads(bs, x_all, dy_all)
    assert_close(_f(got["dws_gate"][i0:i1]), res["dW_gate"][0], BF16_TOL, "bf16 bwd grid dWs_gate [full]")
    assert_close(_f(got["dws_up"][i0:i1]), res["dW_up"][0], BF16_TOL, "bf16 bwd grid dWs_up [full]")
    assert_close(_f(got["dws_down"][:, i0:i1]), res["dW_down"][0], BF16_TOL, "bf16 bwd grid dWs_down [full]")


@pytest.mark.parametrize("name", ["ragged", "skew_256", "one_token", "k_equals_e"])
def test_backward_shared_side_stream_is_bitexact(m, name):
    """shape.bwd_shared_sms runs the shared expert's backward on a side
    stream on that many SMs while the routed dgrad and dX take the others:
    other grids, the same tiles, the same bits as the single-stream
    backward (bwd_shared_sms = 0), with and without the kept store."""
    cfg = SMALL[name]
    inp = W.make_inputs(cfg, "cpu", with_dy=True)
    d = {k: v.to(DEV) for k, v in inp.items()}
    for act_rows in (cfg.R, None):
        base, _ = _fwd_bwd(m, cfg, d, act_rows=act_rows)
        for k in (2, 9, 40):
            got, _ = _fwd_bwd(m, cfg, d, act_rows=act_rows, bwd_shared_sms=k)
            for key, v in base.items():
                if v is not None:
                    assert torch.equal(_bits(v), _bits(got[key])), (k, act_rows, key)


def test_bwd_shared_sms_rule(m):
    """The split mok_moe_bwd uses: none by default or without a shared
    expert, an explicit count capped at a third of the SMs."""
    n = torch.cuda.get_device_properties(0).multi_processor_count
    c4 = W.CONFIGS["dsv3_bf16_fwdbwd"]
    assert m.bwd_shared_sms(m.shape_of(c4)) == 0
    assert m.bwd_shared_sms(m.shape_of(c4.replace(I_shared=0), bwd_shared_sms=20)) == 0
    assert m.bwd_shared_sms(m.shape_of(c4, bwd_shared_sms=1)) == 0
    assert m.bwd_shared_sms(m.shape_of(c4, bwd_shared_sms=4096)) == n // 3
    assert m.bwd_shared_sms(m.shape_of(c4, bwd_shared_sms=20)) == min(20, n // 3)
    with pytest.raises(ValueError):
        m.bwd_shared_sms(m.shape_of(c4, bwd_shared_sms=-1))


def test_backward_shared_side_stream_full_size(m):
    """The DSV3 fwd+bwd layer (T 4096, h, u kept) with the shared expert's
    backward on 40 SMs of a side stream gives the single-stream bits."""
    cfg = W.CONFIGS["dsv3_bf16_fwdbwd"]
    d = W.make_inputs(cfg, DEV, with_dy=True)
    base, _ = _fwd_bwd(m, cfg, d, act_rows=cfg.R)
    base = {k: _bits(v).clone() for k, v in base.items() if v is not None}
    got, _ = _fwd_bwd(m, cfg, d, act_rows=cfg.R, bwd_shared_sms=40)
    for key, v in base.items():
        assert torch.equal(v, _bits(got[key])), key
