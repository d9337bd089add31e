"""GPU parity of the forward path, called through the C ABI, against the oracle.

Integers (routing, plan, E4M3 / E8M0 bytes) must match bit-exactly; floats
within 2e-2 * max(1, |oracle|) per element; two runs must match bitwise.
Small cases are compared element by element; the full-size workloads compare
the integer outputs in full and sampled token rows one by one.
"""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import (BF16_TOL, alloc_plan, assert_close, device_weights_fetch, host, mok, sample_tokens)
from routing_grouped_expert_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")

# small shapes that still span several tiles and ragged expert tails
SMALL = {
    "tiny": W.CONFIGS["tiny"],
    "ragged": W.MoEConfig("ragged", T=300, D=512, I=256, E=5, K=3, I_shared=128),
    "skew_small": W.MoEConfig("skew_small", T=700, D=256, I=128, E=16, K=4, I_shared=0, skew=2.0),
    "one_expert": W.MoEConfig("one_expert", T=200, D=256, I=128, E=1, K=1, I_shared=0),
}


@pytest.fixture(scope="module")
def m():
    return mok()


def _fwd(m, cfg, d, ws=None):
    shape = m.shape_of(cfg)
    if ws is None:
        ws = torch.empty(m.workspace_bytes(shape, m.OP_FWD), dtype=torch.uint8, device=DEV)
    out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    saved = alloc_plan(cfg, DEV)
    m.moe_fwd(shape, m.make_weights(d), d["x"], d["s"], out, ws, m.make_plan_buf(saved))
    m.check_device_status()
    return out, saved


def _plan_ref(s_host, K, E):
    idx, g, _ = O.route(s_host, K)
    counts, offsets, table, route_dst = O.plan(idx, E)
    return idx, g, counts, offsets, table, route_dst


def _check_plan(saved, ref):
    idx, g, counts, offsets, table, route_dst = ref
    assert np.array_equal(saved["topk_idx"].cpu().numpy(), idx)
    assert np.array_equal(saved["g"].cpu().numpy().view(np.uint32), g.astype(np.float32).view(np.uint32))
    assert np.array_equal(saved["counts"].cpu().numpy(), counts)
    assert np.array_equal(saved["offsets"].cpu().numpy(), offsets)
    R = len(route_dst)
    assert np.array_equal(saved["table"][:R].cpu().numpy(), table)
    assert np.array_equal(saved["route_dst"][:R].cpu().numpy(), route_dst)


# ---------------------------------------------------------------- route / plan
@pytest.mark.parametrize("name", ["tiny", "skew_small", "dsv3_bf16_fwd", "skewed_bf16_fwd"])
def test_route_and_plan_bitexact(m, name):
    cfg = SMALL.get(name) or W.CONFIGS[name]
    s = W.make_inputs(cfg.replace(D=256, I=128, I_shared=0), DEV)["s"]  # only s matters here
    T, E, K = cfg.T, cfg.E, cfg.K
    topk = torch.empty(T, K, dtype=torch.int32, device=DEV)
    g = torch.empty(T, K, dtype=torch.float32, device=DEV)
    m.route(s, K, topk, g)
    plan = alloc_plan(cfg, DEV)
    plan["topk_idx"], plan["g"] = topk, g
    ws = torch.empty(m.workspace_bytes(m.shape_of(cfg), m.OP_PLAN), dtype=torch.uint8, device=DEV)
    m.plan(topk, E, plan["counts"], plan["offsets"], plan["table"], plan["route_dst"], ws)
    m.check_device_status()
    _check_plan(plan, _plan_ref(s.cpu().numpy(), K, E))


def test_route_ties_lowest_index(m):
    T, E, K = 64, 256, 8
    rng = np.random.default_rng(5)
    s = rng.choice(np.array([0.25, 0.5, 0.125, 0.0], dtype=np.float32), size=(T, E))
    s[3] = 0.5  # a row of all-equal scores
    sd = torch.from_numpy(s).to(DEV)
    topk = torch.empty(T, K, dtype=torch.int32, device=DEV)
    g = torch.empty(T, K, dtype=torch.float32, device=DEV)
    m.route(sd, K, topk, g)
    idx, gr, _ = O.route(s, K)
    assert np.array_equal(topk.cpu().numpy(), idx)
    assert np.array_equal(g.cpu().numpy(), gr)
    assert topk[3].tolist() == list(range(8))


def test_plan_reports_bad_route(m):
    T, E, K = 40, 8, 2
    topk = torch.randint(0, E, (T, K), dtype=torch.int32, device=DEV)
    topk[7, 1] = E  # out of range
    R = T * K
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    table = torch.empty(R, 3, dtype=torch.int32, device=DEV)
    route_dst = torch.empty(R, dtype=torch.int32, device=DEV)
    ws = torch.empty(1 << 16, dtype=torch.uint8, device=DEV)
    m.plan(topk, E, counts, offsets, table, route_dst, ws)
    assert m.get_error() == m.MOK_ERR_BAD_ROUTE
    assert m.get_error() == m.MOK_OK  # cleared


# ---------------------------------------------------------------- dispatch / combine
@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_dispatch_exact(m, name):
    cfg = SMALL[name]
    inp = W.make_inputs(cfg, "cpu")
    h = host(inp)
    ref = _plan_ref(h["s"], cfg.K, cfg.E)
    table = torch.from_numpy(ref[4]).to(DEV)
    x = inp["x"].to(DEV)
    xg = torch.empty(cfg.R, cfg.D, dtype=torch.bfloat16, device=DEV)
    m.dispatch(m.shape_of(cfg), x, table, torch.from_numpy(ref[5]).to(DEV), xg)
    want = O.gather(h["x"], ref[4], cfg.K)
    assert np.array_equal(W.bf16_bits(xg), want)


@pytest.mark.parametrize("name,shared,weights", [("tiny", True, True), ("ragged", False, True),
                                                 ("ragged", True, False)])
def test_combine_matches_oracle(m, name, shared, weights):
    cfg = SMALL[name]
    gen = torch.Generator().manual_seed(3)
    yg = torch.randn(cfg.R, cfg.D, generator=gen).to(torch.bfloat16)
    ys = torch.randn(cfg.T, cfg.D, generator=gen).to(torch.bfloat16) if shared else None
    inp = W.make_inputs(cfg, "cpu")
    idx, g, _ = O.route(W.f32_host(inp["s"]), cfg.K)
    _, _, _, route_dst = O.plan(idx, cfg.E)
    out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    gd = torch.from_numpy(g).to(DEV) if weights else None
    m.combine(m.shape_of(cfg), yg.to(DEV), ys.to(DEV) if shared else None, gd,
              torch.from_numpy(route_dst).to(DEV), out)
    y_ref = O.bf16_to_f32(W.bf16_bits(yg))
    ys_ref = O.bf16_to_f32(W.bf16_bits(ys)) if shared else None
    ref = O.combine(y_ref, ys_ref, g if weights else np.ones_like(g), route_dst)
    assert_close(out.float().cpu().numpy(), ref, BF16_TOL, "combine")


# ---------------------------------------------------------------- expert FFN
@pytest.mark.parametrize("name", list(SMALL))
def test_expert_ffn_elementwise(m, name):
    cfg = SMALL[name]
    inp = W.make_inputs(cfg, "cpu")
    h = host(inp)
    ref_fwd = O.moe_forward(h, cfg.K)
    d = {k: v.to(DEV) for k, v in inp.items()}
    xg = torch.from_numpy(O.f32_to_bf16_bits(ref_fwd["xg"]).view(np.int16)).view(torch.bfloat16).to(DEV)
    offsets = torch.from_numpy(ref_fwd["offsets"]).to(DEV)
    a = torch.empty(cfg.R, cfg.I, dtype=torch.bfloat16, device=DEV)
    yg = torch.empty(cfg.R, cfg.D, dtype=torch.bfloat16, device=DEV)
    m.expert_ffn(m.shape_of(cfg), m.make_weights(d), xg, offsets, yg, a_out=a)
    m.check_device_status()
    assert_close(a.float().cpu().numpy(), ref_fwd["a"], BF16_TOL, "a")
    assert_close(yg.float().cpu().numpy(), ref_fwd["y"], BF16_TOL, "y")


@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_shared_ffn_elementwise(m, name):
    cfg = SMALL[name]
    inp = W.make_inputs(cfg, "cpu")
    h = host(inp)
    d = {k: v.to(DEV) for k, v in inp.items()}
    ys = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(m.workspace_bytes(m.shape_of(cfg), m.OP_SHARED_FFN), dtype=torch.uint8, device=DEV)
    m.shared_ffn(m.shape_of(cfg), m.make_weights(d), d["x"], ys, ws)
    ref = O.shared_ffn(O.bf16_to_f32(h["x"]), h["ws_gate"], h["ws_up"], h["ws_down"])
    assert_close(ys.float().cpu().numpy(), ref, BF16_TOL, "ys")


# ---------------------------------------------------------------- whole forward
@pytest.mark.parametrize("name", list(SMALL))
def test_moe_fwd_elementwise_and_deterministic(m, name):
    cfg = SMALL[name]
    inp = W.make_inputs(cfg, "cpu")
    h = host(inp)
    d = {k: v.to(DEV) for k, v in inp.items()}
    out1, saved = _fwd(m, cfg, d)
    ref = O.moe_forward(h, cfg.K)
    _check_plan(saved, (ref["topk_idx"], ref["g"], ref["counts"], ref["offsets"], ref["table"],
                        ref["route_dst"]))
    assert_close(out1.float().cpu().numpy(), ref["out"], BF16_TOL, f"bf16 fwd out [{name}]")
    out2, _ = _fwd(m, cfg, d)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16)), "run-to-run mismatch"


@pytest.mark.parametrize("name", ["dsv3_bf16_fwd", "skewed_bf16_fwd"])
def test_moe_fwd_full_size_sampled(m, name):
    """mok_moe_fwd's out rows of 512 seeded tokens (always the first and the
    last) against the oracle's forward of those tokens."""
    from concurrent.futures import ThreadPoolExecutor
    cfg = W.CONFIGS[name]
    d = W.make_inputs(cfg, DEV)
    out, saved = _fwd(m, cfg, d)
    s_host = d["s"].cpu().numpy()
    _check_plan(saved, _plan_ref(s_host, cfg.K, cfg.E))
    toks = sample_tokens(cfg.T, 512, seed=0)
    x_rows = W.bf16_bits(d["x"][torch.from_numpy(toks).to(DEV)])
    with ThreadPoolExecutor(max_workers=16) as pool:
        ref = O.moe_forward_tokens(toks, x_rows, s_host[toks], device_weights_fetch(d), cfg.K, map_fn=pool.map)
    assert_close(out[torch.from_numpy(toks).to(DEV)].float().cpu().numpy(), ref["out"], BF16_TOL,
                 f"bf16 fwd out [{name}]")
    out2, _ = _fwd(m, cfg, d)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), "run-to-run mismatch"


def test_expert_ffn_full_size_sampled_rows(m):
    """Grouped GEMM rows at the DSV3 shape, checked route by route."""
    cfg = W.CONFIGS["dsv3_bf16_fwd"]
    d = W.make_inputs(cfg, DEV)
    s_host = d["s"].cpu().numpy()
    idx, g, counts, offsets, table, route_dst = _plan_ref(s_host, cfg.K, cfg.E)
    shape = m.shape_of(cfg)
    xg = torch.empty(cfg.R, cfg.D, dtype=torch.bfloat16, device=DEV)
    m.dispatch(shape, d["x"], torch.from_numpy(table).to(DEV), torch.from_numpy(route_dst).to(DEV), xg)
    a = torch.empty(cfg.R, cfg.I, dtype=torch.bfloat16, device=DEV)
    yg = torch.empty(cfg.R, cfg.D, dtype=torch.bfloat16, device=DEV)
    m.expert_ffn(shape, m.make_weights(d), xg, torch.from_numpy(offsets).to(DEV), yg, a_out=a)
    m.check_device_status()
    # the first and last row of the first, a middle and the last expert
    picks = []
    for e in (0, cfg.E // 2, cfg.E - 1):
        picks += [int(offsets[e]), int(offsets[e + 1]) - 1]
    fetch = device_weights_fetch(d).fetch
    for p in picks:
        e = int(table[p, 1])
        t = int(table[p, 0]) // cfg.K
        Wg, Wu, Wd = fetch(e)
        _, _, a_ref, y_ref = O.expert_ffn_rows(W.bf16_bits(d["x"][t:t + 1]), Wg, Wu, Wd)
        assert_close(a[p].float().cpu().numpy(), a_ref[0], BF16_TOL, f"a row {p}")
        assert_close(yg[p].float().cpu().numpy(), y_ref[0], BF16_TOL, f"y row {p}")


# ---------------------------------------------------------------- argument checks
def test_zero_tokens_is_a_noop(m):
    cfg = SMALL["tiny"].replace(T=0)
    shape = m.shape_of(cfg)
    ws = torch.empty(1024, dtype=torch.uint8, device=DEV)
    z = torch.empty(0, cfg.D, dtype=torch.bfloat16, device=DEV)
    m.moe_fwd(shape, m.Weights(), z, torch.empty(0, cfg.E, device=DEV), z, ws)


def test_invalid_shapes_rejected(m):
    import ctypes
    lib = m._lib_handle()
    for bad in [dict(D=200), dict(I=100), dict(K=9), dict(E=0), dict(chunk_rows=100), dict(chunk_rows=-2)]:
        kw = dict(T=16, D=256, I=128, E=8, K=2, I_shared=0)
        kw.update(bad)
        sh = m.make_shape(**kw)
        assert lib.mok_moe_fwd(ctypes.byref(sh), ctypes.byref(m.Weights()), None, None, None, None, None, 0,
                               None) == m.MOK_ERR_INVALID_ARG


def test_split_expert_entry_points_match_expert_ffn(m):
    cfg = SMALL["ragged"]
    inp = W.make_inputs(cfg, "cpu")
    ref = O.moe_forward(host(inp), cfg.K)
    d = {k: v.to(DEV) for k, v in inp.items()}
    shape = m.shape_of(cfg)
    xg = torch.from_numpy(O.f32_to_bf16_bits(ref["xg"]).view(np.int16)).view(torch.bfloat16).to(DEV)
    off = torch.from_numpy(ref["offsets"]).to(DEV)
    a1 = torch.empty(cfg.R, cfg.I, dtype=torch.bfloat16, device=DEV)
    y1 = torch.empty(cfg.R, cfg.D, dtype=torch.bfloat16, device=DEV)
    m.expert_ffn(shape, m.make_weights(d), xg, off, y1, a_out=a1)
    a2 = torch.empty_like(a1)
    y2 = torch.empty_like(y1)
    m.expert_upgate(shape, m.make_weights(d), xg, off, a2)
    m.expert_down(shape, m.make_weights(d), a2, off, y2)
    assert torch.equal(a1.view(torch.int16), a2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    # the shared expert inside the same launches gives the bytes of mok_shared_ffn
    a3, y3 = torch.empty_like(a1), torch.empty_like(y1)
    as_ = torch.empty(cfg.T, cfg.I_shared, dtype=torch.bfloat16, device=DEV)
    ys1 = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    m.expert_upgate(shape, m.make_weights(d), xg, off, a3, x_shared=d["x"], a_shared=as_)
    m.expert_down(shape, m.make_weights(d), a3, off, y3, a_shared=as_, ys=ys1)
    ys2 = torch.empty_like(ys1)
    sws = torch.empty(m.workspace_bytes(shape, m.OP_SHARED_FFN), dtype=torch.uint8, device=DEV)
    m.shared_ffn(shape, m.make_weights(d), d["x"], ys2, sws)
    # the shared expert's up/gate alone (routed operands NULL) on a second stream
    as2 = torch.empty_like(as_)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    m.expert_upgate(shape, m.make_weights(d), None, None, None, x_shared=d["x"], a_shared=as2, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    m.check_device_status()
    assert torch.equal(a1.view(torch.int16), a3.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))
    assert torch.equal(ys1.view(torch.int16), ys2.view(torch.int16))
    assert torch.equal(as_.view(torch.int16), as2.view(torch.int16))
    with pytest.raises(m.MokError):  # no routed operands and no shared expert: nothing to run
        m.expert_upgate(shape, m.make_weights(d), None, None, None)


RING_REUSE = W.MoEConfig("ring_reuse", T=1024, D=256, I=128, E=16, K=4, I_shared=128)


@pytest.mark.parametrize("name,chunk", [("tiny", 512), ("ragged", 512), ("skew_small", 512),
                                        ("skew_small", 2048), ("ring_reuse", 512), ("ring_reuse", 32768)])
def test_ring_upgate_bitexact_vs_dispatch(m, name, chunk):
    """The dispatch fused into the up/gate as a ring of chunk-row slots (4
    slots: R > 4 chunks reuses them) gives the bytes of the explicit gather
    followed by the dense-A GEMM."""
    cfg = RING_REUSE if name == "ring_reuse" else SMALL[name]
    inp = W.make_inputs(cfg, "cpu")
    ref = O.moe_forward(host(inp), cfg.K)
    d = {k: v.to(DEV) for k, v in inp.items()}
    shape = m.shape_of(cfg, chunk_rows=chunk)
    table = torch.from_numpy(ref["table"]).to(DEV)
    off = torch.from_numpy(ref["offsets"]).to(DEV)
    xg = torch.empty(cfg.R, cfg.D, dtype=torch.bfloat16, device=DEV)
    m.dispatch(shape, d["x"], table, torch.from_numpy(ref["route_dst"]).to(DEV), xg)
    a1 = torch.empty(cfg.R, cfg.I, dtype=torch.bfloat16, device=DEV)
    m.expert_upgate(shape, m.make_weights(d), xg, off, a1)
    ws = torch.empty(m.workspace_bytes(shape, m.OP_RING), dtype=torch.uint8, device=DEV)
    for _ in range(2):  # the counters start from zero on every call
        a2 = torch.full_like(a1, float("nan"))
        m.expert_upgate_ring(shape, m.make_weights(d), d["x"], table, off, a2, ws)
        m.check_device_status()
        assert torch.equal(a1.view(torch.int16), a2.view(torch.int16))
    assert_close(a2.float().cpu().numpy(), ref["a"], BF16_TOL, "a")


@pytest.mark.parametrize("name", ["ragged", "ring_reuse"])
def test_moe_fwd_ring_matches_whole_batch_dispatch(m, name):
    """mok_moe_fwd with a chunk size (ring dispatch) equals the whole-batch
    dispatch bit for bit, and the oracle within tolerance."""
    cfg = RING_REUSE if name == "ring_reuse" else SMALL[name]
    inp = W.make_inputs(cfg, "cpu")
    ref = O.moe_forward(host(inp), cfg.K)
    d = {k: v.to(DEV) for k, v in inp.items()}
    outs = []
    for chunk in (-1, 512, 512):
        shape = m.shape_of(cfg, chunk_rows=chunk)
        ws = torch.empty(m.workspace_bytes(shape, m.OP_FWD), dtype=torch.uint8, device=DEV)
        out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
        m.moe_fwd(shape, m.make_weights(d), d["x"], d["s"], out, ws)
        m.check_device_status()
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[1].view(torch.int16), outs[2].view(torch.int16))
    assert_close(outs[1].float().cpu().numpy(), ref["out"], BF16_TOL, "out")


BIG_GROUPS = W.MoEConfig("big_groups", T=1100, D=256, I=256, E=2, K=1, I_shared=128)


def test_moe_fwd_automatic_ring_for_large_groups(m):
    """chunk_rows 0 on a layer of 550 routed rows per expert gathers through
    the ring (b = 2048, one chunk holding every row), with the kept h, u
    store written as by the whole-batch dispatch (chunk_rows -1): out, h and
    u bit-identical, and out within tolerance of the oracle."""
    cfg = BIG_GROUPS
    inp = W.make_inputs(cfg, "cpu")
    ref = O.moe_forward(host(inp), cfg.K)
    d = {k: v.to(DEV) for k, v in inp.items()}
    res = []
    for chunk in (-1, 0):
        shape = m.shape_of(cfg, chunk_rows=chunk)
        ws = torch.empty(m.workspace_bytes(shape, m.OP_FWD), dtype=torch.uint8, device=DEV)
        out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
        saved = alloc_plan(cfg, DEV)
        saved["act"] = torch.full((cfg.R, 2 * cfg.I), float("nan"), device=DEV)
        m.moe_fwd(shape, m.make_weights(d), d["x"], d["s"], out, ws, m.make_plan_buf(saved))
        m.check_device_status()
        res.append((out, saved["act"]))
    assert torch.equal(res[0][0].view(torch.int16), res[1][0].view(torch.int16))
    assert torch.equal(res[0][1].view(torch.int32), res[1][1].view(torch.int32))
    assert_close(res[1][0].float().cpu().numpy(), ref["out"], BF16_TOL, "out")


@pytest.mark.parametrize("config,chunks", [("dsv3_bf16_fwd", (0, 512, 2048, 32768)),
                                           ("skewed_bf16_fwd", (0, 512, 2048, 8192, 32768))])
def test_moe_fwd_ring_full_size_bitexact(m, config, chunks):
    """Full-size layers: every chunk size of the ring, and the automatic
    choice (chunk_rows 0: the whole-batch dispatch for DSV3, the ring of
    2048-row chunks for the skewed layer's 1024 rows per expert), give the
    whole-batch dispatch's output bit for bit (hot and empty experts
    included)."""
    cfg = W.CONFIGS[config]
    d = W.make_inputs(cfg, DEV)
    w = m.make_weights(d)
    outs = []
    for chunk in (-1,) + chunks:
        shape = m.shape_of(cfg, chunk_rows=chunk)
        ws = torch.empty(m.workspace_bytes(shape, m.OP_FWD), dtype=torch.uint8, device=DEV)
        out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
        m.moe_fwd(shape, w, d["x"], d["s"], out, ws)
        m.check_device_status()
        outs.append(out)
        del ws
    for o in outs[1:]:
        assert torch.equal(outs[0].view(torch.int16), o.view(torch.int16))


@pytest.mark.parametrize("name,producer_sms", [("tiny", 8), ("dsv3_bf16_fwd", 40), ("dsv3_mxfp8_fwd", 40)])
def test_producer_sms_split_is_bitexact(m, name, producer_sms):
    """shape.producer_sms leaves SMs free for route, plan and the dispatch
    while the shared expert's launches run on the rest: a different grid,
    the same tiles, the same bytes."""
    cfg = W.CONFIGS[name]
    d = W.make_inputs(cfg, DEV if cfg.T > 1024 else "cpu")
    d = {k: v.to(DEV) for k, v in d.items()}
    if cfg.dtype == "mxfp8":
        from test_gpu_mxfp8 import mx_weights
        d = mx_weights(m, d)
    outs = []
    for ps in (0, producer_sms):
        shape = m.shape_of(cfg, producer_sms=ps)
        ws = torch.empty(m.workspace_bytes(shape, m.OP_FWD), dtype=torch.uint8, device=DEV)
        out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
        m.moe_fwd(shape, m.make_weights(d), d["x"], d["s"], out, ws)
        m.check_device_status()
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
