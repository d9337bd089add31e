"""GPU parity of the MXFP8 path (E4M3 codes, E8M0 1x32 scales) against the oracle.

Forward and backward, small shapes element by element and the DSV3 layers on
sampled tokens and experts.

Codes and scales of quantised inputs (the quantiser, the dispatch with fused
quantisation) must match bit-exactly.  Floats from the MXFP8 GEMMs must be
within 6e-2 * max(1, |oracle|) per element.  The codes of a (quantised in the
up/gate epilogue) must match except in blocks whose bf16 value of a is a
rounding decision fp32 summation order does not fix (oracle bf16_flip_ulp).
"""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import (MXFP8_TOL, alloc_plan, assert_close, assert_close_ranged, device_weights_fetch, host, mok,
                     sample_experts, sample_tokens)
from routing_grouped_expert_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")

SMALL = {
    "tiny": W.CONFIGS["tiny"],
    "ragged": W.MoEConfig("ragged", T=301, D=512, I=256, E=5, K=3, I_shared=128, dtype="mxfp8"),
    "skew_small": W.MoEConfig("skew_small", T=700, D=256, I=128, E=16, K=4, I_shared=0, skew=2.0,
                              dtype="mxfp8"),
    # experts of 512 or more routed rows on average: the row-major down form
    "big_experts": W.MoEConfig("big_experts", T=1100, D=256, I=256, E=2, K=1, I_shared=128, dtype="mxfp8"),
}


@pytest.fixture(scope="module")
def m():
    return mok()


def scale_positions(rows: int, offsets=None) -> np.ndarray:
    """Word index (within one 128-column group) of each row's scale word:
    plain layout, or grouped by expert when offsets are given (mok.h)."""
    r = np.arange(rows, dtype=np.int64)
    if offsets is not None:
        off = np.asarray(offsets, dtype=np.int64)
        e = np.searchsorted(off, r, side="right") - 1
        r = 128 * (off[e] // 128 + e) + r - off[e]
    return (r & ~127) | ((r & 31) << 2) | ((r >> 5) & 3)


def words_to_bytes(words: torch.Tensor, rows: int, cols: int, offsets=None) -> np.ndarray:
    """Scale words [cols/128][ld] -> E8M0 bytes [rows][cols/32] (the oracle's order)."""
    w = words.cpu().numpy().view(np.uint32)
    w = w.reshape(cols // 128, w.size // (cols // 128))[:, scale_positions(rows, offsets)]
    return np.ascontiguousarray(w).view(np.uint8).reshape(cols // 128, rows, 4).transpose(1, 0, 2).reshape(
        rows, cols // 32)


def quantize(m, t: torch.Tensor):
    rows, cols = t.shape
    q = torch.empty(rows, cols, dtype=torch.uint8, device=DEV)
    sc = torch.empty(m.mx_scale_words(rows, cols), dtype=torch.int32, device=DEV)
    m.quantize_mxfp8(t, q, sc)
    return q, sc


def mx_weights(m, d, pair=False):
    """The forward's MXFP8 weight copies; pair: also the paired W_up / W_gate
    scale blocks, so that the up/gate takes the routed rows as N when the
    experts average fewer than 512 rows (the library's other up/gate form;
    test_upgate_routed_rows_as_n_bitexact holds it to this one's bytes)."""
    out = dict(d)
    E, I, D = d["w_gate"].shape
    for name, key in (("gate", "w_gate"), ("up", "w_up"), ("down", "w_down")):
        w = d[key]
        q, sc = quantize(m, w.reshape(-1, w.shape[-1]))
        out["q_" + name], out["sc_" + name] = q, sc
    if pair:
        out["sc_gu_pair"] = torch.empty(m.mx_scale_words(2 * E * I, D), dtype=torch.int32, device=DEV)
        m.mxfp8_pair_scales(m.make_shape(T=1, D=D, I=I, E=E, K=1), m.make_weights(out), out["sc_gu_pair"])
    return out


@pytest.mark.parametrize("cols", [128, 384, 512, 640, 1024, 1152])
def test_quantize_bitexact(m, cols):
    """Row lengths that fill a warp pass (512 columns) exactly, partly, or
    leave part of the warp idle (128, 384: 8 or 24 lanes of 32)."""
    gen = torch.Generator().manual_seed(9)
    v = (torch.randn(301, cols, generator=gen) * torch.logspace(-3, 3, cols)).to(torch.bfloat16)
    v[5, :32] = 0
    v[6, 64:96] = -0.0
    q, sc = quantize(m, v.to(DEV))
    qr, sr = O.mxfp8_quantize(O.bf16_to_f32(W.bf16_bits(v)))
    assert np.array_equal(words_to_bytes(sc, 301, cols), sr)
    assert np.array_equal(q.cpu().numpy(), qr)


@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_dispatch_mxfp8_bitexact(m, name):
    cfg = SMALL[name].replace(dtype="mxfp8")
    inp = W.make_inputs(cfg, "cpu")
    h = host(inp)
    idx, _, _ = O.route(h["s"], cfg.K)
    _, offsets, table, route_dst = O.plan(idx, cfg.E)
    xq = torch.empty(cfg.R, cfg.D, dtype=torch.uint8, device=DEV)
    xs = torch.empty(m.mx_scale_words(cfg.R, cfg.D, cfg.E), dtype=torch.int32, device=DEV)
    m.dispatch(m.shape_of(cfg), inp["x"].to(DEV), torch.from_numpy(table).to(DEV),
               torch.from_numpy(route_dst).to(DEV), xq, xs, offsets=torch.from_numpy(offsets).to(DEV))
    qr, sr = O.mxfp8_quantize(O.gather(O.bf16_to_f32(h["x"]), table, cfg.K))
    assert np.array_equal(xq.cpu().numpy(), qr)
    assert np.array_equal(words_to_bytes(xs, cfg.R, cfg.D, offsets), sr)


def _check_a_codes(aq_gpu, asc_gpu, ref_rows, rows_idx, R, I, offsets):
    """a codes and scales equal the oracle's except in blocks holding an
    ambiguous bf16 rounding of a."""
    aq = aq_gpu.cpu().numpy()[rows_idx]
    sb = words_to_bytes(asc_gpu, R, I, offsets)[rows_idx]
    amb = (O.bf16_flip_ulp(ref_rows["a_pre"]) > 0).reshape(len(rows_idx), I // 32, 32).any(-1)
    ok_blocks = ~amb
    assert np.array_equal(sb[ok_blocks], ref_rows["asc"][ok_blocks])
    codes_ok = np.repeat(ok_blocks, 32, axis=1)
    assert np.array_equal(aq[codes_ok], ref_rows["aq"][codes_ok])
    # across all blocks, the codes that differ are the rare flipped roundings
    assert np.mean(aq != ref_rows["aq"]) < 0.01


@pytest.mark.parametrize("name", list(SMALL))
def test_expert_ffn_mxfp8_elementwise(m, name):
    cfg = SMALL[name].replace(dtype="mxfp8")
    inp = W.make_inputs(cfg, "cpu")
    h = host(inp)
    d = mx_weights(m, {k: v.to(DEV) for k, v in inp.items()})
    idx, _, _ = O.route(h["s"], cfg.K)
    _, offsets, table, route_dst = O.plan(idx, cfg.E)
    shape = m.shape_of(cfg)
    off = torch.from_numpy(offsets).to(DEV)
    xq = torch.empty(cfg.R, cfg.D, dtype=torch.uint8, device=DEV)
    xs = torch.empty(m.mx_scale_words(cfg.R, cfg.D, cfg.E), dtype=torch.int32, device=DEV)
    m.dispatch(shape, d["x"], torch.from_numpy(table).to(DEV), torch.from_numpy(route_dst).to(DEV), xq, xs,
               offsets=off)
    aq = torch.empty(cfg.R, cfg.I, dtype=torch.uint8, device=DEV)
    asc = torch.empty(m.mx_scale_words(cfg.R, cfg.I, cfg.E), dtype=torch.int32, device=DEV)
    yg = torch.empty(cfg.R, cfg.D, dtype=torch.bfloat16, device=DEV)
    w = m.make_weights(d)
    m.expert_upgate(shape, w, xq, off, aq, xg_scale=xs, a_scale=asc)
    m.expert_down(shape, w, aq, off, yg, a_scale=asc)
    m.check_device_status()
    for e in range(cfg.E):
        p0, p1 = int(offsets[e]), int(offsets[e + 1])
        if p0 == p1:
            continue
        rows = h["x"][table[p0:p1, 0] // cfg.K]
        ref = O.expert_ffn_rows_mxfp8(rows, h["w_gate"][e], h["w_up"][e], h["w_down"][e])
        assert_close(yg[p0:p1].float().cpu().numpy(), ref["y"], MXFP8_TOL, f"y expert {e}")
        _check_a_codes(aq, asc, ref, np.arange(p0, p1), cfg.R, cfg.I, offsets)
    # mok_expert_ffn (both halves, a kept in the workspace) gives the same bytes
    ws = torch.empty(m.workspace_bytes(shape, m.OP_EXPERT_FFN), dtype=torch.uint8, device=DEV)
    y2 = torch.empty_like(yg)
    m.expert_ffn(shape, w, xq, off, y2, ws=ws, xg_scale=xs)
    assert torch.equal(yg.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("name", list(SMALL))
def test_moe_fwd_mxfp8_elementwise_and_deterministic(m, name):
    cfg = SMALL[name].replace(dtype="mxfp8")
    inp = W.make_inputs(cfg, "cpu")
    h = host(inp)
    d = mx_weights(m, {k: v.to(DEV) for k, v in inp.items()})
    shape = m.shape_of(cfg)
    ws = torch.empty(m.workspace_bytes(shape, m.OP_FWD), dtype=torch.uint8, device=DEV)
    outs = []
    for _ in range(2):
        out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
        saved = alloc_plan(cfg, DEV)
        m.moe_fwd(shape, m.make_weights(d), d["x"], d["s"], out, ws, m.make_plan_buf(saved))
        m.check_device_status()
        outs.append(out)
    ref = O.moe_forward_mxfp8(h, cfg.K)
    assert np.array_equal(saved["table"][:cfg.R].cpu().numpy(), ref["table"])
    assert_close(outs[0].float().cpu().numpy(), ref["out"], MXFP8_TOL, f"mxfp8 fwd out [{name}]")
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_mxfp8_full_size_sampled_rows(m):
    """DSV3 shapes: grouped MXFP8 GEMM rows of three experts, route by route."""
    cfg = W.CONFIGS["dsv3_mxfp8_fwd"]
    d = W.make_inputs(cfg, DEV)
    d = mx_weights(m, d)
    s_host = d["s"].cpu().numpy()
    idx, _, _ = O.route(s_host, cfg.K)
    counts, offsets, table, route_dst = O.plan(idx, cfg.E)
    shape = m.shape_of(cfg)
    out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(m.workspace_bytes(shape, m.OP_FWD), dtype=torch.uint8, device=DEV)
    saved = alloc_plan(cfg, DEV)
    m.moe_fwd(shape, m.make_weights(d), d["x"], d["s"], out, ws, m.make_plan_buf(saved))
    m.check_device_status()
    assert np.array_equal(saved["table"].cpu().numpy(), table)
    xq = torch.empty(cfg.R, cfg.D, dtype=torch.uint8, device=DEV)
    xs = torch.empty(m.mx_scale_words(cfg.R, cfg.D, cfg.E), dtype=torch.int32, device=DEV)
    m.dispatch(shape, d["x"], torch.from_numpy(table).to(DEV), torch.from_numpy(route_dst).to(DEV), xq, xs,
               offsets=torch.from_numpy(offsets).to(DEV))
    yg = torch.empty(cfg.R, cfg.D, dtype=torch.bfloat16, device=DEV)
    fws = torch.empty(m.workspace_bytes(shape, m.OP_EXPERT_FFN), dtype=torch.uint8, device=DEV)
    m.expert_ffn(shape, m.make_weights(d), xq, torch.from_numpy(offsets).to(DEV), yg, ws=fws, xg_scale=xs)
    m.check_device_status()
    for e in (0, int(np.argmax(counts)), cfg.E - 1):
        p0, p1 = int(offsets[e]), int(offsets[e + 1])
        picks = np.array(sorted({p0, p0 + 1, (p0 + p1) // 2, p1 - 1}))
        rows = W.bf16_bits(d["x"][torch.from_numpy(table[picks, 0] // cfg.K).to(DEV)])
        ref = O.expert_ffn_rows_mxfp8(rows, W.bf16_bits(d["w_gate"][e]), W.bf16_bits(d["w_up"][e]),
                                      W.bf16_bits(d["w_down"][e]))
        assert_close(yg[torch.from_numpy(picks).to(DEV)].float().cpu().numpy(), ref["y"], MXFP8_TOL,
                     f"y expert {e}")


def test_moe_fwd_mxfp8_full_size_sampled_tokens(m):
    """The DSV3 MXFP8 forward through mok_moe_fwd: out rows of 512 seeded
    tokens against the oracle's MXFP8 forward of those tokens."""
    from concurrent.futures import ThreadPoolExecutor
    cfg = W.CONFIGS["dsv3_mxfp8_fwd"]
    d = mx_weights(m, W.make_inputs(cfg, DEV))
    shape = m.shape_of(cfg)
    out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(m.workspace_bytes(shape, m.OP_FWD), dtype=torch.uint8, device=DEV)
    saved = alloc_plan(cfg, DEV)
    m.moe_fwd(shape, m.make_weights(d), d["x"], d["s"], out, ws, m.make_plan_buf(saved))
    m.check_device_status()
    s_host = d["s"].cpu().numpy()
    toks = sample_tokens(cfg.T, 512, seed=3)
    x_rows = W.bf16_bits(d["x"][torch.from_numpy(toks).to(DEV)])
    with ThreadPoolExecutor(max_workers=16) as pool:
        ref = O.moe_forward_tokens(toks, x_rows, s_host[toks], device_weights_fetch(d), cfg.K, mxfp8=True,
                                   map_fn=pool.map)
    assert_close(out[torch.from_numpy(toks).to(DEV)].float().cpu().numpy(), ref["out"], MXFP8_TOL,
                 "mxfp8 fwd out [full]")


def _mx_fwd_chunk(m, cfg, d, chunk, act=False):
    """mok_moe_fwd (MXFP8) with the given chunk_rows: out and, with act, the
    kept h, u store."""
    shape = m.shape_of(cfg, chunk_rows=chunk)
    ws = torch.empty(m.workspace_bytes(shape, m.OP_FWD), dtype=torch.uint8, device=DEV)
    out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    saved = alloc_plan(cfg, DEV)
    if act:
        saved["act"] = torch.full((cfg.R, 2 * cfg.I), float("nan"), device=DEV)
    m.moe_fwd(shape, m.make_weights(d), d["x"], d["s"], out, ws, m.make_plan_buf(saved))
    m.check_device_status()
    return out, saved.get("act")


RING_REUSE_MX = W.MoEConfig("ring_reuse_mx", T=1024, D=256, I=128, E=16, K=4, I_shared=128, dtype="mxfp8")


@pytest.mark.parametrize("name,chunk", [("tiny", 512), ("ragged", 512), ("skew_small", 2048), ("big_experts", 512),
                                        ("ring_reuse", 512), ("ring_reuse", 32768)])
def test_moe_fwd_mxfp8_ring_bitexact(m, name, chunk):
    """The quantising dispatch fused into the up/gate as a ring (producer
    warps quantise routed rows into 4 slots of chunk rows, reused when R >
    4 chunks) gives the whole-batch dispatch's out and kept h, u bit for
    bit, and the oracle within tolerance."""
    cfg = RING_REUSE_MX if name == "ring_reuse" else SMALL[name].replace(dtype="mxfp8")
    inp = W.make_inputs(cfg, "cpu")
    d = mx_weights(m, {k: v.to(DEV) for k, v in inp.items()})
    out0, act0 = _mx_fwd_chunk(m, cfg, d, -1, act=True)
    for _ in range(2):  # the counters start from zero on every call
        out1, act1 = _mx_fwd_chunk(m, cfg, d, chunk, act=True)
        assert torch.equal(out0.view(torch.int16), out1.view(torch.int16))
        assert torch.equal(act0.view(torch.int32), act1.view(torch.int32))
    ref = O.moe_forward_mxfp8(host(inp), cfg.K)
    assert_close(out1.float().cpu().numpy(), ref["out"], MXFP8_TOL, f"mxfp8 ring out [{name}]")


def test_moe_fwd_mxfp8_ring_full_size_bitexact(m):
    """DSV3 MXFP8 forward: the ring of 512- and 2048-row chunks gives the
    whole-batch quantising dispatch's output bit for bit."""
    cfg = W.CONFIGS["dsv3_mxfp8_fwd"]
    d = mx_weights(m, W.make_inputs(cfg, DEV))
    out0, _ = _mx_fwd_chunk(m, cfg, d, -1)
    for chunk in (512, 2048):
        out1, _ = _mx_fwd_chunk(m, cfg, d, chunk)
        assert torch.equal(out0.view(torch.int16), out1.view(torch.int16))


# ---------------------------------------------------------------- backward
BWD = {
    "ragged": W.MoEConfig("ragged_bwd", T=300, D=512, I=256, E=5, K=3, I_shared=128, dtype="mxfp8"),
    # empty experts, a hot expert and ragged expert ends
    "skew": W.MoEConfig("skew_bwd", T=700, D=512, I=256, E=32, K=4, I_shared=256, skew=2.0, dtype="mxfp8"),
    "one_token": W.MoEConfig("one_token_bwd", T=1, D=256, I=256, E=8, K=2, I_shared=256, dtype="mxfp8"),
    # the largest E and K the boundary accepts: most experts empty
    "max_e_k": W.MoEConfig("max_e_k_bwd", T=40, D=256, I=256, E=1024, K=32, I_shared=0, dtype="mxfp8"),
    # experts of 512 or more routed rows on average: t and dX in the
    # row-major form (t with its fp32 outputs on stages of two K blocks)
    "big_experts": W.MoEConfig("big_experts_bwd", T=1100, D=256, I=256, E=2, K=1, I_shared=256, dtype="mxfp8"),
}


def bwd_weights(m, cfg, d, pair=False):
    """The forward's MXFP8 copies plus the backward's (W_down^T along D,
    [W_gate^T | W_up^T] along 2I) from mok_quantize_mxfp8_bwd_weights."""
    out = mx_weights(m, d, pair=pair)
    E, I, D = cfg.E, cfg.I, cfg.D
    out["qt_down"] = torch.empty(E * I, D, dtype=torch.uint8, device=DEV)
    out["sct_down"] = torch.empty(m.mx_scale_words(E * I, D), dtype=torch.int32, device=DEV)
    out["qt_gu"] = torch.empty(E * D, 2 * I, dtype=torch.uint8, device=DEV)
    out["sct_gu"] = torch.empty(m.mx_scale_words(E * D, 2 * I), dtype=torch.int32, device=DEV)
    m.quantize_mxfp8_bwd_weights(m.shape_of(cfg), m.make_weights(out), out["qt_down"], out["sct_down"],
                                 out["qt_gu"], out["sct_gu"])
    return out


def test_bwd_weight_copies_bitexact(m):
    cfg = BWD["ragged"]
    inp = W.make_inputs(cfg, "cpu")
    h = host(inp)
    d = bwd_weights(m, cfg, {k: v.to(DEV) for k, v in inp.items()})
    E, I, D = cfg.E, cfg.I, cfg.D
    wd_t = O.bf16_to_f32(h["w_down"]).transpose(0, 2, 1).reshape(E * I, D)
    q, sc = O.mxfp8_quantize(wd_t)
    assert np.array_equal(d["qt_down"].cpu().numpy(), q)
    assert np.array_equal(words_to_bytes(d["sct_down"], E * I, D), sc)
    wgu_t = np.concatenate([O.bf16_to_f32(h["w_gate"]).transpose(0, 2, 1),
                            O.bf16_to_f32(h["w_up"]).transpose(0, 2, 1)], axis=2).reshape(E * D, 2 * I)
    q, sc = O.mxfp8_quantize(wgu_t)
    assert np.array_equal(d["qt_gu"].cpu().numpy(), q)
    assert np.array_equal(words_to_bytes(d["sct_gu"], E * D, 2 * I), sc)


def _mx_fwd_bwd(m, cfg, d, act_rows=None, bwd_shared_sms=0, act_shared=False):
    shape = m.shape_of(cfg, bwd_shared_sms=bwd_shared_sms)
    w = m.make_weights(d)
    ws = torch.empty(max(m.workspace_bytes(shape, m.OP_FWD), m.workspace_bytes(shape, m.OP_BWD)),
                     dtype=torch.uint8, device=DEV)
    out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    saved = alloc_plan(cfg, DEV)
    if act_rows is not None:
        saved["act"] = torch.full((act_rows, 2 * cfg.I), float("nan"), dtype=torch.float32, device=DEV)
    if act_shared and cfg.I_shared:
        saved["act_shared"] = torch.full((cfg.T, 2 * cfg.I_shared), float("nan"), dtype=torch.float32, device=DEV)
    pb = m.make_plan_buf(saved)
    m.moe_fwd(shape, w, d["x"], d["s"], out, ws, pb)
    bf = torch.bfloat16
    T, D, I, E, K, Is = cfg.T, cfg.D, cfg.I, cfg.E, cfg.K, cfg.I_shared
    g = dict(dx=torch.empty(T, D, dtype=bf, device=DEV), dw_gate=torch.empty(E, I, D, dtype=bf, device=DEV),
             dw_up=torch.empty(E, I, D, dtype=bf, device=DEV), dw_down=torch.empty(E, D, I, dtype=bf, device=DEV),
             dws_gate=torch.empty(Is, D, dtype=bf, device=DEV), dws_up=torch.empty(Is, D, dtype=bf, device=DEV),
             dws_down=torch.empty(D, Is, dtype=bf, device=DEV), ds=torch.empty(T, E, device=DEV),
             dg=torch.empty(T, K, device=DEV))
    for v in g.values():
        v.fill_(float("nan"))
    m.moe_bwd(shape, w, d["x"], d["s"], pb, d["dy"], g["dx"], g["dw_gate"], g["dw_up"], g["dw_down"],
              g["dws_gate"], g["dws_up"], g["dws_down"], g["ds"], g["dg"], ws)
    m.check_device_status()
    return g


@pytest.mark.parametrize("name", list(BWD))
def test_backward_mxfp8_elementwise_and_deterministic(m, name):
    cfg = BWD[name]
    inp = W.make_inputs(cfg, "cpu", with_dy=True)
    h = host(inp)
    d = bwd_weights(m, cfg, {k: v.to(DEV) for k, v in inp.items()})
    got = _mx_fwd_bwd(m, cfg, d)
    ref = O.moe_backward_mxfp8(h, h["dy"], cfg.K, ranges=True)
    f = lambda t: t.float().cpu().numpy()
    for k, r in (("dx", "dX"), ("dg", "dg"), ("ds", "ds")):
        assert_close(f(got[k]), ref[r], MXFP8_TOL, f"mxfp8 bwd {r} [{name}]")
    pairs = [("dw_gate", "dW_gate"), ("dw_up", "dW_up"), ("dw_down", "dW_down")]
    if cfg.I_shared:
        pairs += [("dws_gate", "dWs_gate"), ("dws_up", "dWs_up"), ("dws_down", "dWs_down")]
    for k, r in pairs:
        assert_close_ranged(f(got[k]), ref[r], ref["range"][r], MXFP8_TOL, f"mxfp8 bwd {r} [{name}]")
    if name == "skew":
        empty = np.flatnonzero(np.bincount(O.route(h["s"], cfg.K)[0].reshape(-1), minlength=cfg.E) == 0)
        assert len(empty) > 0 and torch.all(got["dw_gate"][torch.from_numpy(empty).to(DEV)] == 0)
    again = _mx_fwd_bwd(m, cfg, d)
    for k, v in got.items():
        bits = (lambda t: t.view(torch.int16)) if v.dtype == torch.bfloat16 else (lambda t: t.view(torch.int32))
        assert torch.equal(bits(v), bits(again[k])), k



@pytest.mark.parametrize("name", ["ragged", "skew"])
def test_backward_mxfp8_kept_activations(m, name):
    """MXFP8: the forward keeps h, u (fp32, from its block-scaled up/gate) of
    the experts that fit; the backward replays only the others.  Every
    capacity, with or without the shared expert's store, gives the
    all-replay path's bytes."""
    cfg = BWD[name]
    inp = W.make_inputs(cfg, "cpu", with_dy=True)
    d = bwd_weights(m, cfg, {k: v.to(DEV) for k, v in inp.items()})
    base = _mx_fwd_bwd(m, cfg, d)
    for rows, keep_shared in ((cfg.R, True), (cfg.R, False), (cfg.R // 2, True)):
        got = _mx_fwd_bwd(m, cfg, d, act_rows=rows, act_shared=keep_shared)
        for k, v in base.items():
            bits = (lambda t: t.view(torch.int16)) if v.dtype == torch.bfloat16 else (lambda t: t.view(torch.int32))
            assert torch.equal(bits(v), bits(got[k])), (rows, k)


def test_backward_mxfp8_full_size_sampled(m):
    """The DSV3 fwd+bwd layer (T 4096, 256 experts) with MXFP8 routed experts:
    dX, dg and ds of 512 seeded tokens, and whole weight gradients of four
    experts (the fullest, the emptiest and two seeded ones), each from the
    oracle's MXFP8 backward of those rows.  The oracle quantises every
    touched expert's weights, so the calls run on a thread pool."""
    from concurrent.futures import ThreadPoolExecutor
    cfg = W.CONFIGS["dsv3_mxfp8_fwdbwd"]
    d = bwd_weights(m, cfg, W.make_inputs(cfg, DEV))
    got = _mx_fwd_bwd(m, cfg, d)
    s_host = d["s"].cpu().numpy()
    idx, g, den = O.route(s_host, cfg.K)
    counts, offsets, table, _ = O.plan(idx, cfg.E)
    f = lambda t: t.float().cpu().numpy()
    hw = device_weights_fetch(d)
    x_all = W.bf16_bits(d["x"])
    dy_all = W.bf16_bits(d["dy"])
    toks = sample_tokens(cfg.T, 512, seed=2)
    sel = torch.from_numpy(toks).to(DEV)
    with ThreadPoolExecutor(max_workers=16) as pool:
        ref = O.moe_backward_tokens(x_all[toks], dy_all[toks], s_host[toks], hw, cfg.K, mxfp8=True,
                                    map_fn=pool.map)
        assert_close(f(got["dx"][sel]), ref["dX"], MXFP8_TOL, "mxfp8 bwd dX [full]")
        assert_close(f(got["dg"][sel]), ref["dg"], MXFP8_TOL, "mxfp8 bwd dg [full]")
        assert_close(f(got["ds"][sel]), ref["ds"], MXFP8_TOL, "mxfp8 bwd ds [full]")
        experts = sample_experts(counts, 4, seed=4)

        def expert_grads(e):
            p0, p1 = int(offsets[e]), int(offsets[e + 1])
            if p0 == p1:
                return None
            toks_e = table[p0:p1, 0] // cfg.K
            gr = g[toks_e, table[p0:p1, 0] % cfg.K]
            b = O.route_backward_rows_mxfp8(x_all[toks_e], dy_all[toks_e], gr, *hw.fetch(e), ranges=True)
            X = O.bf16_to_f32(x_all[toks_e])
            dY = O.bf16_to_f32(dy_all[toks_e])
            rg = b["ranges"]
            lo, hi = O.sum_range(b["a_g"], rg["a_g"], dY)
            return {"dW_down": (O.round_bf16(dY.T @ b["a_g"]), (lo.T, hi.T)),
                    "dW_gate": (O.round_bf16(b["dh"].T @ X), O.sum_range(b["dh"], rg["dh"], X)),
                    "dW_up": (O.round_bf16(b["du"].T @ X), O.sum_range(b["du"], rg["du"], X))}

        for e, res in zip(experts, pool.map(expert_grads, experts)):
            if counts[e] == 0:
                assert torch.all(got["dw_down"][e] == 0) and torch.all(got["dw_gate"][e] == 0)
                continue
            for k, r in (("dw_down", "dW_down"), ("dw_gate", "dW_gate"), ("dw_up", "dW_up")):
                assert_close_ranged(f(got[k][e]), res[r][0], res[r][1], MXFP8_TOL, f"mxfp8 bwd {r} [full, expert {e}]")


@pytest.mark.parametrize("name", ["ragged", "skew"])
def test_backward_mxfp8_grid_inputs_bare_tolerance(m, name):
    """MXFP8 on grid inputs (x, dY, weights exact in E4M3 at their block
    scales; exact fp32 product sums): every output within 6e-2 * max(1,
    |oracle|) with no other allowance."""
    cfg = BWD[name].replace(values="grid")
    inp = W.make_inputs(cfg, "cpu", with_dy=True)
    h = host(inp)
    d = bwd_weights(m, cfg, {k: v.to(DEV) for k, v in inp.items()})
    got = _mx_fwd_bwd(m, cfg, d, act_rows=cfg.R)
    ref = O.moe_backward_mxfp8(h, h["dy"], cfg.K)
    f = lambda t: t.float().cpu().numpy()
    pairs = [("dx", "dX"), ("dg", "dg"), ("ds", "ds"), ("dw_gate", "dW_gate"), ("dw_up", "dW_up"),
             ("dw_down", "dW_down"), ("dws_gate", "dWs_gate"), ("dws_up", "dWs_up"), ("dws_down", "dWs_down")]
    for k, r in pairs:
        assert_close(f(got[k]), ref[r], MXFP8_TOL, f"mxfp8 bwd grid {r} [{name}]")


def test_pair_scales_are_the_permutation():
    """mok_mxfp8_pair_scales: block b = e (I/64) + s of the paired copy holds
    the scale words of W_up rows e I + 64 s .. + 63, then of the same W_gate
    rows, in the 128-row block order (row 32 c + l at word 4 l + c)."""
    m = mok()
    cfg = BWD["ragged"]
    d = mx_weights(m, {k: v.to(DEV) for k, v in W.make_inputs(cfg, "cpu").items()}, pair=True)
    E, I, D = cfg.E, cfg.I, cfg.D
    pos = lambda r: (r & ~127) | ((r & 31) << 2) | ((r >> 5) & 3)
    sg = d["sc_gate"].cpu().numpy().reshape(D // 128, -1)
    su = d["sc_up"].cpu().numpy().reshape(D // 128, -1)
    sp = d["sc_gu_pair"].cpu().numpy().reshape(D // 128, -1)
    v = np.arange(2 * E * I)
    b, mm = v >> 7, v & 127
    r = (b // (I // 64)) * I + 64 * (b % (I // 64)) + (mm & 63)
    want = np.where(mm[None, :] < 64, su[:, pos(r)], sg[:, pos(r)])
    assert np.array_equal(sp[:, pos(v)], want)


@pytest.mark.parametrize("name", ["tiny", "ragged", "skew_small", "dsv3_mxfp8_fwd", "dsv3_mxfp8_fwdbwd"])
def test_upgate_routed_rows_as_n_bitexact(m, name):
    """The MXFP8 up/gate with the routed rows as N (paired scales) gives the
    row-major kernel's bytes: a codes, a scale words, y and the forward's
    out; on the fwd+bwd layer also the kept h, u and every gradient."""
    if name in CONFIG_NAMES:
        cfg = W.CONFIGS[name]
        inp = W.make_inputs(cfg, DEV)
    else:
        cfg = SMALL[name].replace(dtype="mxfp8")
        inp = {k: v.to(DEV) for k, v in W.make_inputs(cfg, "cpu").items()}
    dp = mx_weights(m, inp, pair=True)
    dr = mx_weights(m, inp, pair=False)
    shape = m.shape_of(cfg)
    res = []
    for d in (dp, dr):
        ws = torch.zeros(m.workspace_bytes(shape, m.OP_FWD), dtype=torch.uint8, device=DEV)
        out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
        saved = alloc_plan(cfg, DEV)
        saved["act"] = torch.zeros(cfg.R, 2 * cfg.I, dtype=torch.float32, device=DEV)
        m.moe_fwd(shape, m.make_weights(d), inp["x"], inp["s"], out, ws, m.make_plan_buf(saved))
        m.check_device_status()
        res.append((out, saved["act"], ws))
    assert torch.equal(res[0][0].view(torch.int16), res[1][0].view(torch.int16)), "out"
    assert torch.equal(res[0][1].view(torch.int32), res[1][1].view(torch.int32)), "kept h, u"
    assert torch.equal(res[0][2], res[1][2]), "workspace (a codes, a scales, y)"
    if cfg.backward:
        dp = bwd_weights(m, cfg, inp, pair=True)
        dr = dict(dp)
        del dr["sc_gu_pair"]
        gp = _mx_fwd_bwd(m, cfg, dp, act_rows=cfg.R)
        gr = _mx_fwd_bwd(m, cfg, dr, act_rows=cfg.R)
        for k, v in gp.items():
            bits = (lambda t: t.view(torch.int16)) if v.dtype == torch.bfloat16 else (lambda t: t.view(torch.int32))
            assert torch.equal(bits(v), bits(gr[k])), k


CONFIG_NAMES = ("dsv3_mxfp8_fwd", "dsv3_mxfp8_fwdbwd")


@pytest.mark.parametrize("name", ["ragged", "skew"])
def test_backward_mxfp8_shared_side_stream_is_bitexact(m, name):
    """The MXFP8 backward with the shared expert's backward on a side stream
    (t, the activation gradient and dX of the routed experts on the other
    SMs) gives the single-stream bits."""
    cfg = BWD[name]
    inp = W.make_inputs(cfg, "cpu", with_dy=True)
    d = bwd_weights(m, cfg, {k: v.to(DEV) for k, v in inp.items()})
    base = _mx_fwd_bwd(m, cfg, d, act_rows=cfg.R)
    for k in (10, 40):
        got = _mx_fwd_bwd(m, cfg, d, act_rows=cfg.R, bwd_shared_sms=k)
        for key, v in base.items():
            bits = (lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32))
            assert torch.equal(bits(v), bits(got[key])), (k, key)
