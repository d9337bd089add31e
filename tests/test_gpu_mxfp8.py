"""GPU parity of the MXFP8 path (E4M3 codes, E8M0 1x32 scales) against the oracle.

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
from helpers import MXFP8_TOL, alloc_plan, assert_close, host, mok
from routing_grouped_expert_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")

SMALL = {
    "tiny": W.CONFIGS["tiny"],
    "ragged": W.MoEConfig("ragged", T=301, D=512, I=256, E=5, K=3, I_shared=128, dtype="mxfp8"),
    "skew_small": W.MoEConfig("skew_small", T=700, D=256, I=128, E=16, K=4, I_shared=0, skew=2.0,
                              dtype="mxfp8"),
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


def mx_weights(m, d):
    out = dict(d)
    E, I, D = d["w_gate"].shape
    for name, key in (("gate", "w_gate"), ("up", "w_up"), ("down", "w_down")):
        w = d[key]
        q, sc = quantize(m, w.reshape(-1, w.shape[-1]))
        out["q_" + name], out["sc_" + name] = q, sc
    return out


def test_quantize_bitexact(m):
    gen = torch.Generator().manual_seed(9)
    v = (torch.randn(301, 512, generator=gen) * torch.logspace(-3, 3, 512)).to(torch.bfloat16)
    v[5, :32] = 0
    v[6, 64:96] = -0.0
    q, sc = quantize(m, v.to(DEV))
    qr, sr = O.mxfp8_quantize(O.bf16_to_f32(W.bf16_bits(v)))
    assert np.array_equal(words_to_bytes(sc, 301, 512), sr)
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
    assert_close(outs[0].float().cpu().numpy(), ref["out"], MXFP8_TOL, "out")
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
