"""Degenerate and maximum shapes through the C ABI against the oracle: one
token, every expert selected (K = E), the largest E and K the API accepts,
a ring chunk larger than all routed rows, MXFP8 and the router at T = 1."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import BF16_TOL, MXFP8_TOL, alloc_plan, assert_close, host, mok
from routing_grouped_expert_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")

SHAPES = {
    "one_token": W.MoEConfig("one_token", T=1, D=256, I=128, E=8, K=2, I_shared=128),
    "one_token_one_expert": W.MoEConfig("one_token_one_expert", T=1, D=256, I=128, E=1, K=1, I_shared=0),
    "k_equals_e": W.MoEConfig("k_equals_e", T=65, D=256, I=128, E=8, K=8, I_shared=128),
    "max_e_k": W.MoEConfig("max_e_k", T=40, D=256, I=128, E=1024, K=32, I_shared=0),
}


@pytest.fixture(scope="module")
def m():
    return mok()


def _fwd(m, cfg, d, chunk=0, dtype=None):
    shape = m.shape_of(cfg, dtype=dtype, chunk_rows=chunk)
    ws = torch.empty(max(1, m.workspace_bytes(shape, m.OP_FWD)), dtype=torch.uint8, device=DEV)
    out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    saved = alloc_plan(cfg, DEV)
    m.moe_fwd(shape, m.make_weights(d), d["x"], d["s"], out, ws, m.make_plan_buf(saved))
    m.check_device_status()
    return out, saved


@pytest.mark.parametrize("name", list(SHAPES))
def test_degenerate_shapes_forward(m, name):
    cfg = SHAPES[name]
    inp = W.make_inputs(cfg, "cpu")
    ref = O.moe_forward(host(inp), cfg.K)
    d = {k: v.to(DEV) for k, v in inp.items()}
    out, saved = _fwd(m, cfg, d)
    assert np.array_equal(saved["topk_idx"].cpu().numpy(), ref["topk_idx"])
    assert np.array_equal(saved["table"].cpu().numpy(), ref["table"])
    assert np.array_equal(saved["offsets"].cpu().numpy(), ref["offsets"])
    assert_close(out.float().cpu().numpy(), ref["out"], BF16_TOL, "out")
    if cfg.K == cfg.E:  # every expert selected: g = s / sum(s) over all experts
        s = inp["s"].numpy()
        g = saved["g"].cpu().numpy()
        order = saved["topk_idx"].cpu().numpy()
        assert np.allclose(np.take_along_axis(s, order, axis=1) / s.sum(axis=1, keepdims=True), g, rtol=1e-6)


@pytest.mark.parametrize("name", ["one_token", "k_equals_e"])
def test_ring_chunk_larger_than_all_rows(m, name):
    cfg = SHAPES[name]
    inp = W.make_inputs(cfg, "cpu")
    d = {k: v.to(DEV) for k, v in inp.items()}
    out0, _ = _fwd(m, cfg, d, chunk=-1)
    out1, _ = _fwd(m, cfg, d, chunk=32768)
    assert torch.equal(out0.view(torch.int16), out1.view(torch.int16))


def test_mxfp8_one_token(m):
    cfg = SHAPES["one_token"].replace(dtype="mxfp8")
    inp = W.make_inputs(cfg, "cpu")
    d = {k: v.to(DEV) for k, v in inp.items()}
    for name, key in (("gate", "w_gate"), ("up", "w_up"), ("down", "w_down")):
        wt = d[key].reshape(-1, d[key].shape[-1])
        q = torch.empty(wt.shape, dtype=torch.uint8, device=DEV)
        sc = torch.empty(m.mx_scale_words(*wt.shape), dtype=torch.int32, device=DEV)
        m.quantize_mxfp8(wt, q, sc)
        d["q_" + name], d["sc_" + name] = q, sc
    out, _ = _fwd(m, cfg, d)
    ref = O.moe_forward_mxfp8(host(inp), cfg.K)
    assert_close(out.float().cpu().numpy(), ref["out"], MXFP8_TOL, "out")


def test_router_one_token(m):
    cfg = SHAPES["one_token"]
    x = W.make_inputs(cfg, "cpu")["x"]
    w = W.make_router_weights(cfg)
    s = torch.empty(1, cfg.E, dtype=torch.float32, device=DEV)
    topk = torch.empty(1, cfg.K, dtype=torch.int32, device=DEV)
    g = torch.empty(1, cfg.K, dtype=torch.float32, device=DEV)
    m.router(m.shape_of(cfg), x.to(DEV), w.to(DEV), s, topk, g)
    m.check_device_status()
    _, s_ref = O.router_scores(W.bf16_bits(x), W.bf16_bits(w))
    s_gpu = s.cpu().numpy()
    assert np.all(np.abs(s_gpu - s_ref) <= 2e-4 * s_ref + 1e-9)
    idx, gr, _ = O.route(s_gpu, cfg.K)
    assert np.array_equal(topk.cpu().numpy(), idx)
