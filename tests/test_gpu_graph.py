"""mok_moe_fwd captured in a CUDA graph (after one eager call on the device,
which creates the side stream) replays to the eager output bit for bit:
the side-stream fork/join, the ring's counter reset and cooperative launch,
and the MXFP8 path are all stream-ordered work without host syncs.  The
same holds for a forward + backward step (BF16 and MXFP8) in one graph."""
import numpy as np
import pytest
import torch

from helpers import mok
from routing_grouped_expert_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def m():
    return mok()


def _mx(m, d):
    d = dict(d)
    for name, key in (("gate", "w_gate"), ("up", "w_up"), ("down", "w_down")):
        wt = d[key].reshape(-1, d[key].shape[-1])
        q = torch.empty(wt.shape, dtype=torch.uint8, device=DEV)
        sc = torch.empty(m.mx_scale_words(*wt.shape), dtype=torch.int32, device=DEV)
        m.quantize_mxfp8(wt, q, sc)
        d["q_" + name], d["sc_" + name] = q, sc
    return d


@pytest.mark.parametrize("dtype,chunk", [(None, 0), (None, 512), ("mxfp8", 0), ("mxfp8", 512)])
def test_moe_fwd_graph_replay_matches_eager(m, dtype, chunk):
    cfg = W.MoEConfig("g", T=700, D=512, I=256, E=16, K=4, I_shared=256)
    d = {k: v.to(DEV) for k, v in W.make_inputs(cfg, "cpu").items()}
    if dtype == "mxfp8":
        d = _mx(m, d)
    shape = m.shape_of(cfg, dtype=dtype, chunk_rows=chunk)
    w = m.make_weights(d)
    ws = torch.empty(m.workspace_bytes(shape, m.OP_FWD), dtype=torch.uint8, device=DEV)
    eager = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    m.moe_fwd(shape, w, d["x"], d["s"], eager, ws)
    m.check_device_status()
    out = torch.empty_like(eager)
    s_in = d["s"].clone()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            m.moe_fwd(shape, w, d["x"], s_in, out, ws, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    m.check_device_status()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    # new inputs in the captured buffers flow through the replay
    s_in.copy_(torch.softmax(torch.randn(cfg.T, cfg.E, device=DEV), dim=1))
    g.replay()
    ref = torch.empty_like(eager)
    m.moe_fwd(shape, w, d["x"], s_in, ref, ws)
    torch.cuda.synchronize()
    m.check_device_status()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def _mx_bwd(m, cfg, d):
    d = _mx(m, d)
    E, I, D = cfg.E, cfg.I, cfg.D
    d["qt_down"] = torch.empty(E * I, D, dtype=torch.uint8, device=DEV)
    d["sct_down"] = torch.empty(m.mx_scale_words(E * I, D), dtype=torch.int32, device=DEV)
    d["qt_gu"] = torch.empty(E * D, 2 * I, dtype=torch.uint8, device=DEV)
    d["sct_gu"] = torch.empty(m.mx_scale_words(E * D, 2 * I), dtype=torch.int32, device=DEV)
    m.quantize_mxfp8_bwd_weights(m.shape_of(cfg), m.make_weights(d), d["qt_down"], d["sct_down"], d["qt_gu"],
                                 d["sct_gu"])
    return d


@pytest.mark.parametrize("dtype", [None, "mxfp8"])
def test_moe_fwd_bwd_graph_replay_matches_eager(m, dtype):
    """mok_moe_fwd + mok_moe_bwd in one captured graph: the replayed
    gradients equal the eager ones bit for bit."""
    cfg = W.MoEConfig("gb", T=700, D=512, I=256, E=16, K=4, I_shared=256)
    d = {k: v.to(DEV) for k, v in W.make_inputs(cfg, "cpu", with_dy=True).items()}
    if dtype == "mxfp8":
        d = _mx_bwd(m, cfg, d)
    shape = m.shape_of(cfg, dtype=dtype)
    w = m.make_weights(d)
    ws = torch.empty(max(m.workspace_bytes(shape, m.OP_FWD), m.workspace_bytes(shape, m.OP_BWD)),
                     dtype=torch.uint8, device=DEV)
    T, D, I, E, K, Is = cfg.T, cfg.D, cfg.I, cfg.E, cfg.K, cfg.I_shared
    bf = torch.bfloat16

    def buffers():
        saved = dict(topk_idx=torch.empty(T, K, dtype=torch.int32, device=DEV),
                     g=torch.empty(T, K, device=DEV), counts=torch.empty(E, dtype=torch.int32, device=DEV),
                     offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV),
                     table=torch.empty(T * K, 3, dtype=torch.int32, device=DEV),
                     route_dst=torch.empty(T * K, dtype=torch.int32, device=DEV))
        g = dict(out=torch.empty(T, D, dtype=bf, device=DEV), dx=torch.empty(T, D, dtype=bf, device=DEV),
                 dw_gate=torch.empty(E, I, D, dtype=bf, device=DEV), dw_up=torch.empty(E, I, D, dtype=bf, device=DEV),
                 dw_down=torch.empty(E, D, I, dtype=bf, device=DEV), dws_gate=torch.empty(Is, D, dtype=bf, device=DEV),
                 dws_up=torch.empty(Is, D, dtype=bf, device=DEV), dws_down=torch.empty(D, Is, dtype=bf, device=DEV),
                 ds=torch.empty(T, E, device=DEV), dg=torch.empty(T, K, device=DEV))
        return saved, g

    def run(saved, g, stream=None):
        pb = m.make_plan_buf(saved)
        m.moe_fwd(shape, w, d["x"], d["s"], g["out"], ws, pb, stream=stream)
        m.moe_bwd(shape, w, d["x"], d["s"], pb, d["dy"], g["dx"], g["dw_gate"], g["dw_up"], g["dw_down"],
                  g["dws_gate"], g["dws_up"], g["dws_down"], g["ds"], g["dg"], ws, stream=stream)

    es, eg = buffers()
    run(es, eg)
    torch.cuda.synchronize()
    m.check_device_status()
    gs, gg = buffers()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            run(gs, gg, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        for v in gg.values():
            v.zero_()
        graph.replay()
    torch.cuda.synchronize()
    m.check_device_status()
    for k, v in eg.items():
        bits = (lambda t: t.view(torch.int16)) if v.dtype == bf else (lambda t: t.view(torch.int32))
        assert torch.equal(bits(gg[k]), bits(v)), k
