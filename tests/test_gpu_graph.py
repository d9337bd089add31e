"""mok_moe_fwd captured in a CUDA graph (after one eager call on the device,
which creates the side stream) replays to the eager output bit for bit:
the side-stream fork/join, the ring's counter reset and cooperative launch,
and the MXFP8 path are all stream-ordered work without host syncs."""
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


@pytest.mark.parametrize("dtype,chunk", [(None, 0), (None, 512), ("mxfp8", 0)])
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
