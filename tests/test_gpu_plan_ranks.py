"""GPU parity of the pull schedule with several virtual source ranks
(mok_plan_ranks) against the oracle's general schedule, bit for bit, and the
layer's output unchanged by the row order it produces."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import host, mok
from routing_grouped_expert_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def m():
    return mok()


def _plan_ranks(m, topk, E, ranks):
    T, K = topk.shape
    R = T * K
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    table = torch.empty(max(R, 1), 3, dtype=torch.int32, device=DEV)
    route_dst = torch.empty(max(R, 1), dtype=torch.int32, device=DEV)
    ws = torch.empty(m.plan_ranks_workspace_bytes(T, E, K, ranks), dtype=torch.uint8, device=DEV)
    m.plan_ranks(torch.from_numpy(topk).to(DEV), E, ranks, counts, offsets, table, route_dst, ws)
    m.check_device_status()
    return counts.cpu().numpy(), offsets.cpu().numpy(), table.cpu().numpy()[:R], route_dst.cpu().numpy()[:R]


@pytest.mark.parametrize("T,E,K,ranks,skew", [(256, 8, 2, 4, 0.0), (300, 5, 3, 3, 0.0), (512, 64, 8, 8, 2.0),
                                              (1024, 256, 8, 64, 0.0), (7168, 256, 8, 8, 0.0), (64, 4, 4, 64, 0.0)])
def test_plan_ranks_matches_oracle_schedule(m, T, E, K, ranks, skew):
    cfg = W.MoEConfig("p", T=T, D=256, I=128, E=E, K=K, I_shared=0, skew=skew)
    s = W.make_inputs(cfg, "cpu")["s"].numpy()
    topk, _, _ = O.route(s, K)
    counts, offsets, table, route_dst = _plan_ranks(m, topk, E, ranks)
    N = T // ranks
    Tc, M, S, Phi = O.pull_schedule(topk.reshape(ranks, N, K), c=0, L=E)
    assert np.array_equal(counts, Tc)
    assert np.array_equal(offsets[:E], S) and offsets[E] == T * K
    # Phi holds (source rank, i*K + k); the global route id is (r*N + i)*K + k
    src = Phi[:, 0] * N * K + Phi[:, 1]
    assert np.array_equal(table[:, 0], src)
    assert np.array_equal(table[:, 1], topk.reshape(-1)[src])
    assert np.array_equal(table[:, 2], np.arange(T * K))
    assert np.array_equal(route_dst[src], np.arange(T * K))


def test_plan_ranks_one_rank_is_plan_and_layer_output_is_order_free(m):
    cfg = W.MoEConfig("p", T=512, D=256, I=128, E=16, K=4, I_shared=0)
    inp = W.make_inputs(cfg, "cpu")
    topk, g, _ = O.route(inp["s"].numpy(), cfg.K)
    _, _, table1, rd1 = _plan_ranks(m, topk, cfg.E, 1)
    _, _, tref, rdref = O.plan(topk, cfg.E)
    assert np.array_equal(table1, tref) and np.array_equal(rd1, rdref)
    # the layer through the split entry points with an 8-rank schedule gives
    # the one-rank output bit for bit (each row's FFN is independent of order)
    d = {k: v.to(DEV) for k, v in inp.items()}
    shape = m.shape_of(cfg)
    w = m.make_weights(d)
    outs = []
    for ranks in (1, 8):
        counts, offsets, table, route_dst = _plan_ranks(m, topk, cfg.E, ranks)
        tab = torch.from_numpy(table).to(DEV)
        off = torch.from_numpy(offsets).to(DEV)
        xg = torch.empty(cfg.R, cfg.D, dtype=torch.bfloat16, device=DEV)
        m.dispatch(shape, d["x"], tab, torch.from_numpy(route_dst).to(DEV), xg)
        yg = torch.empty(cfg.R, cfg.D, dtype=torch.bfloat16, device=DEV)
        fws = torch.empty(m.workspace_bytes(shape, m.OP_EXPERT_FFN), dtype=torch.uint8, device=DEV)
        m.expert_ffn(shape, w, xg, off, yg, ws=fws)
        out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
        m.combine(shape, yg, None, torch.from_numpy(g.astype(np.float32)).to(DEV),
                  torch.from_numpy(route_dst).to(DEV), out)
        m.check_device_status()
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
