"""GPU parity of mok_router: s = softmax(x W_r^T) against the oracle, and the
top-K / g taken from it bit-exactly equal to the oracle's route on the same s.

s tolerance: |s_gpu - s_oracle| <= 2e-4 * s_oracle + 1e-9.  The logits differ
only in fp32 summation order (tensor cores vs numpy), the softmax uses the
fast exponential (a few ulp), so the expected error is below 1e-5 relative.
"""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import mok
from routing_grouped_expert_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
CASES = {
    "tiny": W.CONFIGS["tiny"],
    "ragged_e5": W.MoEConfig("ragged_e5", T=300, D=512, I=256, E=5, K=3, I_shared=0),
    "e16": W.MoEConfig("e16", T=700, D=256, I=128, E=16, K=4, I_shared=0),
    "e256": W.MoEConfig("e256", T=1000, D=1024, I=128, E=256, K=8, I_shared=0),
}


@pytest.fixture(scope="module")
def m():
    return mok()


def _run(m, cfg, x, w):
    s = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=DEV)
    topk = torch.empty(cfg.T, cfg.K, dtype=torch.int32, device=DEV)
    g = torch.empty(cfg.T, cfg.K, dtype=torch.float32, device=DEV)
    m.router(m.shape_of(cfg), x, w, s, topk, g)
    m.check_device_status()
    return s.cpu().numpy(), topk.cpu().numpy(), g.cpu().numpy()


def _check(s_gpu, topk, g, s_ref, K):
    assert np.all(np.abs(s_gpu - s_ref) <= 2e-4 * s_ref + 1e-9)
    idx, gr, _ = O.route(s_gpu, K)
    assert np.array_equal(topk, idx)
    assert np.array_equal(g.view(np.uint32), gr.astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("name", list(CASES))
def test_router_scores_and_route(m, name):
    cfg = CASES[name]
    x = W.make_inputs(cfg, "cpu")["x"]
    w = W.make_router_weights(cfg)
    s_gpu, topk, g = _run(m, cfg, x.to(DEV), w.to(DEV))
    _, s_ref = O.router_scores(W.bf16_bits(x), W.bf16_bits(w))
    _check(s_gpu, topk, g, s_ref, cfg.K)
    # deterministic
    s2, topk2, _ = _run(m, cfg, x.to(DEV), w.to(DEV))
    assert np.array_equal(s_gpu.view(np.uint32), s2.view(np.uint32)) and np.array_equal(topk, topk2)


def test_router_full_size_sampled_rows(m):
    """DSV3 shapes (T 7168, D 7168, E 256): every route bit-exact on the GPU's
    s, s checked against the oracle on 512 seeded rows."""
    cfg = W.CONFIGS["dsv3_bf16_fwd"]
    x = W.make_inputs(cfg, DEV)["x"]
    w = W.make_router_weights(cfg, DEV)
    s_gpu, topk, g = _run(m, cfg, x, w)
    rows = np.sort(np.random.default_rng(11).choice(cfg.T, 512, replace=False))
    _, s_ref = O.router_scores(W.bf16_bits(x[torch.from_numpy(rows).to(DEV)]), W.bf16_bits(w))
    assert np.all(np.abs(s_gpu[rows] - s_ref) <= 2e-4 * s_ref + 1e-9)
    idx, gr, _ = O.route(s_gpu, cfg.K)
    assert np.array_equal(topk, idx)
    assert np.array_equal(g.view(np.uint32), gr.astype(np.float32).view(np.uint32))


def test_router_rejects_more_than_256_experts(m):
    cfg = W.MoEConfig("e512", T=64, D=256, I=128, E=512, K=8, I_shared=0)
    with pytest.raises(m.MokError):
        _run(m, cfg, torch.zeros(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV),
             torch.zeros(cfg.E, cfg.D, dtype=torch.bfloat16, device=DEV))
