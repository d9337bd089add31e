"""Pins of the oracle's router scores s = softmax(x W_r^T) against closed
forms, invariants and an independent library softmax."""
import numpy as np
import torch

import oracle as O
from routing_grouped_expert_device_gb300 import workloads as W


def _bits(a: np.ndarray) -> np.ndarray:
    return O.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def test_softmax_rows_sum_to_one_and_match_torch_fp64():
    rng = np.random.default_rng(3)
    logits = rng.normal(size=(64, 37)) * 3
    s64 = O.softmax_rows(logits, O.FP64_SHADOW)
    assert np.allclose(s64.sum(axis=1), 1.0, atol=1e-14)
    ref = torch.softmax(torch.from_numpy(logits), dim=1).numpy()
    assert np.allclose(s64, ref, rtol=1e-13, atol=1e-16)
    s32 = O.softmax_rows(logits.astype(np.float32), O.FP32)
    assert s32.dtype == np.float32
    assert np.all(np.abs(s32.sum(axis=1) - 1.0) < 4e-7 * 37)
    assert np.allclose(s32, ref, rtol=2e-6, atol=1e-9)


def test_softmax_closed_forms():
    # shift invariance
    rng = np.random.default_rng(4)
    l = rng.normal(size=(8, 5))
    assert np.allclose(O.softmax_rows(l, O.FP64_SHADOW), O.softmax_rows(l + 7.25, O.FP64_SHADOW), rtol=1e-14)
    # two experts: s0 = 1 / (1 + e^(l1 - l0)), the logistic function
    l2 = np.array([[0.3, -1.2], [5.0, 5.0], [-2.0, 1.0]])
    s = O.softmax_rows(l2, O.FP64_SHADOW)
    assert np.allclose(s[:, 0], 1.0 / (1.0 + np.exp(l2[:, 1] - l2[:, 0])), rtol=1e-15)
    # one expert: s = 1
    assert np.array_equal(O.softmax_rows(np.array([[-3.0], [9.0]]), O.FP64_SHADOW), np.ones((2, 1)))


def test_router_logits_one_hot_rows_pick_weight_columns_exactly():
    rng = np.random.default_rng(5)
    D, E = 64, 8
    w = (rng.normal(size=(E, D)) / 8).astype(np.float32)
    x = np.zeros((D, D), dtype=np.float32)
    x[np.arange(D), np.arange(D)] = 1.0
    logits, _ = O.router_scores(_bits(x), _bits(w))
    assert np.array_equal(logits, O.bf16_to_f32(_bits(w)).T)


def test_router_permuting_experts_permutes_scores():
    cfg = W.MoEConfig("r", T=16, D=256, I=128, E=12, K=2, I_shared=0)
    x = W.bf16_bits(W.make_inputs(cfg)["x"])
    w = W.bf16_bits(W.make_router_weights(cfg))
    perm = np.random.default_rng(6).permutation(cfg.E)
    _, s = O.router_scores(x, w, O.FP64_SHADOW)
    _, sp = O.router_scores(x, w[perm], O.FP64_SHADOW)
    assert np.allclose(sp, s[:, perm], rtol=1e-14)


def test_router_fp32_within_bound_of_fp64():
    cfg = W.MoEConfig("r", T=64, D=512, I=128, E=16, K=2, I_shared=0)
    x = W.bf16_bits(W.make_inputs(cfg)["x"])
    w = W.bf16_bits(W.make_router_weights(cfg))
    l32, s32 = O.router_scores(x, w)
    l64, s64 = O.router_scores(x, w, O.FP64_SHADOW)
    assert np.max(np.abs(l32 - l64)) < 1e-4
    assert np.max(np.abs(s32 - s64) / s64) < 1e-4
