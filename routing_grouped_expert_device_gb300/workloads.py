"""Seeded synthetic MoE-layer workloads.

This module only draws inputs: token activations x, expert weights, router
scores s and the upstream gradient dY.  It holds none of the layer's
arithmetic, so both the CUDA path and the CPU oracle can be fed the same bytes.

Distributions (Mixture-of-Kittens, "Overlapping computation and communication
in MoE": notation D, I, E, s; the layer benchmarks use standard-normal router
inputs):
  * x ~ N(0, 1), drawn in fp32 and rounded to bf16 (round-to-nearest-even);
  * every weight matrix ~ N(0, 1/fan_in) (std 1/sqrt(fan_in)), fan_in = D for
    W_gate/W_up and I (or I_shared) for W_down, rounded to bf16;
  * router logits ~ N(0, 1) in fp32, plus b_e = -2 ln(e+1) for the skewed
    workload; s = softmax(logits) over all E experts, kept in fp32;
  * dY ~ N(0, 1), rounded to bf16.

Draw order from one generator seeded with ``seed``: x, W_gate, W_up, W_down,
shared W_gate, shared W_up, shared W_down, logits, dY.  The router projection
W_r [E][D] ~ N(0, 1/D) (``make_router_weights``) comes from a second
generator seeded with ``seed + 7919``, so it leaves every tensor above as is;
with x ~ N(0, 1) its logits x W_r^T are again about N(0, 1).  Large tensors are drawn
in fixed-size slabs so that peak memory stays bounded; the slab size is part of
the recipe, so the bytes are a pure function of (config, seed, device).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    """One MoE layer shape.  T tokens, D model dim, I expert intermediate dim,
    E routed experts, K experts per token, I_shared shared-expert intermediate
    dim (0 = no shared expert)."""

    name: str
    T: int
    D: int
    I: int
    E: int
    K: int
    I_shared: int
    dtype: str = "bf16"          # "bf16" or "mxfp8" (routed experts)
    skew: float = 0.0            # logit bias b_e = -skew * ln(e + 1)
    backward: bool = False
    chunks: Tuple[int, ...] = ()
    # "normal": the distributions above.  "grid": x, dY and every weight are
    # small integers times a power of two (x, dY: j / 2; W_gate, W_up,
    # W_shared_gate/up: j 2^-8; W_down, W_shared_down: j 2^-7; j uniform in
    # -3..3: at D = 7168, I = 2048 standard deviations of 1 and 0.66-0.7 of
    # the normal weights'), so every product sum of the layer's GEMMs over D
    # or I is exact in fp32 whatever the summation order.
    values: str = "normal"

    @property
    def R(self) -> int:
        return self.T * self.K

    def fwd_flops(self) -> float:
        """Algorithmic forward FLOPs: 2*M*N*K for each of the three GEMMs of
        every route plus the shared expert over all tokens."""
        return 6.0 * self.R * self.D * self.I + 6.0 * self.T * self.D * self.I_shared

    def bwd_flops(self) -> float:
        """Algorithmic backward FLOPs: twice the forward (dgrad + wgrad),
        excluding the recomputation of h and u."""
        return 2.0 * self.fwd_flops()

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


CONFIGS: Dict[str, MoEConfig] = {
    "tiny": MoEConfig("tiny", T=256, D=256, I=128, E=8, K=2, I_shared=128),
    "dsv3_bf16_fwd": MoEConfig("dsv3_bf16_fwd", T=7168, D=7168, I=2048, E=256, K=8, I_shared=2048),
    "skewed_bf16_fwd": MoEConfig("skewed_bf16_fwd", T=16384, D=4096, I=1536, E=128, K=8, I_shared=0,
                                 skew=2.0, chunks=(512, 2048, 8192, 32768)),
    "dsv3_mxfp8_fwd": MoEConfig("dsv3_mxfp8_fwd", T=7168, D=7168, I=2048, E=256, K=8, I_shared=2048,
                                dtype="mxfp8"),
    # 1/8 of the DSV3 layer (32 experts, same rows per expert): a profiling
    # case for the same kernels that still exceeds L2
    "dsv3_slice_bf16_fwd": MoEConfig("dsv3_slice_bf16_fwd", T=896, D=7168, I=2048, E=32, K=8, I_shared=2048),
    # the same slice with MXFP8 expert GEMMs
    "dsv3_slice_mxfp8_fwd": MoEConfig("dsv3_slice_mxfp8_fwd", T=896, D=7168, I=2048, E=32, K=8, I_shared=2048,
                                      dtype="mxfp8"),
    # 1/8 of the fwd+bwd layer (32 experts, 128 rows per expert): a
    # profiling case for the backward kernels that still exceeds L2
    "dsv3_slice_bf16_fwdbwd": MoEConfig("dsv3_slice_bf16_fwdbwd", T=512, D=7168, I=2048, E=32, K=8,
                                        I_shared=2048, backward=True),
    "dsv3_bf16_fwdbwd": MoEConfig("dsv3_bf16_fwdbwd", T=4096, D=7168, I=2048, E=256, K=8, I_shared=2048,
                                  backward=True),
    # the same layer with the routed experts in MXFP8, forward and backward
    "dsv3_mxfp8_fwdbwd": MoEConfig("dsv3_mxfp8_fwdbwd", T=4096, D=7168, I=2048, E=256, K=8, I_shared=2048,
                                   backward=True, dtype="mxfp8"),
}

_SLAB = 1 << 26  # elements drawn per randn call


def _draw(gen: torch.Generator, shape, std: float, device, out_dtype=torch.bfloat16) -> torch.Tensor:
    """N(0, std^2) in fp32, drawn slab by slab along dim 0, cast to out_dtype."""
    out = torch.empty(shape, dtype=out_dtype, device=device)
    flat = out.view(shape[0], -1)
    row = flat.shape[1]
    rows_per = max(1, _SLAB // max(row, 1))
    for r0 in range(0, shape[0], rows_per):
        r1 = min(shape[0], r0 + rows_per)
        v = torch.randn((r1 - r0, row), generator=gen, dtype=torch.float32, device=device)
        if std != 1.0:
            v.mul_(std)
        flat[r0:r1].copy_(v)  # fp32 -> bf16 copy rounds to nearest even
    return out


def _draw_grid(gen: torch.Generator, shape, scale: float, device) -> torch.Tensor:
    """Integers uniform in -3..3 times `scale` (a power of two), bf16."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    row = flat.shape[1]
    rows_per = max(1, _SLAB // max(row, 1))
    for r0 in range(0, shape[0], rows_per):
        r1 = min(shape[0], r0 + rows_per)
        v = torch.randint(-3, 4, (r1 - r0, row), generator=gen, device=device).to(torch.float32)
        flat[r0:r1].copy_(v * scale)  # exact in bf16
    return out


def make_inputs(cfg: MoEConfig, device="cpu", seed: int = 0, with_dy: Optional[bool] = None) -> Dict[str, torch.Tensor]:
    """Draw one layer's inputs on ``device``.

    Returns bf16 tensors x [T][D], w_gate/w_up [E][I][D], w_down [E][D][I],
    ws_gate/ws_up [I_s][D], ws_down [D][I_s] (absent when I_shared == 0),
    fp32 s [T][E] and, for backward workloads, bf16 dy [T][D].
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    T, D, I, E, Is = cfg.T, cfg.D, cfg.I, cfg.E, cfg.I_shared
    out: Dict[str, torch.Tensor] = {}
    if cfg.values == "grid":
        draw = lambda shape, scale: _draw_grid(gen, shape, scale, device)
        sx, sgu, sd = 0.5, 2.0 ** -8, 2.0 ** -7
    else:
        draw = lambda shape, std: _draw(gen, shape, std, device)
        sx, sgu, sd = 1.0, 1.0 / math.sqrt(D), None
    out["x"] = draw((T, D), sx)
    out["w_gate"] = draw((E, I, D), sgu)
    out["w_up"] = draw((E, I, D), sgu)
    out["w_down"] = draw((E, D, I), sd if sd else 1.0 / math.sqrt(I))
    if Is > 0:
        out["ws_gate"] = draw((Is, D), sgu)
        out["ws_up"] = draw((Is, D), sgu)
        out["ws_down"] = draw((D, Is), sd if sd else 1.0 / math.sqrt(Is))
    logits = torch.randn((T, E), generator=gen, dtype=torch.float32, device=device)
    if cfg.skew != 0.0:
        bias = -cfg.skew * torch.log(torch.arange(1, E + 1, dtype=torch.float32, device=device))
        logits = logits + bias
    out["s"] = torch.softmax(logits, dim=1).contiguous()
    if with_dy is None:
        with_dy = cfg.backward
    if with_dy:
        out["dy"] = draw((T, D), sx)
    return out


def make_router_weights(cfg: MoEConfig, device="cpu", seed: int = 0) -> torch.Tensor:
    """Router projection W_r [E][D] bf16, N(0, 1/D)."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 7919)
    return _draw(gen, (cfg.E, cfg.D), 1.0 / math.sqrt(cfg.D), device)


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a bf16 tensor's bit patterns (marshalling only)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


def f32_host(t: torch.Tensor):
    """Host numpy float32 copy of an fp32 tensor."""
    assert t.dtype == torch.float32
    return t.detach().contiguous().cpu().numpy()
