"""CPU oracle for the single-GPU MoE layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

The oracle is a plain, slow, step-by-step numpy evaluation of the layer as the
Mixture-of-Kittens pages define it.  It shares no code with the CUDA path.

Pinned (see ``tests/test_oracle_*.py``): bf16 rounding, top-k routing, the pull
schedule / plan, the forward (dense single-expert closed form, hand-computed
identity-weight case, relabelling and permutation invariants, W_up = 0
reduction, fp64 shadow error bound), the MXFP8 quantiser (exhaustive against a
nearest-value search and the PyTorch float8_e4m3fn cast) and the backward
(central finite differences in the fp64 shadow, scale-invariance identity of
ds, dense-matmul weight gradients).
"""
from .moe_oracle import *  # noqa: F401,F403
