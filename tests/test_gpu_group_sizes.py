"""Grouped expert GEMMs at group sizes around every tile boundary, through
mok_expert_ffn with explicit offsets, against the oracle.

Groups of 0, 1, 15, 16, 17, 31, 32, 33, 127, 128, 129, 255, 256, 257, 272,
511, 512 and 513 rows: a tile takes up to 256 rows of a group (rounded up to
16 where the rows are the MMA's N dimension), the epilogue stores a chunk of
32 rows as a whole or row by row, and a group's last tile may hold one row.
With those groups alone the layer averages fewer than 512 rows per expert,
which runs the kernels with the rows as N; one more group of 7000 rows lifts
the average over 512, which runs the row-major kernels.  Both must match the
oracle, and each other bit for bit on the common groups (the tensor core
sums each output over K in the same order either way).
"""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import BF16_TOL, assert_close, mok

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SIZES = [0, 1, 15, 16, 17, 31, 32, 33, 127, 128, 129, 255, 256, 257, 272, 511, 512, 513]
D, I = 256, 128


@pytest.fixture(scope="module")
def m():
    return mok()


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def _inputs(sizes, rng):
    E, R = len(sizes), int(sum(sizes))
    bits = O.f32_to_bf16_bits
    return dict(xg=bits(rng.standard_normal((R, D)).astype(np.float32)),
                wg=bits((rng.standard_normal((E, I, D)) / np.sqrt(D)).astype(np.float32)),
                wu=bits((rng.standard_normal((E, I, D)) / np.sqrt(D)).astype(np.float32)),
                wd=bits((rng.standard_normal((E, D, I)) / np.sqrt(I)).astype(np.float32)))


def _run(m, sizes, inp):
    """The first len(sizes) groups of inp, with these sizes."""
    E, R = len(sizes), int(sum(sizes))
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    xg, wg, wu, wd = inp["xg"][:R], inp["wg"][:E], inp["wu"][:E], inp["wd"][:E]
    w = {"w_gate": _bf16(wg), "w_up": _bf16(wu), "w_down": _bf16(wd)}
    a = torch.full((R, I), float("nan"), dtype=torch.bfloat16, device=DEV)
    y = torch.full((R, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    shape = m.make_shape(R, D, I, E, 1, 0, m.MOK_BF16, 0)
    m.expert_ffn(shape, m.make_weights(w), _bf16(xg), torch.from_numpy(offsets).to(DEV), y, a_out=a)
    m.check_device_status()
    a_ref, y_ref = O.expert_ffn(xg, offsets, wg, wu, wd)
    assert_close(a.float().cpu().numpy(), a_ref, BF16_TOL, "a")
    assert_close(y.float().cpu().numpy(), y_ref, BF16_TOL, "y")
    return a, y


def test_group_sizes_both_tilings(m):
    big_sizes = SIZES + [7000]
    assert sum(SIZES) < 512 * len(SIZES) and sum(big_sizes) >= 512 * len(big_sizes)
    inp = _inputs(big_sizes, np.random.default_rng(11))
    small = _run(m, SIZES, inp)   # fewer than 512 rows per expert: rows as N
    big = _run(m, big_sizes, inp)  # the same groups first, then 7000 rows: row-major
    R = sum(SIZES)
    for got_small, got_big, what in zip(small, big, ("a", "y")):
        assert torch.equal(got_small.view(torch.int16), got_big[:R].view(torch.int16)), what
