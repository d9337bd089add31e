"""Pins of the oracle's number formats against library routines and brute force.

bf16 rounding -> torch's float32 -> bfloat16 cast; E4M3 encoding -> an
exhaustive nearest-value search and torch's float8_e4m3fn cast; the E8M0 scale
rule -> its definition (smallest e with amax <= 448 * 2^e) at every boundary.
"""
import numpy as np
import pytest
import torch

import oracle as O


def _torch_bf16_bits(v32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_round_matches_torch_cast_random_and_ties():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    # exact halfway points (low half = 0x8000) with both parities of the kept lsb
    ties = (rng.integers(0, 2**16, size=1 << 16, dtype=np.uint64).astype(np.uint32) << 16) | np.uint32(0x8000)
    allbits = np.concatenate([bits, ties, ties ^ np.uint32(0x10000)])
    v = allbits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) < 3.0e38)]
    assert np.array_equal(O.f32_to_bf16_bits(v), _torch_bf16_bits(v))


def test_bf16_bits_roundtrip_exact():
    b = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = O.bf16_to_f32(b)
    fin = np.isfinite(f)
    assert np.array_equal(O.f32_to_bf16_bits(f[fin]), b[fin])
    assert np.array_equal(f[fin], torch.from_numpy(b[fin].view(np.int16)).view(torch.bfloat16).float().numpy())


def _all_bf16_values_upto(limit):
    b = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = O.bf16_to_f32(b)
    return f[np.isfinite(f) & (np.abs(f) <= limit)]


def test_e4m3_code_table():
    v = O.e4m3_code_values()
    assert v[0x7E] == 448.0 and v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.all(np.diff(v[:127]) > 0)
    assert np.count_nonzero(np.isfinite(v)) == 254


def test_e4m3_encode_exhaustive_vs_torch_cast():
    v = _all_bf16_values_upto(448.0)
    ours = O.e4m3_encode(v)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_vs_nearest_search():
    """Brute force: nearest finite code value, ties to the even mantissa."""
    vals = O.e4m3_code_values()
    finite = [c for c in range(256) if np.isfinite(vals[c])]
    rng = np.random.default_rng(2)
    v = _all_bf16_values_upto(448.0)
    sample = np.concatenate([rng.choice(v, 3000), (vals[1:126] + vals[2:127]) / 2])  # incl. exact midpoints
    got = O.e4m3_encode(sample)
    for x, c in zip(sample, got):
        best = None
        for code in finite:
            if np.signbit(vals[code]) != np.signbit(x) and vals[code] != 0:
                continue
            d = abs(vals[code] - x)
            if best is None or d < best[0] or (d == best[0] and (code & 1) == 0 and (best[1] & 1) == 1):
                best = (d, code)
        want = best[1] | (0x80 if np.signbit(x) else 0)
        assert int(c) == want, (x, c, want)


def test_e4m3_round_is_the_encoders_value():
    """The closed form (3 mantissa bits, ties to even) against the value of
    the code e4m3_encode picks: every bf16 value up to 448, both signs,
    scaled by powers of two into the subnormal range, and the exact
    midpoints between neighbouring codes."""
    vals = O.e4m3_code_values()
    v = _all_bf16_values_upto(448.0).astype(np.float64)
    mids = (vals[1:126] + vals[2:127]) / 2
    cases = [v, v * 2.0 ** -7, v * 2.0 ** -12, mids, -mids]
    for c in cases:
        c = c[np.abs(c) <= 448.0]
        want = vals[O.e4m3_encode(c)]
        got = O.e4m3_round(c)
        assert np.array_equal(got, want)
        assert np.array_equal(np.signbit(got[want == 0]), np.signbit(c[want == 0]))


def test_mxfp8_roundtrip_is_quantize_then_dequantize():
    rng = np.random.default_rng(5)
    v = O.round_bf16((rng.standard_normal((96, 256)) * 10.0 ** rng.uniform(-5, 5, (96, 1))).astype(np.float32))
    v[3, 64:96] = 0.0
    want = O.mxfp8_dequantize(*O.mxfp8_quantize(v)).astype(np.float32)
    assert np.array_equal(O.mxfp8_roundtrip(v), want)


@pytest.mark.parametrize("k", range(-20, 21, 3))
def test_mx_scale_rule_boundaries(k):
    b = 448.0 * 2.0 ** k
    assert O.mx_scale_exponent(b) == k
    assert O.mx_scale_exponent(np.nextafter(b, np.inf)) == k + 1
    assert O.mx_scale_exponent(np.nextafter(b, 0)) == k


def test_mx_scale_rule_definition_random():
    rng = np.random.default_rng(3)
    amax = np.abs(rng.standard_normal(20000)) * 10.0 ** rng.uniform(-6, 6, 20000)
    e = O.mx_scale_exponent(amax).astype(np.float64)
    assert np.all(amax <= 448.0 * 2.0 ** e)
    assert np.all(amax > 448.0 * 2.0 ** (e - 1))
    assert O.mx_scale_exponent(0.0) == -127


def test_mxfp8_quantize_roundtrip_error_bound():
    rng = np.random.default_rng(4)
    v = O.round_bf16(rng.standard_normal((64, 256)).astype(np.float32))
    q, sc = O.mxfp8_quantize(v)
    assert q.shape == v.shape and sc.shape == (64, 8)
    d = O.mxfp8_dequantize(q, sc)
    blocks = np.abs(v).reshape(64, 8, 32).max(-1)
    # E4M3 keeps 3 mantissa bits: error <= 2^-4 * |v| in the normal range,
    # <= half the smallest subnormal step (2^-10 * 2^e) below it
    e = sc.astype(np.int64) - 127
    floor = (2.0 ** -10 * 2.0 ** e)[..., None]
    err = np.abs(d - v).reshape(64, 8, 32)
    assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(v).reshape(64, 8, 32), floor) + 0)
    # the block maximum is representable without overflow
    assert np.all(np.abs(d).reshape(64, 8, 32).max(-1) <= 448.0 * 2.0 ** e + 0)
    assert np.all(blocks > 0)


def test_mxfp8_zero_block_and_signed_zero():
    v = np.zeros((1, 64), dtype=np.float32)
    v[0, 40] = -0.0
    v[0, 33] = 1.5
    q, sc = O.mxfp8_quantize(v)
    assert sc[0, 0] == 0
    assert np.all(q[0, :32] == 0)
    assert q[0, 40] == 0x80


def test_bf16_flip_ulp_marks_only_near_midpoints():
    one = np.float32(1.0)
    ulp = 2.0 ** -7  # bf16 spacing in [1, 2)
    mid = np.float32(1.0 + ulp / 2)  # exact rounding midpoint
    assert O.bf16_flip_ulp(mid) == ulp
    assert O.bf16_flip_ulp(np.nextafter(mid, np.float32(2))) == ulp
    assert O.bf16_flip_ulp(one) == 0.0
    assert O.bf16_flip_ulp(np.float32(1.0 + ulp / 4)) == 0.0
    rng = np.random.default_rng(7)
    v = rng.standard_normal(100000).astype(np.float32)
    f = O.bf16_flip_ulp(v)
    frac = np.mean(f > 0)
    assert 0.001 < frac < 0.05  # ~ 2 * 2^-14 / 2^-8 of values sit near a midpoint
    nz = f > 0
    assert np.allclose(f[nz], np.abs(O.round_bf16(v[nz] * (1 + 2.0 ** -14)) - O.round_bf16(v[nz] * (1 - 2.0 ** -14))))
