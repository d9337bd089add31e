"""Pins of the oracle's MXFP8 backward (route_backward_rows_mxfp8,
moe_backward_mxfp8).

* With the quantiser switched off and small-integer inputs (every product
  exact), it is the BF16 backward: the same dh, du, a_g, dg, weight
  gradients and ds bit for bit, dX within one bf16 ulp (the fp32 sum over
  [dh | du] runs in another order).
* Quantisation axes: inputs whose rows are each one binade (so every 1x32
  block along the row is exact in E4M3 at the block's scale, and every
  fp32 sum of a row pair's products is exact) while the other axis mixes
  binades 2^14 apart (inexact there).  The replay h, u and t then equal the
  exact products, bit for bit and unrounded (the pages put no rounding point
  on them), and a quantiser along the other axis would not (checked, so the
  construction has teeth); likewise the weights of the dX product along 2I.
  Activations that E4M3 does not hold exactly enter the replay and t
  quantised per row (and unquantised they would give other h, t).
* Random inputs: within the MXFP8 error of the BF16 backward.
"""
import numpy as np

import oracle as O


def _rows_binades(rng, r, c, lo_exp=-14):
    """[r][c] values (1 + j/8) * 2^k * sign, k = 0 on even rows and lo_exp on
    odd rows: every block of 32 along c is one binade."""
    j = rng.integers(0, 8, size=(r, c))
    sgn = rng.choice([-1.0, 1.0], size=(r, c))
    k = np.where(np.arange(r) % 2 == 0, 0, lo_exp)[:, None]
    return (sgn * (1 + j / 8.0) * np.ldexp(1.0, k)).astype(np.float32)


def _int_problem(seed, T=10, D=64, I=64, E=3, K=2, Is=32):
    rng = np.random.default_rng(seed)
    ints = lambda *shape: rng.integers(-2, 3, size=shape).astype(np.float32)
    bits = O.f32_to_bf16_bits
    inp = dict(x=bits(ints(T, D)), w_gate=bits(ints(E, I, D)), w_up=bits(ints(E, I, D)),
               w_down=bits(ints(E, D, I)), ws_gate=bits(ints(Is, D)), ws_up=bits(ints(Is, D)),
               ws_down=bits(ints(D, Is)))
    logits = rng.standard_normal((T, E))
    inp["s"] = (np.exp(logits) / np.exp(logits).sum(1, keepdims=True)).astype(np.float32)
    dy = bits(ints(T, D))
    return inp, dy, K


def test_quantiser_off_is_the_bf16_backward():
    for seed in range(3):
        inp, dy, K = _int_problem(seed)
        a = O.moe_backward_mxfp8(inp, dy, K, deq=lambda v: np.asarray(v, dtype=np.float32))
        b = O.moe_backward(inp, dy, K)
        for k in ("dW_gate", "dW_up", "dW_down", "dWs_gate", "dWs_up", "dWs_down", "dg", "ds"):
            assert np.array_equal(a[k], b[k]), k
        assert np.allclose(a["dX"], b["dX"], rtol=2.0 ** -7, atol=0), "dX"
        assert np.abs(b["dX"]).max() > 1.0  # not a trivially zero case


def _exact(a, b_t):
    """The fp64 product a @ b_t.T as float32 (exact for one-binade rows)."""
    return (a.astype(np.float64) @ b_t.astype(np.float64).T).astype(np.float32)


def test_replay_and_t_quantised_along_d():
    rng = np.random.default_rng(7)
    n, D, I = 64, 64, 64
    x = _rows_binades(rng, n, D)
    dy = _rows_binades(rng, n, D)
    Wg = _rows_binades(rng, I, D)
    Wu = _rows_binades(rng, I, D)
    WdT = _rows_binades(rng, I, D)        # W_down^T: blocks along D are one binade
    Wd = np.ascontiguousarray(WdT.T)      # [D][I]
    g = np.full(n, 0.5, np.float32)
    r = O.route_backward_rows_mxfp8(x, dy, g, Wg, Wu, Wd)
    assert r["h"].dtype == np.float32 and r["t"].dtype == np.float32
    assert np.array_equal(r["h"], _exact(x, Wg))
    assert np.array_equal(r["u"], _exact(x, Wu))
    assert np.array_equal(r["t"], _exact(dy, WdT))
    # not rounded to bf16 anywhere: the exact products carry more than 8 bits
    assert not np.array_equal(r["h"], O.round_bf16(r["h"]))
    assert not np.array_equal(r["t"], O.round_bf16(r["t"]))
    # the same operands quantised along the other axis lose the small binade
    close = lambda a, b: np.allclose(a, b, rtol=2.0 ** -12, atol=0)
    wrong = O.mxfp8_roundtrip(Wg.T).T
    assert not close(x @ wrong.T, r["h"])
    wrong_d = O.mxfp8_roundtrip(Wd)       # W_down along I
    assert not close(dy @ wrong_d, r["t"])
    wrong_x = O.mxfp8_roundtrip(x.T).T    # x along the token axis
    assert not close(wrong_x @ Wg.T, r["h"])
    # activations that E4M3 does not hold exactly enter quantised per row
    xr = O.round_bf16(rng.standard_normal((n, D)).astype(np.float32))
    dyr = O.round_bf16(rng.standard_normal((n, D)).astype(np.float32))
    r2 = O.route_backward_rows_mxfp8(xr, dyr, g, Wg, Wu, Wd)
    assert close(r2["h"], _exact(O.mxfp8_roundtrip(xr), Wg))
    assert close(r2["t"], _exact(O.mxfp8_roundtrip(dyr), WdT))
    assert not close(r2["h"], _exact(xr, Wg))
    assert not close(r2["t"], _exact(dyr, WdT))


def test_dx_weights_quantised_along_2i():
    rng = np.random.default_rng(8)
    n, D, I = 40, 64, 64
    x = O.round_bf16(rng.standard_normal((n, D)).astype(np.float32))
    dy = O.round_bf16(rng.standard_normal((n, D)).astype(np.float32))
    # W_gate^T and W_up^T rows (fixed d) are one binade along I
    Wg = np.ascontiguousarray(_rows_binades(rng, D, I).T)   # [I][D]
    Wu = np.ascontiguousarray(_rows_binades(rng, D, I).T)
    Wd = O.round_bf16((rng.standard_normal((D, I)) / 8).astype(np.float32))
    g = np.full(n, 0.25, np.float32)
    r = O.route_backward_rows_mxfp8(x, dy, g, Wg, Wu, Wd)
    dhu = O.mxfp8_roundtrip(np.concatenate([r["dh"], r["du"]], axis=1))
    wgu = np.concatenate([Wg, Wu], axis=0)   # [2I][D]: the exact weights
    want = O.round_bf16((dhu.astype(np.float64) @ wgu.astype(np.float64)).astype(np.float32))
    assert np.allclose(r["dx"], want, rtol=2.0 ** -7, atol=0)
    # quantising [W_gate^T | W_up^T] along D instead would not be exact
    wrong = O.mxfp8_roundtrip(wgu)           # along D
    assert not np.allclose(O.round_bf16(dhu @ wrong), r["dx"], rtol=2.0 ** -7, atol=0)


def test_random_inputs_within_mxfp8_error_of_bf16():
    rng = np.random.default_rng(3)
    T, D, I, E, K = 24, 128, 64, 4, 2
    bits = O.f32_to_bf16_bits
    inp = dict(x=bits(rng.standard_normal((T, D)).astype(np.float32)),
               w_gate=bits((rng.standard_normal((E, I, D)) / np.sqrt(D)).astype(np.float32)),
               w_up=bits((rng.standard_normal((E, I, D)) / np.sqrt(D)).astype(np.float32)),
               w_down=bits((rng.standard_normal((E, D, I)) / np.sqrt(I)).astype(np.float32)))
    logits = rng.standard_normal((T, E))
    inp["s"] = (np.exp(logits) / np.exp(logits).sum(1, keepdims=True)).astype(np.float32)
    dy = bits(rng.standard_normal((T, D)).astype(np.float32))
    a = O.moe_backward_mxfp8(inp, dy, K)
    b = O.moe_backward(inp, dy, K)
    for k in ("dX", "dW_gate", "dW_up", "dW_down", "dg"):
        err = np.abs(a[k] - b[k]).max() / max(1e-6, np.abs(b[k]).max())
        assert err < 0.15, (k, err)
    assert not np.array_equal(a["dX"], b["dX"])  # the quantisation is on
