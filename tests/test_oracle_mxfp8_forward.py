"""Pins of the quantisation axes of the oracle's MXFP8 forward
(expert_ffn_rows_mxfp8, moe_forward_mxfp8, moe_forward_tokens with MXFP8
experts).

Mixture-of-Kittens paper note, "The production details": MXFP8 with the
quantisation fused into the dispatch (x per token row, along D), the grouped
GEMMs (W_gate, W_up along D; W_down along I) and the gated activation
(a = bf16(SiLU(h) u), quantised along I).

With normal weights every 1x32 block along either axis gets about the same
E8M0 scale, so an axis mistake would be invisible.  Here every row of x,
W_gate, W_up and W_down holds one binade (values (1 + j/8) 2^k, exact in
E4M3 at the block's scale, and every fp32 sum over a row pair is exact),
while consecutive rows sit 2^14 apart, so a block along the other axis mixes
binades and loses the small one.  The oracle must then give h and u as the
exact products and y as the exact down projection of its own quantised a;
the same steps with any operand quantised along the other axis must not.
"""
import numpy as np

import oracle as O


def _rows_binades(rng, r, c, lo_exp=-14):
    j = rng.integers(0, 8, size=(r, c))
    sgn = rng.choice([-1.0, 1.0], size=(r, c))
    k = np.where(np.arange(r) % 2 == 0, 0, lo_exp)[:, None]
    return (sgn * (1 + j / 8.0) * np.ldexp(1.0, k)).astype(np.float32)


def _exact(a, b_t):
    return (a.astype(np.float64) @ b_t.astype(np.float64).T).astype(np.float32)


def _close(a, b):
    return np.allclose(a, b, rtol=2.0 ** -12, atol=0)


def _down(a, Wd):
    """bf16(y) of the down projection of a (quantised along I) with exact W_down."""
    return O.round_bf16(_exact(O.mxfp8_roundtrip(a), Wd))


def test_expert_rows_quantisation_axes():
    rng = np.random.default_rng(11)
    n, D, I = 64, 64, 64
    x = _rows_binades(rng, n, D)
    Wg = _rows_binades(rng, I, D)
    Wu = _rows_binades(rng, I, D)
    Wd = _rows_binades(rng, D, I)          # rows of W_down: blocks along I one binade
    r = O.expert_ffn_rows_mxfp8(x, Wg, Wu, Wd)
    h, u = _exact(x, Wg), _exact(x, Wu)
    a = O.round_bf16(O.silu(h) * u)
    assert np.array_equal(r["a"], a)
    # a is quantised along I: codes and E8M0 bytes per 1x32 block of a row
    q, sc = O.mxfp8_quantize(a)
    assert np.array_equal(r["aq"], q) and np.array_equal(r["asc"], sc)
    assert r["asc"].shape == (n, I // 32)
    # y from that quantised a, W_down along I (exact): at most one bf16 ulp
    # from the fp64 evaluation of the same operands
    want = _down(a, Wd)
    assert _close(r["y"], want)
    # teeth: each operand along the other axis changes the result
    wrong_h = _exact(O.mxfp8_roundtrip(x.T).T, Wg)             # x along tokens
    assert not _close(wrong_h, h)
    wrong_h = _exact(x, O.mxfp8_roundtrip(Wg.T).T)             # W_gate along I
    assert not _close(wrong_h, h)
    wrong_u = _exact(x, O.mxfp8_roundtrip(Wu.T).T)             # W_up along I
    assert not _close(wrong_u, u)
    wrong_y = O.round_bf16(_exact(O.mxfp8_roundtrip(a), O.mxfp8_roundtrip(Wd.T).T))  # W_down along D
    assert not _close(wrong_y, want)
    wrong_y = O.round_bf16(_exact(O.mxfp8_roundtrip(a.T).T, Wd))   # a along tokens
    assert not _close(wrong_y, want)


def _layer(rng, T=96, D=64, I=64, E=3, K=2):
    bits = O.f32_to_bf16_bits
    inp = dict(x=bits(_rows_binades(rng, T, D)),
               w_gate=bits(np.stack([_rows_binades(rng, I, D) for _ in range(E)])),
               w_up=bits(np.stack([_rows_binades(rng, I, D) for _ in range(E)])),
               w_down=bits(np.stack([_rows_binades(rng, D, I) for _ in range(E)])))
    logits = rng.standard_normal((T, E))
    inp["s"] = (np.exp(logits) / np.exp(logits).sum(1, keepdims=True)).astype(np.float32)
    return inp, K


def test_layer_quantisation_axes():
    rng = np.random.default_rng(12)
    inp, K = _layer(rng)
    r = O.moe_forward_mxfp8(inp, K)
    x = O.bf16_to_f32(inp["x"])
    # x quantised per token row along D: exact for one-binade rows
    assert np.array_equal(O.mxfp8_dequantize(r["xq"], r["xs"]).astype(np.float32), x)
    assert r["xs"].shape == (x.shape[0], x.shape[1] // 32)
    for e in range(inp["w_gate"].shape[0]):
        p0, p1 = int(r["offsets"][e]), int(r["offsets"][e + 1])
        assert p1 > p0
        xe = x[r["table"][p0:p1, 0] // K]
        Wg, Wu, Wd = (O.bf16_to_f32(inp[k][e]) for k in ("w_gate", "w_up", "w_down"))
        a = O.round_bf16(O.silu(_exact(xe, Wg)) * _exact(xe, Wu))
        assert np.array_equal(r["a"][p0:p1], a)
        assert _close(r["y"][p0:p1], _down(a, Wd))
        assert not _close(O.round_bf16(_exact(O.mxfp8_roundtrip(a), O.mxfp8_roundtrip(Wd.T).T)), r["y"][p0:p1])
    # the token-sampled forward (MXFP8 experts) gives the same per-route y
    toks = [0, 7, 50, 95]
    part = O.moe_forward_tokens(toks, inp["x"][toks], inp["s"][toks], O.HostWeights.from_arrays(inp), K,
                                mxfp8=True)
    rd = r["route_dst"].reshape(-1, K)
    for j, t in enumerate(toks):
        for k in range(K):
            assert np.array_equal(part["y"][j, k], r["y"][rd[t, k]])
    assert np.array_equal(part["out"], r["out"][toks])
