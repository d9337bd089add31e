"""Plain CPU oracle of the Mixture-of-Kittens (MoK) MoE layer, single GPU view.

TEST INFRASTRUCTURE ONLY (see the package docstring).  No blocking, fusion or
reordering beyond what the definitions state; a numpy matmul is the only
library primitive used for the contractions.

Sources (the pages' own titles and sections):
  [blog]  "Mixture-of-Kittens: our open-source MoE megakernel for NVL72s"
          (Cursor blog), sections "Overlapping computation and communication
          in MoE" (notation, the MoE(x, s) equation, g_i) and "Scheduling"
          (the pull-schedule algorithm: counts T, M, offsets S, table Phi).
  [note]  "Mixture-of-Kittens: MoE Megakernel for NVL72s" (paper note),
          sections "Pull dispatch, push combine" (sort key of the schedule:
          local expert, per-source ordinal, source rank), "The production
          details" (determinism, MXFP8, BF16 shared expert, SonicMoE router
          gradient).

Readings where the pages are silent or garbled (each is also listed in the
design notes):
  * the router weights s enter as fp32 [T][E]; top-k picks the K largest,
    lowest expert index first on ties, output in descending-score order;
  * g_k = s_k / (((s_0 + s_1) + s_2) + ...) summed in fp32 in k order, IEEE
    division;
  * rounding points: a = bf16(SiLU(h) * u); y = bf16(W_down a) per expert
    output; shared expert output bf16; out = bf16(fp32 sum in the order
    shared, k = 0..K-1);
  * the garbled in-rank position of the schedule reads
    p = sum_r' min(M[l, r'], o) + |{r' < r : M[l, r'] > o}|;
  * MXFP8: E4M3 (OCP "fn") codes with one E8M0 scale per 1x32 block along the
    reduction dim, scale 2^e with e the smallest integer such that
    amax <= 448 * 2^e (all-zero block: byte 0); a is rounded to bf16 before it
    is quantised along I; the shared expert stays BF16.

Numerics: the default is fp32 arithmetic with the bf16 rounding points above.
``FP64_SHADOW`` evaluates the same steps in fp64 with every rounding point
switched off; it bounds the fp32 oracle's own error and drives the
finite-difference checks of the backward.

bf16 tensors are passed as numpy uint16 bit patterns; fp32 tensors as float32.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Dict, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "Numerics", "FP32", "FP64_SHADOW",
    "bf16_to_f32", "round_bf16", "f32_to_bf16_bits", "bf16_flip_ulp",
    "silu", "softmax_rows", "router_scores", "route", "pull_schedule", "plan", "gather",
    "expert_ffn_rows", "expert_ffn", "shared_ffn", "combine", "moe_forward",
    "HostWeights", "moe_forward_tokens",
    "route_backward_rows", "rounding_ranges", "sum_range", "moe_backward", "moe_backward_tokens", "router_grad",
    "e4m3_code_values", "e4m3_encode", "e4m3_round", "mx_scale_exponent", "mxfp8_quantize",
    "mxfp8_dequantize", "expert_ffn_rows_mxfp8", "moe_forward_mxfp8",
    "mxfp8_roundtrip", "route_backward_rows_mxfp8", "moe_backward_mxfp8",
]


# --------------------------------------------------------------------------
# numerics
# --------------------------------------------------------------------------
def bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_bf16(v) -> np.ndarray:
    """Round float32 values to the nearest bf16 value, ties to even.

    Returned as float32 holding bf16-representable values.  Adding 0x7FFF plus
    the lowest kept bit and truncating the low 16 bits is round-half-to-even on
    the binary representation (finite inputs)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    keep_lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + keep_lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def bf16_flip_ulp(v, rel: float = 2.0 ** -14) -> np.ndarray:
    """Where a bf16 rounding decision is not fixed by fp32 arithmetic.

    An fp32 value that is the sum of many products differs between two
    correct evaluations (other summation orders) by far less than 2^-14 of
    its size.  If rounding v * (1 - rel) and v * (1 + rel) to bf16 gives
    different values, either rounding of v is a correct result; return that
    one-ulp difference there and 0 elsewhere."""
    v = np.asarray(v, dtype=np.float64)
    lo = round_bf16((v * (1.0 - rel)).astype(np.float32))
    hi = round_bf16((v * (1.0 + rel)).astype(np.float32))
    return np.abs(hi.astype(np.float64) - lo.astype(np.float64))


def f32_to_bf16_bits(v) -> np.ndarray:
    return (round_bf16(v).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


@dataclasses.dataclass(frozen=True)
class Numerics:
    """Arithmetic type plus whether the bf16 rounding points are applied."""

    dtype: type
    round_points: bool

    def rnd(self, v) -> np.ndarray:
        if self.round_points:
            return round_bf16(np.asarray(v, dtype=np.float32))
        return np.asarray(v, dtype=self.dtype)

    def w(self, bits_or_values) -> np.ndarray:
        """Weight / activation operand: bf16 bits -> arithmetic type."""
        a = np.asarray(bits_or_values)
        if a.dtype == np.uint16:
            a = bf16_to_f32(a)
        return a.astype(self.dtype, copy=False)


FP32 = Numerics(np.float32, True)
FP64_SHADOW = Numerics(np.float64, False)


def silu(h: np.ndarray) -> np.ndarray:
    """SiLU(h) = h / (1 + exp(-h)) in h's type ([blog] layer equation)."""
    with np.errstate(over="ignore"):
        return h / (h.dtype.type(1) + np.exp(-h))


# --------------------------------------------------------------------------
# router scores, routing and the pull schedule
# --------------------------------------------------------------------------
def softmax_rows(logits: np.ndarray, num: Numerics = FP32) -> np.ndarray:
    """Row softmax exp(l - max l) / sum exp(l - max l) in num's type."""
    lv = np.asarray(logits, dtype=num.dtype)
    e = np.exp(lv - lv.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def router_scores(x, w_router, num: Numerics = FP32):
    """Router scores s = softmax(x W_r^T) over the E routed experts.

    [blog] "Overlapping computation and communication in MoE": the gate g is
    formed from router weights s over the routed experts; the pages show only
    s, so the router is read as the usual projection of a DeepSeek-V3-style
    layer, logits[t, e] = sum_d x[t, d] W_r[e, d] (x, W_r bf16; sums in num's
    type), followed by a softmax over e.  Returns (logits, s), both [T][E].
    """
    logits = num.w(x) @ num.w(w_router).T
    return logits, softmax_rows(logits, num)


def route(s: np.ndarray, K: int, num: Numerics = FP32):
    """Top-K experts per token and their renormalised weights.

    [blog] "Overlapping computation and communication in MoE": a router
    selects the top-k routed experts of each token; g_i = s_i / sum_{j in topk} s_j.
    Order: descending s, lowest index first among equal s (stable sort of -s).
    Returns topk_idx int32 [T][K], g [T][K], den [T].
    """
    s = np.asarray(s, dtype=num.dtype)
    order = np.argsort(-s, axis=1, kind="stable")[:, :K].astype(np.int32)
    sel = np.take_along_axis(s, order, axis=1)
    den = sel[:, 0].copy()
    for k in range(1, K):
        den = den + sel[:, k]
    g = sel / den[:, None]
    return order, g, den


def pull_schedule(routing: np.ndarray, c: int, L: int):
    """Pull-based dispatch schedule of one destination rank.

    [blog] "Scheduling": inputs the routing tensor E[r, i, k] (global expert of
    route k of token i on source rank r), local rank c and L experts per rank.
    Pass 1 counts T[l] and M[l, r]; S is the exclusive scan of T; pass 2 gives
    route (r, i, k) of local expert l the slot S[l] + p, with o its ordinal
    among (l, r) routes and p = sum_r' min(M[l, r'], o) + |{r' < r : M[l, r'] > o}|
    (round-robin over source ranks, the sort key (local expert, ordinal,
    source rank) of [note] "Pull dispatch, push combine").

    Returns T [L], M [L][R], S [L], Phi [sum T][2] = (src_rank, i*K + k).
    """
    routing = np.asarray(routing)
    R, N, K = routing.shape
    T = np.zeros(L, dtype=np.int64)
    M = np.zeros((L, R), dtype=np.int64)
    for r in range(R):
        for i in range(N):
            for k in range(K):
                e = int(routing[r, i, k])
                if e // L == c:
                    l = e - c * L
                    T[l] += 1
                    M[l, r] += 1
    S = np.zeros(L, dtype=np.int64)
    for l in range(1, L):
        S[l] = S[l - 1] + T[l - 1]
    C = np.zeros((L, R), dtype=np.int64)
    Phi = np.full((int(T.sum()), 2), -1, dtype=np.int64)
    for r in range(R):
        for i in range(N):
            for k in range(K):
                e = int(routing[r, i, k])
                if e // L != c:
                    continue
                l = e - c * L
                o = C[l, r]
                p = int(np.minimum(M[l], o).sum()) + int(np.count_nonzero(M[l, :r] > o))
                Phi[S[l] + p] = (r, i * K + k)
                C[l, r] += 1
    return T, M, S, Phi


def plan(topk_idx: np.ndarray, E: int):
    """Device-plan outputs for one GPU (the pull schedule with one source rank,
    c = 0, L = E).

    counts[e] = routes to expert e; offsets = exclusive scan, offsets[E] = R;
    table[dst] = (src_index = t*K + k, expert, dst); route_dst[t*K + k] = dst.
    With one source the position is the route's ordinal within its expert, so
    routes of an expert land contiguously in (t, k) scan order.
    """
    topk_idx = np.asarray(topk_idx)
    T, K = topk_idx.shape
    if topk_idx.size and (topk_idx.min() < 0 or topk_idx.max() >= E):
        raise ValueError("expert index out of range")
    counts, _, S, Phi = pull_schedule(topk_idx[None, :, :], c=0, L=E)
    R = T * K
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[:E] = S
    offsets[E] = R
    table = np.zeros((R, 3), dtype=np.int32)
    route_dst = np.zeros(R, dtype=np.int32)
    flat = topk_idx.reshape(-1)
    for dst in range(R):
        src = int(Phi[dst, 1])
        table[dst] = (src, flat[src], dst)
        route_dst[src] = dst
    return counts.astype(np.int32), offsets.astype(np.int32), table, route_dst


def gather(x: np.ndarray, table: np.ndarray, K: int) -> np.ndarray:
    """xg[p] = x[table[p].src_index // K]: rows land expert-contiguous
    ([blog] "Scheduling": zero local copies)."""
    return np.asarray(x)[np.asarray(table)[:, 0] // K]


# --------------------------------------------------------------------------
# expert FFNs and combine
# --------------------------------------------------------------------------
def expert_ffn_rows(xrows, Wg, Wu, Wd, num: Numerics = FP32):
    """E_i(x) = W_down (SiLU(W_gate x) * (W_up x)) for a batch of rows of one
    expert ([blog] layer equation).  W_gate, W_up are [I][D], W_down [D][I].
    Returns (h, u, a, y) with a and y at their rounding points."""
    X = num.w(xrows)
    h = X @ num.w(Wg).T
    u = X @ num.w(Wu).T
    a = num.rnd(silu(h) * u)
    y = num.rnd(a.astype(num.dtype) @ num.w(Wd).T)
    return h, u, a.astype(num.dtype), y.astype(num.dtype)


def expert_ffn(xg, offsets, w_gate, w_up, w_down, num: Numerics = FP32):
    """Grouped expert FFN over the expert-ordered rows: expert e owns rows
    [offsets[e], offsets[e+1]).  Returns a [R][I] and y [R][D]."""
    R = xg.shape[0]
    E = len(offsets) - 1
    I = w_gate.shape[1]
    D = w_gate.shape[2]
    a = np.zeros((R, I), dtype=num.dtype)
    y = np.zeros((R, D), dtype=num.dtype)
    for e in range(E):
        p0, p1 = int(offsets[e]), int(offsets[e + 1])
        if p0 == p1:
            continue
        _, _, a[p0:p1], y[p0:p1] = expert_ffn_rows(xg[p0:p1], w_gate[e], w_up[e], w_down[e], num)
    return a, y


def shared_ffn(x, ws_gate, ws_up, ws_down, num: Numerics = FP32):
    """E_shared(x): the same SwiGLU FFN over every token, kept in BF16
    ([note] "The production details")."""
    return expert_ffn_rows(x, ws_gate, ws_up, ws_down, num)[3]


def combine(y, ys, g, route_dst, num: Numerics = FP32):
    """out[t] = bf16(ys[t] + sum_k g[t,k] * y[route_dst[t,k]]), accumulated in
    the fixed order shared, k = 0..K-1 ([blog] layer equation; [note]
    determinism: fixed-order reduction)."""
    g = np.asarray(g, dtype=num.dtype)
    T, K = g.shape
    rd = np.asarray(route_dst).reshape(T, K)
    acc = np.zeros((T, y.shape[1]), dtype=num.dtype) if ys is None else np.asarray(ys, dtype=num.dtype).copy()
    for k in range(K):
        acc = acc + g[:, k:k + 1] * np.asarray(y, dtype=num.dtype)[rd[:, k]]
    return num.rnd(acc).astype(num.dtype)


def moe_forward(inp: Dict[str, np.ndarray], K: int, num: Numerics = FP32) -> Dict[str, np.ndarray]:
    """MoE(x, s) = E_shared(x) + sum_{i in topk} g_i E_i(x), step by step:
    route -> plan -> gather -> grouped expert FFN -> shared FFN -> combine.

    ``inp``: x [T][D] bits, s [T][E] f32, w_gate/w_up [E][I][D] bits,
    w_down [E][D][I] bits, optional ws_gate/ws_up/ws_down bits."""
    s = inp["s"]
    E = s.shape[1]
    topk_idx, g, den = route(s, K, num)
    counts, offsets, table, route_dst = plan(topk_idx, E)
    x = num.w(inp["x"])
    xg = gather(x, table, K)
    a, y = expert_ffn(xg, offsets, inp["w_gate"], inp["w_up"], inp["w_down"], num)
    ys = None
    if inp.get("ws_gate") is not None:
        ys = shared_ffn(x, inp["ws_gate"], inp["ws_up"], inp["ws_down"], num)
    out = combine(y, ys, g, route_dst, num)
    return dict(topk_idx=topk_idx, g=g, den=den, counts=counts, offsets=offsets, table=table,
                route_dst=route_dst, xg=xg, a=a, y=y, ys=ys, out=out)


@dataclasses.dataclass
class HostWeights:
    """Expert weights reachable one expert at a time (bits, uint16).  ``fetch``
    returns (W_gate [I][D], W_up [I][D], W_down [D][I]) of expert e."""

    fetch: Callable[[int], Tuple[np.ndarray, np.ndarray, np.ndarray]]
    shared: Optional[Tuple[np.ndarray, np.ndarray, np.ndarray]] = None

    @staticmethod
    def from_arrays(inp: Dict[str, np.ndarray]) -> "HostWeights":
        sh = None
        if inp.get("ws_gate") is not None:
            sh = (inp["ws_gate"], inp["ws_up"], inp["ws_down"])
        return HostWeights(lambda e: (inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e]), sh)


def moe_forward_tokens(tokens: Sequence[int], x_rows, s_rows, weights: HostWeights, K: int,
                       num: Numerics = FP32, mxfp8: bool = False, map_fn: Callable = map):
    """The forward for a sample of tokens, one route at a time (routing is
    per token, so the sampled rows need no other token).  mxfp8: the routed
    experts as expert_ffn_rows_mxfp8 (x quantised per token row, so a
    sampled row is quantised as in the whole layer); the shared expert stays
    BF16.  map_fn maps the per-expert evaluations (e.g. a thread pool's map;
    the arithmetic is the same).  Returns topk_idx, g, per-route
    a [n][K][I], y [n][K][D], ys and out [n][D]."""
    n = len(tokens)
    topk_idx, g, _ = route(s_rows, K, num)
    X = num.w(x_rows)
    by_expert: Dict[int, list] = {}
    for j in range(n):
        for k in range(K):
            by_expert.setdefault(int(topk_idx[j, k]), []).append((j, k))
    def one_expert(item):
        e, lst = item
        Wg, Wu, Wd = weights.fetch(e)
        rows = np.array([j for j, _ in lst])
        if mxfp8:
            rr = expert_ffn_rows_mxfp8(X[rows], Wg, Wu, Wd)
            return rr["a"], rr["y"]
        return expert_ffn_rows(X[rows], Wg, Wu, Wd, num)[2:]

    items = sorted(by_expert.items())
    a = y = None
    for (e, lst), (ae, ye) in zip(items, map_fn(one_expert, items)):
        if a is None:
            a = np.zeros((n, K, ae.shape[1]), dtype=num.dtype)
            y = np.zeros((n, K, ye.shape[1]), dtype=num.dtype)
        for q, (j, k) in enumerate(lst):
            a[j, k] = ae[q]
            y[j, k] = ye[q]
    ys = None
    if weights.shared is not None:
        ys = shared_ffn(X, *weights.shared, num)
    acc = np.zeros_like(y[:, 0]) if ys is None else np.asarray(ys, dtype=num.dtype).copy()
    for k in range(K):
        acc = acc + np.asarray(g[:, k:k + 1], dtype=num.dtype) * y[:, k]
    out = num.rnd(acc).astype(num.dtype)
    return dict(topk_idx=topk_idx, g=g, a=a, y=y, ys=ys, out=out)


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------
# Bounds on how far another correct evaluation of the backward's products
# (a different fp32 summation order: the tensor cores' K-serial accumulation)
# and of its exponential and division can land from this oracle's, used to
# mark the bf16 rounding points whose decision the arithmetic does not fix.
#   products: |delta| <= sqrt(K) 2^-24 sum_k |a_k b_k| (an fp32 sum of K
#             terms in another order; measured on the GPU: at most 0.18 of it
#             at K = 512 and K = 7168);
#   sigma = 1 / (1 + exp(-h)): relative (8 + 1.2 |h|) 2^-24 (fast exponential
#             and reciprocal on the GPU, libm here);
#   each further product / sum: 8 ulp relative.
_U32 = 2.0 ** -24


def _bf16_range(v, dv):
    """bf16 values that rounding v + e, |e| <= dv, can give: (lo, hi) in
    float32 (equal to round_bf16(v) where the decision is fixed)."""
    v = np.asarray(v, dtype=np.float64)
    lo = round_bf16((v - dv).astype(np.float32))
    hi = round_bf16((v + dv).astype(np.float32))
    return np.minimum(lo, hi), np.maximum(lo, hi)


def rounding_ranges(X, dY, g, Wg, Wu, Wd, h, u, t, a):
    """For rows of one expert: the admissible bf16 values of dh, du, a and
    a_g under the bounds above, as (lo, hi) pairs (lo == hi == the oracle's
    value where the rounding decision is fixed).  All inputs float32 as the
    oracle computed them (Wd is [D][I])."""
    f = lambda z: np.asarray(z, dtype=np.float64)
    X, dY, Wg, Wu, Wd, h, u, t, a = map(f, (X, dY, Wg, Wu, Wd, h, u, t, a))
    gcol = f(g).reshape(-1, 1)
    eps = np.sqrt(X.shape[1]) * _U32
    dh_ = eps * (np.abs(X) @ np.abs(Wg).T)
    du_ = eps * (np.abs(X) @ np.abs(Wu).T)
    dt_ = eps * (np.abs(dY) @ np.abs(Wd))
    sig = 1.0 / (1.0 + np.exp(-h))
    dsig = sig * (8.0 + 1.2 * np.abs(h)) * _U32
    silu_v = h * sig
    dsilu = np.abs(sig * (1.0 + h * (1.0 - sig))) * dh_ + np.abs(h) * dsig
    a_pre = silu_v * u
    da_pre = np.abs(u) * dsilu + np.abs(silu_v) * du_ + 8 * _U32 * np.abs(a_pre)
    sp = sig * (1.0 + h * (1.0 - sig))                       # SiLU'(h)
    dsp = np.abs(sig * (1.0 - sig) * (2.0 + h * (1.0 - 2.0 * sig))) * dh_ + np.abs(1.0 + h - 2.0 * h * sig) * dsig
    dh_pre = gcol * t * u * sp
    ddh = np.abs(gcol) * (np.abs(u * sp) * dt_ + np.abs(t * sp) * du_ + np.abs(t * u) * dsp) + 8 * _U32 * np.abs(dh_pre)
    du_pre = gcol * t * silu_v
    ddu = np.abs(gcol) * (np.abs(silu_v) * dt_ + np.abs(t) * dsilu) + 8 * _U32 * np.abs(du_pre)
    a_lo, a_hi = _bf16_range(a_pre, da_pre)
    ag_ends = np.stack([gcol * a_lo, gcol * a_hi])
    ag_lo, _ = _bf16_range(ag_ends.min(0), 8 * _U32 * np.abs(ag_ends).max(0))
    _, ag_hi = _bf16_range(ag_ends.max(0), 8 * _U32 * np.abs(ag_ends).max(0))
    return dict(dh=_bf16_range(dh_pre, ddh), du=_bf16_range(du_pre, ddu), a=(a_lo, a_hi), a_g=(ag_lo, ag_hi))


def sum_range(vals, rng, other):
    """Range of bf16(sum_p v[p, i] * other[p, j]) shifts when each v[p, i]
    may be any bf16 value in [lo, hi] (rng) instead of vals: returns
    (lo_shift, hi_shift) [I][J] of the fp32 sum before its final rounding."""
    v = np.asarray(vals, dtype=np.float64)
    lo = np.asarray(rng[0], dtype=np.float64) - v
    hi = np.asarray(rng[1], dtype=np.float64) - v
    o = np.asarray(other, dtype=np.float64)
    op, on = np.maximum(o, 0.0), np.minimum(o, 0.0)
    return lo.T @ op + hi.T @ on, hi.T @ op + lo.T @ on


def route_backward_rows(xrows, dyrows, g, Wg, Wu, Wd, num: Numerics = FP32, ranges: bool = False):
    """Backward of g * E_i(x) for a batch of rows of one expert.

    Recomputes h, u (forward replay), t = W_down^T dY; the router-weight
    gradient is dg = <t, SiLU(h) u> ([note] "The production details":
    SonicMoE's inner product of the gated activation with the
    down-projection input gradient; the down-projection output is never
    formed), with the gated activation taken unrounded: the pages put no
    rounding point inside the inner product.  With da = g t and
    SiLU'(h) = sig(h) (1 + h (1 - sig(h))):
        dh = bf16(da * u * SiLU'(h)),  du = bf16(da * SiLU(h)),
        a = bf16(SiLU(h) u), a_g = bf16(g * a),  dx = bf16(dh W_gate + du W_up).
    Returns dict(h, u, a, t, dg, dh, du, a_g, dx); ranges (fp32 numerics):
    also "ranges", rounding_ranges of dh, du, a, a_g."""
    X = num.w(xrows)
    dY = num.w(dyrows)
    gcol = np.asarray(g, dtype=num.dtype).reshape(-1, 1)
    Wg_, Wu_, Wd_ = num.w(Wg), num.w(Wu), num.w(Wd)
    h = X @ Wg_.T
    u = X @ Wu_.T
    a_pre = silu(h) * u
    a = num.rnd(a_pre).astype(num.dtype)
    t = dY @ Wd_
    dg = np.sum(t * a_pre, axis=1)
    da = gcol * t
    one = num.dtype(1)
    with np.errstate(over="ignore"):
        sig = one / (one + np.exp(-h))
    dh = num.rnd(da * u * sig * (one + h * (one - sig))).astype(num.dtype)
    du = num.rnd(da * h * sig).astype(num.dtype)
    a_g = num.rnd(gcol * a).astype(num.dtype)
    dx = num.rnd(dh @ Wg_ + du @ Wu_).astype(num.dtype)
    out = dict(h=h, u=u, a=a, t=t, dg=dg, dh=dh, du=du, a_g=a_g, dx=dx)
    if ranges:
        out["ranges"] = rounding_ranges(X, dY, g, Wg_, Wu_, Wd_, h, u, t, a)
    return out


def router_grad(dg, g, den, topk_idx, E, num: Numerics = FP32):
    """ds[t, j] for the renormalised weights g_k = s_k / den:
    dg_k/ds_j = (delta_kj - g_k) / den, so
    ds[t, topk[t,k]] = (dg[t,k] - sum_k' g[t,k'] dg[t,k']) / den[t], 0 elsewhere."""
    dg = np.asarray(dg, dtype=num.dtype)
    g = np.asarray(g, dtype=num.dtype)
    T, K = g.shape
    dot = np.zeros(T, dtype=num.dtype)
    for k in range(K):
        dot = dot + g[:, k] * dg[:, k]
    ds = np.zeros((T, E), dtype=num.dtype)
    val = (dg - dot[:, None]) / np.asarray(den, dtype=num.dtype)[:, None]
    np.put_along_axis(ds, np.asarray(topk_idx, dtype=np.int64), val, axis=1)
    return ds


def moe_backward(inp: Dict[str, np.ndarray], dy, K: int, num: Numerics = FP32,
                 fwd: Optional[Dict[str, np.ndarray]] = None,
                 routed_rows: Optional[Callable] = None, ranges: bool = False) -> Dict[str, np.ndarray]:
    """Gradients of L = <dY, MoE(x, s)> w.r.t. x, every weight and s.

    Routing is recomputed (or taken from ``fwd``); gradients do not flow
    through the top-k choice.  Per expert (rows [offsets[e], offsets[e+1])):
      dW_down[e] = bf16(sum_p dY_p (x) a_g_p), dW_gate[e] = bf16(sum_p dh_p (x) x_p),
      dW_up[e] = bf16(sum_p du_p (x) x_p);
    the shared expert likewise with g = 1 over all tokens;
    dX[t] = bf16(dx_shared[t] + sum_k dx[route_dst[t,k]]) in k order.

    routed_rows: the per-expert backward of the routed experts (default
    route_backward_rows; moe_backward_mxfp8 passes the MXFP8 one), called
    as routed_rows(x_rows, dy_rows, g_rows, W_gate[e], W_up[e], W_down[e],
    ranges=...).

    ranges (fp32 numerics): also out["range"][name] = (lo_shift, hi_shift)
    of each weight gradient: how far its fp32 sum can move when the dh, du
    or a_g points whose bf16 rounding the arithmetic does not fix
    (rounding_ranges) round the other way, term by term (sum_range)."""
    if fwd is None:
        s = inp["s"]
        topk_idx, g, den = route(s, K, num)
        counts, offsets, table, route_dst = plan(topk_idx, s.shape[1])
    else:
        topk_idx, g, den = fwd["topk_idx"], fwd["g"], fwd["den"]
        offsets, table, route_dst = fwd["offsets"], fwd["table"], fwd["route_dst"]
    E = len(offsets) - 1
    x = num.w(inp["x"])
    dY = num.w(dy)
    T, D = x.shape
    I = inp["w_gate"].shape[1]
    R = T * K
    src_tok = np.asarray(table)[:, 0] // K
    src_k = np.asarray(table)[:, 0] % K
    g_route = np.asarray(g, dtype=num.dtype)[src_tok, src_k]
    dx_r = np.zeros((R, D), dtype=num.dtype)
    dg_route = np.zeros(R, dtype=num.dtype)
    dW_gate = np.zeros((E, I, D), dtype=num.dtype)
    dW_up = np.zeros((E, I, D), dtype=num.dtype)
    dW_down = np.zeros((E, D, I), dtype=num.dtype)
    rng: Dict[str, tuple] = {}
    for e in range(E):
        p0, p1 = int(offsets[e]), int(offsets[e + 1])
        if p0 == p1:
            continue
        rows = src_tok[p0:p1]
        if routed_rows is None:
            b = route_backward_rows(x[rows], dY[rows], g_route[p0:p1],
                                    inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e], num, ranges=ranges)
        else:
            b = routed_rows(x[rows], dY[rows], g_route[p0:p1], inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e],
                            ranges=ranges)
        dx_r[p0:p1] = b["dx"]
        dg_route[p0:p1] = b["dg"]
        dW_down[e] = num.rnd(dY[rows].T @ b["a_g"])
        dW_gate[e] = num.rnd(b["dh"].T @ x[rows])
        dW_up[e] = num.rnd(b["du"].T @ x[rows])
        if ranges:
            rg = b["ranges"]
            for name, (lo, hi) in (("dW_down", sum_range(b["a_g"], rg["a_g"], dY[rows])),
                                   ("dW_gate", sum_range(b["dh"], rg["dh"], x[rows])),
                                   ("dW_up", sum_range(b["du"], rg["du"], x[rows]))):
                if name == "dW_down":
                    lo, hi = lo.T, hi.T
                rng.setdefault(name, (np.zeros(dW_down.shape if name == "dW_down" else dW_gate.shape),
                                      np.zeros(dW_down.shape if name == "dW_down" else dW_gate.shape)))
                rng[name][0][e], rng[name][1][e] = lo, hi
    out = dict(dW_gate=dW_gate, dW_up=dW_up, dW_down=dW_down, dx_r=dx_r)
    acc = np.zeros((T, D), dtype=num.dtype)
    if inp.get("ws_gate") is not None:
        bs = route_backward_rows(x, dY, np.ones(T, dtype=num.dtype),
                                 inp["ws_gate"], inp["ws_up"], inp["ws_down"], num, ranges=ranges)
        acc = bs["dx"].copy()
        out["dWs_down"] = num.rnd(dY.T @ bs["a_g"]).astype(num.dtype)
        out["dWs_gate"] = num.rnd(bs["dh"].T @ x).astype(num.dtype)
        out["dWs_up"] = num.rnd(bs["du"].T @ x).astype(num.dtype)
        if ranges:
            rg = bs["ranges"]
            lo, hi = sum_range(bs["a_g"], rg["a_g"], dY)
            rng["dWs_down"] = (lo.T, hi.T)
            rng["dWs_gate"] = sum_range(bs["dh"], rg["dh"], x)
            rng["dWs_up"] = sum_range(bs["du"], rg["du"], x)
    rd = np.asarray(route_dst).reshape(T, K)
    for k in range(K):
        acc = acc + dx_r[rd[:, k]]
    out["dX"] = num.rnd(acc).astype(num.dtype)
    dg = np.zeros((T, K), dtype=num.dtype)
    dg[src_tok, src_k] = dg_route
    out["dg"] = dg
    out["ds"] = router_grad(dg, g, den, topk_idx, E, num)
    if ranges:
        for name in ("dW_gate", "dW_up", "dW_down"):
            rng.setdefault(name, (np.zeros(out[name].shape), np.zeros(out[name].shape)))
        out["range"] = rng
    return out


def moe_backward_tokens(x_rows, dy_rows, s_rows, weights: HostWeights, K: int, mxfp8: bool = False,
                        map_fn: Callable = map) -> Dict[str, np.ndarray]:
    """The backward restricted to a sample of tokens: dX rows, dg and ds of
    those tokens (each depends only on its own routes), the same steps as
    moe_backward.  Every route of the sample runs route_backward_rows (or
    route_backward_rows_mxfp8) with its expert's weights, grouped by expert;
    the shared expert (BF16, g = 1) runs over the sampled rows; then
    dX = bf16(dx_shared + sum_k dx_k) in k order and ds from dg.  map_fn
    maps the per-expert evaluations.  Returns dX [n][D], dg [n][K], ds [n][E]."""
    num = FP32
    topk_idx, g, den = route(s_rows, K, num)
    n = topk_idx.shape[0]
    X = num.w(x_rows)
    dY = num.w(dy_rows)
    by_expert: Dict[int, list] = {}
    for j in range(n):
        for k in range(K):
            by_expert.setdefault(int(topk_idx[j, k]), []).append((j, k))
    rows_fn = route_backward_rows_mxfp8 if mxfp8 else route_backward_rows

    def one_expert(item):
        e, lst = item
        rows = np.array([j for j, _ in lst])
        ks = np.array([k for _, k in lst])
        b = rows_fn(X[rows], dY[rows], g[rows, ks], *weights.fetch(e))
        return b["dx"], b["dg"]

    items = sorted(by_expert.items())
    dx_route = np.zeros((n, K, X.shape[1]), dtype=np.float32)
    dg = np.zeros((n, K), dtype=np.float32)
    for (e, lst), (dxe, dge) in zip(items, map_fn(one_expert, items)):
        for q, (j, k) in enumerate(lst):
            dx_route[j, k] = dxe[q]
            dg[j, k] = dge[q]
    acc = np.zeros_like(X)
    if weights.shared is not None:
        acc = route_backward_rows(X, dY, np.ones(n, dtype=np.float32), *weights.shared)["dx"].copy()
    for k in range(K):
        acc = acc + dx_route[:, k]
    dX = round_bf16(acc)
    return dict(topk_idx=topk_idx, g=g, dX=dX, dg=dg, ds=router_grad(dg, g, den, topk_idx, s_rows.shape[1]))


# --------------------------------------------------------------------------
# MXFP8 (E4M3 payload, E8M0 1x32 block scales)
# --------------------------------------------------------------------------
def e4m3_code_values() -> np.ndarray:
    """Value of every E4M3 ("fn": bias 7, no infinities, S.1111.111 = NaN)
    byte, as float64; NaN for the two NaN codes."""
    c = np.arange(256)
    sign = np.where(c >> 7, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(ex == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (ex - 7.0))
    v = sign * mag
    v[(c & 0x7F) == 0x7F] = np.nan
    return v


_E4M3_POS = e4m3_code_values()[:127]  # codes 0x00..0x7E, ascending, 0 .. 448


def e4m3_encode(v) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to the even code (even mantissa);
    requires |v| <= 448.  The sign bit is kept, so -0 and negative values that
    round to zero give 0x80."""
    v = np.asarray(v, dtype=np.float64)
    mag = np.abs(v)
    if np.any(mag > 448.0) or np.any(np.isnan(v)):
        raise ValueError("e4m3_encode: |v| must be <= 448")
    hi = np.clip(np.searchsorted(_E4M3_POS, mag, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    d_lo = mag - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return code | (np.signbit(v).astype(np.uint8) << np.uint8(7))


def e4m3_round(v) -> np.ndarray:
    """The value e4m3_encode picks, computed without codes: E4M3 keeps 3
    mantissa bits, so in binade [2^q, 2^(q+1)) (q >= -6) its values are
    n 2^(q-3) for integers n in [8, 16), and below 2^-6 the subnormals are
    n 2^-9 (n in [0, 8)).  Rounding |v| / step to the nearest integer with
    ties to even is ties to the even mantissa in both cases (n even iff the
    mantissa is even; n = 16 is the next binade's even mantissa 0).
    |v| <= 448; float64 out, sign kept."""
    v = np.asarray(v, dtype=np.float64)
    mag = np.abs(v)
    if np.any(mag > 448.0) or np.any(np.isnan(v)):
        raise ValueError("e4m3_round: |v| must be <= 448")
    _, q = np.frexp(mag)  # mag = m 2^q with m in [0.5, 1): binade 2^(q - 1)
    step = np.ldexp(1.0, np.maximum(q - 1, -6) - 3)
    return np.copysign(np.rint(mag / step) * step, v)


def mx_scale_exponent(amax) -> np.ndarray:
    """Smallest integer e with amax <= 448 * 2^e, from frexp (no floating
    log2): amax = m 2^q with m in [0.5, 1) and 448 = 0.875 * 2^9, so
    e = q - 9 when m <= 0.875, else q - 8.  amax = 0 gives -127; clamped to
    the E8M0 range [-127, 127]."""
    amax = np.asarray(amax, dtype=np.float64)
    m, q = np.frexp(amax)
    e = np.where(m <= 0.875, q - 9, q - 8)
    e = np.where(amax == 0.0, -127, e)
    return np.clip(e, -127, 127).astype(np.int32)


def mxfp8_quantize(v) -> Tuple[np.ndarray, np.ndarray]:
    """Quantise along the last axis in 1x32 blocks: codes uint8 (same shape)
    and E8M0 scale bytes uint8 [..., n/32] (byte = e + 127)."""
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[-1]
    if n % 32:
        raise ValueError("last dim must be a multiple of 32")
    blocks = v.reshape(v.shape[:-1] + (n // 32, 32))
    e = mx_scale_exponent(np.max(np.abs(blocks), axis=-1))
    scaled = blocks * np.ldexp(1.0, -e)[..., None]
    codes = e4m3_encode(scaled).reshape(v.shape)
    return codes, (e + 127).astype(np.uint8)


def mxfp8_dequantize(codes, scales) -> np.ndarray:
    """codes * 2^(scale - 127), float64 (exact)."""
    codes = np.asarray(codes, dtype=np.uint8)
    n = codes.shape[-1]
    vals = e4m3_code_values()[codes].reshape(codes.shape[:-1] + (n // 32, 32))
    e = np.asarray(scales, dtype=np.int32) - 127
    return (vals * np.ldexp(1.0, e)[..., None]).reshape(codes.shape)


def expert_ffn_rows_mxfp8(xrows, Wg, Wu, Wd):
    """One expert's FFN with MXFP8 operands for a batch of rows ([note]
    "The production details"): x quantised per row along D, W_gate / W_up
    along D, W_down along I, a = bf16(SiLU(h) u) quantised along I; every
    GEMM contracts the exactly dequantised values in fp32.  Inputs are bf16
    bits (or float values).  Returns dict(a_pre, a, aq, asc, y)."""
    X, Wgd, Wud, Wdd = (mxfp8_roundtrip(FP32.w(v)) for v in (xrows, Wg, Wu, Wd))
    h = X @ Wgd.T
    u = X @ Wud.T
    a_pre = silu(h) * u
    a = round_bf16(a_pre)
    aq, asc = mxfp8_quantize(a)
    y = round_bf16(mxfp8_dequantize(aq, asc).astype(np.float32) @ Wdd.T)
    return dict(a_pre=a_pre, a=a, aq=aq, asc=asc, y=y)


def moe_forward_mxfp8(inp: Dict[str, np.ndarray], K: int, quant: Optional[Dict[str, tuple]] = None,
                      experts: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """The layer with routed experts in MXFP8 ([note] "The production details":
    quantisation fused into dispatch, the grouped GEMMs and the gated
    activation; the shared expert stays BF16).

    x is quantised per token row along D; W_gate, W_up along D; W_down along I;
    a = bf16(SiLU(h) u) is quantised along I before the down projection.  Each
    GEMM contracts the exactly dequantised values in fp32.  ``quant`` may hold
    precomputed (codes, scales) of the weights keyed 'w_gate', 'w_up', 'w_down'.
    ``experts`` restricts the routed FFN to a subset (other rows stay zero)."""
    num = FP32
    s = inp["s"]
    E = s.shape[1]
    topk_idx, g, den = route(s, K, num)
    counts, offsets, table, route_dst = plan(topk_idx, E)
    x = num.w(inp["x"])
    xq, xs = mxfp8_quantize(x)
    xd = mxfp8_dequantize(xq, xs).astype(np.float32)
    xg_d = gather(xd, table, K)
    R, D = xg_d.shape
    I = inp["w_gate"].shape[1]
    a = np.zeros((R, I), dtype=np.float32)
    aq = np.zeros((R, I), dtype=np.uint8)
    asc = np.zeros((R, I // 32), dtype=np.uint8)
    y = np.zeros((R, D), dtype=np.float32)
    quant = quant or {}
    todo = range(E) if experts is None else experts
    for e in todo:
        p0, p1 = int(offsets[e]), int(offsets[e + 1])
        if p0 == p1:
            continue
        if "w_gate" in quant:
            Wg = mxfp8_dequantize(quant["w_gate"][0][e], quant["w_gate"][1][e])
            Wu = mxfp8_dequantize(quant["w_up"][0][e], quant["w_up"][1][e])
            Wd = mxfp8_dequantize(quant["w_down"][0][e], quant["w_down"][1][e])
        else:
            Wg = mxfp8_roundtrip(bf16_to_f32(inp["w_gate"][e]))
            Wu = mxfp8_roundtrip(bf16_to_f32(inp["w_up"][e]))
            Wd = mxfp8_roundtrip(bf16_to_f32(inp["w_down"][e]))
        X = xg_d[p0:p1]
        h = X @ Wg.astype(np.float32).T
        u = X @ Wu.astype(np.float32).T
        ae = round_bf16(silu(h) * u)
        qe, se = mxfp8_quantize(ae)
        a[p0:p1], aq[p0:p1], asc[p0:p1] = ae, qe, se
        y[p0:p1] = round_bf16(mxfp8_dequantize(qe, se).astype(np.float32) @ Wd.astype(np.float32).T)
    ys = None
    if inp.get("ws_gate") is not None:
        ys = shared_ffn(x, inp["ws_gate"], inp["ws_up"], inp["ws_down"], num)
    out = combine(y, ys, g, route_dst, num)
    return dict(topk_idx=topk_idx, g=g, counts=counts, offsets=offsets, table=table, route_dst=route_dst,
                xq=xq, xs=xs, a=a, aq=aq, asc=asc, y=y, ys=ys, out=out)


def mxfp8_roundtrip(v) -> np.ndarray:
    """Quantise along the last axis and dequantise exactly, as float32: the
    values a block-scaled GEMM contracts.  The same values as
    mxfp8_dequantize(*mxfp8_quantize(v)), taken through e4m3_round (no codes)."""
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[-1]
    if n % 32:
        raise ValueError("last dim must be a multiple of 32")
    blocks = v.reshape(v.shape[:-1] + (n // 32, 32))
    e = mx_scale_exponent(np.max(np.abs(blocks), axis=-1))[..., None]
    vals = np.ldexp(e4m3_round(np.ldexp(blocks, -e)), e)
    return vals.reshape(v.shape).astype(np.float32)


def route_backward_rows_mxfp8(xrows, dyrows, g, Wg, Wu, Wd, deq: Optional[Callable] = None, ranges: bool = False):
    """Backward of g * E_i(x) for rows of one expert with MXFP8 routed GEMMs
    ([note] "The production details": MXFP8 with quantisation fused into the
    dispatch, the grouped GEMMs and the gated activation; the router gradient
    as the inner product of the gated activation with the down-projection
    input gradient).  Each GEMM contracts operands quantised along its own
    reduction dim, exactly dequantised, in fp32:
      replay  h = X W_gate^T, u = X W_up^T : x, W_gate, W_up along D (the
              forward's quantisation);
      t = dY W_down                        : dY along D, W_down^T along D;
      dx = [dh | du] [W_gate ; W_up]       : [dh | du] along 2I,
              [W_gate^T | W_up^T] along 2I; dx = bf16.
    h, u and t stay the fp32 products: the pages put no rounding point
    there.  The activation gradient is the BF16 backward's, on those values:
      a = bf16(SiLU(h) u), dg = <t, SiLU(h) u> (unrounded), da = g t,
      dh = bf16(da u SiLU'(h)), du = bf16(da SiLU(h)), a_g = bf16(g a).
    ``deq`` is the quantise-dequantise step along the last axis (default
    mxfp8_roundtrip); the identity turns the quantisation off.  Inputs are
    bf16 bits or float values.  Returns dict(h, u, a, t, dg, dh, du, a_g, dx)
    and with ranges also rounding_ranges of dh, du, a, a_g (products of the
    quantised operands)."""
    deq = mxfp8_roundtrip if deq is None else deq
    X = deq(FP32.w(xrows))
    dY = deq(FP32.w(dyrows))
    gcol = np.asarray(g, dtype=np.float32).reshape(-1, 1)
    Wg_, Wu_, Wd_ = FP32.w(Wg), FP32.w(Wu), FP32.w(Wd)
    Wgq, Wuq, WdqT = deq(Wg_), deq(Wu_), deq(np.ascontiguousarray(Wd_.T))
    h = X @ Wgq.T
    u = X @ Wuq.T
    t = dY @ WdqT.T
    a_pre = silu(h) * u
    a = round_bf16(a_pre)
    dg = np.sum(t * a_pre, axis=1, dtype=np.float32)
    da = gcol * t
    one = np.float32(1)
    with np.errstate(over="ignore"):
        sig = one / (one + np.exp(-h))
    dh = round_bf16(da * u * sig * (one + h * (one - sig)))
    du = round_bf16(da * h * sig)
    a_g = round_bf16(gcol * a)
    dhu = deq(np.concatenate([dh, du], axis=1))
    wgu_t = deq(np.concatenate([Wg_.T, Wu_.T], axis=1))  # [D][2I]
    dx = round_bf16(dhu @ wgu_t.T)
    out = dict(h=h, u=u, a=a, t=t, dg=dg, dh=dh, du=du, a_g=a_g, dx=dx)
    if ranges:
        out["ranges"] = rounding_ranges(X, dY, g, Wgq, Wuq, np.ascontiguousarray(WdqT.T), h, u, t, a)
    return out


def moe_backward_mxfp8(inp: Dict[str, np.ndarray], dy, K: int,
                       fwd: Optional[Dict[str, np.ndarray]] = None,
                       deq: Optional[Callable] = None, ranges: bool = False) -> Dict[str, np.ndarray]:
    """The backward with the routed experts' GEMMs in MXFP8
    (route_backward_rows_mxfp8); the weight gradients are BF16 products of
    the bf16 x, dY and the MXFP8 path's bf16 dh, du, a_g, as in moe_backward;
    the shared expert is BF16 ([note] "The production details")."""
    return moe_backward(inp, dy, K, FP32, fwd=fwd, ranges=ranges,
                        routed_rows=lambda *a, ranges=False: route_backward_rows_mxfp8(*a, deq=deq, ranges=ranges))
