"""Pins of the oracle's routing and plan.

route -> repeated-argmax brute force (lowest index on ties), exact g special
cases, sum g = 1; plan -> numpy's stable argsort (a library counting-sort
equivalent) plus the plan invariants; the general pull schedule -> Python's
sorted() on the key (local expert, per-source ordinal, source rank).
"""
import numpy as np
import pytest

import oracle as O


def _brute_topk(row, K):
    chosen = []
    for _ in range(K):
        best = None
        for e, v in enumerate(row):
            if e in chosen:
                continue
            if best is None or v > row[best]:
                best = e
        chosen.append(best)
    return chosen


def test_route_matches_repeated_argmax():
    rng = np.random.default_rng(0)
    for T, E, K in [(64, 8, 2), (32, 16, 4), (16, 5, 5), (16, 7, 1)]:
        s = rng.random((T, E), dtype=np.float32)
        idx, g, den = O.route(s, K)
        for t in range(T):
            assert list(idx[t]) == _brute_topk(list(s[t]), K)


def test_route_ties_lowest_index_first():
    s = np.array([[0.1, 0.3, 0.3, 0.2, 0.3],
                  [0.2, 0.2, 0.2, 0.2, 0.2],
                  [0.0, 0.0, 0.5, 0.0, 0.0]], dtype=np.float32)
    idx, g, _ = O.route(s, 2)
    assert idx.tolist() == [[1, 2], [0, 1], [2, 0]]
    idx3, _, _ = O.route(s, 3)
    assert idx3.tolist() == [[1, 2, 4], [0, 1, 2], [2, 0, 1]]
    for t in range(3):
        assert list(idx3[t]) == _brute_topk(list(s[t]), 3)


def test_route_g_exact_cases():
    rng = np.random.default_rng(5)
    s = rng.random((50, 9), dtype=np.float32) + np.float32(0.01)
    _, g1, _ = O.route(s, 1)
    assert np.all(g1 == 1.0)
    for K in (2, 4):
        eq = np.full((4, 6), 0.125, dtype=np.float32)
        _, g, _ = O.route(eq, K)
        assert np.all(g == np.float32(1.0 / K))
    _, g, _ = O.route(np.array([[0.375, 0.125, 0.0625]], dtype=np.float32), 2)
    assert g.tolist() == [[0.75, 0.25]]


def test_route_g_sums_to_one():
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((1000, 64)).astype(np.float32)
    s = np.exp(logits) / np.exp(logits).sum(1, keepdims=True)
    for K in (2, 8):
        _, g, _ = O.route(s.astype(np.float32), K)
        assert np.all(np.abs(g.sum(1, dtype=np.float64) - 1.0) <= K * 2.0 ** -23)
        assert np.all(np.diff(g, axis=1) <= 0)


def _random_topk(rng, T, E, K, skew=0.0):
    logits = rng.standard_normal((T, E)) - skew * np.log(np.arange(1, E + 1))
    s = np.exp(logits)
    s /= s.sum(1, keepdims=True)
    return O.route(s.astype(np.float32), K)[0]


@pytest.mark.parametrize("T,E,K,skew", [(256, 8, 2, 0.0), (300, 16, 4, 2.0), (97, 5, 3, 0.0), (1, 4, 4, 0.0)])
def test_plan_matches_stable_sort_and_invariants(T, E, K, skew):
    rng = np.random.default_rng(T + E)
    idx = _random_topk(rng, T, E, K, skew)
    counts, offsets, table, route_dst = O.plan(idx, E)
    flat = idx.reshape(-1)
    R = T * K
    assert np.array_equal(table[:, 0], np.argsort(flat, kind="stable"))
    assert counts.sum() == R and np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and offsets[E] == R and np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(table[:, 2], np.arange(R))
    assert np.array_equal(table[:, 1], flat[table[:, 0]])
    assert np.all(np.diff(table[:, 1]) >= 0)
    assert np.array_equal(np.sort(table[:, 0]), np.arange(R))
    assert np.array_equal(route_dst[table[:, 0]], np.arange(R))
    for e in range(E):
        src = table[offsets[e]:offsets[e + 1], 0]
        assert np.all(np.diff(src) > 0)


def test_plan_skewed_has_empty_experts():
    rng = np.random.default_rng(11)
    idx = _random_topk(rng, 512, 128, 8, skew=2.0)
    counts, offsets, table, _ = O.plan(idx, 128)
    assert (counts == 0).any() and counts[0] == 512


def test_plan_rejects_bad_expert():
    with pytest.raises(ValueError):
        O.plan(np.array([[0, 9]], dtype=np.int32), 8)


@pytest.mark.parametrize("R,N,K,L,c", [(3, 5, 2, 4, 1), (4, 7, 3, 3, 0), (2, 9, 4, 2, 2), (5, 3, 1, 4, 3)])
def test_pull_schedule_matches_sort_key(R, N, K, L, c):
    rng = np.random.default_rng(R * 100 + N)
    n_ranks_total = max(c + 1, 4)
    routing = rng.integers(0, n_ranks_total * L, size=(R, N, K))
    Tcnt, M, S, Phi = O.pull_schedule(routing, c, L)
    keyed = []
    ordinal = {}
    for r in range(R):
        for i in range(N):
            for k in range(K):
                e = int(routing[r, i, k])
                if e // L != c:
                    continue
                l = e - c * L
                o = ordinal.get((l, r), 0)
                ordinal[(l, r)] = o + 1
                keyed.append(((l, o, r), (r, i * K + k)))
    want = [v for _, v in sorted(keyed)]
    assert [tuple(map(int, p)) for p in Phi] == want
    assert Tcnt.sum() == len(want)
    assert np.array_equal(M.sum(1), Tcnt)
    assert np.array_equal(S, np.concatenate([[0], np.cumsum(Tcnt)[:-1]]))


def test_pull_schedule_one_rank_is_plan():
    rng = np.random.default_rng(3)
    idx = _random_topk(rng, 40, 6, 2)
    Tc, M, S, Phi = O.pull_schedule(idx[None], 0, 6)
    _, offsets, table, _ = O.plan(idx, 6)
    assert np.array_equal(Phi[:, 1], table[:, 0]) and np.all(Phi[:, 0] == 0)
    assert np.array_equal(S, offsets[:-1])


def test_route_many_ties_wide_rows():
    """Rows of 256 scores drawn from 3 levels: ties everywhere."""
    rng = np.random.default_rng(12)
    s = rng.choice(np.array([0.25, 0.5, 0.125], dtype=np.float32), size=(64, 256))
    idx, _, _ = O.route(s, 8)
    for t in range(64):
        assert list(idx[t]) == _brute_topk(list(s[t]), 8)
