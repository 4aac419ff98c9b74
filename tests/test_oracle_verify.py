"""Pins of the oracle's verification (no GPU).

Losslessness ("the distribution is mathematically identical to running the
target model alone", kimi-k3-dspark-gguf intro) is pinned by exact
enumeration: every uniform of the verify step acts through a threshold or a
monotone map, so each outcome owns an integer interval of uniform values. The
intervals are found by bisection on the oracle itself (black box), and the
emitted-token distribution they imply must equal the target's.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import identities as I
from oracle import sampling as S

U32 = 1 << 32
W24 = 1 << 24


def test_greedy_accept_length_two_ways():
    rng = np.random.default_rng(0)
    B, V = 7, 50
    for trial in range(200):
        P = rng.standard_normal((B + 1, V)).astype(np.float32)
        g = [int(np.argmax(P[i])) for i in range(B + 1)]
        k = int(rng.integers(0, B + 1))
        tokens = np.array([g[i] if i < k else (g[i] + 1 + int(rng.integers(0, V - 1))) % V
                           for i in range(B)], dtype=np.int32)
        if trial % 3 == 0:  # matches after the first mismatch do not count
            tokens[min(k + 1, B - 1):] = np.array(g[min(k + 1, B - 1):B])
        a, out = S.verify_greedy(P, tokens)
        match = [int(tokens[i]) == g[i] for i in range(B)]
        assert a == I.accepted_prefix(match) == I.accepted_prefix_by_products(match)
        assert out[:a].tolist() == tokens[:a].tolist()
        assert out[a] == g[a]
        assert np.all(out[a + 1:] == -1)


def test_equal_distributions_always_accept():
    rng = np.random.default_rng(1)
    B, V = 7, 64
    ell = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    P = np.concatenate([ell, rng.standard_normal((1, V)).astype(np.float32)])
    for step in range(20):
        tokens = rng.integers(0, V, B).astype(np.int32)
        E = [S.row_weights(ell[i], 1.0) for i in range(B)]
        ok = all(E[i][tokens[i]] > 0 for i in range(B))
        a, out = S.verify_prob(P, ell, tokens, 0, 1.0, 1.0, seed=3, seq=0, step=step)
        if ok:
            assert a == B and out[:B].tolist() == tokens.tolist()


def _dist(logits, T, top_p):
    """Exact target/draft distribution of the spec as Fractions (from the oracle's weights)."""
    E = S.row_weights(np.asarray(logits, dtype=np.float32), T)
    nu = S.nucleus(E, top_p)
    keys = (E.astype(object) << 18) | np.array([(1 << 18) - 1 - v for v in range(E.size)], dtype=object)
    return [Fraction(int(E[v]), nu.Sn) if keys[v] >= nu.kstar else Fraction(0) for v in range(E.size)]


def _first(pred, lo, hi):
    """Smallest x in [lo, hi) with pred(x) true (pred monotone), hi if none."""
    while lo < hi:
        mid = (lo + hi) // 2
        if pred(mid):
            hi = mid
        else:
            lo = mid + 1
    return lo


def _interval_dist(f, V):
    """Probabilities of a monotone non-decreasing map W (24-bit) -> token."""
    out = [Fraction(0)] * V
    start = 0
    for v in range(V):
        end = _first(lambda w: f(w) > v, start, W24)
        out[v] = Fraction(end - start, W24)
        start = end
    assert start == W24
    return out


def _enumerate(P_of, ell_of, q_tables, V, B, T, top_p, draft_greedy):
    """Exact emitted-token law of the oracle's verify for every draft sequence.

    Returns first[v] = P(out[0] = v) and, for B = 2, nxt[v][w] = P(out[1] = w | accept_len >= 1, out[0] = v).
    """
    first = [Fraction(0)] * V
    reach = [Fraction(0)] * V
    nxt = [[Fraction(0)] * V for _ in range(V)]
    bonus_ok = True

    def run(t, U, Wres, Wb):
        P = P_of(t)
        ell = ell_of(t)
        return S.verify_prob_core(P, ell, np.array(t, dtype=np.int32), draft_greedy, T, top_p,
                                  np.array(U, dtype=np.uint32), np.array(Wres, dtype=np.uint32), Wb)

    drafts = [(t1,) for t1 in range(V)] if B == 1 else [(t1, t2) for t1 in range(V) for t2 in range(V)]
    for t in drafts:
        q1 = q_tables[0]
        prob_t = q1[t[0]]
        if B == 2:
            prob_t *= q_tables[1][t[0]][t[1]]
        if prob_t == 0:
            continue
        # position 1: acceptance threshold on U1
        thr1 = _first(lambda u: run(t, [u] + [0] * (B - 1), [0] * B, 0)[0] < 1, 0, U32)
        acc1 = Fraction(thr1, U32)
        if thr1 < U32:
            res1 = _interval_dist(lambda w: run(t, [U32 - 1] + [0] * (B - 1), [w] + [0] * (B - 1), 0)[1][0], V)
            for v in range(V):
                first[v] += prob_t * (1 - acc1) * res1[v]
        first[t[0]] += prob_t * acc1
        if B == 1:
            if thr1 > 0:
                bon = _interval_dist(lambda w: run(t, [0], [0], w)[1][1], V)
                exp = _dist(P_of(t)[1], T, top_p)
                bonus_ok &= all(abs(bon[v] - exp[v]) <= Fraction(1, W24) for v in range(V))
            continue
        if thr1 == 0:
            continue
        reach[t[0]] += prob_t * acc1
        thr2 = _first(lambda u: run(t, [0, u], [0, 0], 0)[0] < 2, 0, U32)
        acc2 = Fraction(thr2, U32)
        if thr2 < U32:
            res2 = _interval_dist(lambda w: run(t, [0, U32 - 1], [0, w], 0)[1][1], V)
            for w in range(V):
                nxt[t[0]][w] += prob_t * acc1 * (1 - acc2) * res2[w]
        nxt[t[0]][t[1]] += prob_t * acc1 * acc2
        if thr2 > 0:
            bon = _interval_dist(lambda w: run(t, [0, 0], [0, 0], w)[1][2], V)
            exp = _dist(P_of(t)[2], T, top_p)
            bonus_ok &= all(abs(bon[v] - exp[v]) <= Fraction(1, W24) for v in range(V))
    for v in range(V):
        if reach[v] > 0:
            nxt[v] = [x / reach[v] for x in nxt[v]]
    return first, nxt, bonus_ok, reach


@pytest.mark.parametrize("V,B,T,top_p,draft_greedy,seed", [
    (3, 1, 1.0, 1.0, 0, 0),
    (4, 1, 0.8, 0.9, 0, 1),
    (5, 1, 1.0, 0.95, 1, 2),
    (3, 2, 1.0, 1.0, 0, 3),
    (4, 2, 1.3, 0.85, 0, 4),
    (3, 2, 1.0, 0.95, 1, 5),
])
def test_verify_is_lossless_by_exact_enumeration(V, B, T, top_p, draft_greedy, seed):
    rng = np.random.default_rng(seed)
    lp = lambda: (rng.standard_normal(V) * 1.5).astype(np.float32)
    # prefix-conditional target tables p(.), p(.|t1), p(.|t1,t2) and draft tables q(.), q(.|t1)
    p1 = lp()
    p2 = {a: lp() for a in range(V)}
    p3 = {(a, b): lp() for a in range(V) for b in range(V)}
    q1 = lp()
    q2 = {a: lp() for a in range(V)}
    if B == 1:
        P_of = lambda t: np.stack([p1, p2[t[0]]])
        ell_of = lambda t: np.stack([q1])
    else:
        P_of = lambda t: np.stack([p1, p2[t[0]], p3[(t[0], t[1])]])
        ell_of = lambda t: np.stack([q1, q2[t[0]]])
    if draft_greedy:
        qd1 = [Fraction(int(v == S.argmax(q1))) for v in range(V)]
        qd2 = {a: [Fraction(int(v == S.argmax(q2[a]))) for v in range(V)] for a in range(V)}
    else:
        qd1 = _dist(q1, T, top_p)
        qd2 = {a: _dist(q2[a], T, top_p) for a in range(V)}
    first, nxt, bonus_ok, reach = _enumerate(P_of, ell_of, [qd1, qd2], V, B, T, top_p, draft_greedy)
    tol = Fraction(V, W24)
    target1 = _dist(p1, T, top_p)
    assert all(abs(first[v] - target1[v]) <= tol for v in range(V)), (first, target1)
    assert bonus_ok
    if B == 2:
        assert any(r > 0 for r in reach)
        for v in range(V):
            if reach[v] == 0:  # no accepted draft can emit v first (e.g. a greedy draft)
                continue
            t2 = _dist(p2[v], T, top_p)
            assert all(abs(nxt[v][w] - t2[w]) <= tol for w in range(V)), (v, nxt[v], t2)


def test_probabilistic_verify_uses_spec_uniforms():
    rng = np.random.default_rng(8)
    B, V = 7, 200
    ell = (rng.standard_normal((B, V)) * 1.5).astype(np.float32)
    P = (np.concatenate([ell, ell[-1:]]) + rng.standard_normal((B + 1, V)) * 0.5).astype(np.float32)
    tokens = np.array([S.argmax(ell[i]) for i in range(B)], dtype=np.int32)
    for step in range(10):
        a, out = S.verify_prob(P, ell, tokens, 0, 1.0, 0.95, seed=42, seq=3, step=step)
        U = [S.uniform_u32(42, 3, step, i, 2) for i in range(B)]
        Wr = [S.uniform_u32(42, 3, step, i, 3) >> 8 for i in range(B)]
        Wb = S.uniform_u32(42, 3, step, B, 4) >> 8
        a2, out2 = S.verify_prob_core(P, ell, tokens, 0, 1.0, 0.95, U, Wr, Wb)
        assert a == a2 and np.array_equal(out, out2)
        assert 0 <= a <= B and np.all(out[a + 1:] == -1) and 0 <= out[a] < V


def test_planted_role_swap_fails_the_enumeration(monkeypatch):
    """A verify that swaps the target's and the draft's roles (accepting with q/p and
    resampling from max(0, q - p)), planted on the CPU, no longer reproduces the
    target's law under exact enumeration."""
    real = S.verify_prob_core

    def swapped(P, ell, tokens, draft_greedy, T, top_p, U, Wres, Wbonus):
        B = ell.shape[0]
        P2 = np.concatenate([ell, P[B:]], axis=0).astype(np.float32)
        return real(P2, np.ascontiguousarray(P[:B]), tokens, draft_greedy, T, top_p, U, Wres, Wbonus)

    monkeypatch.setattr(S, "verify_prob_core", swapped)
    V, T, top_p = 3, 1.0, 1.0
    rng = np.random.default_rng(21)
    p1 = (rng.standard_normal(V) * 1.5).astype(np.float32)
    p2 = (rng.standard_normal(V) * 1.5).astype(np.float32)
    q1 = (rng.standard_normal(V) * 1.5).astype(np.float32)
    first, _, _, _ = _enumerate(lambda t: np.stack([p1, p2]), lambda t: np.stack([q1]), [_dist(q1, T, top_p), {}],
                                V, 1, T, top_p, 0)
    target1 = _dist(p1, T, top_p)
    assert max(abs(first[v] - target1[v]) for v in range(V)) > Fraction(1, 100)
