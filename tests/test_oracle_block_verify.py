"""Pins of the oracle's block verification (no GPU).

Losslessness by exact enumeration: for every drafted block, the acceptance
decisions are thresholds on 32-bit uniforms (their exact probabilities follow
from h_i) and the final token is a monotone map of a 24-bit uniform (its law is
found by bisection on the oracle itself). The law of the emitted sequence must
make every emitted token, given the tokens before it, distributed as the
target's row for that prefix ("kimi-k3-dspark-gguf" intro: the distribution is
identical to the target alone). Block verification must also accept at least as
many tokens on average as token-by-token verification (the point of the method,
"Kimi-K3-DSpark-NVFP4", Sampling options), and strictly more somewhere.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import sampling as S

U32 = 1 << 32
W24 = 1 << 24


def _dist(logits, T, top_p):
    E = S.row_weights(np.asarray(logits, dtype=np.float32), T)
    nu = S.nucleus(E, top_p)
    keys = (E.astype(object) << 18) | np.array([(1 << 18) - 1 - v for v in range(E.size)], dtype=object)
    return [Fraction(int(E[v]), nu.Sn) if keys[v] >= nu.kstar else Fraction(0) for v in range(E.size)]


def _first(pred, lo, hi):
    while lo < hi:
        mid = (lo + hi) // 2
        if pred(mid):
            hi = mid
        else:
            lo = mid + 1
    return lo


def _interval_dist(f, V):
    out, start = [Fraction(0)] * V, 0
    for v in range(V):
        end = _first(lambda w: f(w) > v, start, W24)
        out[v] = Fraction(end - start, W24)
        start = end
    assert start == W24
    return out


def _p_eta(h):
    """P(U < h * 2^32) for a uniform 32-bit U."""
    return Fraction(min(U32, math.ceil(Fraction(h) * U32)), U32)


def _tables(V, B, rng):
    lp = lambda: (rng.standard_normal(V) * 1.5).astype(np.float32)
    target = {pre: lp() for n in range(B + 1) for pre in itertools.product(range(V), repeat=n)}
    draft = {pre: lp() for n in range(B) for pre in itertools.product(range(V), repeat=n)}
    return target, draft


def _law(V, B, T, top_p, dg, target, draft):
    """Exact law of the emitted sequence, and E[tau] of block and of token-by-token verification."""
    qd = {pre: ([Fraction(int(v == S.argmax(draft[pre]))) for v in range(V)] if dg else _dist(draft[pre], T, top_p))
          for pre in draft}
    law, e_block, e_token = {}, Fraction(0), Fraction(0)
    for t in itertools.product(range(V), repeat=B):
        qt = Fraction(1)
        for i in range(B):
            qt *= qd[t[:i]][t[i]]
        if qt == 0:
            continue
        P = np.stack([target[t[:i]] for i in range(B + 1)])
        ell = np.stack([draft[t[:i]] for i in range(B)])
        pi, h = S.block_stats(P, ell, t, dg, T, top_p)
        pe = [None] + [_p_eta(h[i]) for i in range(1, B + 1)]
        # token-by-token: position i accepted with min(1, p/q) given the earlier ones
        acc, run = Fraction(0), Fraction(1)
        for i in range(B):
            pt = _dist(target[t[:i]], T, top_p)[t[i]]
            run *= min(Fraction(1), pt / qd[t[:i]][t[i]])
            acc += run
        e_token += qt * acc
        core = lambda U, Wr, Wb: S.verify_block_core(P, ell, t, dg, T, top_p, U, Wr, Wb)
        for j in range(B + 1):
            pj = pe[j] if j > 0 else Fraction(1)
            for k in range(j + 1, B + 1):
                pj *= 1 - pe[k]
            if pj == 0:
                continue
            e_block += qt * pj * j
            U = [0 if i + 1 == j else (U32 - 1 if i + 1 > j else 0) for i in range(B)]
            assert core(U, [0] * B, 0)[0] == j
            if j == B:
                tok = _interval_dist(lambda w: core(U, [0] * B, w)[1][B], V)
            else:
                tok = _interval_dist(lambda w: core(U, [w if i == j else 0 for i in range(B)], 0)[1][j], V)
            for y in range(V):
                if tok[y]:
                    seq = t[:j] + (y,)
                    law[seq] = law.get(seq, Fraction(0)) + qt * pj * tok[y]
    return law, e_block, e_token


@pytest.mark.parametrize("V,B,T,top_p,dg,seed", [
    (3, 1, 1.0, 1.0, 0, 0),
    (3, 2, 1.0, 1.0, 0, 1),
    (4, 2, 0.8, 0.9, 0, 2),
    (3, 3, 1.0, 1.0, 0, 3),
    (3, 2, 1.0, 0.95, 1, 4),
    (4, 3, 1.3, 0.85, 0, 5),
])
def test_block_verify_is_lossless_by_exact_enumeration(V, B, T, top_p, dg, seed):
    rng = np.random.default_rng(seed)
    target, draft = _tables(V, B, rng)
    law, _, _ = _law(V, B, T, top_p, dg, target, draft)
    assert abs(sum(law.values()) - 1) < Fraction(1, 10 ** 12)
    tol = Fraction(4 * V, W24)
    for n in range(1, B + 2):
        reach, nxt = {}, {}  # P(len >= n, first n - 1 tokens), P(len >= n, first n tokens)
        for seq, pr in law.items():
            if len(seq) >= n:
                reach[seq[:n - 1]] = reach.get(seq[:n - 1], Fraction(0)) + pr
                nxt[seq[:n]] = nxt.get(seq[:n], Fraction(0)) + pr
        assert n > 1 or reach[()] == sum(law.values())
        for pre, r in reach.items():
            want = _dist(target[pre], T, top_p)
            for y in range(V):
                got = nxt.get(pre + (y,), Fraction(0))
                assert abs(got - r * want[y]) <= tol, (n, pre, y, float(got), float(r * want[y]))


def test_block_accepts_at_least_as_much_as_token_verification():
    gains = []
    for seed in range(6):
        rng = np.random.default_rng(100 + seed)
        target, draft = _tables(3, 3, rng)
        _, eb, et = _law(3, 3, 1.0, 1.0, 0, target, draft)
        assert eb >= et - Fraction(3 * 3, U32), (seed, float(eb), float(et))
        gains.append(float(eb - et))
    assert max(gains) > 1e-3


def test_equal_distributions_accept_the_whole_block():
    rng = np.random.default_rng(9)
    B, V = 7, 64
    ell = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    P = np.concatenate([ell, rng.standard_normal((1, V)).astype(np.float32)])
    for step in range(10):
        tokens = np.array([S.sample_nucleus(S.row_weights(ell[i], 1.0), 0, int(S.row_weights(ell[i], 1.0).sum()),
                                            (step * 7919 + i * 104729) % W24) for i in range(B)], dtype=np.int32)
        pi, h = S.block_stats(P, ell, tokens, 0, 1.0, 1.0)
        assert np.all(pi == 1.0) and h[B] == 1.0
        a, out = S.verify_block(P, ell, tokens, 0, 1.0, 1.0, seed=5, seq=0, step=step)
        assert a == B and out[:B].tolist() == tokens.tolist()
