"""Pins of the oracle's uniforms, own exp and sampling spec (no GPU)."""
import math

import numpy as np
import pytest

from oracle import sampling as S
from tests.helpers import golden


def test_philox_known_answers():
    g = golden("philox_kat.json")
    for vec in g["vectors"]:
        ctr = [int(x, 16) for x in vec["ctr"]]
        key = [int(x, 16) for x in vec["key"]]
        out = [int(x, 16) for x in vec["out"]]
        assert list(S.philox4x32_10(ctr, key)) == out


def test_philox_uniformity_and_keying():
    words = np.array([S.uniform_u32(7, seq, 3, pos, 2) for seq in range(64) for pos in range(64)], dtype=np.uint64)
    # 16 equal bins of the top 4 bits: chi-square with 15 dof stays well below the 0.999 quantile (37.7)
    counts = np.bincount((words >> 28).astype(np.int64), minlength=16)
    expect = words.size / 16
    chi2 = float(((counts - expect) ** 2 / expect).sum())
    assert chi2 < 37.7
    # every field of the counter and the key changes the word
    base = S.uniform_u32(1, 2, 3, 4, 1)
    assert base != S.uniform_u32(2, 2, 3, 4, 1)
    assert base != S.uniform_u32(1 << 32 | 1, 2, 3, 4, 1)
    assert base != S.uniform_u32(1, 3, 3, 4, 1)
    assert base != S.uniform_u32(1, 2, 4, 4, 1)
    assert base != S.uniform_u32(1, 2, 3, 5, 1)
    assert base != S.uniform_u32(1, 2, 3, 4, 2)


def test_exp_hat_accuracy():
    xs = np.concatenate([np.linspace(-23.0, 0.0, 20001, dtype=np.float32),
                         -np.logspace(-8, 1.3, 2000).astype(np.float32)])
    worst = 0.0
    prev = None
    for x in np.sort(xs):
        e = S.exp_hat(float(x))
        ref = math.exp(float(x))
        worst = max(worst, abs(e - ref) / float(np.spacing(np.float32(ref))))
        if prev is not None:
            assert e >= prev  # monotone on the sorted grid
        prev = e
    assert worst <= 1.0
    assert S.exp_hat(0.0) == 1.0
    assert S.exp_hat(-23.5) == 0.0
    assert S.exp_hat(float("-inf")) == 0.0


def test_row_weights_definition():
    rng = np.random.default_rng(0)
    l = (rng.standard_normal(1000) * 3).astype(np.float32)
    for T in (1.0, 0.7, 2.5):
        E = S.row_weights(l, T)
        y = (l / np.float32(T)).astype(np.float32)
        m = y.max()
        assert E[int(np.argmax(y))] == 1 << 32
        ref = np.exp((y - m).astype(np.float64)) * 2.0 ** 32
        # floor of 2^32 e^x with an own exp within 1 ulp: relative error below 2^-22 where E > 2^20
        big = ref > 2 ** 20
        assert np.all(np.abs(E[big] - ref[big]) <= ref[big] * 2.0 ** -22 + 1)
        assert np.all(E[ref < 2.0 ** 32 * math.exp(-23.5)] == 0)
    with pytest.raises(S.OracleError):
        S.row_weights(np.array([0.0, np.nan], dtype=np.float32), 1.0)
    with pytest.raises(S.OracleError):
        S.row_weights(np.array([0.0, np.inf], dtype=np.float32), 1.0)


def _keys(E):
    v = np.arange(E.size, dtype=np.uint64)
    return (E.astype(np.uint64) << np.uint64(18)) | (np.uint64((1 << 18) - 1) - v)


@pytest.mark.parametrize("top_p", [0.05, 0.5, 0.9, 0.95, 1.0])
def test_nucleus_is_the_shortest_heaviest_run(top_p):
    rng = np.random.default_rng(int(top_p * 100))
    for trial in range(5):
        V = int(rng.integers(2, 3000))
        l = (rng.standard_normal(V) * rng.uniform(0.1, 4)).astype(np.float32)
        if trial == 4:
            l = np.round(l)  # many exact ties in E
        E = S.row_weights(l, 1.0)
        nu = S.nucleus(E, top_p)
        keys = _keys(E)
        inside = keys >= np.uint64(nu.kstar)
        assert int(inside.sum()) == nu.size
        assert int(E.sum(dtype=np.uint64)) == nu.S
        assert int(E[inside].sum(dtype=np.uint64)) == nu.Sn
        tau = max(1, (nu.S * S.top_p_q32(top_p)) >> 32)
        assert nu.Sn >= tau
        # dropping the lightest member falls short of tau: the run is the shortest
        assert nu.Sn - int(E[keys == np.uint64(nu.kstar)][0]) < tau
        # every member outranks every non-member
        if (~inside).any():
            assert keys[inside].min() > keys[~inside].max()
        if top_p == 1.0:
            assert np.array_equal(inside, E > 0)


def test_nucleus_keeps_at_least_one_token():
    E = S.row_weights(np.array([0.0, -1.0, -2.0], dtype=np.float32), 1.0)
    nu = S.nucleus(E, 1e-9)
    assert nu.size == 1 and nu.Sn == 1 << 32


def test_sampling_frequencies_are_exact():
    """The draw is monotone in W; each token owns a W-interval whose length is
    S_n-proportional (up to 1 of 2^24)."""
    rng = np.random.default_rng(5)
    V = 37
    l = (rng.standard_normal(V) * 2).astype(np.float32)
    E = S.row_weights(l, 1.0)
    nu = S.nucleus(E, 0.9)
    inside = _keys(E) >= np.uint64(nu.kstar)

    def draw(w):
        return S.sample_nucleus(E, nu.kstar, nu.Sn, w)

    # boundary search: first W whose draw exceeds v
    counts = np.zeros(V)
    lo_w = 0
    for v in range(V):
        lo, hi = lo_w, 1 << 24
        while lo < hi:
            mid = (lo + hi) // 2
            if draw(mid) > v:
                hi = mid
            else:
                lo = mid + 1
        counts[v] = lo - lo_w
        lo_w = lo
    assert lo_w == 1 << 24
    p = np.where(inside, E.astype(np.float64), 0.0) / float(nu.Sn)
    assert np.all(np.abs(counts / 2.0 ** 24 - p) <= 2.0 ** -24 + 1e-15)
    assert np.all(counts[~inside] == 0)
    assert draw(0) == int(np.flatnonzero(inside & (E > 0))[0])
    assert draw((1 << 24) - 1) == int(np.flatnonzero(inside & (E > 0))[-1])


def test_argmax_lowest_id_on_ties():
    assert S.argmax(np.array([1.0, 3.0, 3.0, 2.0], dtype=np.float32)) == 1
    assert S.argmax(np.array([-0.0, 0.0], dtype=np.float32)) == 0
    assert S.argmax(np.array([0.0, -0.0], dtype=np.float32)) == 0
    assert S.argmax(np.array([-5.0], dtype=np.float32)) == 0
    rng = np.random.default_rng(1)
    x = rng.standard_normal(100000).astype(np.float32)
    assert S.argmax(x) == int(np.argmax(x))
    with pytest.raises(S.OracleError):
        S.argmax(np.array([1.0, np.nan], dtype=np.float32))
