"""Pins of the oracle's low-rank Markov rollout (no GPU)."""
import numpy as np
import torch

from oracle import sampling as S
from tests.helpers import golden


def _bf16(a) -> torch.Tensor:
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def test_hand_worked_case():
    g = golden("markov_v8_r2.json")
    w1 = _bf16(g["w1"])
    w2 = _bf16(g["w2"])
    assert torch.equal(w1.float(), torch.tensor(g["w1"], dtype=torch.float32))  # exact in bf16
    z = np.array(g["z"], dtype=np.float32)
    tokens, ell = S.markov_rollout(z, w1, w2, g["anchor"])
    assert tokens.tolist() == g["expected_tokens"]
    assert np.array_equal(ell, np.array(g["expected_ell"], dtype=np.float32))


def test_zero_w2_reduces_to_per_position_argmax():
    rng = np.random.default_rng(3)
    V, r, B = 500, 8, 7
    z = rng.standard_normal((B, V)).astype(np.float32)
    w1 = _bf16(rng.standard_normal((V, r)))
    w2 = torch.zeros((r, V), dtype=torch.bfloat16)
    tokens, ell = S.markov_rollout(z, w1, w2, 11)
    assert np.array_equal(ell, z)
    assert tokens.tolist() == [int(np.argmax(z[i])) for i in range(B)]


def test_delta_chain_is_the_low_rank_product():
    """ell - z equals w2^T w1[t_prev] up to the rounding of an r-term fp32 chain."""
    rng = np.random.default_rng(4)
    V, r, B = 2000, 32, 7
    z = (rng.standard_normal((B, V)) * 1.7).astype(np.float32)
    w1 = _bf16(rng.standard_normal((V, r)) * 0.5)
    w2 = _bf16(rng.standard_normal((r, V)) * 0.5)
    anchor = 123
    tokens, ell = S.markov_rollout(z, w1, w2, anchor)
    W1 = w1.double().numpy()
    W2 = w2.double().numpy()
    prev = anchor
    for i in range(B):
        delta = W1[prev] @ W2
        bound = (r + 1) * 2.0 ** -24 * (np.abs(W1[prev]) @ np.abs(W2) + np.abs(z[i]))
        assert np.all(np.abs(ell[i] - (z[i].astype(np.float64) + delta)) <= bound)
        prev = int(tokens[i])
        assert prev == int(np.argmax(ell[i]))
    # the chain depends on the previous token: a different anchor changes row 0
    _, ell2 = S.markov_rollout(z, w1, w2, 124)
    assert not np.array_equal(ell2[0], ell[0])


def test_probabilistic_draft_uses_its_own_uniforms():
    rng = np.random.default_rng(6)
    V, r, B = 300, 8, 7
    z = (rng.standard_normal((B, V)) * 1.5).astype(np.float32)
    w1 = _bf16(rng.standard_normal((V, r)) * 0.3)
    w2 = _bf16(rng.standard_normal((r, V)) * 0.3)
    t_a, ell_a = S.markov_rollout(z, w1, w2, 5, draft_mode=1, T=1.0, top_p=0.95, seed=9, seq=0, step=0)
    t_b, _ = S.markov_rollout(z, w1, w2, 5, draft_mode=1, T=1.0, top_p=0.95, seed=9, seq=0, step=0)
    assert np.array_equal(t_a, t_b)
    # each drawn token is the spec's draw from its own row with the DRAFT uniform of that position
    for i in range(B):
        E = S.row_weights(ell_a[i], 1.0)
        nu = S.nucleus(E, 0.95)
        W = S.uniform_u32(9, 0, 0, i, 1) >> 8
        assert t_a[i] == S.sample_nucleus(E, nu.kstar, nu.Sn, W)
    # a nucleus of one token is the greedy choice when the top logit is well separated
    z2 = z.copy()
    for i in range(B):
        z2[i, (7 * i + 3) % V] += 30.0
    t_g, _ = S.markov_rollout(z2, w1, w2, 5, draft_mode=0)
    t_p, _ = S.markov_rollout(z2, w1, w2, 5, draft_mode=1, T=1.0, top_p=1e-6, seed=1)
    assert np.array_equal(t_g, t_p)
