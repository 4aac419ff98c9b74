"""The samplers' output law over many counter-based uniforms at the full
vocabulary (163,840), through the C ABI: a chi-squared test of the emitted
tokens against the target distribution.

Lossless verification ("kimi-k3-dspark-gguf", intro: the output distribution
equals the target's) means the token emitted at the first block position is
distributed as the target's nucleus distribution p, whatever the draft. Every
call is bit-exact against the oracle elsewhere; this test checks the law over
many (sequence, step) counters of Philox4x32-10, which no single-call test
reaches. Expected probabilities come from the oracle's integer weights
(p_v = E_v / S_n inside the nucleus). The samples are deterministic (fixed
seeds), so the test does not flake; the bound is a chi-squared tail of 1e-6.
"""
import numpy as np
import pytest
import torch
from dataclasses import replace

from oracle import sampling as S
from synthetic import generate as gen
from synthetic.configs import FULL_STEP

pytestmark = pytest.mark.gpu
BS = 32


@pytest.fixture(scope="module")
def M():
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build
    build.build()
    return M


def small_full_vocab():
    G = replace(FULL_STEP.geom, hidden=64, n_aux=1, n_layers=1, n_heads=1, q_lora=64, kv_lora=64, d_nope=16,
                d_rope=16, d_v=64, inter=64)
    return G, replace(FULL_STEP, geom=G)


def peaked_row(V, seed):
    """Logits with a dozen clear favourites over a flat tail."""
    l = gen.normal((V,), 1.0, seed, "chi2_row", "cpu", dtype=torch.float32).numpy().astype(np.float32)
    top = np.random.default_rng(seed).choice(V, 12, replace=False)
    l[top] += np.linspace(6.0, 9.0, 12).astype(np.float32)
    return l, top


def chi2_stat(counts, probs, n):
    e = probs * n
    return float(((counts - e) ** 2 / e).sum())


def chi2_tail_ok(stat, dof):
    # Wilson-Hilferty: the 1e-6 upper tail of chi^2_dof is ~ dof (1 - 2/(9 dof) + 4.753 sqrt(2/(9 dof)))^3
    z = 4.753
    bound = dof * (1 - 2 / (9 * dof) + z * np.sqrt(2 / (9 * dof))) ** 3
    return stat < bound, bound


def binned(tokens, probs_full, nbins=20):
    order = np.argsort(-probs_full)
    keep = order[:nbins]
    counts = np.array([(tokens == v).sum() for v in keep] + [0], dtype=np.float64)
    counts[-1] = len(tokens) - counts[:-1].sum()
    probs = np.concatenate([probs_full[keep], [1.0 - probs_full[keep].sum()]])
    return counts, probs


@pytest.mark.parametrize("T,top_p", [(1.0, 1.0), (1.0, 0.95), (0.8, 0.9)])
def test_verify_emits_the_target_law(M, T, top_p):
    G, w = small_full_vocab()
    V, B = G.vocab, G.block
    W = gen.make_weights(w, "cuda")
    ds = M.DSpark(G, W, max_bs=BS)
    l, top = peaked_row(V, 3)
    P1 = np.tile(l, (B + 1, 1)).astype(np.float32)
    P = torch.from_numpy(np.tile(P1[None], (BS, 1, 1))).cuda()
    ell = torch.zeros(BS, B, V, dtype=torch.float32, device="cuda")
    # a greedy draft on the 6th favourite: accepted with probability p(t), else the residual
    tok = int(top[5])
    tokens = torch.full((BS, B), tok, dtype=torch.int32, device="cuda")
    acc = torch.empty(BS, dtype=torch.int32, device="cuda")
    out = torch.empty(BS, B + 1, dtype=torch.int32, device="cuda")
    draws = []
    for step in range(600):
        ds.verify(P, ell, tokens, M.Sample(M.GREEDY, M.PROBABILISTIC, T, top_p, 2024, step), acc, out, BS)
        draws.append(out[:, 0].clone())
    assert ds.check() == 0
    x = torch.cat(draws).cpu().numpy()
    E = S.row_weights(l, T)
    nu = S.nucleus(E, top_p)
    keys = (E.astype(np.uint64) << np.uint64(18)) | (np.uint64((1 << 18) - 1) - np.arange(V, dtype=np.uint64))
    inside = keys >= np.uint64(nu.kstar)
    p = np.where(inside, E.astype(np.float64), 0.0) / float(nu.Sn)
    assert (x >= 0).all() and inside[x].all()  # every emitted token lies in the target's nucleus
    counts, probs = binned(x, p)
    stat = chi2_stat(counts, probs, len(x))
    ok, bound = chi2_tail_ok(stat, len(counts) - 1)
    assert ok, (stat, bound)


def test_probabilistic_draft_law(M):
    """The rollout's first draw, over many sequences and steps, follows the nucleus
    law of its Markov-corrected logits (z + the delta of the anchor, here zero)."""
    G, w = small_full_vocab()
    V, B = G.vocab, G.block
    W = gen.make_weights(w, "cuda")
    W["markov_w1"] = torch.zeros_like(W["markov_w1"])  # delta = 0: ell = z exactly
    ds = M.DSpark(G, W, max_bs=BS)
    l, _ = peaked_row(V, 5)
    z = torch.from_numpy(np.tile(l, (BS, B, 1)).astype(np.float32)).cuda()
    anchor = torch.zeros(BS, dtype=torch.int32, device="cuda")
    tokens = torch.empty(BS, B, dtype=torch.int32, device="cuda")
    ell = torch.empty(BS, B, V, dtype=torch.float32, device="cuda")
    draws = []
    for step in range(100):
        ds.markov_rollout(z, anchor, M.Sample(M.PROBABILISTIC, M.PROBABILISTIC, 1.0, 0.95, 77, step), tokens, ell, BS)
        draws.append(tokens.clone().reshape(-1))  # all 7 positions share the law (delta = 0)
    assert ds.check() == 0
    x = torch.cat(draws).cpu().numpy()
    E = S.row_weights(l, 1.0)
    nu = S.nucleus(E, 0.95)
    keys = (E.astype(np.uint64) << np.uint64(18)) | (np.uint64((1 << 18) - 1) - np.arange(V, dtype=np.uint64))
    inside = keys >= np.uint64(nu.kstar)
    p = np.where(inside, E.astype(np.float64), 0.0) / float(nu.Sn)
    assert inside[x].all()
    counts, probs = binned(x, p)
    stat = chi2_stat(counts, probs, len(x))
    ok, bound = chi2_tail_ok(stat, len(counts) - 1)
    assert ok, (stat, bound)
