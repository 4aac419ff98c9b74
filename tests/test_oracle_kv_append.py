"""Pins of the oracle's latent-cache append (no GPU): a closed form with unit
weights, the RoPE rotation at a known position, agreement with the block
latents the layer itself forms, page placement and untouched entries."""
import math
from dataclasses import replace

import numpy as np

from oracle import network as N
from synthetic.configs import TINY


def _unit_layer(G):
    """Gains 1; kv_a rows select input k for output k (q_a rows zero)."""
    kvd = G.kv_lora + G.d_rope
    w = np.zeros((G.q_lora + kvd, G.hidden))
    for k in range(kvd):
        w[G.q_lora + k, k] = 1.0
    return {"attn_norm": np.ones(G.hidden), "w_qkv_a": w, "kv_a_norm": np.ones(G.kv_lora)}


def test_closed_form_with_unit_weights():
    # x = c * ones: the attention norm gives ones, kv = ones, the latent norm keeps ones,
    # and the rope pair (1, 1) turns by pos * inv_freq[0] (inv_freq[0] = 1 for pair 0).
    G = replace(TINY, hidden=64, q_lora=16, kv_lora=16, d_rope=2, eps=0.0)
    L = _unit_layer(G)
    x = np.full((2, G.hidden), 3.5)
    e = N.kv_entries(x, L, G, np.array([0, 5]))
    assert np.allclose(e[0], 1.0, atol=1e-12)
    assert np.allclose(e[1, :16], 1.0, atol=1e-12)
    c, s = math.cos(5.0), math.sin(5.0)
    assert np.allclose(e[1, 16:], [c - s, s + c], atol=1e-12)


def test_entries_match_the_layers_block_latents():
    # the append forms the same entry as the layer's own block-row latent: check through
    # attention of a single query that sees only that one cached entry (softmax of one key).
    rng = np.random.default_rng(3)
    G = replace(TINY, n_layers=1)
    kvd = G.kv_lora + G.d_rope
    L = {k: rng.normal(0, 0.05, s) for k, s in [("w_qkv_a", (G.q_lora + kvd, G.hidden))]}
    L.update(attn_norm=1 + rng.normal(0, 0.1, G.hidden), kv_a_norm=1 + rng.normal(0, 0.1, G.kv_lora))
    x = rng.normal(0, 1, (3, G.hidden))
    pos = np.array([7, 64, 130])
    e = N.kv_entries(x, L, G, pos)
    inv_freq = N.rope_inv_freq(G.d_rope, G.rope_theta)
    for i in range(3):
        h = x[i] / math.sqrt(np.mean(x[i] ** 2) + G.eps) * L["attn_norm"]
        kv = L["w_qkv_a"][G.q_lora:] @ h
        ckv = kv[:G.kv_lora] / math.sqrt(np.mean(kv[:G.kv_lora] ** 2) + G.eps) * L["kv_a_norm"]
        assert np.allclose(e[i, :G.kv_lora], ckv, atol=1e-12)
        # rotation preserves each pair's norm and turns it by pos * inv_freq
        kr, er = kv[G.kv_lora:].reshape(-1, 2), e[i, G.kv_lora:].reshape(-1, 2)
        assert np.allclose(np.linalg.norm(kr, axis=1), np.linalg.norm(er, axis=1), atol=1e-12)
        ang = np.arctan2(er[:, 1], er[:, 0]) - np.arctan2(kr[:, 1], kr[:, 0])
        d = np.angle(np.exp(1j * (ang - pos[i] * inv_freq)))
        assert np.allclose(d, 0.0, atol=1e-9)


def test_page_placement_and_untouched_entries():
    rng = np.random.default_rng(5)
    G = replace(TINY, n_layers=2)
    kvd = G.kv_lora + G.d_rope
    layers = []
    for _ in range(G.n_layers):
        layers.append({"w_qkv_a": rng.normal(0, 0.05, (G.q_lora + kvd, G.hidden)), "attn_norm": np.ones(G.hidden),
                       "kv_a_norm": np.ones(G.kv_lora)})
    n_pages, P = 12, 64
    pools = [rng.normal(0, 1, (n_pages, P, kvd)) for _ in range(G.n_layers)]
    page_table = np.array([[3, 7, 1, 0], [5, 2, 9, 11]])
    ctx = np.array([62, 128])
    n_new = np.array([4, 0])          # sequence 0 crosses from page 3 into page 7; sequence 1 appends nothing
    x = rng.normal(0, 1, (2, 5, G.hidden))
    out, ctx2 = N.kv_append(x, layers, G, pools, page_table, ctx, n_new)
    assert list(ctx2) == [66, 128]
    for l in range(G.n_layers):
        e = N.kv_entries(x[0, :4], layers[l], G, np.arange(62, 66))
        assert np.array_equal(out[l][3, 62], e[0]) and np.array_equal(out[l][3, 63], e[1])
        assert np.array_equal(out[l][7, 0], e[2]) and np.array_equal(out[l][7, 1], e[3])
        mask = np.ones((n_pages, P), bool)
        mask[3, 62:] = False
        mask[7, :2] = False
        assert np.array_equal(out[l][mask], pools[l][mask])
        # the appended tokens read back in order through the page table
        assert np.array_equal(N.gather_cache(out[l], page_table[0], 66)[62:], e)
