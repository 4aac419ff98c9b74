"""Pins of the oracle's network definition (no GPU)."""
import math

import numpy as np
import pytest

from oracle import network as N
from synthetic.configs import TINY, Geometry


def test_rmsnorm_properties():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 64)) * 3
    g = np.ones(64)
    y = N.rmsnorm(x, g, 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-12)
    assert np.allclose(N.rmsnorm(7.0 * x, g, 0.0), y, atol=1e-12)  # scale invariant
    g2 = rng.standard_normal(64)
    assert np.allclose(N.rmsnorm(x, g2, 0.0), y * g2)
    # eps sits inside the root: a zero row stays zero, a tiny row is damped
    assert np.all(N.rmsnorm(np.zeros((1, 8)), np.ones(8), 1e-6) == 0)
    small = np.full((1, 4), 1e-4)
    assert np.allclose(N.rmsnorm(small, np.ones(4), 1e-6), 1e-4 / math.sqrt(1e-8 + 1e-6))


def test_silu_values():
    assert N.silu(np.array([0.0]))[0] == 0.0
    assert abs(N.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(N.silu(np.array([-30.0]))[0]) < 1e-11


def test_rope_identities():
    rng = np.random.default_rng(1)
    d = 16
    inv = N.rope_inv_freq(d, 10000.0)
    assert inv[0] == 1.0 and abs(inv[1] - 10000.0 ** (-2.0 / d)) < 1e-15
    x = rng.standard_normal((3, d))
    # position 0 is the identity; rotations keep the norm
    assert np.allclose(N.apply_rope(x, np.zeros(3), inv), x)
    y = N.apply_rope(x, np.array([5.0, 77.0, 1000.0]), inv)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1))
    # interleaved pairs: pair 0 rotates by the position itself (inv_freq 1)
    e0 = np.zeros((1, d)); e0[0, 0] = 1.0
    r = N.apply_rope(e0, np.array([0.3]), inv)
    assert abs(r[0, 0] - math.cos(0.3)) < 1e-15 and abs(r[0, 1] - math.sin(0.3)) < 1e-15
    # relative position: q(m).k(n) depends on m - n only
    q = rng.standard_normal((1, d)); k = rng.standard_normal((1, d))
    dots = [float((N.apply_rope(q, np.array([m + 10.0]), inv) @ N.apply_rope(k, np.array([m + 3.0]), inv).T)[0, 0])
            for m in (0, 100, 4000)]
    assert np.allclose(dots, dots[0], atol=1e-10)


def test_yarn_reduces_and_ramps():
    d = 64
    plain = N.rope_inv_freq(d, 10000.0)
    assert np.array_equal(N.rope_inv_freq(d, 10000.0, 1.0), plain)
    y = N.rope_inv_freq(d, 10000.0, 16.0, 65536, 1.0, 32.0)
    rot = 65536 * plain / (2 * math.pi)  # rotations over the original context
    assert np.allclose(y[rot > 32], plain[rot > 32])            # fast pairs untouched
    assert np.allclose(y[rot < 1], plain[rot < 1] / 16.0)       # slow pairs interpolated by s
    mid = (rot >= 1) & (rot <= 32)
    assert np.all((y[mid] <= plain[mid] + 1e-18) & (y[mid] >= plain[mid] / 16.0 - 1e-18))
    assert N.yarn_attention_factor(1.0) == 1.0
    assert abs(N.yarn_attention_factor(16.0) - (0.1 * math.log(16.0) + 1.0) ** 2) < 1e-15


def _mla_inputs(rng, T=7, h=4, dn=8, dr=4, dv=6, c=12, J=20):
    return (rng.standard_normal((T, h, dn)), rng.standard_normal((T, h, dr)), rng.standard_normal((J, c)),
            rng.standard_normal((J, dr)), rng.standard_normal((h, dn, c)), rng.standard_normal((h, dv, c)))


def test_absorbed_equals_unabsorbed():
    rng = np.random.default_rng(2)
    args = _mla_inputs(rng)
    a = N.mla_attention(*args, scale=0.3, absorbed=True)
    b = N.mla_attention(*args, scale=0.3, absorbed=False)
    assert np.max(np.abs(a - b)) <= 1e-12 * np.max(np.abs(b))


def test_single_head_is_textbook_attention():
    """n_h = 1: softmax(q.K / sqrt-scale) V with K = [W_kb c || k_r], V = W_vb c, by loops."""
    rng = np.random.default_rng(3)
    q_nope, q_rope, c_kv, k_r, w_kb, w_vb = _mla_inputs(rng, h=1, J=9)
    scale = 0.25
    out = N.mla_attention(q_nope, q_rope, c_kv, k_r, w_kb, w_vb, scale)
    T, J = q_nope.shape[0], c_kv.shape[0]
    for t in range(T):
        keys = [np.concatenate([w_kb[0] @ c_kv[j], k_r[j]]) for j in range(J)]
        vals = [w_vb[0] @ c_kv[j] for j in range(J)]
        q = np.concatenate([q_nope[t, 0], q_rope[t, 0]])
        s = [scale * float(q @ keys[j]) for j in range(J)]
        m = max(s)
        w = [math.exp(x - m) for x in s]
        o = sum(w[j] * vals[j] for j in range(J)) / sum(w)
        assert np.allclose(out[t, 0], o, atol=1e-12)


def test_attention_is_non_causal_and_permutation_invariant():
    rng = np.random.default_rng(4)
    q_nope, q_rope, c_kv, k_r, w_kb, w_vb = _mla_inputs(rng, J=15)
    out = N.mla_attention(q_nope, q_rope, c_kv, k_r, w_kb, w_vb, 0.2)
    perm = rng.permutation(15)
    out2 = N.mla_attention(q_nope, q_rope, c_kv[perm], k_r[perm], w_kb, w_vb, 0.2)
    assert np.allclose(out, out2, atol=1e-12)
    # changing the last key (a later block row) changes the first query's output
    c2 = c_kv.copy(); c2[-1] += 1.0
    out3 = N.mla_attention(q_nope, q_rope, c2, k_r, w_kb, w_vb, 0.2)
    assert not np.allclose(out3[0], out[0])


def _rand_layer(rng, G: Geometry, std=0.05):
    H = G.hidden
    return {
        "attn_norm": np.ones(H), "q_a_norm": np.ones(G.q_lora), "kv_a_norm": np.ones(G.kv_lora),
        "mlp_norm": np.ones(H),
        "w_qkv_a": rng.standard_normal((G.qkv_a_out, H)) * std,
        "w_q_b": rng.standard_normal((G.n_heads * G.q_head_dim, G.q_lora)) * std,
        "w_kv_b": rng.standard_normal((G.n_heads * (G.d_nope + G.d_v), G.kv_lora)) * std,
        "w_o": rng.standard_normal((H, G.n_heads * G.d_v)) * std,
        "w_gate": rng.standard_normal((G.inter, H)) * std,
        "w_up": rng.standard_normal((G.inter, H)) * std,
        "w_down": rng.standard_normal((H, G.inter)) * std,
    }


def test_layer_composition_special_cases():
    G = TINY
    rng = np.random.default_rng(5)
    L = _rand_layer(rng, G)
    x = rng.standard_normal((7, G.hidden))
    cache = rng.standard_normal((30, G.kv_dim))
    pos = np.arange(7) + 30.0
    # with o_proj and down_proj zero the residual stream passes through unchanged
    Z = dict(L, w_o=np.zeros_like(L["w_o"]), w_down=np.zeros_like(L["w_down"]))
    assert np.array_equal(N.layer(x, Z, G, cache[:, :G.kv_lora], cache[:, G.kv_lora:], pos), x)
    # with only the MLP live the update is W_d(silu(W_g n(x)) * W_u n(x)) on the pre-norm of x
    M = dict(L, w_o=np.zeros_like(L["w_o"]))
    h = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + G.eps)
    g = h @ M["w_gate"].T
    upd = ((g / (1 + np.exp(-g))) * (h @ M["w_up"].T)) @ M["w_down"].T
    assert np.allclose(N.layer(x, M, G, cache[:, :G.kv_lora], cache[:, G.kv_lora:], pos), x + upd, atol=1e-12)
    # absorbed and decompressed layers agree
    a = N.layer(x, L, G, cache[:, :G.kv_lora], cache[:, G.kv_lora:], pos, absorbed=True)
    b = N.layer(x, L, G, cache[:, :G.kv_lora], cache[:, G.kv_lora:], pos, absorbed=False)
    assert np.max(np.abs(a - b)) < 1e-12 * np.max(np.abs(b))


def test_draft_block_absorbed_vs_unabsorbed_and_logits():
    G = TINY
    rng = np.random.default_rng(6)
    layers = [_rand_layer(rng, G) for _ in range(G.n_layers)]
    x = rng.standard_normal((7, G.hidden))
    caches = [rng.standard_normal((40, G.kv_dim)) for _ in range(G.n_layers)]
    w_lm = rng.standard_normal((G.vocab, G.hidden)) * 0.02
    h1, z1 = N.draft_block(x, layers, np.ones(G.hidden), w_lm, G, caches, 40, absorbed=True)
    h2, z2 = N.draft_block(x, layers, np.ones(G.hidden), w_lm, G, caches, 40, absorbed=False)
    assert np.max(np.abs(h1 - h2)) < 1e-10
    assert np.allclose(np.sqrt(np.mean(h1 * h1, axis=-1)), 1.0, atol=1e-6)
    assert np.allclose(z1, h1 @ w_lm.T)


def test_fuse_ctx_is_concatenation():
    rng = np.random.default_rng(7)
    aux = rng.standard_normal((7, 5, 16))
    w = rng.standard_normal((16, 80))
    x = N.fuse_ctx(w, aux)
    for t in range(7):
        assert np.allclose(x[t], sum(w[:, 16 * a:16 * (a + 1)] @ aux[t, a] for a in range(5)))


def test_confidence_special_cases():
    rng = np.random.default_rng(8)
    h = rng.standard_normal((7, 32))
    assert np.allclose(N.confidence(h, np.zeros(32), 0.0), 0.5)
    assert np.allclose(N.confidence(h, np.zeros(32), math.log(3.0)), 0.75)
    w = rng.standard_normal(32)
    c = N.confidence(h, w, 0.0)
    assert np.allclose(c + N.confidence(h, -w, 0.0), 1.0)


def test_gather_cache_follows_page_table():
    pool = np.arange(4 * 3 * 2).reshape(4, 3, 2).astype(np.float64)
    out = N.gather_cache(pool, np.array([2, 0, 3]), 7)
    assert out.tolist() == [pool[2, 0].tolist(), pool[2, 1].tolist(), pool[2, 2].tolist(),
                            pool[0, 0].tolist(), pool[0, 1].tolist(), pool[0, 2].tolist(), pool[3, 0].tolist()]
    assert N.gather_cache(pool, np.array([1]), 0).shape == (0, 2)


def _uniform_err():
    """Relative error of the oracle layer against its closed form when every query is zero."""
    G = TINY
    rng = np.random.default_rng(11)
    L = dict(_rand_layer(rng, G, std=0.1))
    L["w_q_b"] = np.zeros_like(L["w_q_b"])
    x = rng.standard_normal((7, G.hidden))
    ctx = 23
    cache = rng.standard_normal((ctx, G.kv_dim))
    got = N.layer(x, L, G, cache[:, :G.kv_lora], cache[:, G.kv_lora:], np.arange(7) + float(ctx))
    h = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + G.eps)
    kv = (h @ L["w_qkv_a"].T)[:, G.q_lora:G.q_lora + G.kv_lora]
    c_blk = kv / np.sqrt(np.mean(kv * kv, axis=-1, keepdims=True) + G.eps)
    mean_c = (cache[:, :G.kv_lora].sum(axis=0) + c_blk.sum(axis=0)) / (ctx + 7)
    per = G.d_nope + G.d_v
    o = np.concatenate([L["w_kv_b"][hh * per + G.d_nope:(hh + 1) * per] @ mean_c for hh in range(G.n_heads)])
    x1 = x + (L["w_o"] @ o)[None, :]
    h2 = x1 / np.sqrt(np.mean(x1 * x1, axis=-1, keepdims=True) + G.eps)
    g = h2 @ L["w_gate"].T
    want = x1 + ((g / (1 + np.exp(-g))) * (h2 @ L["w_up"].T)) @ L["w_down"].T
    return np.max(np.abs(got - want)) / np.max(np.abs(want))


def test_layer_with_zero_queries_attends_uniformly_to_cache_and_block():
    """q = 0 makes every score 0, so each query row's attention is the plain mean of the
    latents of all ctx cache rows and all 7 block rows (non-causal: every row sees the
    whole block), absorbed by each head's v_b (rows d_nope.. of the head's kv_b block),
    concatenated head by head into o_proj. The planted mistakes below (a causal mask, a
    dropped block, swapped k_b / v_b halves, a reversed head order) each break it."""
    assert _uniform_err() < 1e-12


def test_layer_is_invariant_to_a_consistent_head_permutation():
    """Renumbering the heads in q_b (row blocks), kv_b (row blocks) and o_proj (column
    blocks) together leaves the layer unchanged; renumbering only q_b does not (each
    head's queries must meet its own k_b / v_b and o_proj columns)."""
    G = TINY
    rng = np.random.default_rng(12)
    L = _rand_layer(rng, G, std=0.1)
    x = rng.standard_normal((7, G.hidden))
    cache = rng.standard_normal((19, G.kv_dim))
    pos = np.arange(7) + 19.0
    base = N.layer(x, L, G, cache[:, :G.kv_lora], cache[:, G.kv_lora:], pos)
    perm = rng.permutation(G.n_heads)
    assert not np.array_equal(perm, np.arange(G.n_heads))

    def rows(w, per):
        return np.concatenate([w[p * per:(p + 1) * per] for p in perm])

    qhd, kvh = G.d_nope + G.d_rope, G.d_nope + G.d_v
    w_o = np.concatenate([L["w_o"][:, p * G.d_v:(p + 1) * G.d_v] for p in perm], axis=1)
    P = dict(L, w_q_b=rows(L["w_q_b"], qhd), w_kv_b=rows(L["w_kv_b"], kvh), w_o=w_o)
    out = N.layer(x, P, G, cache[:, :G.kv_lora], cache[:, G.kv_lora:], pos)
    assert np.max(np.abs(out - base)) < 1e-12 * np.max(np.abs(base))
    Q = dict(L, w_q_b=rows(L["w_q_b"], qhd))
    assert np.max(np.abs(N.layer(x, Q, G, cache[:, :G.kv_lora], cache[:, G.kv_lora:], pos) - base)) > 1e-6


def test_planted_mistakes_fail_the_composition_pin(monkeypatch):
    """Mistakes planted in the oracle (on the CPU) each break the zero-query pin."""
    assert _uniform_err() < 1e-12
    real_attn, real_split = N.mla_attention, N.split_kv_b

    def drop_block(q_nope, q_rope, c_kv, k_r, w_kb, w_vb, scale, absorbed=True):
        T = q_nope.shape[0]  # attends to the cache only
        return real_attn(q_nope, q_rope, c_kv[:-T], k_r[:-T], w_kb, w_vb, scale, absorbed)

    def causal(q_nope, q_rope, c_kv, k_r, w_kb, w_vb, scale, absorbed=True):
        T, J = q_nope.shape[0], c_kv.shape[0]  # block row t sees the cache and block rows <= t
        return np.stack([real_attn(q_nope[t:t + 1], q_rope[t:t + 1], c_kv[:J - T + t + 1], k_r[:J - T + t + 1],
                                   w_kb, w_vb, scale, absorbed)[0] for t in range(T)])

    def heads_reversed(*a, **k):
        return real_attn(*a, **k)[:, ::-1, :]

    def kb_vb_swapped(w, n_heads, d_nope, d_v, kv_lora):
        kb, vb = real_split(w, n_heads, d_nope, d_v, kv_lora)
        return vb, kb

    for name, fn in (("mla_attention", drop_block), ("mla_attention", causal),
                     ("mla_attention", heads_reversed), ("split_kv_b", kb_vb_swapped)):
        with monkeypatch.context() as m:
            m.setattr(N, name, fn)
            assert _uniform_err() > 1e-6, fn.__name__


def _shift_err(cache_of=None):
    """Largest difference between the draft block and the same step with every position
    shifted by 1000 (cache keys roped at j + 1000, block row i at ctx + i + 1000)."""
    G = TINY
    rng = np.random.default_rng(13)
    layers = [_rand_layer(rng, G, std=0.1) for _ in range(G.n_layers)]
    x = rng.standard_normal((7, G.hidden))
    ctx, shift = 17, 1000.0
    inv = N.rope_inv_freq(G.d_rope, G.rope_theta)
    lat = [rng.standard_normal((ctx, G.kv_lora)) for _ in range(G.n_layers)]
    raw = [rng.standard_normal((ctx, G.d_rope)) for _ in range(G.n_layers)]
    caches = [np.concatenate([lat[l], N.apply_rope(raw[l], np.arange(ctx, dtype=np.float64), inv)], axis=1)
              for l in range(G.n_layers)]
    if cache_of is not None:
        caches = [caches[cache_of(l)] for l in range(G.n_layers)]
    w_lm = rng.standard_normal((G.vocab, G.hidden)) * 0.02
    h1, _ = N.draft_block(x, layers, np.ones(G.hidden), w_lm, G, caches, ctx)
    x2 = x
    for l, L in enumerate(layers):
        kr = N.apply_rope(raw[l], np.arange(ctx, dtype=np.float64) + shift, inv)
        x2 = N.layer(x2, L, G, lat[l], kr, np.arange(7.0) + ctx + shift)
    h2 = N.rmsnorm(x2, np.ones(G.hidden), G.eps)
    return np.max(np.abs(h1 - h2))


def test_positions_are_relative_and_the_block_follows_its_cache():
    """RoPE makes scores depend on relative positions only. With no cache, shifting the
    block's positions leaves a layer unchanged; with a cache whose keys were roped at
    positions 0..ctx-1, the draft block (block row i at ctx + i, layer l reading cache l)
    equals the same step with every position shifted by 1000. Placing the block at i
    instead of ctx + i, or giving every layer the same cache, breaks it (planted below)."""
    G = TINY
    rng = np.random.default_rng(14)
    L = _rand_layer(rng, G, std=0.1)
    x = rng.standard_normal((7, G.hidden))
    empty = np.zeros((0, G.kv_lora)), np.zeros((0, G.d_rope))
    a = N.layer(x, L, G, *empty, np.arange(7.0))
    b = N.layer(x, L, G, *empty, np.arange(7.0) + 1000.0)
    assert np.max(np.abs(a - b)) < 1e-9 * np.max(np.abs(a))
    assert _shift_err() < 1e-9
    assert _shift_err(cache_of=lambda l: 0) > 1e-6  # every layer reading layer 0's cache


def test_planted_position_mistake_fails_the_pin(monkeypatch):
    real_layer = N.layer

    def block_at_zero(x, L, geom, ckv, kr, positions, absorbed=True):
        return real_layer(x, L, geom, ckv, kr, positions - positions[0], absorbed)

    monkeypatch.setattr(N, "layer", block_at_zero)
    assert _shift_err() > 1e-6
