"""ORACLE (test infrastructure only): the DSpark drafter network written out as
its plain definition in float64 numpy. Slow by design; no blocking, fusion or
reordering beyond what the definition states. Only tests, the smoke check and
the benchmark's CPU-baseline leg may use it. It shares no code with the CUDA
library.

Pages (Kimi-K3-DSpark model cards):
  * fc over the 5 captured target states -- "Kimi K3 DSpark Q8_0 GGUF",
    "Architecture metadata" (fc.weight consumes five captured hidden states);
    "Kimi-K3-DSpark-NVFP4", "What is quantized to what" (context_proj).
  * 5 dense block-diffusion layers, non-causal attention over a 7-token block,
    MLA latent KV of 576 per token shared with the target -- "Kimi-K3-DSpark-
    NVFP4", "Original model card / Model Overview".
  * MLA tensors q_a, kv_a_with_mqa, k_b, v_b; split RoPE dims (nope + rope);
    decompression of the latent through kv_b -- "kimi-k3-dspark-gguf",
    "Runtime status" / "What's needed from llama.cpp".
  * fused q_a + kv_a, kv_b absorbed, norms high precision, SwiGLU gate/up/down,
    o_proj, q_b_proj -- "Kimi-K3-DSpark-NVFP4", "What is quantized to what".
  * lm_head is the target's unembedding -- "Kimi-K3-DSpark-NVFP4",
    "Measurement" (the real target lm_head).
  * confidence head -- "kimi-k3-dspark-gguf", "How it works".
Readings where the pages are silent (RMSNorm eps 1e-6 with the eps inside the
root; RoFormer interleaved RoPE pairs, theta 10000, block row i at position
ctx + i; YaRN per Peng et al. 2023; softmax scale 1/sqrt(d_nope + d_rope); no
bias and no pre-norm on fc; confidence = sigmoid(w.h + b) per position) are
listed with the design notes.

Weights are passed as float64 arrays (the same bf16 bytes the GPU reads,
converted exactly). Shapes follow the row-major [out, in] convention.
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence, Tuple

import numpy as np


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def rope_inv_freq(d_rope: int, theta: float, yarn_factor: float = 1.0, orig_ctx: int = 65536,
                  alpha: float = 1.0, beta: float = 32.0) -> np.ndarray:
    """Per-pair angular frequencies theta_j = theta^(-2j/d).

    With yarn_factor s > 1 (YaRN, Peng et al. 2023, "NTK-by-parts"): for each
    pair the number of rotations over the original context r_j = L / lambda_j
    (lambda_j = 2 pi / theta_j) sets a ramp gamma = clip((r - alpha)/(beta - alpha), 0, 1)
    and theta'_j = (1 - gamma) theta_j / s + gamma theta_j.
    """
    j = np.arange(d_rope // 2, dtype=np.float64)
    inv = theta ** (-2.0 * j / d_rope)
    if yarn_factor > 1.0:
        lam = 2.0 * math.pi / inv
        r = orig_ctx / lam
        gamma = np.clip((r - alpha) / (beta - alpha), 0.0, 1.0)
        inv = (1.0 - gamma) * inv / yarn_factor + gamma * inv
    return inv


def yarn_attention_factor(yarn_factor: float) -> float:
    """Multiplier on the attention logits: (0.1 ln s + 1)^2 for s > 1, else 1."""
    if yarn_factor <= 1.0:
        return 1.0
    m = 0.1 * math.log(yarn_factor) + 1.0
    return m * m


def apply_rope(x: np.ndarray, positions: np.ndarray, inv_freq: np.ndarray) -> np.ndarray:
    """Rotate interleaved pairs (2j, 2j+1) of the last axis by positions * inv_freq[j].

    x has shape [T, ..., d]; positions has shape [T].
    """
    ang = positions.astype(np.float64)[:, None] * inv_freq[None, :]  # [T, d/2]
    shape = (x.shape[0],) + (1,) * (x.ndim - 2) + (inv_freq.shape[0],)
    c = np.cos(ang).reshape(shape)
    s = np.sin(ang).reshape(shape)
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def softmax(s: np.ndarray, axis: int = -1) -> np.ndarray:
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def split_kv_b(w_kv_b: np.ndarray, n_heads: int, d_nope: int, d_v: int, kv_lora: int):
    """kv_b_proj rows per head: d_nope rows of k_b followed by d_v rows of v_b."""
    w = w_kv_b.reshape(n_heads, d_nope + d_v, kv_lora)
    return w[:, :d_nope, :], w[:, d_nope:, :]  # W_kb [h, d_nope, c], W_vb [h, d_v, c]


def mla_attention(q_nope, q_rope, c_kv, k_r, w_kb, w_vb, scale: float, absorbed: bool = True):
    """Non-causal MLA attention of the block's queries over every key j.

    q_nope [T, h, d_nope], q_rope [T, h, d_rope], c_kv [J, c], k_r [J, d_rope].
    Unabsorbed (decompressed): K_h,j = [W_kb,h c_j || k_r,j], V_h,j = W_vb,h c_j.
    Absorbed: score = (W_kb,h^T q_nope) . c_j + q_rope . k_r,j; output W_vb,h (sum_j p c_j).
    Returns o [T, h, d_v].
    """
    if absorbed:
        q_lat = np.einsum("thd,hdc->thc", q_nope, w_kb)
        s = np.einsum("thc,jc->htj", q_lat, c_kv) + np.einsum("thr,jr->htj", q_rope, k_r)
        p = softmax(scale * s, axis=-1)
        o_lat = np.einsum("htj,jc->thc", p, c_kv)
        return np.einsum("thc,hvc->thv", o_lat, w_vb)
    k_nope = np.einsum("hdc,jc->hjd", w_kb, c_kv)
    v = np.einsum("hvc,jc->hjv", w_vb, c_kv)
    s = np.einsum("thd,hjd->htj", q_nope, k_nope) + np.einsum("thr,jr->htj", q_rope, k_r)
    p = softmax(scale * s, axis=-1)
    return np.einsum("htj,hjv->thv", p, v)


def fuse_ctx(w_fc: np.ndarray, aux: np.ndarray) -> np.ndarray:
    """x = W_fc [a_1 || ... || a_n] per block row. aux [T, n_aux, H] -> x [T, H]."""
    T = aux.shape[0]
    return aux.reshape(T, -1) @ w_fc.T


def layer(x: np.ndarray, L: Dict[str, np.ndarray], geom, cache_ckv: np.ndarray, cache_kr: np.ndarray,
          positions: np.ndarray, absorbed: bool = True) -> np.ndarray:
    """One block-diffusion layer: pre-norm MLA attention + residual, pre-norm SwiGLU MLP + residual."""
    G = geom
    T = x.shape[0]
    inv_freq = rope_inv_freq(G.d_rope, G.rope_theta, G.yarn_factor, G.yarn_orig_ctx, G.yarn_alpha, G.yarn_beta)
    scale = yarn_attention_factor(G.yarn_factor) / math.sqrt(G.d_nope + G.d_rope)

    h = rmsnorm(x, L["attn_norm"], G.eps)
    qkv = h @ L["w_qkv_a"].T
    c_q = rmsnorm(qkv[:, :G.q_lora], L["q_a_norm"], G.eps)
    kv = qkv[:, G.q_lora:]
    c_kv_blk = rmsnorm(kv[:, :G.kv_lora], L["kv_a_norm"], G.eps)
    k_r_blk = apply_rope(kv[:, G.kv_lora:], positions, inv_freq)
    q = (c_q @ L["w_q_b"].T).reshape(T, G.n_heads, G.q_head_dim)
    q_nope = q[:, :, :G.d_nope]
    q_rope = apply_rope(q[:, :, G.d_nope:], positions, inv_freq)

    c_kv = np.concatenate([cache_ckv, c_kv_blk], axis=0)
    k_r = np.concatenate([cache_kr, k_r_blk], axis=0)
    w_kb, w_vb = split_kv_b(L["w_kv_b"], G.n_heads, G.d_nope, G.d_v, G.kv_lora)
    o = mla_attention(q_nope, q_rope, c_kv, k_r, w_kb, w_vb, scale, absorbed)
    x = x + o.reshape(T, G.n_heads * G.d_v) @ L["w_o"].T

    h2 = rmsnorm(x, L["mlp_norm"], G.eps)
    a = silu(h2 @ L["w_gate"].T) * (h2 @ L["w_up"].T)
    return x + a @ L["w_down"].T


def draft_block(x: np.ndarray, layers: Sequence[Dict[str, np.ndarray]], final_norm: np.ndarray,
                w_lm: np.ndarray, geom, caches: Sequence[np.ndarray], ctx_len: int,
                absorbed: bool = True, with_logits: bool = True) -> Tuple[np.ndarray, np.ndarray]:
    """5 (n_layers) layers over the block, final norm, lm_head.

    x [T, H]; caches[l] [ctx_len, kv_lora + d_rope] (normalised latent || roped key);
    block row i sits at position ctx_len + i. Returns (h_out [T, H], z [T, V]).
    """
    G = geom
    T = x.shape[0]
    positions = np.arange(T, dtype=np.float64) + ctx_len
    for l, L in enumerate(layers):
        cache = caches[l][:ctx_len]
        x = layer(x, L, G, cache[:, :G.kv_lora], cache[:, G.kv_lora:], positions, absorbed)
    h_out = rmsnorm(x, final_norm, G.eps)
    z = h_out @ w_lm.T if with_logits else None
    return h_out, z


def confidence(h_out: np.ndarray, w_conf: np.ndarray, b_conf: float) -> np.ndarray:
    """c_i = sigmoid(w_c . h_out_i + b_c)."""
    return 1.0 / (1.0 + np.exp(-(h_out @ w_conf + b_conf)))


def gather_cache(pool: np.ndarray, page_table_row: np.ndarray, ctx_len: int) -> np.ndarray:
    """Token j of a sequence lives at pool[page_table[j // P], j % P]."""
    P = pool.shape[1]
    j = np.arange(ctx_len)
    return pool[np.asarray(page_table_row)[j // P], j % P]


def kv_entries(x: np.ndarray, L: Dict[str, np.ndarray], geom, positions: np.ndarray) -> np.ndarray:
    """Latent cache entries [c_kv || k_r] (kv_lora + d_rope each) of tokens with
    context features x [n, H] at the given positions, for one layer: the layer's
    attention pre-norm, the kv_a rows of the fused q_a || kv_a projection, the
    latent norm and RoPE on the rope part -- the same entry the layer forms for
    its block rows ("Kimi-K3-DSpark-NVFP4", Model Overview: draft and target
    share one 576-element latent layout, so the draft's pages unify with the
    target's cache)."""
    G = geom
    inv_freq = rope_inv_freq(G.d_rope, G.rope_theta, G.yarn_factor, G.yarn_orig_ctx, G.yarn_alpha, G.yarn_beta)
    h = rmsnorm(x, L["attn_norm"], G.eps)
    kv = h @ L["w_qkv_a"][G.q_lora:].T
    c_kv = rmsnorm(kv[:, :G.kv_lora], L["kv_a_norm"], G.eps)
    k_r = apply_rope(kv[:, G.kv_lora:], positions, inv_freq)
    return np.concatenate([c_kv, k_r], axis=1)


def kv_append(x_new: np.ndarray, layers: Sequence[Dict[str, np.ndarray]], geom, pools: Sequence[np.ndarray],
              page_table: np.ndarray, ctx_len: np.ndarray, n_new: np.ndarray):
    """Append the latent entries of newly verified tokens to every layer's paged
    cache. Sequence b's token j < n_new[b] (context features x_new[b, j]) goes
    to position ctx_len[b] + j, i.e. pool[page_table[b, pos // P], pos % P].
    Returns new pools (copies) and the new context lengths ctx_len + n_new."""
    out = [p.copy() for p in pools]
    P = out[0].shape[1]
    for b in range(x_new.shape[0]):
        n = int(n_new[b])
        if n == 0:
            continue
        pos = int(ctx_len[b]) + np.arange(n)
        for l, L in enumerate(layers):
            e = kv_entries(x_new[b, :n], L, geom, pos)
            out[l][np.asarray(page_table[b])[pos // P], pos % P] = e
    return out, np.asarray(ctx_len) + np.asarray(n_new)
