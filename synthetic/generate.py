"""Seeded synthetic inputs for the DSpark draft-and-verify step.

The real drafter weights, target hidden states, tokenizer and benchmark
streams are not available, so every tensor here is drawn from a seeded
generator with the shapes and value distributions the model cards describe
(Kimi-K3-DSpark-NVFP4, "Measurement": aux regimes gauss / heavy; "Speculator
acceptance": ~95k-token AA-LCR prompts and 10k-token SPEED-Bench inputs).

This module holds no arithmetic of the method; it is imported by the oracle
tests and by the GPU path alike. Each tensor is drawn from its own
``torch.Generator`` seeded from (workload seed, tensor name), so adding a tensor
never shifts another one. Values drawn on a CUDA device differ from values
drawn on the CPU for the same seed; a test draws once and hands the same bytes
to both sides.
"""
from __future__ import annotations

import math
import zlib
from typing import Dict, List, Optional

import torch

from .configs import Geometry, Workload

_CHUNK = 1 << 26  # elements per randn call, bounds the fp32 temporary (256 MB)


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + zlib.crc32(name.encode())) & 0x7FFF_FFFF_FFFF)
    return g


def normal(shape, std: float, seed: int, name: str, device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    """N(0, std^2) draws rounded to ``dtype``; generated in chunks to bound memory."""
    g = _gen(seed, name, device)
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        t = torch.randn(hi - lo, generator=g, device=device, dtype=torch.float32)
        flat[lo:hi].copy_(t.mul_(std))
    return out


def student_t3_unit_rms(shape, seed: int, name: str, device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    """Heavy-tailed draws: Z / sqrt(chi2_3 / 3), then divided by the tensor's RMS."""
    g = _gen(seed, name, device)
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float64)
    c = torch.randn((3,) + tuple(shape), generator=g, device=device, dtype=torch.float64)
    chi2 = (c * c).sum(0)
    t = z / torch.sqrt(chi2 / 3.0)
    t = t / torch.sqrt((t * t).mean())
    return t.to(dtype)


def make_weights(w: Workload, device="cpu") -> Dict[str, torch.Tensor]:
    """Drafter weight set. Matrices bf16 row-major [out, in]; norm gains and the
    confidence head fp32 (the cards keep norms and the confidence head at high
    precision: "Kimi K3 DSpark Q8_0 GGUF", "Conversion result")."""
    G, s, std = w.geom, w.weight_seed, w.weight_std
    H = G.hidden
    W: Dict[str, torch.Tensor] = {}
    W["w_fc"] = normal((H, G.n_aux * H), std, s, "fc", device)
    for l in range(G.n_layers):
        p = f"l{l}."
        W[p + "attn_norm"] = torch.ones(H, dtype=torch.float32, device=device)
        W[p + "w_qkv_a"] = normal((G.qkv_a_out, H), std, s, p + "qkv_a", device)
        W[p + "q_a_norm"] = torch.ones(G.q_lora, dtype=torch.float32, device=device)
        W[p + "kv_a_norm"] = torch.ones(G.kv_lora, dtype=torch.float32, device=device)
        W[p + "w_q_b"] = normal((G.n_heads * G.q_head_dim, G.q_lora), std, s, p + "q_b", device)
        W[p + "w_kv_b"] = normal((G.n_heads * (G.d_nope + G.d_v), G.kv_lora), std, s, p + "kv_b", device)
        W[p + "w_o"] = normal((H, G.n_heads * G.d_v), std, s, p + "o", device)
        W[p + "mlp_norm"] = torch.ones(H, dtype=torch.float32, device=device)
        W[p + "w_gate"] = normal((G.inter, H), std, s, p + "gate", device)
        W[p + "w_up"] = normal((G.inter, H), std, s, p + "up", device)
        W[p + "w_down"] = normal((H, G.inter), std, s, p + "down", device)
    W["final_norm"] = torch.ones(H, dtype=torch.float32, device=device)
    W["w_lm"] = normal((G.vocab, H), std, s, "lm_head", device)
    W["markov_w1"] = normal((G.vocab, G.rank), std, s, "markov_w1", device)
    W["markov_w2"] = normal((G.rank, G.vocab), std, s, "markov_w2", device)
    W["w_conf"] = normal((H,), std, s, "conf", device, dtype=torch.float32)
    W["b_conf"] = torch.tensor([0.1], dtype=torch.float32, device=device)
    return W


def context_lengths(w: Workload) -> List[int]:
    if w.ctx:
        assert len(w.ctx) in (1, w.bs)
        return list(w.ctx) * (w.bs if len(w.ctx) == 1 else 1)
    lo, hi = w.extra["ctx_lo"], w.extra["ctx_hi"]
    g = _gen(w.input_seed, "ctx_len", "cpu")
    return torch.randint(lo, hi + 1, (w.bs,), generator=g).tolist()


def make_inputs(w: Workload, device="cpu") -> Dict[str, object]:
    """Per-step inputs: aux states, paged latent KV, page table, context lengths, anchors."""
    G, s = w.geom, w.input_seed
    ctx = context_lengths(w)
    P = G.page_size
    pages_per_seq = [max(1, math.ceil(c / P)) for c in ctx]
    n_pages = sum(pages_per_seq)
    max_pages = max(pages_per_seq)
    # Pages of all sequences come from one pool, assigned by a seeded permutation.
    if w.random_pages:
        perm = torch.randperm(n_pages, generator=_gen(s, "pages", "cpu"))
    else:
        perm = torch.arange(n_pages)
    table = torch.zeros((w.bs, max_pages), dtype=torch.int32)
    k = 0
    for b, npg in enumerate(pages_per_seq):
        table[b, :npg] = perm[k:k + npg].to(torch.int32)
        k += npg
    if w.aux_dist == "normal":
        aux = normal((w.bs, G.block, G.n_aux, G.hidden), w.aux_std, s, "aux", device)
    else:
        aux = student_t3_unit_rms((w.bs, G.block, G.n_aux, G.hidden), s, "aux", device)
    pools = [normal((n_pages, P, G.kv_dim), w.kv_std, s, f"kv{l}", device) for l in range(G.n_layers)]
    anchor = torch.randint(0, G.vocab, (w.bs,), generator=_gen(s, "anchor", "cpu"), dtype=torch.int32)
    return {
        "aux": aux,
        "kv_pools": pools,
        "page_table": table.to(device),
        "ctx_len": torch.tensor(ctx, dtype=torch.int32, device=device),
        "ctx_list": ctx,
        "anchor": anchor.to(device),
        "n_pages": n_pages,
        "max_pages": max_pages,
    }


def draft_logits(bs: int, block: int, vocab: int, seed: int, std: float = 1.7, device="cpu",
                 name: str = "z") -> torch.Tensor:
    """Stand-in lm_head logits z [bs, block, vocab] fp32 (std ~ sqrt(H) * 0.02 for the full drafter)."""
    return normal((bs, block, vocab), std, seed, name, device, dtype=torch.float32)


def noise(shape, std: float, seed: int, name: str = "target_noise", device="cpu") -> torch.Tensor:
    """fp32 N(0, std^2) noise used to build target logits from drafter logits."""
    return normal(shape, std, seed, name, device, dtype=torch.float32)


def uniform_tokens(shape, vocab: int, seed: int, name: str = "tokens") -> torch.Tensor:
    return torch.randint(0, vocab, shape, generator=_gen(seed, name, "cpu"), dtype=torch.int32)
