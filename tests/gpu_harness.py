"""Shared set-up for the GPU parity tests: draw a workload with the seeded
generators, run the CUDA path through the C ABI, run the oracle on the same
bytes. Marshalling only; the arithmetic lives in oracle/ and in libdspark."""
from __future__ import annotations

from dataclasses import replace
from typing import List

import numpy as np
import torch

from oracle import network as N
from synthetic import generate as gen
from synthetic.configs import Geometry, Workload
from tests.helpers import f64, oracle_layers

# Small geometries with several tiles and ragged tails for the GEMMs and a
# split KV loop for attention (latent widths covered by the attention kernel).
MID = Geometry(hidden=1024, n_aux=5, n_layers=2, n_heads=16, q_lora=256, kv_lora=256, d_nope=64, d_rope=32,
               d_v=64, inter=2048, vocab=8192, rank=32)
# The full latent width (512 + 64): the tensor-core attention path, with 40
# heads so a sequence's 280 query rows span three 128-row tiles (the last ragged).
MIDLAT = Geometry(hidden=1024, n_aux=2, n_layers=1, n_heads=40, q_lora=256, kv_lora=512, d_nope=32, d_rope=64,
                  d_v=32, inter=1024, vocab=4096, rank=32)
MID128 = Geometry(hidden=768, n_aux=3, n_layers=1, n_heads=12, q_lora=192, kv_lora=128, d_nope=48, d_rope=32,
                  d_v=48, inter=1536, vocab=6144, rank=24, block=5)


def workload(G: Geometry, bs: int, ctx, seed: int, **kw) -> Workload:
    return Workload(f"test_{G.hidden}_{bs}", G, bs=bs, ctx=tuple(ctx), weight_seed=seed, input_seed=seed + 100, **kw)


def draw(w: Workload, device="cpu"):
    W = gen.make_weights(w, device)
    I = gen.make_inputs(w, device)
    return W, I


def to_cuda(d):
    out = {}
    for k, v in d.items():
        if torch.is_tensor(v):
            out[k] = v.cuda()
        elif isinstance(v, list) and v and torch.is_tensor(v[0]):
            out[k] = [t.cuda() for t in v]
        else:
            out[k] = v
    return out


def gpu_draft(ds, w: Workload, I):
    """fc fusion + draft block through the C ABI. Returns x (after the layers), h_out, z."""
    G, bs = w.geom, w.bs
    x = torch.empty(bs, G.block, G.hidden, dtype=torch.float32, device="cuda")
    ds.fuse_ctx(I["aux"], x, bs)
    x0 = x.clone()
    kv = ds.make_kv(I["kv_pools"], I["page_table"], I["ctx_len"], max(I["ctx_list"]))
    h_out = torch.empty_like(x)
    z = torch.empty(bs, G.block, G.vocab, dtype=torch.float32, device="cuda")
    ds.draft_block(x, kv, h_out, z, bs)
    st = ds.check()
    return x0, h_out, z, st


def oracle_draft(w: Workload, W, I, with_logits=True):
    """Oracle fc fusion + draft block per sequence on the same bytes (float64)."""
    G = w.geom
    layers = oracle_layers(W, G)
    w_fc, fin = f64(W["w_fc"]), f64(W["final_norm"])
    w_lm = f64(W["w_lm"]) if with_logits else None
    aux = f64(I["aux"])
    pools = [f64(p) for p in I["kv_pools"]]
    table = I["page_table"].cpu().numpy()
    xs, hs, zs = [], [], []
    for b, ctx in enumerate(I["ctx_list"]):
        x = N.fuse_ctx(w_fc, aux[b])
        caches = [N.gather_cache(p, table[b], ctx) for p in pools]
        h, z = N.draft_block(x, layers, fin, w_lm, G, caches, ctx, with_logits=with_logits)
        xs.append(x)
        hs.append(h)
        zs.append(z)
    return np.stack(xs), np.stack(hs), (np.stack(zs) if with_logits else None)


def u32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)
