"""Weight-only FP8, NVFP4 and MXFP4 at the full drafter geometry (hidden 7168,
5 layers, vocabulary 163,840; the weight-format sweep workload) through the C
ABI, against the oracle on the decoded weights ("Kimi-K3-DSpark-NVFP4", header
and "What is quantized to what": fc, q_b, o_proj and the MLP weight-only).

This is the launch configuration the benchmark times for these formats: K up
to 35,840, the stream-K split over every SM, NVFP4 group-scale rows of 2,240
bytes. Compared: the fc fusion on every channel, h_out on every element and
the logits on 4096 sampled vocabulary rows, at relative L2 <= 3e-2."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import network as N
from synthetic import generate as gen
from synthetic import quantize as Q
from synthetic.configs import FORMAT_FP8, FORMAT_MXFP4, FORMAT_NVFP4, FP8_STEP
from tests.helpers import rel_l2

pytestmark = pytest.mark.gpu
TOL = 3e-2
CODES = {"fp8": FORMAT_FP8, "nvfp4": FORMAT_NVFP4, "mxfp4": FORMAT_MXFP4}
KEYS = ("attn_norm", "w_qkv_a", "q_a_norm", "kv_a_norm", "w_q_b", "w_kv_b", "w_o", "mlp_norm", "w_gate", "w_up",
        "w_down")


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def decode(v, fmt):
    """Oracle-side decoding of one matrix entry (bf16 tensor or quantised triple) to float64."""
    if not isinstance(v, tuple):
        return f64(v)
    d, sc, g = v
    d, sc = d.cpu().numpy(), sc.cpu().numpy()
    if fmt == "fp8":
        return F.dequant_fp8(d, sc)
    if fmt == "mxfp4":
        return F.dequant_mxfp4(d, sc)
    return F.dequant_nvfp4(d, sc, g)


@pytest.fixture(scope="module")
def M():
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build
    build.build()
    return M


@pytest.fixture(scope="module")
def bf16_weights():
    return gen.make_weights(FP8_STEP, "cuda")


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4", "mxfp4"])
def test_full_geometry_weight_only_draft(M, bf16_weights, fmt):
    w = FP8_STEP
    G = w.geom
    W = bf16_weights
    Wq = Q.quantise_weights(W, fmt, G.n_layers)
    I = gen.make_inputs(w, "cuda")
    ctx = I["ctx_list"][0]
    ds = M.DSpark(G, Wq, max_bs=1, max_ctx=ctx, weight_format=CODES[fmt])
    x = torch.empty(1, G.block, G.hidden, dtype=torch.float32, device="cuda")
    ds.fuse_ctx(I["aux"], x, 1)
    x0 = x.clone()
    kv = ds.make_kv(I["kv_pools"], I["page_table"], I["ctx_len"], ctx)
    h = torch.empty_like(x)
    z = torch.empty(1, G.block, G.vocab, dtype=torch.float32, device="cuda")
    ds.draft_block(x, kv, h, z, 1)
    assert ds.check() == 0
    # oracle on the decoded weights, layer by layer (one layer's float64 weights at a time)
    ox = N.fuse_ctx(decode(Wq["w_fc"], fmt), f64(I["aux"][0]))
    assert rel_l2(x0[0].cpu().numpy(), ox) < TOL
    table = I["page_table"][0]
    pages = table[: (ctx + G.page_size - 1) // G.page_size].long()
    pos = np.arange(G.block, dtype=np.float64) + ctx
    xo = ox
    for l in range(G.n_layers):
        L = {k: decode(Wq[f"l{l}.{k}"], fmt) for k in KEYS}
        pool = f64(I["kv_pools"][l][pages])
        cache = N.gather_cache(pool, np.arange(pool.shape[0]), ctx)
        xo = N.layer(xo, L, G, cache[:, :G.kv_lora], cache[:, G.kv_lora:], pos)
        del L
    oh = N.rmsnorm(xo, f64(W["final_norm"]), G.eps)
    rows = np.sort(np.random.default_rng(5).choice(G.vocab, 4096, replace=False))
    oz = oh @ f64(W["w_lm"][torch.as_tensor(rows, device="cuda")]).T
    assert rel_l2(h[0].cpu().numpy(), oh) < TOL
    assert rel_l2(z[0].cpu().numpy()[:, rows], oz) < TOL
