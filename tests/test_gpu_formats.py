"""Weight-only FP8, NVFP4 and MXFP4 through the C ABI against the oracle on the
decoded weights ("Kimi-K3-DSpark-NVFP4": FP8 per-channel and NVFP4 group-16
weight-only; MXFP4 the cards' third format). Tolerance: relative L2 <= 3e-2 on
hidden states and logits."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import network as N
from synthetic import generate as gen
from synthetic import quantize as Q
from synthetic.configs import FORMAT_FP8, FORMAT_MXFP4, FORMAT_NVFP4, TINY_STEP
from tests.gpu_harness import MID, workload
from tests.helpers import f64, rel_l2

pytestmark = pytest.mark.gpu
TOL = 3e-2
FMTS = {"fp8": FORMAT_FP8, "nvfp4": FORMAT_NVFP4, "mxfp4": FORMAT_MXFP4}
MIDMX = replace(MID, q_lora=512)  # every quantised input dimension a multiple of 512
KEYS = ("attn_norm", "w_qkv_a", "q_a_norm", "kv_a_norm", "w_q_b", "w_kv_b", "w_o", "mlp_norm", "w_gate", "w_up",
        "w_down")


@pytest.fixture(scope="module")
def M():
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build
    build.build()
    return M


def decode(v, fmt):
    """Oracle-side decoding of one matrix entry to float64."""
    if not isinstance(v, tuple):
        return f64(v)
    d, sc, g = v
    if fmt == "fp8":
        return F.dequant_fp8(d.cpu().numpy(), sc.cpu().numpy())
    if fmt == "mxfp4":
        return F.dequant_mxfp4(d.cpu().numpy(), sc.cpu().numpy())
    return F.dequant_nvfp4(d.cpu().numpy(), sc.cpu().numpy(), g)


def to_dev(Wq):
    out = {}
    for k, v in Wq.items():
        out[k] = tuple(x.cuda() if torch.is_tensor(x) else x for x in v) if isinstance(v, tuple) else v.cuda()
    return out


@pytest.mark.parametrize("fmt,w", [("fp8", TINY_STEP), ("fp8", workload(MID, 2, (300, 90), seed=9)),
                                   ("nvfp4", workload(MID, 2, (300, 90), seed=9)),
                                   ("mxfp4", workload(MIDMX, 2, (300, 90), seed=9))],
                         ids=["fp8_tiny", "fp8_mid", "nvfp4_mid", "mxfp4_mid"])
def test_weight_only_draft(M, fmt, w):
    G, bs = w.geom, w.bs
    W = gen.make_weights(w, "cpu")
    I = gen.make_inputs(w, "cpu")
    Wq = Q.quantise_weights(W, fmt, G.n_layers)
    ds = M.DSpark(G, to_dev(Wq), max_bs=bs, max_ctx=max(I["ctx_list"]), weight_format=FMTS[fmt])
    x = torch.empty(bs, G.block, G.hidden, dtype=torch.float32, device="cuda")
    ds.fuse_ctx(I["aux"].cuda(), x, bs)
    x0 = x.clone()
    kv = ds.make_kv([p.cuda() for p in I["kv_pools"]], I["page_table"].cuda(), I["ctx_len"].cuda(),
                    max(I["ctx_list"]))
    h = torch.empty_like(x)
    z = torch.empty(bs, G.block, G.vocab, dtype=torch.float32, device="cuda")
    ds.draft_block(x, kv, h, z, bs)
    assert ds.check() == 0
    layers = [{k: decode(Wq[f"l{l}.{k}"], fmt) for k in KEYS} for l in range(G.n_layers)]
    w_fc = decode(Wq["w_fc"], fmt)
    pools = [f64(p) for p in I["kv_pools"]]
    table = I["page_table"].numpy()
    for b, ctx in enumerate(I["ctx_list"]):
        ox = N.fuse_ctx(w_fc, f64(I["aux"][b]))
        assert rel_l2(x0[b].cpu().numpy(), ox) < TOL
        caches = [N.gather_cache(p, table[b], ctx) for p in pools]
        oh, oz = N.draft_block(ox, layers, f64(W["final_norm"]), f64(W["w_lm"]), G, caches, ctx)
        assert rel_l2(h[b].cpu().numpy(), oh) < TOL, b
        assert rel_l2(z[b].cpu().numpy(), oz) < TOL, b


def test_nvfp4_rejects_unaligned_geometry(M):
    G = TINY_STEP.geom  # q_lora 128: group-scale rows of 8 bytes are not TMA strides
    W = gen.make_weights(TINY_STEP, "cpu")
    Wq = Q.quantise_weights(W, "nvfp4", G.n_layers)
    with pytest.raises(M.DSparkError) as e:
        M.DSpark(G, to_dev(Wq), max_bs=1, weight_format=FORMAT_NVFP4)
    assert e.value.status == 4


def test_activation_beyond_f16_range_is_reported(M):
    """The NVFP4 / MXFP4 GEMMs take activations in f16: a magnitude above 65504 is
    reported as DSPARK_ERR_BAD_INPUT (17), and a clean call afterwards is OK."""
    w = workload(MID, 1, (64,), seed=9)
    G = w.geom
    W = gen.make_weights(w, "cpu")
    I = gen.make_inputs(w, "cpu")
    ds = M.DSpark(G, to_dev(Q.quantise_weights(W, "nvfp4", G.n_layers)), max_bs=1, weight_format=FORMAT_NVFP4)
    x = torch.empty(1, G.block, G.hidden, dtype=torch.float32, device="cuda")
    aux = I["aux"].cuda()
    bad = aux.clone()
    bad.view(-1)[5] = 70000.0
    ds.fuse_ctx(bad, x, 1)
    assert ds.check() == 17
    ds.fuse_ctx(aux, x, 1)
    assert ds.check() == 0


def test_mxfp4_scale_out_of_f16_range_is_reported(M):
    """An MXFP4 scale below 2^-22 (E8M0 byte 104) cannot be decoded exactly in f16:
    DSPARK_ERR_BAD_INPUT (17); a clean call afterwards is OK."""
    w = workload(MIDMX, 1, (64,), seed=9)
    G = w.geom
    W = gen.make_weights(w, "cpu")
    I = gen.make_inputs(w, "cpu")
    Wq = Q.quantise_weights(W, "mxfp4", G.n_layers)
    d, sc, g = Wq["w_fc"]
    bad = sc.clone()
    bad[0, 0] = 104
    Wb = dict(Wq)
    Wb["w_fc"] = (d, bad, g)
    x = torch.empty(1, G.block, G.hidden, dtype=torch.float32, device="cuda")
    ds = M.DSpark(G, to_dev(Wb), max_bs=1, weight_format=FORMAT_MXFP4)
    ds.fuse_ctx(I["aux"].cuda(), x, 1)
    assert ds.check() == 17
    ds2 = M.DSpark(G, to_dev(Wq), max_bs=1, weight_format=FORMAT_MXFP4)
    ds2.fuse_ctx(I["aux"].cuda(), x, 1)
    assert ds2.check() == 0


@pytest.mark.parametrize("bs", [1, 2, 3], ids=["rows7", "rows14", "rows21"])
def test_fp8_fc_split_is_exact(M, bs):
    """FP8 weights go to the tensor core as stored and every bf16 activation as the
    sum of two E4M3 terms with a power-of-two scale per row and 128-k chunk, which
    is exact within 2^13 of the chunk maximum. So the fc fusion equals the
    float64 product of the decoded weights and the bf16 activations up to fp32
    summation (relative L2 below 1e-5, where the 3e-2 format tolerance allows for
    the quantisation itself), also for activations spread over 32 binades and
    beyond the f16 range. Rows 7, 14 and 21 take the 8-, 16- and 32-row activation tiles."""
    w = workload(MID, bs, (64,) * bs, seed=21)
    G = w.geom
    W = gen.make_weights(w, "cpu")
    I = gen.make_inputs(w, "cpu")
    Wq = Q.quantise_weights(W, "fp8", G.n_layers)
    w_fc = decode(Wq["w_fc"], "fp8")
    aux = I["aux"]
    g = torch.Generator().manual_seed(5)
    e = torch.randint(-24, 9, aux.shape, generator=g).to(torch.float32)
    wide = (aux.to(torch.float32) * torch.pow(2.0, e)).to(torch.bfloat16)
    big = aux.clone()
    big.view(-1)[3] = 70000.0
    ds = M.DSpark(G, to_dev(Wq), max_bs=bs, max_ctx=64, weight_format=FORMAT_FP8)
    for a in (aux, wide, big):
        x = torch.empty(bs, G.block, G.hidden, dtype=torch.float32, device="cuda")
        ds.fuse_ctx(a.cuda(), x, bs)
        assert ds.check() == 0
        for b in range(bs):
            assert rel_l2(x[b].cpu().numpy(), N.fuse_ctx(w_fc, f64(a[b]))) < 1e-5, b


def test_fp8_nonfinite_activation_is_reported(M):
    """An infinite activation reaching the FP8 GEMM is DSPARK_ERR_BAD_INPUT (17);
    a clean call afterwards is OK."""
    w = TINY_STEP
    G = w.geom
    W = gen.make_weights(w, "cpu")
    I = gen.make_inputs(w, "cpu")
    ds = M.DSpark(G, to_dev(Q.quantise_weights(W, "fp8", G.n_layers)), max_bs=1, weight_format=FORMAT_FP8)
    x = torch.empty(1, G.block, G.hidden, dtype=torch.float32, device="cuda")
    aux = I["aux"].cuda()
    bad = aux.clone()
    bad.view(-1)[11] = float("inf")
    ds.fuse_ctx(bad, x, 1)
    assert ds.check() == 17
    ds.fuse_ctx(aux, x, 1)
    assert ds.check() == 0
