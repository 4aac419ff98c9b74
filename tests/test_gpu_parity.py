"""GPU path vs the oracle, element by element, through the C ABI.

Hidden states and logits: relative L2 <= 1e-2 (bf16 weights; the oracle is
float64 on the same bf16 bytes). Markov tokens and logits, verify decisions:
bit-exact on the same inputs and uniforms.
"""
import numpy as np
import pytest
import torch

from oracle import network as N
from oracle import sampling as S
from synthetic import generate as gen
from synthetic.configs import TINY, TINY_STEP
from tests.gpu_harness import MID, MID128, MIDLAT, draw, gpu_draft, oracle_draft, to_cuda, u32, workload
from tests.helpers import f64, rel_l2

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def M():
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return M


def _draft_case(M, w):
    W, I = draw(w, "cpu")
    Wd, Id = to_cuda(W), to_cuda(I)
    ds = M.DSpark(w.geom, Wd, max_bs=w.bs, max_ctx=max(I["ctx_list"]))
    x0, h_out, z, st = gpu_draft(ds, w, Id)
    assert st == 0
    ox, oh, oz = oracle_draft(w, W, I)
    return ds, (x0, h_out, z), (ox, oh, oz), W, I


def test_tiny_step_draft(M):
    ds, (x0, h, z), (ox, oh, oz), _, _ = _draft_case(M, TINY_STEP)
    assert rel_l2(x0.cpu().numpy(), ox) < TOL
    assert rel_l2(h.cpu().numpy(), oh) < TOL
    assert rel_l2(z.cpu().numpy(), oz) < TOL
    # deterministic: a second run gives the same bytes
    x2, h2, z2, st = gpu_draft(ds, TINY_STEP, to_cuda(gen.make_inputs(TINY_STEP, "cpu")))
    assert st == 0 and torch.equal(h2, h) and torch.equal(z2, z)


@pytest.mark.parametrize("G,bs,ctx", [
    (MID, 3, (1000, 77, 300)),     # split KV loop, ragged pages, three sequences
    (MID, 1, (0,)),                # empty context: only the block's own latents
    (MID128, 2, (130, 4000)),      # block 5, 3 aux states, long/short mix
    (MIDLAT, 3, (1000, 77, 4097)),  # tensor-core attention: partial pages, a one-token last page, splits
    (MIDLAT, 1, (0,)),             # tensor-core attention: only the block's own latents
    (MIDLAT, 2, (64, 640)),        # tensor-core attention: contexts ending on page boundaries
    # 26 sequences fill the GPU with unsplit CTAs, so the split plan caps the chunks per
    # CTA: long contexts take two splits, short ones leave their second split empty
    (MIDLAT, 26, (4000, 10, 1600, 0, 500, 2047, 64, 3900, 1535, 2049, 77, 3100, 128, 250, 1800, 999,
                  2500, 5, 1400, 2222, 640, 1600, 300, 2800, 1, 2048)),
])
def test_mid_draft(M, G, bs, ctx):
    w = workload(G, bs, ctx, seed=7)
    _, (x0, h, z), (ox, oh, oz), _, _ = _draft_case(M, w)
    assert rel_l2(x0.cpu().numpy(), ox) < TOL
    for b in range(bs):
        assert rel_l2(h[b].cpu().numpy(), oh[b]) < TOL, b
        assert rel_l2(z[b].cpu().numpy(), oz[b]) < TOL, b


def _rollout_inputs(G, bs, seed, std=1.7):
    W = gen.make_weights(workload(G, bs, (0,) * bs, seed), "cpu")
    z = gen.draft_logits(bs, G.block, G.vocab, seed, std=std)
    anchor = gen.uniform_tokens((bs,), G.vocab, seed, "anchor")
    return W, z, anchor


@pytest.mark.parametrize("mode,T,top_p", [(0, 1.0, 1.0), (1, 1.0, 0.95), (1, 0.7, 0.5), (1, 1.3, 1.0)])
@pytest.mark.parametrize("G,bs", [(TINY, 1), (TINY, 3), (MID, 9)])
def test_rollout_bit_exact(M, G, bs, mode, T, top_p):
    W, z, anchor = _rollout_inputs(G, bs, seed=11 + bs)
    Wd = to_cuda(W)
    ds = M.DSpark(G, Wd, max_bs=bs)
    tokens = torch.empty(bs, G.block, dtype=torch.int32, device="cuda")
    ell = torch.empty(bs, G.block, G.vocab, dtype=torch.float32, device="cuda")
    smp = M.Sample(mode, mode, T, top_p, 1234567, 9)
    ds.markov_rollout(z.cuda(), anchor.cuda(), smp, tokens, ell, bs)
    assert ds.check() == 0
    for b in range(bs):
        t_o, ell_o = S.markov_rollout(z[b].numpy(), W["markov_w1"], W["markov_w2"], int(anchor[b]), mode, T, top_p,
                                      seed=1234567, seq=b, step=9)
        assert tokens[b].cpu().numpy().tolist() == t_o.tolist(), b
        assert np.array_equal(u32(ell[b].cpu().numpy()), u32(ell_o)), b


def _verify_inputs(G, bs, seed, draft_mode, T, top_p, noise):
    W, z, anchor = _rollout_inputs(G, bs, seed)
    toks, ells, Ps = [], [], []
    for b in range(bs):
        t, l = S.markov_rollout(z[b].numpy(), W["markov_w1"], W["markov_w2"], int(anchor[b]), draft_mode, T, top_p,
                                seed=seed, seq=b, step=3)
        n = gen.noise((G.block + 1, G.vocab), noise[b % len(noise)], seed, f"tn{b}").numpy()
        P = np.concatenate([l, l[-1:]], axis=0) + n
        toks.append(t)
        ells.append(l)
        Ps.append(P.astype(np.float32))
    return W, np.stack(toks), np.stack(ells), np.stack(Ps)


@pytest.mark.parametrize("vmode,dmode,T,top_p", [(0, 0, 1.0, 1.0), (1, 0, 1.0, 0.95), (1, 1, 1.0, 0.95),
                                                  (1, 1, 0.8, 1.0), (2, 1, 1.0, 0.95), (2, 0, 1.0, 1.0),
                                                  (2, 1, 0.7, 0.9)])
@pytest.mark.parametrize("G,bs", [(TINY, 4), (MID, 3)])
def test_verify_bit_exact(M, G, bs, vmode, dmode, T, top_p):
    W, toks, ells, Ps = _verify_inputs(G, bs, 21, dmode, T, top_p, noise=(0.0, 0.02, 0.5, 2.0))
    ds = M.DSpark(G, to_cuda(W), max_bs=bs)
    acc = torch.empty(bs, dtype=torch.int32, device="cuda")
    out = torch.empty(bs, G.block + 1, dtype=torch.int32, device="cuda")
    seen = set()
    for step in range(3):
        smp = M.Sample(dmode, vmode, T, top_p, 777, step)
        ds.verify(torch.from_numpy(Ps).cuda(), torch.from_numpy(ells).cuda(), torch.from_numpy(toks).cuda(), smp,
                  acc, out, bs)
        assert ds.check() == 0
        for b in range(bs):
            if vmode == 0:
                a, o = S.verify_greedy(Ps[b], toks[b])
            elif vmode == 1:
                a, o = S.verify_prob(Ps[b], ells[b], toks[b], int(dmode == 0), T, top_p, seed=777, seq=b, step=step)
            else:  # block verification
                a, o = S.verify_block(Ps[b], ells[b], toks[b], int(dmode == 0), T, top_p, seed=777, seq=b, step=step)
            assert int(acc[b]) == a, (b, step)
            assert out[b].cpu().numpy().tolist() == o.tolist(), (b, step)
            seen.add(a)
    if vmode == 0:
        assert G.block in seen  # the zero-noise sequence accepts the whole block


def test_confidence(M):
    G = TINY
    W = gen.make_weights(TINY_STEP, "cpu")
    h = gen.normal((2, G.block, G.hidden), 1.0, 5, "h_out", dtype=torch.float32)
    ds = M.DSpark(G, to_cuda(W), max_bs=2)
    conf = torch.empty(2, G.block, dtype=torch.float32, device="cuda")
    ds.confidence(h.cuda(), conf, 2)
    ref = N.confidence(f64(h), f64(W["w_conf"]), float(W["b_conf"]))
    assert np.max(np.abs(conf.cpu().numpy() - ref)) < 1e-5


def test_device_errors_are_reported(M):
    """Non-finite logits, out-of-range tokens, anchors and pages set the error word (no fault)."""
    G = TINY
    W = gen.make_weights(TINY_STEP, "cpu")
    ds = M.DSpark(G, to_cuda(W), max_bs=1, max_ctx=128)
    z = gen.draft_logits(1, G.block, G.vocab, 3).cuda()
    tokens = torch.empty(1, G.block, dtype=torch.int32, device="cuda")
    ell = torch.empty_like(z)
    smp = M.Sample(0, 0, 1.0, 1.0, 1, 0)
    zb = z.clone()
    zb[0, 2, 17] = float("nan")
    ds.markov_rollout(zb, torch.zeros(1, dtype=torch.int32, device="cuda"), smp, tokens, ell, 1)
    assert ds.check() == 17
    ds.markov_rollout(z, torch.full((1,), G.vocab, dtype=torch.int32, device="cuda"), smp, tokens, ell, 1)
    assert ds.check() == 18
    P = torch.cat([z, z[:, -1:]], dim=1).contiguous()
    bad_tok = torch.full((1, G.block), -3, dtype=torch.int32, device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    out = torch.empty(1, G.block + 1, dtype=torch.int32, device="cuda")
    ds.verify(P, z, bad_tok, smp, acc, out, 1)
    assert ds.check() == 18
    Pn = P.clone()
    Pn[0, 0, 5] = float("inf")
    ds.verify(Pn, z, bad_tok.abs(), smp, acc, out, 1)
    assert ds.check() == 17
    # a page table entry outside the pool
    I = to_cuda(gen.make_inputs(TINY_STEP, "cpu"))
    I["page_table"][0, 1] = 10_000
    x = torch.empty(1, G.block, G.hidden, dtype=torch.float32, device="cuda")
    ds.fuse_ctx(I["aux"], x, 1)
    kv = ds.make_kv(I["kv_pools"], I["page_table"], I["ctx_len"], 128)
    ds.draft_block(x, kv, torch.empty_like(x), torch.empty(1, G.block, G.vocab, device="cuda"), 1)
    assert ds.check() == 18
    # the library still works afterwards
    ds.markov_rollout(z, torch.zeros(1, dtype=torch.int32, device="cuda"), smp, tokens, ell, 1)
    assert ds.check() == 0


def test_host_errors_on_device_handle(M):
    G = TINY
    ds = M.DSpark(G, to_cuda(gen.make_weights(TINY_STEP, "cpu")), max_bs=1)
    x = torch.empty(1, G.block, G.hidden, dtype=torch.float32, device="cuda")
    aux = torch.empty(1, G.block, G.n_aux, G.hidden, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(M.DSparkError) as e:
        ds.fuse_ctx(aux, x, 2)  # workspace sized for one sequence
    assert e.value.status == 6
    with pytest.raises(M.DSparkError) as e:
        ds.fuse_ctx(aux, x.view(-1)[1:], 1)
    assert e.value.status == 2
    with pytest.raises(M.DSparkError) as e:
        ds.fuse_ctx(aux, x, 0)
    assert e.value.status == 3
