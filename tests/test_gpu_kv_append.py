"""Latent-cache append through the C ABI against the oracle: appended entries
within bf16 rounding (rel-L2 <= 1e-2 per entry), every other pool entry
byte-identical, ctx_len advanced exactly; out-of-range counts reported."""
import numpy as np
import pytest
import torch

from oracle import network as N
from synthetic import generate as gen
from synthetic.configs import TINY
from tests.gpu_harness import MID, MIDLAT, workload
from tests.helpers import f64, oracle_layers, rel_l2

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def M():
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build
    build.build()
    return M


def _setup(G, bs, ctx, n_max, seed):
    """Seeded weights and cache plus one spare page per sequence for the new tokens."""
    w = workload(G, bs, ctx, seed=seed)
    W = gen.make_weights(w, "cpu")
    I = gen.make_inputs(w, "cpu")
    P = G.page_size
    npg = [max(1, -(-c // P)) for c in ctx]
    spare = torch.arange(I["n_pages"], I["n_pages"] + bs, dtype=torch.int32)
    table = torch.cat([I["page_table"], torch.zeros((bs, 1), dtype=torch.int32)], dim=1)
    for b in range(bs):
        table[b, npg[b]:] = spare[b]
    pools = [torch.cat([p, gen.normal((bs, P, G.kv_dim), 1.0, seed, f"spare{l}", "cpu")])
             for l, p in enumerate(I["kv_pools"])]
    x_new = gen.normal((bs, n_max, G.hidden), 1.0, seed, "x_new", "cpu").float()
    return W, pools, table, x_new


@pytest.mark.parametrize("G,bs,ctx,n_new,n_max", [
    (TINY, 2, (62, 128), (4, 0), 5),             # crosses a page boundary; one sequence appends nothing
    (MID, 3, (1000, 77, 300), (8, 1, 3), 8),
    (MIDLAT, 2, (4094, 0), (7, 8), 8),           # full latent width; an empty context
])
def test_kv_append_matches_oracle(M, G, bs, ctx, n_new, n_max):
    W, pools, table, x_new = _setup(G, bs, ctx, n_max, seed=21)
    ds = M.DSpark(G, {k: v.cuda() for k, v in W.items()}, max_bs=bs, max_ctx=max(ctx) + n_max)
    pools_d = [p.cuda() for p in pools]
    ctx_d = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    table_d = table.cuda()  # the KV struct holds raw pointers: keep every tensor alive
    kv = ds.make_kv(pools_d, table_d, ctx_d, max(ctx) + n_max)
    ds.kv_append(x_new.cuda(), torch.tensor(n_new, dtype=torch.int32, device="cuda"), kv, bs)
    assert ds.check() == 0
    assert ctx_d.cpu().tolist() == [c + n for c, n in zip(ctx, n_new)]

    want, ctx2 = N.kv_append(f64(x_new), oracle_layers(W, G), G, [f64(p) for p in pools], table.numpy(),
                             np.array(ctx), np.array(n_new))
    assert list(ctx2) == ctx_d.cpu().tolist()
    P = G.page_size
    for l in range(G.n_layers):
        got = pools_d[l].cpu()
        touched = torch.zeros(got.shape[:2], dtype=torch.bool)
        for b in range(bs):
            for j in range(n_new[b]):
                pos = ctx[b] + j
                pg, off = int(table[b, pos // P]), pos % P
                touched[pg, off] = True
                assert rel_l2(got[pg, off].double().numpy(), want[l][pg, off]) < TOL, (l, b, j)
        assert torch.equal(got[~touched], pools[l][~touched])


def test_kv_append_reports_bad_counts(M):
    G, bs, ctx, n_max = TINY, 2, (10, 20), 4
    W, pools, table, x_new = _setup(G, bs, ctx, n_max, seed=22)
    ds = M.DSpark(G, {k: v.cuda() for k, v in W.items()}, max_bs=bs, max_ctx=64)
    pools_d = [p.cuda() for p in pools]
    ctx_d = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    table_d = table.cuda()
    kv = ds.make_kv(pools_d, table_d, ctx_d, 64)
    ds.kv_append(x_new.cuda(), torch.tensor([2, n_max + 1], dtype=torch.int32, device="cuda"), kv, bs)
    assert ds.check() == 18
    assert ctx_d.cpu().tolist() == [12, 20]     # the bad sequence keeps its length
    for l in range(G.n_layers):                 # and none of its slots were written
        got = pools_d[l].cpu()
        for j in range(n_max + 1):
            pos = ctx[1] + j
            assert torch.equal(got[int(table[1, pos // 64]), pos % 64], pools[l][int(table[1, pos // 64]), pos % 64])
