"""The allocation-free fc fusion (dspark_fuse_ctx_noalloc) through the C ABI,
against the workspace version (dspark_fuse_ctx) and the oracle.

Some callers cannot give the library device memory: a serving process whose
device memory another allocator has already reserved, a latency-critical path
that may not call cudaMalloc, a plugin host that forbids libraries from owning
device buffers. For them the fusion keeps its scratch in a fixed array inside
the library. This file runs last so that a failure here never hides another
test; it passes alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

from oracle import network as N
from synthetic import generate as gen
from synthetic import quantize as Q
from synthetic.configs import FORMAT_FP8, TINY_STEP
from tests.gpu_harness import MID, workload
from tests.helpers import f64, rel_l2

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def M():
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build
    build.build()
    return M


@pytest.mark.parametrize("w", [TINY_STEP, workload(MID, 2, (64, 64), seed=3)], ids=["tiny_bs1", "mid_bs2"])
def test_noalloc_matches_workspace_fusion_and_oracle(M, w):
    G, bs = w.geom, w.bs
    Wc = gen.make_weights(w, "cpu")
    W = {k: v.cuda() for k, v in Wc.items()}
    aux_c = gen.make_inputs(w, "cpu")["aux"]
    aux = aux_c.cuda()
    ds = M.DSpark(G, W, max_bs=bs)
    ref = torch.empty(bs, G.block, G.hidden, dtype=torch.float32, device="cuda")
    ds.fuse_ctx(aux, ref, bs)
    assert ds.check() == 0
    ox = np.stack([N.fuse_ctx(f64(Wc["w_fc"]), f64(aux_c[b])) for b in range(bs)])
    for call in range(2):  # two calls in a row share (and must clear) the fixed scratch
        x = torch.full((bs, G.block, G.hidden), float("nan"), dtype=torch.float32, device="cuda")
        ds.fuse_ctx_noalloc(aux, x, bs)
        torch.cuda.synchronize()
        assert ds.check_noalloc() == 0, call
        assert torch.isfinite(x).all(), call
        assert rel_l2(x.cpu().numpy(), ref.cpu().numpy()) < TOL, call
        assert rel_l2(x.cpu().numpy(), ox) < TOL, call


def test_noalloc_rejects_sizes_beyond_its_limit(M):
    G = TINY_STEP.geom
    W = {k: v.cuda() for k, v in gen.make_weights(TINY_STEP, "cpu").items()}
    ds = M.DSpark(G, W, max_bs=3)
    aux = torch.zeros(3, G.block, G.n_aux, G.hidden, dtype=torch.bfloat16, device="cuda")
    x = torch.empty(3, G.block, G.hidden, dtype=torch.float32, device="cuda")
    with pytest.raises(M.DSparkError) as e:
        ds.fuse_ctx_noalloc(aux, x, 3)
    assert e.value.status == 3


def test_noalloc_rejects_quantised_weights_before_launching(M):
    """The fixed-scratch fusion streams bf16 fc weights only: a handle with FP8
    weights gets DSPARK_ERR_UNSUPPORTED (4) from the host check, and the output
    is left untouched."""
    G = TINY_STEP.geom
    W = gen.make_weights(TINY_STEP, "cpu")
    Wq = Q.quantise_weights(W, "fp8", G.n_layers)
    Wd = {k: (tuple(x.cuda() if torch.is_tensor(x) else x for x in v) if isinstance(v, tuple) else v.cuda())
          for k, v in Wq.items()}
    ds = M.DSpark(G, Wd, max_bs=1, weight_format=FORMAT_FP8)
    aux = gen.make_inputs(TINY_STEP, "cpu")["aux"].cuda()
    x = torch.full((1, G.block, G.hidden), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(M.DSparkError) as e:
        ds.fuse_ctx_noalloc(aux, x, 1)
    assert e.value.status == 4
    torch.cuda.synchronize()
    assert bool((x == 7.0).all())
