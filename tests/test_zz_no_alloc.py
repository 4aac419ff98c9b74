"""The allocation-free fc fusion (dspark_fuse_ctx_noalloc) against the
workspace version (dspark_fuse_ctx), through the C ABI.

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

from synthetic import generate as gen
from synthetic.configs import TINY_STEP
from tests.gpu_harness import MID, workload
from tests.helpers import rel_l2

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def M():
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build
    build.build()
    return M


@pytest.mark.parametrize("w", [TINY_STEP, workload(MID, 2, (64, 64), seed=3)], ids=["tiny_bs1", "mid_bs2"])
def test_noalloc_matches_workspace_fusion(M, w):
    G, bs = w.geom, w.bs
    W = {k: v.cuda() for k, v in gen.make_weights(w, "cpu").items()}
    aux = gen.make_inputs(w, "cpu")["aux"].cuda()
    ds = M.DSpark(G, W, max_bs=bs)
    ref = torch.empty(bs, G.block, G.hidden, dtype=torch.float32, device="cuda")
    ds.fuse_ctx(aux, ref, bs)
    assert ds.check() == 0
    for call in range(2):  # two calls in a row share (and must clear) the fixed scratch
        x = torch.full((bs, G.block, G.hidden), float("nan"), dtype=torch.float32, device="cuda")
        ds.fuse_ctx_noalloc(aux, x, bs)
        torch.cuda.synchronize()
        assert torch.isfinite(x).all(), call
        assert rel_l2(x.cpu().numpy(), ref.cpu().numpy()) < TOL, call


def test_noalloc_rejects_sizes_beyond_its_limit(M):
    G = TINY_STEP.geom
    W = {k: v.cuda() for k, v in gen.make_weights(TINY_STEP, "cpu").items()}
    ds = M.DSpark(G, W, max_bs=3)
    aux = torch.zeros(3, G.block, G.n_aux, G.hidden, dtype=torch.bfloat16, device="cuda")
    x = torch.empty(3, G.block, G.hidden, dtype=torch.float32, device="cuda")
    with pytest.raises(M.DSparkError) as e:
        ds.fuse_ctx_noalloc(aux, x, 3)
    assert e.value.status == 3
