"""The bounded inter-CTA waits give up, report DSPARK_ERR_TIMEOUT and leave the
library usable (failure detection without a GPU fault).

The rollout kernels meet at grid barriers in the workspace. Here the barrier's
arrival word is poisoned so that it can never complete (a flag nothing sets),
and the wait limit in the workspace (bytes 72..79) is set to 1 ms: every CTA
must give up, free its tensor memory and return; dspark_check reports the
time-out; after the workspace is zero-filled again the same call is bit-exact
against the oracle."""
import numpy as np
import pytest
import torch

from oracle import sampling as S
from synthetic import generate as gen
from synthetic.configs import TINY
from tests.gpu_harness import u32, workload

pytestmark = pytest.mark.gpu
TIMEOUT = 16


@pytest.fixture(scope="module")
def M():
    import mla_block_diffusion_gb300 as M
    from mla_block_diffusion_gb300 import build
    build.build()
    return M


def poison(ds, wait_ns: int):
    ws = ds.ws
    ws[72:80].view(torch.int64).fill_(wait_ns)          # wait limit of the sampling kernels
    ws[64:68].view(torch.int32).fill_(0x40000000)        # grid-barrier arrivals: never reaches the grid size


@pytest.mark.parametrize("bs,mode", [(1, 0), (2, 0), (1, 1)], ids=["resident_greedy", "streaming_bs2", "prob_bs1"])
def test_rollout_wait_times_out_and_recovers(M, bs, mode):
    G = TINY
    W = gen.make_weights(workload(G, bs, (0,) * bs, 5), "cpu")
    z = gen.draft_logits(bs, G.block, G.vocab, 5)
    anchor = gen.uniform_tokens((bs,), G.vocab, 5, "anchor")
    ds = M.DSpark(G, {k: v.cuda() for k, v in W.items()}, max_bs=bs)
    tokens = torch.empty(bs, G.block, dtype=torch.int32, device="cuda")
    ell = torch.empty(bs, G.block, G.vocab, dtype=torch.float32, device="cuda")
    smp = M.Sample(mode, mode, 1.0, 0.9, 3, 1)
    poison(ds, 1_000_000)
    ds.markov_rollout(z.cuda(), anchor.cuda(), smp, tokens, ell, bs)
    assert ds.check() == TIMEOUT
    ds.ws.zero_()
    ds.markov_rollout(z.cuda(), anchor.cuda(), smp, tokens, ell, bs)
    assert ds.check() == 0
    for b in range(bs):
        t_o, ell_o = S.markov_rollout(z[b].numpy(), W["markov_w1"], W["markov_w2"], int(anchor[b]), mode, 1.0, 0.9,
                                      seed=3, seq=b, step=1)
        assert tokens[b].cpu().numpy().tolist() == t_o.tolist(), b
        assert np.array_equal(u32(ell[b].cpu().numpy()), u32(ell_o)), b
