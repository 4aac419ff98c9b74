"""Host-side bookkeeping of bench.py (no GPU): the launch count it claims per step
follows the library's choices of kernels, and the algorithmic byte count matches
the sum of the step's parts (weights once, KV once, the small activations)."""
import types

import pytest
import torch

import bench
from synthetic.configs import FULL, TINY


@pytest.fixture
def sms152(monkeypatch):
    monkeypatch.setattr(torch.cuda, "get_device_properties", lambda i: types.SimpleNamespace(multi_processor_count=152))
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)


def _handle(G, ctx, bs=1):
    return types.SimpleNamespace(G=G, max_ctx=ctx, max_bs=bs)


def test_full_geometry_launches_62_kernels(sms152):
    # fc + 5 x 11 (the split combine fused with the v absorption) + final norm,
    # lm_head, rollout, confidence and the two greedy verify kernels; the count the
    # ncu launch list of one step shows
    assert bench.ds_launches_per_step(_handle(FULL, 4096)) == 62
    assert bench.ds_launches_per_step(_handle(FULL, 95000)) == 62


def test_verification_rules_add_their_kernels(sms152):
    # probabilistic: nucleus + accept-and-draw (as many as greedy); block: nucleus,
    # residual masses, decisions (the counts the verify launch list shows)
    assert bench.ds_launches_per_step(_handle(FULL, 95000), draft_mode=1, verify_mode=1) == 62
    assert bench.ds_launches_per_step(_handle(FULL, 4096), draft_mode=1, verify_mode=2) == 63


def test_one_split_at_batch_32(sms152):
    # 32 sequences leave one KV split per row tile and part: the fused kernel then
    # reads the attention's normalised output and only absorbs v (still one launch)
    assert bench.ds_launches_per_step(_handle(FULL, 4096, bs=32)) == 62


def test_other_latent_widths_use_the_unfused_combine(sms152):
    n = bench.ds_launches_per_step(_handle(TINY, 128))
    per_layer = (n - 1 - 6) / TINY.n_layers
    assert per_layer in (11, 12)


@pytest.mark.parametrize("fmt,base", [("bf16", 7.064e9), ("fp8", 4.878e9), ("nvfp4", 3.922e9)])
def test_algorithmic_bytes_full_step(fmt, base):
    # weights once (w2 once) + KV at ctx 4096, worked out by hand for the three
    # formats (bf16 7.064 GB, FP8 4.878 GB, NVFP4 3.922 GB); the bench adds the
    # step's small tensors: z and ell written and read, the target logits, aux
    ab = bench.algorithmic_bytes(FULL, 4096, fmt=fmt)
    small = ab["logits"] + ab["aux"]
    assert 20e6 < small < 30e6
    assert abs(ab["total"] - small - base) < 0.002 * base
