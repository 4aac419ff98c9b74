"""The drift harness's metrics (no GPU): closed forms and the identity between the
per-position sequential agreement and the mean leading run ("Kimi-K3-DSpark-
NVFP4", Measurement: the ceiling is a prefix-run-length statistic)."""
import math

import numpy as np
import torch

import bench


def test_snr_closed_form():
    w = torch.ones(100, dtype=torch.float64)
    assert abs(bench.weight_snr_db(w, w * 0.9) - 20.0) < 1e-9  # error 0.1 of the signal: 20 dB


def test_kl_and_overlap_two_point():
    l_ref = torch.tensor([[0.0, 0.0]], dtype=torch.float64)  # p = (1/2, 1/2)
    l_var = torch.tensor([[math.log(3.0), 0.0]], dtype=torch.float64)  # q = (3/4, 1/4)
    kl, ov = bench.kl_and_overlap(l_ref, l_var)
    want = 0.5 * math.log(0.5 / 0.75) + 0.5 * math.log(0.5 / 0.25)
    assert abs(float(kl[0]) - want) < 1e-12
    assert abs(float(ov[0]) - 0.75) < 1e-12                  # 1 - TV = 1/2 + 1/4
    kl0, ov0 = bench.kl_and_overlap(l_ref, l_ref)
    assert abs(float(kl0[0])) < 1e-15 and abs(float(ov0[0]) - 1.0) < 1e-15


def test_prefix_run_equals_ceiling_of_conditional_agreement():
    rng = np.random.default_rng(0)
    agree = rng.random((5000, 7)) < np.array([0.98, 0.95, 0.9, 0.93, 0.85, 0.9, 0.8])
    runs = bench.prefix_runs(agree)
    s = bench.conditional_agreement(agree)
    assert abs(bench.ceiling_from_agreement(s) - runs.mean()) < 1e-9
    assert bench.prefix_runs(np.array([[1, 1, 0, 1], [0, 1, 1, 1], [1, 1, 1, 1]])).tolist() == [2, 0, 4]


def test_ceiling_reproduces_the_cards_bf16_row():
    s = np.array([98.6, 98.0, 97.1, 96.4, 95.7, 94.6, 93.5]) / 100  # per-position agreement, boot, BF16
    assert abs(bench.ceiling_from_agreement(s) - 6.25) < 0.005


def test_pearson():
    a = np.arange(10.0)
    assert abs(bench.pearson(a, 3 * a + 1) - 1.0) < 1e-12
    assert abs(bench.pearson(a, -a) + 1.0) < 1e-12
