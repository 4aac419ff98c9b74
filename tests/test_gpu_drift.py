"""The drift harness end to end on a small geometry (GPU): the bench's --drift mode
runs every format through the library against the bf16 path; the line parses, its
figures lie in range, the ceiling equals the mean leading run, and the weight SNR
orders the formats as the cards' table does (FP8 > NVFP4 > MXFP4)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_drift_harness_small():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--drift", "--blocks", "6", "--regime", "all",
                        "--drift-geom", "mid"], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert [l["drift"] for l in lines] == ["boot", "heavy", "gauss"]
    for l in lines:
        F = l["formats"]
        assert F["fp8"]["weight_snr_db"] > F["nvfp4"]["weight_snr_db"] > F["mxfp4"]["weight_snr_db"] > 10
        for f, m in F.items():
            assert 0 <= m["greedy_agreement"] <= 1 and 0 <= m["sequential_rollout"] <= 1
            assert 0 <= m["ceiling"] <= 7 and abs(m["ceiling"] - m["mean_leading_run"]) < 1e-9
            assert 0 < m["one_minus_tv"] <= 1 and m["kl_mean"] >= 0 and m["kl_p99"] >= 0
            assert 0 <= m["hidden_rel_err"] < 1 and -1 <= m["confidence_r"] <= 1
