"""Test-side marshalling: torch tensors from the seeded generators to the
float64 numpy arrays the oracle takes. Holds no arithmetic of the method."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy()


def oracle_layers(W: dict, geom) -> list:
    keys = ["attn_norm", "w_qkv_a", "q_a_norm", "kv_a_norm", "w_q_b", "w_kv_b", "w_o", "mlp_norm",
            "w_gate", "w_up", "w_down"]
    return [{k: f64(W[f"l{l}.{k}"]) for k in keys} for l in range(geom.n_layers)]


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
