"""Weight-only FP8 / NVFP4 / MXFP4 versions of the seeded bf16 weights (input preparation).

The model cards ship FP8 and NVFP4 artefacts of the drafter ("Kimi-K3-DSpark-NVFP4":
"compressed-tensors nvfp4-pack-quantized, group-16, E4M3 group scales, weight-only";
FP8 per-channel weight-only as the recommended build) produced by an external
quantiser. This module stands in for that quantiser so the synthetic weights exist in
both formats; it is input preparation, not a step of the path:

* FP8: per output row s = amax / 448, q = round-to-nearest-even(w / s) in E4M3.
* NVFP4: global g = amax_tensor / (448 * 6); per group of 16 along the input dimension
  s = E4M3(amax_group / 6 / g); q = nearest E2M1 value of w / (s * g) (ties to the
  even code), two codes per byte, the even element in the low nibble.

Quantised matrices: fc, q_b, o, gate, up, down ("What is quantized to what"); q_a/kv_a,
kv_b, lm_head, the Markov matrices, norms and the confidence head stay as they are.
"""
from __future__ import annotations

from typing import Dict, Tuple

import torch

QUANTISED = ("w_fc", "w_q_b", "w_o", "w_gate", "w_up", "w_down")

# E2M1 magnitudes by code (bit 3 is the sign)
_E2M1 = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float64)


def quant_fp8(w: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """bf16 [out, in] -> (E4M3 bytes as uint8 [out, in], fp32 scale [out])."""
    wf = w.to(torch.float32)
    amax = wf.abs().amax(dim=1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (wf / scale[:, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), scale.to(torch.float32)


def _e2m1_codes(x: torch.Tensor) -> torch.Tensor:
    """Nearest E2M1 code of each value (|x| clamped to 6), ties to the even code."""
    grid = _E2M1.to(x.device)
    mag = x.abs().clamp(max=6.0).to(torch.float64)
    hi = torch.bucketize(mag, grid).clamp(max=7)          # first code with grid >= mag
    lo = (hi - 1).clamp(min=0)
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = torch.where(pick_hi, hi, lo)
    sign = ((x < 0) & (idx > 0)).to(torch.int64) << 3
    return (idx + sign).to(torch.uint8)


def quant_nvfp4(w: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor, float]:
    """bf16 [out, in] -> (packed E2M1 uint8 [out, in/2], E4M3 group scales uint8 [out, in/16], global fp32)."""
    out_f, in_f = w.shape
    assert in_f % 16 == 0
    wf = w.to(torch.float32)
    amax_t = float(wf.abs().max())
    g = amax_t / (448.0 * 6.0) if amax_t > 0 else 1.0
    grp = wf.view(out_f, in_f // 16, 16)
    amax_g = grp.abs().amax(dim=2)
    s = (amax_g / 6.0 / g).clamp(max=448.0).to(torch.float8_e4m3fn)
    s_val = s.to(torch.float32)
    denom = (s_val * g)[..., None]
    x = torch.where(denom > 0, grp / torch.where(denom > 0, denom, torch.ones_like(denom)), torch.zeros_like(grp))
    codes = _e2m1_codes(x).view(out_f, in_f)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8)
    return packed.contiguous(), s.view(torch.uint8).contiguous(), float(g)


def quant_mxfp4(w: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor, float]:
    """bf16 [out, in] -> (packed E2M1 uint8 [out, in/2], E8M0 scale bytes uint8 [out, in/32], 1.0).
    OCP MX: shared exponent floor(log2(amax_group)) - 2 (the largest E2M1 exponent), elements
    rounded to the nearest E2M1 value of w / 2^shared (ties to the even code), saturating at 6."""
    out_f, in_f = w.shape
    assert in_f % 32 == 0
    wf = w.to(torch.float64)
    grp = wf.view(out_f, in_f // 32, 32)
    amax = grp.abs().amax(dim=2)
    ex = torch.where(amax > 0, torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))) - 2,
                     torch.full_like(amax, -127.0)).clamp(-127, 127)
    x = grp / torch.pow(2.0, ex)[..., None]
    codes = _e2m1_codes(x).view(out_f, in_f)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8)
    return packed.contiguous(), (ex + 127).to(torch.uint8).contiguous(), 1.0


def quantise_weights(W: Dict[str, torch.Tensor], fmt: str, n_layers: int) -> Dict[str, object]:
    """Return a copy of the weight dict where the quantised matrices are replaced by
    (data, scale, global_scale) triples; everything else is shared."""
    out: Dict[str, object] = dict(W)
    names = ["w_fc"] + [f"l{l}.{k}" for l in range(n_layers) for k in QUANTISED[1:]]
    for n in names:
        if fmt == "fp8":
            d, sc = quant_fp8(W[n])
            out[n] = (d, sc, 1.0)
        elif fmt == "nvfp4":
            out[n] = quant_nvfp4(W[n])
        elif fmt == "mxfp4":
            out[n] = quant_mxfp4(W[n])
        else:
            raise ValueError(fmt)
    return out
