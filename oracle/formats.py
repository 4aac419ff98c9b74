"""ORACLE (test infrastructure only): decoders of the weight-only formats, written
from the format definitions, float64 out. The oracle runs the network on the
decoded (dequantised) weights.

* E4M3 (OCP 8-bit floating point): sign, 4 exponent bits (bias 7), 3 mantissa bits;
  exponent 0 is subnormal (m / 8 * 2^-6); exponent 15 with mantissa 7 is NaN; no infinity.
* E2M1 (OCP 4-bit): sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is
  subnormal (m / 2); magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
* FP8 weight-only ("Kimi-K3-DSpark-NVFP4", Considerations: per-channel weight-only FP8):
  w = E4M3(q) * scale[row].
* NVFP4 weight-only ("Kimi-K3-DSpark-NVFP4", header: group-16, E4M3 group scales,
  weight-only): w = E2M1(q) * E4M3(s_group) * global; two codes per byte, the even
  element in the low nibble.
* MXFP4 weight-only (the cards' third format, "Kimi-K3-DSpark-NVFP4", Measurement:
  the MXFP4 column; its encoding is the OCP Microscaling v1.0 MXFP4 element type):
  w = E2M1(q) * 2^(s_group - 127) with an E8M0 scale byte per group of 32 inputs
  (255 is NaN); two codes per byte, the even element in the low nibble.
"""
from __future__ import annotations

import numpy as np


def e4m3_value(code: int) -> float:
    code = int(code) & 0xFF
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e2m1_value(code: int) -> float:
    code = int(code) & 0xF
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m * 0.5
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def dequant_fp8(data: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """data uint8 [out, in] E4M3 codes, scale fp32 [out] -> float64 [out, in]."""
    return E4M3_TABLE[np.asarray(data, dtype=np.uint8)] * np.asarray(scale, dtype=np.float64)[:, None]


def dequant_nvfp4(packed: np.ndarray, scales: np.ndarray, global_scale: float) -> np.ndarray:
    """packed uint8 [out, in/2], scales uint8 [out, in/16] E4M3, global fp32 -> float64 [out, in]."""
    packed = np.asarray(packed, dtype=np.uint8)
    out_f, half = packed.shape
    codes = np.empty((out_f, 2 * half), dtype=np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    s = E4M3_TABLE[np.asarray(scales, dtype=np.uint8)]           # [out, in/16]
    return E2M1_TABLE[codes] * np.repeat(s, 16, axis=1) * float(global_scale)


def e8m0_value(code: int) -> float:
    """E8M0 scale: 2^(code - 127); code 255 is NaN."""
    code = int(code) & 0xFF
    if code == 0xFF:
        return float("nan")
    return 2.0 ** (code - 127)


E8M0_TABLE = np.array([e8m0_value(c) for c in range(256)], dtype=np.float64)


def dequant_mxfp4(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """packed uint8 [out, in/2] (even element low nibble), scales uint8 [out, in/32]."""
    packed = np.asarray(packed, dtype=np.uint8)
    out_f, half = packed.shape
    codes = np.empty((out_f, 2 * half), dtype=np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    vals = E2M1_TABLE[codes]
    s = E8M0_TABLE[np.asarray(scales, dtype=np.uint8)]
    return vals * np.repeat(s, 32, axis=1)
