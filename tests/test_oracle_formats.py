"""Pins of the oracle's weight-format decoders (no GPU)."""
import numpy as np
import torch

from oracle import formats as F
from synthetic import quantize as Q


def test_e4m3_known_codes_and_library_agreement():
    assert F.e4m3_value(0x38) == 1.0
    assert F.e4m3_value(0x7E) == 448.0          # largest finite
    assert F.e4m3_value(0x01) == 2.0 ** -9      # smallest subnormal
    assert F.e4m3_value(0x08) == 2.0 ** -6      # smallest normal
    assert F.e4m3_value(0xB8) == -1.0
    assert np.isnan(F.e4m3_value(0x7F)) and np.isnan(F.e4m3_value(0xFF))
    # every code agrees with the library's float8_e4m3fn (a plain format conversion)
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ok = ~np.isnan(lib)
    assert np.array_equal(F.E4M3_TABLE[ok], lib[ok]) and np.array_equal(np.isnan(F.E4M3_TABLE), ~ok)


def test_e2m1_grid():
    assert F.E2M1_TABLE[:8].tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert F.E2M1_TABLE[8:].tolist() == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_round_trips_are_exact_on_grid_values():
    # rows whose entries are grid values times a power of two quantise and decode exactly
    g = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -6.0, -4.0, -3.0, -2.0, -1.5, -1.0, -0.5, 0.0])
    w = (torch.stack([g * 2.0 ** -k for k in range(4)]) * 0.125).to(torch.bfloat16)
    d, s, glob = Q.quant_nvfp4(w)
    assert np.array_equal(F.dequant_nvfp4(d.numpy(), s.numpy(), glob), w.double().numpy())
    w8 = torch.tensor([[1.0, -2.0, 448.0, 0.5], [3.5, 0.0, -0.25, 1.75]]).to(torch.bfloat16)
    q, sc = Q.quant_fp8(w8)
    assert np.allclose(F.dequant_fp8(q.numpy(), sc.numpy()), w8.double().numpy(), rtol=0, atol=0)


def test_nibble_order_and_group_scales():
    codes = np.arange(16, dtype=np.uint8)
    packed = (codes[0::2] | (codes[1::2] << 4))[None, :]
    scales = np.array([[0x38]], dtype=np.uint8)  # 1.0
    out = F.dequant_nvfp4(packed, scales, 2.0)
    assert out[0].tolist() == (2.0 * F.E2M1_TABLE).tolist()
    scales2 = np.array([[0x40]], dtype=np.uint8)  # 2.0
    assert np.array_equal(F.dequant_nvfp4(packed, scales2, 1.0), out)


def test_quantisation_error_of_gaussian_weights():
    """Weight SNR on N(0, 0.02^2): FP8 per-channel near 31 dB, NVFP4 near 20 dB (the cards report
    31.5 / 20.4 dB on the real weights; these are the synthetic stand-ins, reported not pinned)."""
    w = (torch.randn(256, 1024, generator=torch.Generator().manual_seed(0)) * 0.02).to(torch.bfloat16)
    ref = w.double().numpy()
    q, sc = Q.quant_fp8(w)
    e8 = F.dequant_fp8(q.numpy(), sc.numpy()) - ref
    d, s, g = Q.quant_nvfp4(w)
    e4 = F.dequant_nvfp4(d.numpy(), s.numpy(), g) - ref
    snr = lambda e: 10 * np.log10((ref ** 2).sum() / (e ** 2).sum())
    assert 26 < snr(e8) < 36
    assert 15 < snr(e4) < 25


def test_e8m0_scales():
    assert F.e8m0_value(127) == 1.0
    assert F.e8m0_value(0) == 2.0 ** -127
    assert F.e8m0_value(254) == 2.0 ** 127
    assert F.e8m0_value(130) == 8.0
    assert np.isnan(F.e8m0_value(255))


def test_mxfp4_hand_decoded_row():
    # 64 inputs: group 0 scale 2^-3, group 1 scale 2^2; codes 1 (0.5) and 0xF (-6) alternate
    packed = np.full((1, 32), 0xF1, dtype=np.uint8)   # low nibble 1 (even inputs), high nibble 0xF (odd)
    scales = np.array([[124, 129]], dtype=np.uint8)
    w = F.dequant_mxfp4(packed, scales)
    assert w.shape == (1, 64)
    assert np.all(w[0, 0:32:2] == 0.5 * 2.0 ** -3) and np.all(w[0, 1:32:2] == -6 * 2.0 ** -3)
    assert np.all(w[0, 32::2] == 0.5 * 4) and np.all(w[0, 33::2] == -6 * 4)


def test_mxfp4_round_trip_and_saturation():
    rng = np.random.default_rng(4)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    # groups whose largest magnitude is 6 * 2^k: the shared exponent is k and every value survives
    k = rng.integers(-8, 3, size=(3, 4))
    vals = rng.choice(grid, size=(3, 4, 32)) * rng.choice([-1, 1], size=(3, 4, 32))
    vals[..., 0] = 6.0
    w = (vals * 2.0 ** k[..., None]).reshape(3, 128)
    d, s, _ = Q.quant_mxfp4(torch.tensor(w, dtype=torch.float64))
    assert np.array_equal(F.dequant_mxfp4(d.numpy(), s.numpy()), w)
    # amax 7 * 2^k: shared exponent floor(log2 7) - 2 = 0, so 7 saturates to 6 (the OCP rule)
    w2 = np.zeros((1, 32))
    w2[0, 0] = 7.0
    w2[0, 1] = 0.25
    d, s, _ = Q.quant_mxfp4(torch.tensor(w2, dtype=torch.float64))
    out = F.dequant_mxfp4(d.numpy(), s.numpy())
    assert out[0, 0] == 6.0 and int(s[0, 0]) == 127 and out[0, 1] in (0.0, 0.5)
