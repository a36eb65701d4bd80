"""Pins for the oracle's operand decoders and block-scale dequantisation."""
import math

import numpy as np
import pytest
import torch

from oracle import numerics as on

pytestmark = pytest.mark.cpu


def test_e4m3_all_codes_against_torch():
    """Every one of the 256 E4M3 codes against torch's float8_e4m3fn."""
    codes = np.arange(256, dtype=np.uint8)
    ours = on.decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert int(np.isnan(ours).sum()) == 2          # S.1111.111 only


def test_e4m3_known_codes():
    """Hand-derived values from the bit-field definition."""
    table = {0x00: 0.0, 0x80: -0.0, 0x38: 1.0, 0xB8: -1.0, 0x7E: 448.0, 0xFE: -448.0,
             0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x40: 2.0, 0x3C: 1.5}
    for c, v in table.items():
        got = on.decode_e4m3(np.array([c], np.uint8))[0]
        assert got == v and math.copysign(1, got) == math.copysign(1, v)
    assert np.isnan(on.decode_e4m3(np.array([0x7F, 0xFF], np.uint8))).all()


def test_ue8m0():
    s = np.arange(255, dtype=np.uint8)
    assert np.array_equal(on.decode_ue8m0(s), np.array([math.ldexp(1.0, int(x) - 127) for x in s]))
    assert np.isnan(on.decode_ue8m0(np.array([255], np.uint8))[0])


def test_bf16_exact():
    x = torch.randn(1000, dtype=torch.float32).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(on.decode_bf16(bits), x.to(torch.float64).numpy())


def test_dequant_rows_brute_force():
    """out[r, k] = e4m3(code[r, k]) * 2^(sf[k // 128, r] - 127), element by element."""
    rng = np.random.default_rng(3)
    R, K = 5, 256
    codes = rng.integers(0, 256, (R, K), dtype=np.uint8)
    codes[codes & 0x7F == 0x7F] = 0x11
    sf = rng.integers(100, 150, (K // 128, R), dtype=np.uint8)
    got = on.dequant_rows(codes, sf)
    for r in range(R):
        for k in range(K):
            v = on.decode_e4m3(codes[r:r + 1, k])[0] * 2.0 ** (int(sf[k // 128, r]) - 127)
            assert got[r, k] == v


def test_dequant_weight_brute_force():
    rng = np.random.default_rng(4)
    N, K = 256, 384
    codes = rng.integers(0, 0x7E, (N, K), dtype=np.uint8)
    sf = rng.integers(110, 140, (K // 128, N // 128), dtype=np.uint8)
    got = on.dequant_weight(codes, sf)
    for n in range(0, N, 37):
        for k in range(0, K, 29):
            v = on.decode_e4m3(codes[n:n + 1, k])[0] * 2.0 ** (int(sf[k // 128, n // 128]) - 127)
            assert got[n, k] == v


def test_power_of_two_scale_shifts_exactly():
    """Raising one scale byte by s multiplies exactly that block by 2^s."""
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 0x7E, (128, 256), dtype=np.uint8)
    sf = np.full((2, 1), 127, np.uint8)
    base = on.dequant_weight(codes, sf)
    sf2 = sf.copy()
    sf2[1, 0] = 130
    shifted = on.dequant_weight(codes, sf2)
    assert np.array_equal(shifted[:, :128], base[:, :128])
    assert np.array_equal(shifted[:, 128:], base[:, 128:] * 8.0)
