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


# ---- FP4 E2M1 with per-32 UE8M0 scales
def _minifloat(code, ebits, mbits, bias):
    """Generic sign/exponent/mantissa decoder (no NaN/inf handling), checked
    against torch on two FP8 formats below and then applied to E2M1."""
    sign = (code >> (ebits + mbits)) & 1
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    if e == 0:
        v = m * 2.0 ** (1 - bias - mbits)
    else:
        v = (1 + m * 2.0 ** -mbits) * 2.0 ** (e - bias)
    return -v if sign else v


def test_generic_minifloat_matches_torch_fp8():
    for dt, eb, mb_, bias in ((torch.float8_e4m3fn, 4, 3, 7), (torch.float8_e5m2, 5, 2, 15)):
        codes = np.arange(256, dtype=np.uint8)
        ref = torch.from_numpy(codes).view(dt).to(torch.float64).numpy()
        for c in range(256):
            if np.isfinite(ref[c]):
                assert _minifloat(c, eb, mb_, bias) == ref[c], (dt, c)


def test_e2m1_all_codes():
    codes = np.arange(16)
    got = on.decode_e2m1(codes)
    want = np.array([_minifloat(int(c), 2, 1, 1) for c in codes])
    assert np.array_equal(got, want)
    # the published E2M1 value set: largest finite magnitude 6, smallest 0.5
    assert sorted(set(np.abs(got).tolist())) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(got[8:], -got[:8])


def test_unpack_e2m1_nibble_order():
    packed = np.array([[0x21, 0xF3]], dtype=np.uint8)
    assert on.unpack_e2m1(packed).tolist() == [[0x1, 0x2, 0x3, 0xF]]


def test_dequant_weight_mx4_brute_force():
    rng = np.random.default_rng(12)
    N, K = 6, 128
    packed = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sf = rng.integers(110, 140, (N, K // 32), dtype=np.uint8)
    got = on.dequant_weight_mx4(packed, sf)
    for n in range(N):
        for k in range(K):
            byte = int(packed[n, k // 2])
            code = (byte >> 4) if k % 2 else (byte & 0xF)
            v = _minifloat(code, 2, 1, 1) * 2.0 ** (int(sf[n, k // 32]) - 127)
            assert got[n, k] == v
