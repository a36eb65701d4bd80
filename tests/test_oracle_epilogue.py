"""Pins of the oracle's SwiGLU and FP8 re-quantisation (oracle/epilogue.py)
against facts fixed by mathematics and by the E4M3 / UE8M0 definitions."""
import numpy as np
import pytest
import torch

from oracle import epilogue as oe
from oracle import numerics as on

pytestmark = pytest.mark.cpu


def test_silu_closed_forms():
    x = np.linspace(-40.0, 40.0, 2001)
    s = oe.silu(x)
    assert oe.silu(np.array([0.0]))[0] == 0.0
    # SiLU(x) - SiLU(-x) = x sigmoid(x) + x sigmoid(-x) = x
    assert np.allclose(s - oe.silu(-x), x, rtol=0, atol=1e-12)
    # sigmoid(1) = e / (1 + e)
    assert oe.silu(np.array([1.0]))[0] == pytest.approx(np.e / (1.0 + np.e), rel=1e-15)
    # far tails: SiLU(x) -> x for large x, -> 0 for very negative x (no overflow)
    assert oe.silu(np.array([800.0]))[0] == 800.0
    assert oe.silu(np.array([-800.0]))[0] == pytest.approx(0.0, abs=1e-300)
    # minimum of SiLU near x = -1.2785 is about -0.2785
    assert s.min() == pytest.approx(-0.27846454, abs=1e-6)


def test_swiglu_is_product():
    g = np.array([0.0, 1.0, -2.0, 3.5])
    u = np.array([5.0, -2.0, 0.5, 0.0])
    assert np.array_equal(oe.swiglu(g, u), oe.silu(g) * u)


def test_encode_roundtrips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = on.decode_e4m3(codes)
    assert np.array_equal(oe.encode_e4m3(vals), codes)


def test_encode_rounds_to_nearest_even_and_saturates():
    mags = on.decode_e4m3(np.arange(127, dtype=np.uint8))
    mid = (mags[:-1] + mags[1:]) / 2              # exact midpoints (in float64)
    got = oe.encode_e4m3(mid)
    lo = np.arange(126)
    want = np.where(lo % 2 == 0, lo, lo + 1)      # ties go to the even code
    assert np.array_equal(got, want.astype(np.uint8))
    # just off the midpoint goes to the nearer side
    assert np.array_equal(oe.encode_e4m3(np.nextafter(mid, 0)), lo.astype(np.uint8))
    assert np.array_equal(oe.encode_e4m3(np.nextafter(mid, 1e9)), (lo + 1).astype(np.uint8))
    assert oe.encode_e4m3(np.array([1e9, -1e9, 449.0])).tolist() == [0x7E, 0xFE, 0x7E]
    assert oe.encode_e4m3(np.array([-0.0]))[0] == 0x80


def test_encode_agrees_with_torch_float8_in_range():
    x = torch.randn(20000, dtype=torch.float64, generator=torch.Generator().manual_seed(3)) * 50
    x = x.clamp(-448, 448)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oe.encode_e4m3(x.numpy()), ref)


def test_ue8m0_boundaries():
    k = np.arange(-20, 21)
    a = 448.0 * np.exp2(k.astype(np.float64))
    assert np.array_equal(oe.ue8m0_for_amax(a), (127 + k).astype(np.uint8))           # exactly on the bound
    assert np.array_equal(oe.ue8m0_for_amax(np.nextafter(a, np.inf)), (128 + k).astype(np.uint8))
    assert np.array_equal(oe.ue8m0_for_amax(a * 0.51), (127 + k).astype(np.uint8))   # down to just above half
    assert oe.ue8m0_for_amax(np.array([0.0]))[0] == 127
    assert oe.ue8m0_for_amax(np.array([1e-300]))[0] == 1     # clamped
    assert oe.ue8m0_for_amax(np.array([1e300]))[0] == 254


def test_quantize_blocks_bounds_and_layout():
    rng = np.random.default_rng(0)
    h = rng.standard_normal((5, 256)) * np.exp2(rng.integers(-8, 8, size=(5, 1)))
    h[2, 128:] = 0.0                                          # an all-zero block
    codes, sf = oe.quantize_blocks(h)
    assert sf.shape == (2, 5) and codes.shape == (5, 256)
    assert sf[1, 2] == 127 and np.all(codes[2, 128:] == 0)
    deq = on.decode_e4m3(codes) * np.exp2(np.repeat(sf.T.astype(np.float64), 128, axis=1) - 127)
    amax = np.abs(h.reshape(5, 2, 128)).max(axis=2)
    # the block maximum fits: max|h| <= 448 * scale, and half the scale would not do
    scale = np.exp2(sf.T.astype(np.float64) - 127)
    nz = amax > 0
    assert np.all(amax[nz] <= 448 * scale[nz]) and np.all(amax[nz] > 224 * scale[nz])
    # error of each element: at most half the E4M3 spacing at its magnitude
    # (relative 2^-4 for normals, 2^-10 * scale in the subnormal range)
    s_el = np.repeat(scale, 128, axis=1)
    bound = np.maximum(np.abs(h) * 2.0 ** -4, 2.0 ** -10 * s_el)
    assert np.all(np.abs(deq - h) <= bound * (1 + 1e-12))


def test_gate_up_halves_layout():
    R, F = 3, 256
    H = np.arange(R * 2 * F, dtype=np.float64).reshape(R, 2 * F)
    g, u = oe.gate_up_halves(H)
    # feature f of block j: gate at column 256 j + f % 128, up at 256 j + 128 + f % 128
    for f in (0, 5, 127, 128, 200, 255):
        j, i = divmod(f, 128)
        assert np.array_equal(g[:, f], H[:, 256 * j + i])
        assert np.array_equal(u[:, f], H[:, 256 * j + 128 + i])
