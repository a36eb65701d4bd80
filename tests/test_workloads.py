"""The seeded generators reproduce the documented draws and encode FP8 safely."""
import numpy as np
import pytest
import torch

from moe_grouped_gemm_side_gb300 import workloads as wl
from oracle import numerics as on

pytestmark = pytest.mark.cpu


def test_decode_histogram_draw():
    v = wl.counts_zipf_decode()
    assert v == [0, 1, 6, 20, 38, 31, 2, 13, 200, 27, 1, 0, 27, 85, 3, 0]
    assert sum(v) == 454 and sum(1 for x in v if x) == 13


def test_min_zeros_rule():
    for seed in range(40):
        v = wl.counts_zipf_decode(seed=seed, min_zeros=5)
        assert sum(1 for x in v if x == 0) >= 5 and all(0 <= x <= 256 for x in v)


def test_prefill_histogram_draw():
    c = wl.counts_zipf_prefill()
    c = np.array(c, dtype=np.float64)
    assert c.sum() == 32768 and c.max() == 9578 and c.min() == 55
    assert abs(c.sum() ** 2 / (c ** 2).sum() - 8.47) < 0.01


def test_dirichlet_histogram_draw():
    c = wl.counts_dirichlet()
    assert sum(c) == 65536 and c.count(0) == 2 and max(c) == 16548


def test_fp8_rows_roundtrip_and_range():
    x = wl.normal_f32((37, 512), 7) * 100.0
    x[3, :128] = 0.0
    codes, sf = wl.quantize_rows_fp8(x)
    assert codes.shape == (37, 512) and sf.shape == (4, 37)
    assert int(sf[0, 3]) == 127
    deq = on.dequant_rows(codes.numpy(), sf.numpy())
    assert not np.isnan(deq).any()
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 for normal values
    xe = x.double().numpy()
    big = np.abs(xe) > 1e-2 * np.abs(xe).max()
    assert np.max(np.abs(deq - xe)[big] / np.abs(xe)[big]) <= 2.0 ** -4
    # the block maximum lands in the top binade of E4M3 (224 after rounding down)
    blk = np.abs(codes.view(torch.float8_e4m3fn).float().numpy()).reshape(37, 4, 128).max(axis=2)
    assert ((blk >= 224) | (blk == 0)).all()


def test_fp8_weight_scales_shape():
    w = wl.normal_f32((256, 384), 8)
    codes, sf = wl.quantize_weight_fp8(w)
    assert sf.shape == (3, 2)
    deq = on.dequant_weight(codes.numpy(), sf.numpy())
    assert np.max(np.abs(deq - w.double().numpy())) <= 2.0 ** -4 * float(w.abs().max())


def test_masked_sfa_layout():
    ops = wl.make_masked(3, 32, 128, 256, "fp8", seed=5)
    assert ops.A.shape == (3, 32, 256) and ops.SFA.shape == (3, 2, 32) and ops.SFB.shape == (3, 2, 1)


def test_mx4_weight_generator_round_trips():
    """The FP4 weight generator's bytes decode (oracle) to within half an E2M1
    spacing of the drawn values, with the block maximum inside 6 * scale."""
    from oracle import numerics as on
    w = wl.normal_f32((64, 256), 5, "cpu", 0.1)
    packed, sf = wl.quantize_weight_mx4(w)
    assert packed.shape == (64, 128) and sf.shape == (64, 8)
    deq = on.dequant_weight_mx4(packed.numpy(), sf.numpy())
    x = w.double().numpy()
    scale = np.repeat(np.exp2(sf.numpy().astype(np.float64) - 127), 32, axis=1)
    amax = np.repeat(np.abs(x.reshape(64, 8, 32)).max(axis=2), 32, axis=1)
    assert np.all(amax <= 6 * scale) and np.all(amax > 3 * scale)
    # E2M1 spacing: 0.5 below 2, 1 in [2, 4), 2 in [4, 6]
    y = np.abs(x) / scale
    half = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0))
    assert np.all(np.abs(deq - x) <= half * scale * (1 + 1e-6))


def test_integer_e2m1_values():
    from oracle import numerics as on
    p = wl.integer_e2m1_packed((3, 64), 1)
    vals = on.decode_e2m1(on.unpack_e2m1(p.numpy()))
    assert set(np.unique(vals).tolist()) <= {-2.0, -1.0, 0.0, 1.0, 2.0}
