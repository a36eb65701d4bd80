"""M-grouped contiguous form on the GPU against the oracle."""
import numpy as np
import pytest
import torch

from moe_grouped_gemm_side_gb300 import binding as mb
from moe_grouped_gemm_side_gb300 import workloads as wl
from oracle import gemm as og
from oracle import plan as op
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["auto", "single", "dual", "pair", "pair_dual", "tokm"])
def kernel_policy(request, lib):
    """Run every case on every kernel family: one or two weight blocks per
    tile, on one SM or on a CTA pair sharing each MMA, tokens on the MMA's
    N or M axis.  A family whose tile does not divide N falls back to a
    narrower one."""
    mb.set_kernel_policy(mb.POLICIES[request.param])
    yield request.param
    mb.set_kernel_policy(mb.POLICY_AUTO)


def run_contiguous(counts, N, K, dtype, align_q, tile_q=0, seed=1, integer=False, rows_extra=37,
                   a_std=1.0, b_std=1.0, dev="cuda"):
    """Builds operands with poisoned padding, runs the GPU, returns
    (D bits [rows_cap, N], written mask, reference R, status)."""
    E = len(counts)
    p = op.plan(counts, align_q)
    rows_cap = p.P + rows_extra
    if dtype == "fp8":
        rows_cap = (rows_cap + 15) // 16 * 16
    written = np.zeros(rows_cap, dtype=bool)
    for e, t in enumerate(counts):
        written[p.offsets[e]:p.offsets[e] + t] = True
    if dtype == "bf16":
        if integer:
            A = wl.integer_bf16((rows_cap, K), seed, dev)
            B = wl.integer_bf16((E, N, K), seed + 1, dev)
        else:
            A = wl.normal_bf16((rows_cap, K), seed, dev, a_std)
            B = wl.normal_bf16((E, N, K), seed + 1, dev, b_std)
        SFA = SFB = None
    else:
        if integer:
            A = gu.integer_e4m3((rows_cap, K), seed, dev)
            B = gu.integer_e4m3((E, N, K), seed + 1, dev)
            SFA = gu.rand_scales((K // 128, rows_cap), seed + 2, dev, 126, 128)
            SFB = gu.rand_scales((E, K // 128, N // 128), seed + 3, dev, 126, 128)
        else:
            ops = wl.make_contiguous(E, rows_cap, N, K, "fp8", seed, dev, a_std, b_std)
            A, B, SFA, SFB = ops.A, ops.B, ops.SFA, ops.SFB
    gu.poison_rows_(A, written, dtype == "fp8", SFA)
    gu.poison_experts_(B, [t <= 0 for t in counts], dtype == "fp8", SFB)
    # oracle on the same bytes
    if dtype == "bf16":
        Ad = gu.deq_bf16(A)
        Bd = gu.deq_bf16(B).reshape(E, N, K)
    else:
        Ad = gu.deq_rows_fp8(A, SFA)
        Bd = np.stack([gu.deq_weight_fp8(B[e], SFB[e]) for e in range(E)])
    R, wmask = og.contiguous(Ad, Bd, counts, align_q)
    assert np.array_equal(wmask, written)
    D = gu.sentinel_like((rows_cap, N), dev)
    d_counts = torch.tensor(counts, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mb.mgemm_contiguous(A, B, D, d_counts, align_q, SFA=SFA, SFB=SFB, tile_q=tile_q, status=status)
    torch.cuda.synchronize()
    return gu.bf16_bits(D), written, R, int(status.item())


def assert_sentinels(Dbits, written):
    assert (Dbits[~written] == gu.SENTINEL_BITS).all(), "a row outside the valid segments was written"


@pytest.mark.parametrize("tile_q", [16, 32, 64, 128, 256, 0])
def test_bf16_integer_exact(lib, cuda, tile_q):
    """Small integers: every fp32 partial sum is exact, so the output is the
    bf16 rounding of the exact product, bit for bit."""
    counts = wl.counts_uniformish()
    Dbits, written, R, status = run_contiguous(counts, 256, 256, "bf16", 32, tile_q, integer=True)
    assert status == 0
    assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
    assert_sentinels(Dbits, written)


def test_bf16_uniformish_normal(lib, cuda):
    for tile_q in (0, 16, 32):
        Dbits, written, R, status = run_contiguous(wl.counts_uniformish(), 256, 256, "bf16", 16, tile_q)
        assert status == 0
        gu.check_rows_bf16(Dbits[written], R[written])
        assert_sentinels(Dbits, written)


@pytest.mark.parametrize("seed", range(6))
def test_bf16_random_histograms(lib, cuda, seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 12))
    counts = wl.counts_random(seed, E, int(rng.choice([5, 40, 300, 700])))
    N = int(rng.choice([128, 256, 384]))
    K = int(rng.choice([128, 256, 640]))
    align = int(rng.choice([1, 8, 16, 128]))
    tile_q = int(rng.choice([0, 16, 48, 128, 256]))
    Dbits, written, R, status = run_contiguous(counts, N, K, "bf16", align, tile_q, seed=seed)
    assert status == 0
    if written.any():
        gu.check_rows_bf16(Dbits[written], R[written])
    assert_sentinels(Dbits, written)


def test_bf16_all_experts_empty(lib, cuda):
    Dbits, written, R, status = run_contiguous([0, 0, 0], 128, 128, "bf16", 16)
    assert status == 0 and not written.any()
    assert_sentinels(Dbits, written)


def test_bf16_single_row_and_big_expert(lib, cuda):
    Dbits, written, R, status = run_contiguous([1, 0, 1000, 3], 256, 512, "bf16", 64)
    assert status == 0
    gu.check_rows_bf16(Dbits[written], R[written])
    assert_sentinels(Dbits, written)


@pytest.mark.parametrize("tile_q", [16, 64, 128, 240, 256, 0])
def test_fp8_integer_exact(lib, cuda, tile_q):
    """E4M3 integers with distinct power-of-two scales per (row, K block) and
    per weight block: exact in fp32, so bit-exact after bf16 rounding.  Pins
    the scale layout of both operands."""
    counts = [37, 0, 130, 5, 64]
    Dbits, written, R, status = run_contiguous(counts, 256, 384, "fp8", 16, tile_q, integer=True)
    assert status == 0
    assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
    assert_sentinels(Dbits, written)


@pytest.mark.parametrize("seed", range(4))
def test_fp8_random(lib, cuda, seed):
    rng = np.random.default_rng(100 + seed)
    E = int(rng.integers(1, 10))
    counts = wl.counts_random(100 + seed, E, int(rng.choice([20, 200, 600])))
    N = int(rng.choice([128, 256]))
    K = int(rng.choice([256, 512, 896]))
    Dbits, written, R, status = run_contiguous(counts, N, K, "fp8", 32, 0, seed=seed)
    assert status == 0
    p = op.plan(counts, 32)
    for e, t in enumerate(counts):
        if t:
            o = p.offsets[e]
            gu.check_frobenius(Dbits[o:o + t], R[o:o + t])
    assert_sentinels(Dbits, written)


def test_device_errors(lib, cuda):
    # capacity: rows_cap smaller than the aligned segments
    dev = cuda
    counts = [40, 40]
    A = wl.normal_bf16((64, 128), 1, dev)
    B = wl.normal_bf16((2, 128, 128), 2, dev)
    D = gu.sentinel_like((64, 128), dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mb.mgemm_contiguous(A, B, D, torch.tensor(counts, dtype=torch.int32, device=dev), 32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 4
    # expert 0 fits and is computed; expert 1 does not and writes nothing
    R = (gu.deq_bf16(A)[:40] @ gu.deq_bf16(B).reshape(2, 128, 128)[0].T)
    gu.check_rows_bf16(gu.bf16_bits(D)[:40], R)
    assert (gu.bf16_bits(D)[40:] == gu.SENTINEL_BITS).all()
    # negative count
    D = gu.sentinel_like((64, 128), dev)
    st.zero_()
    mb.mgemm_contiguous(A, B, D, torch.tensor([-1, 10], dtype=torch.int32, device=dev), 16, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 6
    R = gu.deq_bf16(A)[:10] @ gu.deq_bf16(B).reshape(2, 128, 128)[1].T
    gu.check_rows_bf16(gu.bf16_bits(D)[:10], R)
    assert (gu.bf16_bits(D)[10:] == gu.SENTINEL_BITS).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_max_experts(lib, cuda, dtype):
    """E = 1024 (the largest the library takes): the per-CTA schedule in
    shared memory is at its largest, and most experts are tiny or empty."""
    rng = np.random.default_rng(1024)
    counts = [int(c) for c in rng.integers(0, 6, size=1024)]
    counts[5] = 300
    Dbits, written, R, status = run_contiguous(counts, 256, 256, dtype, 16, seed=17, integer=True)
    assert status == 0
    assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
    assert_sentinels(Dbits, written)
