"""GEMM1 with the expert's SwiGLU fused into its epilogue, stored as bf16 or
re-quantised to E4M3 with UE8M0 per-128 scales ("flops/deepgemm-grouped-
masked-moe-gemm", "Workarounds": SwiGLU between the two grouped GEMMs, FP8
activations for the second), against the oracle: the fp64 grouped GEMM, then
oracle/epilogue.py's SwiGLU and block quantiser.

Acceptance.  With integer operands every fp32 partial sum is exact, so the
kernel's g and u equal the oracle's; the only differences left are the fp32
SiLU and, where that moves a value across a rounding midpoint, the rounding.
The fp32 SiLU with the fast exponential and division has relative error
below (8 + 1.2|g|) 2^-23, and it is zero where the true SiLU is below
|g| 2^-126 (e^-|g| under the fp32 normal range is flushed).  So with
r = |y| (8 + 1.2|g|) 2^-23 + |g u| 2^-126 each output must lie between the
oracle's roundings of y - r and y + r: bit-exact except within r of a
midpoint.  Scale bytes likewise lie between the bytes of the block maxima
of |y| - r and |y| + r.
Float operands: bf16 rows by the per-row 1e-2 max-abs rule, E4M3 blocks
within the format's half-spacing plus the fp32 accumulation error.
"""
import numpy as np
import pytest
import torch

from moe_grouped_gemm_side_gb300 import binding as mb
from moe_grouped_gemm_side_gb300 import workloads as wl
from oracle import epilogue as oe
from oracle import gemm as og
from oracle import numerics as on
from oracle import plan as op
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

Q_SENTINEL = 0x01          # an E4M3 code; unwritten rows must keep it
SF_SENTINEL = 0xEE


def slack(y, g, u):
    """Absolute bound on |y_kernel - y| for exact g and u (see above)."""
    return np.abs(y) * (8.0 + 1.2 * np.abs(g)) * 2.0 ** -23 + np.abs(g * u) * 2.0 ** -126


def operands(shape_a, E, N, K, dtype, integer, seed, dev):
    if dtype == "bf16":
        if integer:
            A = wl.integer_bf16(shape_a, seed, dev)
            B = wl.integer_bf16((E, N, K), seed + 1, dev)
        else:
            A = wl.normal_bf16(shape_a, seed, dev)
            B = wl.normal_bf16((E, N, K), seed + 1, dev, 0.05)
        return A, B, None, None
    if integer:
        A = gu.integer_e4m3(shape_a, seed, dev)
        B = gu.integer_e4m3((E, N, K), seed + 1, dev)
        sfa_shape = (K // 128, shape_a[0]) if len(shape_a) == 2 else (shape_a[0], K // 128, shape_a[1])
        SFA = gu.rand_scales(sfa_shape, seed + 2, dev, 126, 128)
        SFB = gu.rand_scales((E, K // 128, N // 128), seed + 3, dev, 126, 128)
        return A, B, SFA, SFB
    if len(shape_a) == 2:
        ops = wl.make_contiguous(E, shape_a[0], N, K, "fp8", seed, dev, 1.0, 0.05)
    else:
        ops = wl.make_masked(E, shape_a[1], N, K, "fp8", seed, dev, 1.0, 0.05)
    return ops.A, ops.B, ops.SFA, ops.SFB


def dequant(A, B, SFA, SFB, E, N, K, dtype):
    if dtype == "bf16":
        return gu.deq_bf16(A), gu.deq_bf16(B).reshape(E, N, K)
    if A.dim() == 2:
        Ad = gu.deq_rows_fp8(A, SFA)
    else:
        Ad = np.stack([gu.deq_rows_fp8(A[e], SFA[e]) for e in range(A.shape[0])])
    Bd = np.stack([gu.deq_weight_fp8(B[e], SFB[e]) for e in range(E)])
    return Ad, Bd


def out_buffers(rows, I, out, dev, lead=None):
    shape = (rows, I) if lead is None else (lead, rows, I)
    if out == "bf16":
        return gu.sentinel_like(shape, dev), None
    Y = torch.full(shape, Q_SENTINEL, dtype=torch.uint8, device=dev)
    sf_shape = (I // 128, rows) if lead is None else (lead, I // 128, rows)
    return Y, torch.full(sf_shape, SF_SENTINEL, dtype=torch.uint8, device=dev)


def check_bf16_exactish(Ybits, y, g, u):
    """Ybits uint16 [n, I] against y [n, I] (fp64); g, u the gate and up values."""
    r = slack(y, g, u)
    lo = on.decode_bf16(gu.round_bf16_bits(y - r))
    hi = on.decode_bf16(gu.round_bf16_bits(y + r))
    got = on.decode_bf16(Ybits)
    ok = (got >= np.minimum(lo, hi)) & (got <= np.maximum(lo, hi))
    assert ok.all(), f"{(~ok).sum()} of {ok.size} bf16 outputs off; first {np.argwhere(~ok)[:3]}"


def check_fp8_exactish(codes, sf_rows, y, g, u):
    """codes uint8 [n, I], sf_rows uint8 [n, I/128] against y, g, u [n, I]."""
    n, I = y.shape
    nb = I // 128
    r = slack(y, g, u)
    a = np.abs(y)
    amax_lo = np.maximum(a - r, 0.0).reshape(n, nb, 128).max(axis=2)
    amax_hi = (a + r).reshape(n, nb, 128).max(axis=2)
    s_lo = oe.ue8m0_for_amax(amax_lo).astype(int)
    s_hi = oe.ue8m0_for_amax(amax_hi).astype(int)
    s = sf_rows.astype(int)
    ok = (s >= s_lo) & (s <= s_hi)
    assert ok.all(), f"{(~ok).sum()} scale bytes off; first {np.argwhere(~ok)[:3]}"
    scale = np.repeat(np.exp2(s - 127.0), 128, axis=1)
    lo = on.decode_e4m3(oe.encode_e4m3((y - r) / scale))
    hi = on.decode_e4m3(oe.encode_e4m3((y + r) / scale))
    got = on.decode_e4m3(codes)
    ok = (got >= np.minimum(lo, hi)) & (got <= np.maximum(lo, hi))
    assert ok.all(), f"{(~ok).sum()} of {ok.size} E4M3 codes off; first {np.argwhere(~ok)[:3]}"


def check_fp8_float(codes, sf_rows, y):
    """Float operands: each element within half an E4M3 spacing (relative
    2^-4, absolute 2^-10 scale in the subnormal range) plus 1e-5 max|y| of
    its block for the fp32 accumulation."""
    n, I = y.shape
    scale = np.repeat(np.exp2(sf_rows.astype(np.float64) - 127.0), 128, axis=1)
    deq = on.decode_e4m3(codes) * scale
    amax = np.repeat(np.abs(y.reshape(n, I // 128, 128)).max(axis=2), 128, axis=1)
    bound = np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10 * scale) + 1e-5 * amax
    ok = np.abs(deq - y) <= bound
    assert ok.all(), f"{(~ok).sum()} of {ok.size} values off"


def run_contiguous_swiglu(counts, N, K, dtype, out, align_q, tile_q=0, integer=True, seed=11,
                          dev="cuda", rows_extra=32, zero_gate_block=None):
    E = len(counts)
    I = N // 2
    p = op.plan(counts, align_q)
    rows_cap = (p.P + rows_extra + 15) // 16 * 16
    written = np.zeros(rows_cap, dtype=bool)
    for e, t in enumerate(counts):
        written[p.offsets[e]:p.offsets[e] + t] = True
    A, B, SFA, SFB = operands((rows_cap, K), E, N, K, dtype, integer, seed, dev)
    if zero_gate_block is not None:
        e, j = zero_gate_block
        B[e, 256 * j:256 * j + 128].zero_()
    gu.poison_rows_(A, written, dtype == "fp8", SFA)
    Ad, Bd = dequant(A, B, SFA, SFB, E, N, K, dtype)
    H, wmask = og.contiguous(Ad, Bd, counts, align_q)
    assert np.array_equal(wmask, written)
    g, u = oe.gate_up_halves(H[written])
    y = oe.swiglu(g, u)
    Y, SFY = out_buffers(rows_cap, I, out, dev)
    d_counts = torch.tensor(counts, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mb.mgemm_contiguous_swiglu(A, B, Y, d_counts, align_q, SFA=SFA, SFB=SFB, SFY=SFY, tile_q=tile_q,
                               status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return Y, SFY, written, y, g, u


def assert_contiguous(Y, SFY, written, y, g, u, out, exact=True):
    if out == "bf16":
        Ybits = gu.bf16_bits(Y)
        assert (Ybits[~written] == gu.SENTINEL_BITS).all(), "a row outside the segments was written"
        if exact:
            check_bf16_exactish(Ybits[written], y, g, u)
        elif written.any():
            gu.check_rows_bf16(Ybits[written], y)
    else:
        codes = Y.cpu().numpy()
        sf = SFY.cpu().numpy()
        assert (codes[~written] == Q_SENTINEL).all(), "a row outside the segments was written"
        assert (sf[:, ~written] == SF_SENTINEL).all(), "a scale outside the segments was written"
        if exact:
            check_fp8_exactish(codes[written], sf[:, written].T, y, g, u)
        else:
            check_fp8_float(codes[written], sf[:, written].T, y)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("out", ["bf16", "fp8"])
@pytest.mark.parametrize("tile_q", [0, 16, 64, 240])
@pytest.mark.parametrize("N", [768, 1024])
def test_contiguous_integer(lib, cuda, dtype, out, tile_q, N):
    """N = 768 runs one SM per tile, N = 1024 CTA pairs."""
    counts = [37, 0, 300, 1, 16, 129]
    K = 256 if dtype == "bf16" else 512
    res = run_contiguous_swiglu(counts, N, K, dtype, out, 16, tile_q)
    assert_contiguous(*res, out)


@pytest.mark.parametrize("seed", range(4))
def test_contiguous_random_histograms(lib, cuda, seed):
    rng = np.random.default_rng(100 + seed)
    E = int(rng.integers(1, 10))
    counts = wl.counts_random(seed, E, int(rng.choice([20, 200, 600])))
    N = int(rng.choice([256, 512, 1024]))
    dtype = ["bf16", "fp8"][seed % 2]
    out = ["fp8", "bf16"][(seed // 2) % 2]
    res = run_contiguous_swiglu(counts, N, 384 if dtype == "bf16" else 256, dtype, out,
                                int(rng.choice([16, 32, 128])), int(rng.choice([0, 32, 128])), seed=seed)
    assert_contiguous(*res, out)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("out", ["bf16", "fp8"])
def test_contiguous_float_operands(lib, cuda, dtype, out):
    res = run_contiguous_swiglu([200, 0, 57, 513], 512, 1024, dtype, out, 32, integer=False)
    assert_contiguous(*res, out, exact=False)


def test_all_zero_block_gets_the_unit_scale(lib, cuda):
    """A block whose gate rows are zero gives y = 0 there: scale byte 127 and
    zero codes."""
    Y, SFY, written, y, g, u = run_contiguous_swiglu([40, 90], 512, 256, "bf16", "fp8", 16,
                                                     zero_gate_block=(1, 1))
    assert_contiguous(Y, SFY, written, y, g, u, "fp8")
    rows1 = np.nonzero(written)[0][40:]
    assert (SFY.cpu().numpy()[1, rows1] == 127).all()
    assert (Y.cpu().numpy()[rows1, 128:256] & 0x7F == 0).all()


def test_empty(lib, cuda):
    res = run_contiguous_swiglu([0, 0, 0], 256, 256, "fp8", "fp8", 16)
    assert_contiguous(*res, "fp8")
    res = run_contiguous_swiglu([0, 0], 1024, 512, "bf16", "bf16", 16)
    assert_contiguous(*res, "bf16")


@pytest.mark.parametrize("policy", ["auto", "single", "dual", "pair", "pair_dual", "tokm"])
@pytest.mark.parametrize("dtype,out", [("fp8", "fp8"), ("bf16", "bf16")])
def test_every_policy(lib, cuda, policy, dtype, out):
    """Every family choice runs a two-block kernel: CTA pairs (each SM one
    gate block and its up block) for auto and pair-dual with N % 512 == 0,
    one SM otherwise; N = 1024 and 768 cover both."""
    try:
        mb.set_kernel_policy(mb.POLICIES[policy])
        for N in (1024, 768):
            res = run_contiguous_swiglu([5, 70, 0, 300], N, 256 if dtype == "bf16" else 512, dtype, out, 16)
            assert_contiguous(*res, out)
    finally:
        mb.set_kernel_policy(mb.POLICY_AUTO)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("out", ["bf16", "fp8"])
def test_masked_integer(lib, cuda, dtype, out):
    E, M, N = 6, 96, 512
    K = 256 if dtype == "bf16" else 512
    I = N // 2
    valid = [96, 0, 17, 1, 64, 50]
    A, B, SFA, SFB = operands((E, M, K), E, N, K, dtype, True, 31, cuda)
    Ad, Bd = dequant(A, B, SFA, SFB, E, N, K, dtype)
    H, written = og.masked(Ad, Bd, valid)
    g, u = oe.gate_up_halves(H[written])
    y = oe.swiglu(g, u)
    Y, SFY = out_buffers(M, I, out, cuda, lead=E)
    d_valid = torch.tensor(valid, dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    mb.mgemm_masked_swiglu(A, B, Y, d_valid, SFA=SFA, SFB=SFB, SFY=SFY, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    if out == "bf16":
        Ybits = gu.bf16_bits(Y).reshape(E, M, I)
        assert (Ybits[~written] == gu.SENTINEL_BITS).all()
        check_bf16_exactish(Ybits[written], y, g, u)
    else:
        codes = Y.cpu().numpy()
        sf = SFY.cpu().numpy().transpose(0, 2, 1)          # [E, M, I/128]
        assert (codes[~written] == Q_SENTINEL).all()
        assert (sf[~written] == SF_SENTINEL).all()
        check_fp8_exactish(codes[written], sf[written], y, g, u)


def test_chain_feeds_the_second_gemm(lib, cuda):
    """E4M3 Y and its scales go straight into the second grouped GEMM as its
    activations (K = N/2): GEMM2 on the kernel's own Y bytes matches the
    oracle's GEMM2 on the same bytes, and Y matches the oracle's SwiGLU."""
    counts = [300, 0, 45, 129]
    E, N, K, H2, align = len(counts), 1024, 512, 384, 32
    Y, SFY, written, y, g, u = run_contiguous_swiglu(counts, N, K, "fp8", "fp8", align)
    assert_contiguous(Y, SFY, written, y, g, u, "fp8")
    I = N // 2
    W2 = gu.integer_e4m3((E, H2, I), 77, cuda)
    SFW2 = gu.rand_scales((E, I // 128, H2 // 128), 78, cuda, 126, 128)
    D = gu.sentinel_like((Y.shape[0], H2), cuda)
    d_counts = torch.tensor(counts, dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    # unwritten rows of Y / SFY still hold sentinels; the GEMM reads only segment rows
    mb.mgemm_contiguous(Y, W2, D, d_counts, align, SFA=SFY, SFB=SFW2, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Yd = gu.deq_rows_fp8(Y, SFY)
    W2d = np.stack([gu.deq_weight_fp8(W2[e], SFW2[e]) for e in range(E)])
    R2, w2 = og.contiguous(Yd, W2d, counts, align)
    assert np.array_equal(w2, written)
    Dbits = gu.bf16_bits(D)
    for e, t in enumerate(counts):
        if t:
            rows = slice(op.plan(counts, align).offsets[e], op.plan(counts, align).offsets[e] + t)
            gu.check_frobenius(Dbits[rows], R2[rows])
    assert (Dbits[~written] == gu.SENTINEL_BITS).all()
