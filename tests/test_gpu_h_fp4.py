"""FP8 x FP4 grouped GEMM ("flops/deepgemm-grouped-masked-moe-gemm",
"Workarounds": FP8xFP4 linear layers): E4M3 activations with one UE8M0 scale
per (row, 128 K), E2M1 weights packed two per byte with one UE8M0 scale per
(row, 32 K), against the oracle's fp64 product of the decoded operands.

Integer-valued operands with power-of-two scales keep every fp32 partial sum
exact, so those outputs must be the bf16 rounding of the exact product, bit
for bit; float operands use the fp8 per-expert Frobenius rule.  Rows the form
does not compute keep the sentinel."""
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
from tests import test_gpu_g_swiglu as sw

pytestmark = pytest.mark.gpu


def fp4_weights(E, N, K, seed, dev, integer=True):
    if integer:
        B = wl.integer_e2m1_packed((E, N, K), seed, dev)
        SFB = gu.rand_scales((E, N, K // 32), seed + 1, dev, 126, 128)
    else:
        B, SFB = wl.make_weights(E, N, K, "fp8xfp4", seed, dev, 0.05)
    Bd = np.stack([on.dequant_weight_mx4(B[e].cpu().numpy(), SFB[e].cpu().numpy()) for e in range(E)])
    return B, SFB, Bd


def contiguous_case(counts, N, K, align_q, tile_q=0, seed=5, integer=True, dev="cuda"):
    E = len(counts)
    p = op.plan(counts, align_q)
    rows_cap = (p.P + 40 + 15) // 16 * 16
    written = np.zeros(rows_cap, dtype=bool)
    for e, t in enumerate(counts):
        written[p.offsets[e]:p.offsets[e] + t] = True
    if integer:
        A = gu.integer_e4m3((rows_cap, K), seed, dev)
        SFA = gu.rand_scales((K // 128, rows_cap), seed + 2, dev, 126, 128)
    else:
        A, SFA = wl.make_rows(rows_cap, K, "fp8", seed, dev)
    B, SFB, Bd = fp4_weights(E, N, K, seed + 10, dev, integer)
    gu.poison_rows_(A, written, True, SFA)
    R, wmask = og.contiguous(gu.deq_rows_fp8(A, SFA), Bd, counts, align_q)
    assert np.array_equal(wmask, written)
    return A, SFA, B, SFB, R, written, rows_cap


@pytest.mark.parametrize("tile_q,K", [(0, 1024), (16, 1024), (64, 1024), (128, 1024), (240, 1024), (0, 1536),
                                      (64, 512)])
def test_contiguous_integer_exact(lib, cuda, tile_q, K):
    counts = [37, 0, 300, 1, 16, 129]
    N = 768
    A, SFA, B, SFB, R, written, rows_cap = contiguous_case(counts, N, K, 16, tile_q)
    D = gu.sentinel_like((rows_cap, N), cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    d_counts = torch.tensor(counts, dtype=torch.int32, device=cuda)
    mb.mgemm_contiguous(A, B, D, d_counts, 16, SFA=SFA, SFB=SFB, tile_q=tile_q, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Dbits = gu.bf16_bits(D)
    assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
    assert (Dbits[~written] == gu.SENTINEL_BITS).all()


@pytest.mark.parametrize("policy", ["single", "dual", "pair", "pair_dual", "tokm"])
def test_every_policy_runs_single_sm_families(lib, cuda, policy):
    """FP4 weights use the single-SM families; the pair policies fall back."""
    counts = [3, 250, 0, 64]
    A, SFA, B, SFB, R, written, rows_cap = contiguous_case(counts, 512, 512, 32, seed=9)
    D = gu.sentinel_like((rows_cap, 512), cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    try:
        mb.set_kernel_policy(mb.POLICIES[policy])
        mb.mgemm_contiguous(A, B, D, torch.tensor(counts, dtype=torch.int32, device=cuda), 32,
                            SFA=SFA, SFB=SFB, status=status)
        torch.cuda.synchronize()
    finally:
        mb.set_kernel_policy(mb.POLICY_AUTO)
    assert int(status.item()) == 0
    Dbits = gu.bf16_bits(D)
    assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
    assert (Dbits[~written] == gu.SENTINEL_BITS).all()


def test_distinct_scales_per_32_columns(lib, cuda):
    """Every (row, 32 K) weight scale different and every code 1: a scale
    applied to the wrong 32-column group or row changes the result."""
    E, N, K, t = 1, 256, 512, 48
    dev = cuda
    A = gu.integer_e4m3((t, K), 3, dev)
    SFA = torch.full((K // 128, t), 127, dtype=torch.uint8, device=dev)
    B = torch.full((E, N, K // 2), 0x22, dtype=torch.uint8, device=dev)           # all codes = 1.0
    g = torch.Generator().manual_seed(4)
    SFB = torch.randint(120, 135, (E, N, K // 32), generator=g, dtype=torch.int32).to(torch.uint8).to(dev)
    Bd = np.stack([on.dequant_weight_mx4(B[0].cpu().numpy(), SFB[0].cpu().numpy())])
    R, written = og.contiguous(gu.deq_rows_fp8(A, SFA), Bd, [t], 16)
    D = gu.sentinel_like((t, N), dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mb.mgemm_contiguous(A, B, D, torch.tensor([t], dtype=torch.int32, device=dev), 16, SFA=SFA, SFB=SFB,
                        status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(gu.bf16_bits(D), gu.round_bf16_bits(R))


@pytest.mark.parametrize("seed", range(3))
def test_contiguous_float_operands(lib, cuda, seed):
    rng = np.random.default_rng(40 + seed)
    counts = wl.counts_random(seed, int(rng.integers(2, 9)), 400)
    A, SFA, B, SFB, R, written, rows_cap = contiguous_case(counts, 1024, 1536, 32, integer=False, seed=seed)
    D = gu.sentinel_like((rows_cap, 1024), cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    mb.mgemm_contiguous(A, B, D, torch.tensor(counts, dtype=torch.int32, device=cuda), 32, SFA=SFA, SFB=SFB,
                        status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Dbits = gu.bf16_bits(D)
    p = op.plan(counts, 32)
    for e, t in enumerate(counts):
        if t:
            rows = slice(p.offsets[e], p.offsets[e] + t)
            gu.check_frobenius(Dbits[rows], R[rows])
    assert (Dbits[~written] == gu.SENTINEL_BITS).all()


@pytest.mark.parametrize("K", [1024, 512, 2560])
def test_masked_integer_exact(lib, cuda, K):
    """(E2M1 weights need K % 512 == 0: whole 16-byte weight-scale rows.)
    K = 512 runs one group of four K-blocks per tile, so the weight-scale
    group ring turns over at every tile."""
    E, M, N = 6, 96, 512
    valid = [96, 0, 17, 1, 64, 50]
    A = gu.integer_e4m3((E, M, K), 21, cuda)
    SFA = gu.rand_scales((E, K // 128, M), 22, cuda, 126, 128)
    B, SFB, Bd = fp4_weights(E, N, K, 23, cuda)
    Ad = np.stack([gu.deq_rows_fp8(A[e], SFA[e]) for e in range(E)])
    R, written = og.masked(Ad, Bd, valid)
    D = gu.sentinel_like((E, M, N), cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    mb.mgemm_masked(A, B, D, torch.tensor(valid, dtype=torch.int32, device=cuda), SFA=SFA, SFB=SFB,
                    status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Dbits = gu.bf16_bits(D).reshape(E, M, N)
    assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
    assert (Dbits[~written] == gu.SENTINEL_BITS).all()


@pytest.mark.parametrize("out", ["bf16", "fp8"])
def test_swiglu_with_fp4_weights(lib, cuda, out):
    counts = [100, 0, 33, 260]
    N, K = 512, 512
    A, SFA, B, SFB, R, written, rows_cap = contiguous_case(counts, N, K, 16, seed=13)
    g, u = oe.gate_up_halves(R[written])
    y = oe.swiglu(g, u)
    Y, SFY = sw.out_buffers(rows_cap, N // 2, out, cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    mb.mgemm_contiguous_swiglu(A, B, Y, torch.tensor(counts, dtype=torch.int32, device=cuda), 16, SFA=SFA,
                               SFB=SFB, SFY=SFY, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sw.assert_contiguous(Y, SFY, written, y, g, u, out)
