"""Masked form on the GPU against the oracle."""
import numpy as np
import pytest
import torch

from moe_grouped_gemm_side_gb300 import binding as mb
from moe_grouped_gemm_side_gb300 import workloads as wl
from oracle import gemm as og
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


def run_masked(valid_m, M_max, N, K, dtype, seed=1, integer=False, dev="cuda"):
    E = len(valid_m)
    if dtype == "bf16":
        if integer:
            A = wl.integer_bf16((E, M_max, K), seed, dev)
            B = wl.integer_bf16((E, N, K), seed + 1, dev)
        else:
            ops = wl.make_masked(E, M_max, N, K, "bf16", seed, dev)
            A, B = ops.A, ops.B
        SFA = SFB = None
    else:
        if integer:
            A = gu.integer_e4m3((E, M_max, K), seed, dev)
            B = gu.integer_e4m3((E, N, K), seed + 1, dev)
            SFA = gu.rand_scales((E, K // 128, M_max), seed + 2, dev, 126, 128)
            SFB = gu.rand_scales((E, K // 128, N // 128), seed + 3, dev, 126, 128)
        else:
            ops = wl.make_masked(E, M_max, N, K, "fp8", seed, dev)
            A, B, SFA, SFB = ops.A, ops.B, ops.SFA, ops.SFB
    # poison invalid rows (and their scales) of every expert
    valid = np.zeros((E, M_max), dtype=bool)
    for e, v in enumerate(valid_m):
        valid[e, :max(0, min(v, M_max))] = True
    gu.poison_rows_(A.view(E * M_max, K), valid.reshape(-1), dtype == "fp8", None)
    if SFA is not None:
        for e in range(E):
            inv = torch.from_numpy(np.nonzero(~valid[e])[0]).to(dev)
            if inv.numel():
                SFA[e].index_fill_(1, inv, wl.UE8M0_NAN_CODE)
    gu.poison_experts_(B, [not 0 < v <= M_max for v in valid_m], dtype == "fp8", SFB)
    if dtype == "bf16":
        Ad = gu.deq_bf16(A).reshape(E, M_max, K)
        Bd = gu.deq_bf16(B).reshape(E, N, K)
    else:
        Ad = np.stack([gu.deq_rows_fp8(A[e], SFA[e]) for e in range(E)])
        Bd = np.stack([gu.deq_weight_fp8(B[e], SFB[e]) for e in range(E)])
    D = gu.sentinel_like((E, M_max, N), dev)
    d_valid = torch.tensor(valid_m, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mb.mgemm_masked(A, B, D, d_valid, SFA=SFA, SFB=SFB, status=status)
    torch.cuda.synchronize()
    ok_valid = [v if 0 <= v <= M_max else 0 for v in valid_m]
    R, written = og.masked(Ad, Bd, ok_valid)
    return gu.bf16_bits(D).reshape(E, M_max, N), written, R, int(status.item())


def test_bf16_integer_exact(lib, cuda):
    v = [0, 1, 6, 20, 38, 31, 2, 13]
    Dbits, written, R, status = run_masked(v, 64, 256, 256, "bf16", integer=True)
    assert status == 0
    assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
    assert (Dbits[~written] == gu.SENTINEL_BITS).all()


def test_fp8_integer_exact(lib, cuda):
    v = [0, 1, 17, 64, 3, 250, 0, 128]
    Dbits, written, R, status = run_masked(v, 256, 256, 384, "fp8", integer=True)
    assert status == 0
    assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
    assert (Dbits[~written] == gu.SENTINEL_BITS).all()


@pytest.mark.parametrize("M_max", [16, 48, 256, 300])
def test_bf16_random(lib, cuda, M_max):
    rng = np.random.default_rng(M_max)
    v = [int(x) for x in rng.integers(0, M_max + 1, size=6)]
    v[1] = 0
    v[2] = M_max
    Dbits, written, R, status = run_masked(v, M_max, 256, 512, "bf16", seed=M_max)
    assert status == 0
    for e in range(len(v)):
        if v[e]:
            gu.check_rows_bf16(Dbits[e, :v[e]], R[e, :v[e]])
    assert (Dbits[~written] == gu.SENTINEL_BITS).all()


def test_fp8_random(lib, cuda):
    v = [0, 1, 6, 20, 38, 31, 2, 13, 200, 27]
    Dbits, written, R, status = run_masked(v, 256, 256, 768, "fp8", seed=3)
    assert status == 0
    for e in range(len(v)):
        if v[e]:
            gu.check_frobenius(Dbits[e, :v[e]], R[e, :v[e]])
    assert (Dbits[~written] == gu.SENTINEL_BITS).all()


def test_invalid_valid_m(lib, cuda):
    v = [3, 99, -2, 5]
    Dbits, written, R, status = run_masked(v, 32, 128, 128, "bf16", seed=9)
    assert status == 6
    for e in (0, 3):
        gu.check_rows_bf16(Dbits[e, :v[e]], R[e, :v[e]])
    assert (Dbits[1] == gu.SENTINEL_BITS).all() and (Dbits[2] == gu.SENTINEL_BITS).all()


def test_max_experts(lib, cuda):
    """E = 1024 masked buffers of 16 rows, most of them empty."""
    rng = np.random.default_rng(7)
    v = [int(x) if x < 17 else 0 for x in rng.integers(0, 40, size=1024)]
    Dbits, written, R, status = run_masked(v, 16, 256, 256, "fp8", seed=5, integer=True)
    assert status == 0
    assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
    assert (Dbits[~written] == gu.SENTINEL_BITS).all()
