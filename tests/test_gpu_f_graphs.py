"""Decode under CUDA graphs ("flops/deepgemm-grouped-masked-moe-gemm",
"Workarounds": the masked form exists so decode can run from a captured
graph).  The plan and the masked GEMM are captured once; each replay reads
the token counts from device memory, so new histograms need no re-capture
and no host round trip: experts with no tokens produce no tiles on the
device, where an early-exit kernel variant or a conditional graph node
would otherwise be needed."""
import ctypes

import numpy as np
import pytest
import torch

from moe_grouped_gemm_side_gb300 import binding as mb
from oracle import gemm as og
from oracle import plan as op
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_plan_and_masked_gemm_replay_with_new_histograms(lib, cuda, dtype):
    E, M, N, K, q = 12, 64, 256, 384, 16
    dev = cuda
    fp8 = dtype == "fp8"
    if fp8:
        A = gu.integer_e4m3((E, M, K), 21, dev)
        B = gu.integer_e4m3((E, N, K), 22, dev)
        SFA = gu.rand_scales((E, K // 128, M), 23, dev, 126, 128)
        SFB = gu.rand_scales((E, K // 128, N // 128), 24, dev, 126, 128)
        Ad = np.stack([gu.deq_rows_fp8(A[e], SFA[e]) for e in range(E)])
        Bd = np.stack([gu.deq_weight_fp8(B[e], SFB[e]) for e in range(E)])
    else:
        from moe_grouped_gemm_side_gb300 import workloads as wl
        A = wl.integer_bf16((E, M, K), 21, dev)
        B = wl.integer_bf16((E, N, K), 22, dev)
        SFA = SFB = None
        Ad = gu.deq_bf16(A).reshape(E, M, K)
        Bd = gu.deq_bf16(B).reshape(E, N, K)
    D = gu.sentinel_like((E, M, N), dev)
    d_valid = torch.zeros(E, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    offsets = torch.zeros(E + 1, dtype=torch.int64, device=dev)
    stats = torch.zeros(48, dtype=torch.uint8, device=dev)
    dt = mb.MG_FP8_E4M3_UE8M0 if fp8 else mb.MG_BF16
    s = torch.cuda.Stream()

    def step(stream):
        sp = ctypes.c_void_p(stream.cuda_stream)
        assert lib.moe_plan(_p(d_valid), E, q, _p(offsets), None, 0, _p(stats), _p(status), sp) == 0
        assert lib.mgemm_masked(dt, _p(A), None if SFA is None else _p(SFA), _p(B),
                                None if SFB is None else _p(SFB), _p(D), _p(d_valid), E, M, N, K,
                                _p(status), sp) == 0

    with torch.cuda.stream(s):      # one eager call first (kernel attributes are set once)
        step(s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)

    rng = np.random.default_rng(5)
    histograms = [[int(v) for v in rng.integers(0, M + 1, size=E)] for _ in range(3)]
    histograms[1][::2] = [0] * len(histograms[1][::2])     # half the experts idle
    histograms.append([0] * E)                              # nothing to do
    for valid in histograms:
        with torch.cuda.stream(s):
            d_valid.copy_(torch.tensor(valid, dtype=torch.int32), non_blocking=False)
            D.view(torch.int16).fill_(gu.SENTINEL_BITS)
            status.zero_()
        s.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        R, written = og.masked(Ad, Bd, valid)
        Dbits = gu.bf16_bits(D).reshape(E, M, N)
        assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
        assert (Dbits[~written] == gu.SENTINEL_BITS).all()
        ref = op.plan(valid, q)
        got = mb.decode_stats(stats)
        assert (got["P"], got["U"], got["sumsq"], got["active"]) == (ref.P, ref.U, ref.sumsq, ref.active)
        assert np.array_equal(offsets.cpu().numpy(), np.asarray(ref.offsets, dtype=np.int64))
