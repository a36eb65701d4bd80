"""Exemplar selector on the GPU ("MoE GroupGEMM padding under expert skew",
"Adapt kernels without adding a CPU stall"): the device choice equals the
oracle's (integer features, so bit for bit), including the hysteresis state
carried across calls; the GEMMs that read the device tactic compute the same
products as the plain calls; and the choice plus the GEMM replay from one
captured CUDA graph as the histogram changes."""
import random

import numpy as np
import pytest
import torch

from moe_grouped_gemm_side_gb300 import binding as mb
from moe_grouped_gemm_side_gb300 import workloads as wl
from oracle import gemm as og
from oracle import plan as op
from oracle import selector as osel
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def random_table(rng, n):
    return [{"lu": rng.randrange(0, 320), "shares": sorted(rng.randrange(0, 65537) for _ in range(16)),
             "tile_q": 16 * rng.randrange(1, 16), "blocks": rng.choice([1, 2])} for _ in range(n)]


def test_device_choice_equals_oracle(lib, cuda):
    rng = random.Random(21)
    tactic = torch.zeros(3, dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    for trial in range(120):
        n = rng.choice([1, 2, 7, 64, 1024])
        entries = random_table(rng, n)
        d_table = mb.exemplar_table_device(mb.exemplar_table(entries), cuda)
        E = rng.choice([1, 2, 5, 16, 64, 100, 1024, 3000, 4096])
        kind = trial % 3
        if kind == 0:
            c = [rng.randrange(0, 300) for _ in range(E)]
        elif kind == 1:
            c = [0] * E
            for _ in range(rng.randrange(0, 4)):
                c[rng.randrange(E)] = rng.randrange(1, 100000)
        else:
            c = [rng.choice([0, 1, 2, 64, 1 << 20]) for _ in range(E)]
        d_counts = torch.tensor(c, dtype=torch.int32, device=cuda)
        mb.select_exemplar(d_counts, d_table, n, tactic, status=status)
        torch.cuda.synchronize()
        want = osel.choose(c, entries)
        got = tactic.cpu().tolist()
        assert got == [entries[want]["tile_q"], entries[want]["blocks"], want], (trial, got, want)
    assert int(status.item()) == 0


def test_hysteresis_state_across_calls(lib, cuda):
    rng = random.Random(4)
    entries = random_table(rng, 12)
    d_table = mb.exemplar_table_device(mb.exemplar_table(entries), cuda)
    tactic = torch.zeros(3, dtype=torch.int32, device=cuda)
    state = torch.full((1,), -1, dtype=torch.int32, device=cuda)
    base = [rng.randrange(0, 400) for _ in range(64)]
    prev = -1
    switches = 0
    for step in range(60):
        c = [max(0, x + rng.randrange(-40, 41)) for x in base]            # neighbouring histograms
        if step % 20 == 19:
            c = [x * 8 for x in c]                                         # a real change of scale
        margin = 20000
        mb.select_exemplar(torch.tensor(c, dtype=torch.int32, device=cuda), d_table, len(entries), tactic,
                           margin=margin, d_state=state)
        torch.cuda.synchronize()
        want = osel.choose(c, entries, prev, margin)
        assert tactic[2].item() == want and state.item() == want
        switches += want != prev
        prev = want


def test_invalid_exemplar_reports_and_writes_no_tactic(lib, cuda):
    entries = [{"lu": 0, "shares": [0] * 16, "tile_q": 24, "blocks": 1}]
    d_table = mb.exemplar_table_device(mb.exemplar_table(entries), cuda)
    tactic = torch.zeros(3, dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    mb.select_exemplar(torch.tensor([3, 4], dtype=torch.int32, device=cuda), d_table, 1, tactic, status=status)
    torch.cuda.synchronize()
    assert tactic.cpu().tolist() == [0, 0, 0] and int(status.item()) == 6


def contiguous_operands(counts, N, K, align_q, dtype, dev, seed=3):
    p = op.plan(counts, align_q)
    rows_cap = (p.P + 32 + 15) // 16 * 16
    written = np.zeros(rows_cap, dtype=bool)
    for e, t in enumerate(counts):
        written[p.offsets[e]:p.offsets[e] + t] = True
    E = len(counts)
    if dtype == "fp8":
        A = gu.integer_e4m3((rows_cap, K), seed, dev)
        B = gu.integer_e4m3((E, N, K), seed + 1, dev)
        SFA = gu.rand_scales((K // 128, rows_cap), seed + 2, dev, 126, 128)
        SFB = gu.rand_scales((E, K // 128, N // 128), seed + 3, dev, 126, 128)
        Ad = gu.deq_rows_fp8(A, SFA)
        Bd = np.stack([gu.deq_weight_fp8(B[e], SFB[e]) for e in range(E)])
    else:
        A = wl.integer_bf16((rows_cap, K), seed, dev)
        B = wl.integer_bf16((E, N, K), seed + 1, dev)
        SFA = SFB = None
        Ad, Bd = gu.deq_bf16(A), gu.deq_bf16(B).reshape(E, N, K)
    gu.poison_rows_(A, written, dtype == "fp8", SFA)
    R, wmask = og.contiguous(Ad, Bd, counts, align_q)
    return A, B, SFA, SFB, R, written, rows_cap


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("tq,blocks", [(16, 1), (64, 2), (128, 1), (240, 2), (256, 2), (48, 2)])
def test_contiguous_tactic_exact(lib, cuda, dtype, tq, blocks):
    counts = [37, 0, 300, 1, 16, 129]
    N, K = 512, 256 if dtype == "bf16" else 512
    A, B, SFA, SFB, R, written, rows_cap = contiguous_operands(counts, N, K, 16, dtype, cuda)
    D = gu.sentinel_like((rows_cap, N), cuda)
    tactic = torch.tensor([tq, blocks, 0], dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    mb.mgemm_contiguous_tactic(A, B, D, torch.tensor(counts, dtype=torch.int32, device=cuda), 16, tactic,
                               SFA=SFA, SFB=SFB, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Dbits = gu.bf16_bits(D)
    assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
    assert (Dbits[~written] == gu.SENTINEL_BITS).all()


def test_invalid_tactic_falls_back(lib, cuda):
    counts = [20, 70]
    A, B, SFA, SFB, R, written, rows_cap = contiguous_operands(counts, 256, 256, 16, "bf16", cuda)
    D = gu.sentinel_like((rows_cap, 256), cuda)
    tactic = torch.tensor([0, 0, 0], dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    mb.mgemm_contiguous_tactic(A, B, D, torch.tensor(counts, dtype=torch.int32, device=cuda), 16, tactic,
                               status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6
    Dbits = gu.bf16_bits(D)
    assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))


def test_masked_tactic_exact(lib, cuda):
    E, M, N, K = 5, 80, 512, 256
    valid = [80, 0, 17, 1, 64]
    A = wl.integer_bf16((E, M, K), 31, cuda)
    B = wl.integer_bf16((E, N, K), 32, cuda)
    R, written = og.masked(gu.deq_bf16(A).reshape(E, M, K), gu.deq_bf16(B).reshape(E, N, K), valid)
    for tq, blocks in ((16, 1), (32, 2), (80, 2)):
        D = gu.sentinel_like((E, M, N), cuda)
        tactic = torch.tensor([tq, blocks, 0], dtype=torch.int32, device=cuda)
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        mb.mgemm_masked_tactic(A, B, D, torch.tensor(valid, dtype=torch.int32, device=cuda), tactic, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        Dbits = gu.bf16_bits(D).reshape(E, M, N)
        assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
        assert (Dbits[~written] == gu.SENTINEL_BITS).all()


def test_select_and_gemm_in_one_graph(lib, cuda):
    """The choice and the GEMM that reads it, captured once; each replay sees
    a new histogram in device memory."""
    rng = random.Random(8)
    entries = [{"lu": 100, "shares": [4096 * k for k in range(1, 17)], "tile_q": 32, "blocks": 1},
               {"lu": 100, "shares": [65536] * 16, "tile_q": 128, "blocks": 2},
               {"lu": 200, "shares": [4096 * k for k in range(1, 17)], "tile_q": 240, "blocks": 2}]
    d_table = mb.exemplar_table_device(mb.exemplar_table(entries), cuda)
    E, N, K, align, cap = 8, 512, 256, 16, 3000
    A = wl.integer_bf16((cap, K), 41, cuda)
    B = wl.integer_bf16((E, N, K), 42, cuda)
    Ad, Bd = gu.deq_bf16(A), gu.deq_bf16(B).reshape(E, N, K)
    D = gu.sentinel_like((cap, N), cuda)
    d_counts = torch.zeros(E, dtype=torch.int32, device=cuda)
    tactic = torch.zeros(3, dtype=torch.int32, device=cuda)
    state = torch.full((1,), -1, dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    s = torch.cuda.Stream()

    def step():
        mb.select_exemplar(d_counts, d_table, len(entries), tactic, margin=0, d_state=state, status=status,
                           stream=s)
        mb.mgemm_contiguous_tactic(A, B, D, d_counts, align, tactic, status=status, stream=s)

    with torch.cuda.stream(s):
        step()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    histograms = [[30] * E, [2000, 0, 0, 0, 0, 0, 0, 0], [300] * E, [rng.randrange(0, 200) for _ in range(E)]]
    prev = int(state.item())
    for c in histograms:
        with torch.cuda.stream(s):
            d_counts.copy_(torch.tensor(c, dtype=torch.int32))
            D.view(torch.int16).fill_(gu.SENTINEL_BITS)
        s.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        want = osel.choose(c, entries, prev, 0)
        prev = want
        assert tactic.cpu().tolist() == [entries[want]["tile_q"], entries[want]["blocks"], want]
        R, written = og.contiguous(Ad, Bd, c, align)
        Dbits = gu.bf16_bits(D)
        assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
        assert (Dbits[~written] == gu.SENTINEL_BITS).all()


def test_masked_exemplar_in_gemm_matches_oracle_and_tactic_call(lib, cuda):
    """mgemm_masked_exemplar: every CTA makes the select kernel's choice
    (margin 0, no history) in its prologue; the choice equals the oracle's and
    the product equals the tactic call's with that choice, bit for bit."""
    rng = random.Random(33)
    M, N, K = 96, 512, 256
    for trial in range(24):
        E = rng.choice([1, 3, 16, 32])
        n = rng.choice([1, 5, 40, 1024])
        entries = random_table(rng, n)
        for x in entries:
            x["tile_q"] = min(x["tile_q"], 240)
        d_table = mb.exemplar_table_device(mb.exemplar_table(entries), cuda)
        valid = [rng.choice([0, 0, 1, 5, 16, 33, 80, 96]) for _ in range(E)]
        A = wl.integer_bf16((E, M, K), 50 + trial, cuda)
        B = wl.integer_bf16((E, N, K), 80 + trial, cuda)
        d_valid = torch.tensor(valid, dtype=torch.int32, device=cuda)
        out = torch.full((3,), -7, dtype=torch.int32, device=cuda)
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        D1 = gu.sentinel_like((E, M, N), cuda)
        mb.mgemm_masked_exemplar(A, B, D1, d_valid, d_table, n, tactic_out=out, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        want = osel.choose(valid, entries)
        assert out.cpu().tolist() == [entries[want]["tile_q"], entries[want]["blocks"], want], trial
        D2 = gu.sentinel_like((E, M, N), cuda)
        mb.mgemm_masked_tactic(A, B, D2, d_valid, out, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(D1.view(torch.int16), D2.view(torch.int16)), trial
        if trial < 4:
            R, written = og.masked(gu.deq_bf16(A).reshape(E, M, K), gu.deq_bf16(B).reshape(E, N, K), valid)
            Dbits = gu.bf16_bits(D1).reshape(E, M, N)
            assert np.array_equal(Dbits[written], gu.round_bf16_bits(R[written]))
            assert (Dbits[~written] == gu.SENTINEL_BITS).all()
