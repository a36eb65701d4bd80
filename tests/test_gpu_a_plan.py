"""Device planning, device tile selection and the bounded-wait self-test."""
import random

import numpy as np
import pytest
import torch

from moe_grouped_gemm_side_gb300 import binding as mb
from oracle import plan as op

pytestmark = pytest.mark.gpu


def _device_plan(counts, q, max_tiles=None, dev="cuda"):
    ref = op.plan([max(0, c) for c in counts], q)
    if max_tiles is None:
        max_tiles = ref.num_tiles
    d = torch.tensor(counts, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    offs, tiles, stats = mb.plan(d, q, max_tiles, status=status)
    torch.cuda.synchronize()
    return ref, offs.cpu().tolist(), [tuple(t) for t in tiles.cpu().tolist()], mb.decode_stats(stats), int(status.item())


def _assert_plan(counts, q):
    ref, offs, tiles, st, status = _device_plan(counts, q)
    assert status == 0
    assert offs == ref.offsets
    assert tiles == ref.tiles
    assert (st["P"], st["U"], st["sumsq"], st["active"], st["num_tiles"]) == (
        ref.P, ref.U, ref.sumsq, ref.active, ref.num_tiles)
    assert float(st["pad_frac"]).hex() == ref.pad_frac.hex()
    assert float(st["eff_experts"]).hex() == ref.eff_experts.hex()


def test_wait_selftest_times_out_cleanly(lib, cuda):
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    mb.wait_selftest(status, 2_000_000)   # 2 ms
    torch.cuda.synchronize()
    assert int(status.item()) == 5        # MG_ERR_TIMEOUT
    # the context is still healthy
    x = torch.ones(1024, device=cuda)
    assert float(x.sum().item()) == 1024.0


def test_device_plan_worked_examples(lib, cuda):
    for counts in ([17, 17, 17, 17, 16, 16, 16, 16], [100, 32, 0, 0, 0, 0, 0, 0]):
        for q in (8, 16, 32):
            _assert_plan(counts, q)


def test_device_plan_random(lib, cuda):
    rng = random.Random(7)
    for _ in range(200):
        E = rng.choice([1, 3, 32, 64, 257, 1500, 3000])
        c = [0 if rng.random() < 0.3 else rng.randint(1, rng.choice([5, 300, 20000])) for _ in range(E)]
        _assert_plan(c, rng.choice([1, 8, 16, 64, 128, 256]))


def test_device_plan_issue_histogram(lib, cuda):
    from moe_grouped_gemm_side_gb300 import workloads as wl
    for q in (8, 16, 32, 64, 128, 256):
        _assert_plan(wl.counts_issue32(), q)


def test_device_plan_maximum_experts(lib, cuda):
    """2^20 experts (the documented maximum: 1024 block-scan passes of the
    one-CTA plan), offsets, tiles and stats bit-exact."""
    rng = random.Random(5)
    _assert_plan([rng.choice([0, 0, 1, 3, 17, 40, 129]) for _ in range(1 << 20)], 16)


def test_device_plan_square_sum_past_int64(lib, cuda):
    """Sums of squares around 2^63 (just below, just above through the
    low-half carry, far above): sumsq saturates, eff_experts stays the
    correctly rounded ratio of the exact integers, as on the host."""
    q = 2 ** 31 - 1
    for counts in ([q, q], [q, q, 92681], [q, q, 92681, 65535], [q] * 3, [q] * 1000 + [0, 7]):
        ref, offs, _, st, status = _device_plan(counts, 1 << 20, max_tiles=0)
        assert status == 0 and offs == ref.offsets
        assert (st["P"], st["U"], st["active"]) == (ref.P, ref.U, ref.active)
        assert st["sumsq"] == min(ref.sumsq, 2 ** 63 - 1)
        assert float(st["pad_frac"]).hex() == ref.pad_frac.hex()
        assert float(st["eff_experts"]).hex() == ref.eff_experts.hex()


def test_device_plan_tile_count_saturates(lib, cuda):
    """sum_e ceil(t_e/q) past 2^31-1 reads 2^31-1, as on the host."""
    m = 2 ** 31 - 1
    for counts, want in (([m, m], m), ([m], m), ([m - 1, 0], m - 1)):
        d = torch.tensor(counts, dtype=torch.int32, device=cuda)
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        _, _, stats = mb.plan(d, 1, 0, status=status)
        torch.cuda.synchronize()
        st = mb.decode_stats(stats)
        assert int(status.item()) == 0 and st["num_tiles"] == want and st["P"] == sum(counts)
        _, _, hst, _ = mb.plan_host(counts, 1, max_tiles=0)
        assert hst.num_tiles == want


def test_device_plan_errors(lib, cuda):
    ref, offs, tiles, st, status = _device_plan([17] * 8, 8, max_tiles=5)
    assert status == 4 and st["P"] == 192 and tiles == ref.tiles[:5] and offs == ref.offsets
    ref, offs, tiles, st, status = _device_plan([5, -3, 7], 4)
    assert status == 6 and offs == op.plan([5, 0, 7], 4).offsets


def test_device_select_matches_host(lib, cuda):
    rng = random.Random(3)
    cases = [[4096] * 64, [1] * 256, [0] * 8, [100, 32, 0, 0, 0, 0, 0, 0]]
    cases += [[rng.randint(0, rng.choice([30, 300, 3000])) for _ in range(rng.randint(1, 128))] for _ in range(40)]
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    for c in cases:
        d = torch.tensor(c, dtype=torch.int32, device=cuda)
        for dt in (mb.MG_BF16, mb.MG_FP8_E4M3_UE8M0):
            for (N, K) in ((4096, 2048), (4096, 7168), (256, 256)):
                got = int(mb.select_tile(dt, d, N, K).item())
                assert got == mb.select_tile_host(dt, c, N, K, nsm)
