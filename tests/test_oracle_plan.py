"""Pins for the oracle's padding accounting (no GPU).

Each check rests on something other than the oracle itself: the numbers the
padding blog prints for its two worked histograms, closed forms, invariants
the pages state, and brute-force enumeration of tiles row by row.
"""
import itertools
import math
import random

import pytest

from oracle import plan as op
from tests.conftest import load_golden

pytestmark = pytest.mark.cpu

GOLD = load_golden("worked_examples.json")


@pytest.mark.parametrize("case", GOLD["padding_cases"], ids=lambda c: f"{c['counts'][:2]}-q{c['q']}")
def test_worked_padding_examples(case):
    """"MoE GroupGEMM padding under expert skew", "Work a near-uniform routing
    example" and "Contrast a concentrated histogram": P, padding rows and the
    printed padding percentage."""
    p = op.plan(case["counts"], case["q"])
    assert p.U == case["U"]
    assert p.P == case["P"]
    if "padding_rows" in case:
        assert p.P - p.U == case["padding_rows"]
    # the page prints percentages rounded to one decimal (two for 31.25)
    pct = 100.0 * p.pad_frac
    assert abs(pct - case["padding_percent"]) <= 0.05 + 1e-12
    if "useful_share_percent" in case:
        assert abs(100.0 * p.U / p.P - case["useful_share_percent"]) <= 0.05 + 1e-12
    for t, r in zip(case["counts"], p.rounded):
        assert r == case["rounded_per_expert"][str(t)]


def test_worked_examples_exact_fractions():
    """The exact values behind the page's rounded percentages."""
    u = [17, 17, 17, 17, 16, 16, 16, 16]
    c = [100, 32, 0, 0, 0, 0, 0, 0]
    assert op.plan(u, 8).pad_frac == 28 / 160 == 0.175
    assert op.plan(u, 16).pad_frac == 0.3125
    assert op.plan(u, 32).pad_frac == 124 / 256 == 0.484375
    assert op.plan(c, 8).pad_frac == 4 / 136
    assert op.plan(c, 32).pad_frac == 28 / 160


@pytest.mark.parametrize("case", GOLD["effective_experts_cases"], ids=lambda c: c["printed"])
def test_worked_effective_experts(case):
    """"Summarize skew without losing the histogram": almost eight for the
    near-uniform histogram, about 1.58 for the concentrated one."""
    eff = op.effective_experts(case["counts"])
    if "below" in case:
        assert eff < case["below"] and round(eff) == case["round_to_integer"]
    if "round_to_2dp" in case:
        assert round(eff, 2) == case["round_to_2dp"]


def test_effective_experts_exact_values():
    assert op.effective_experts([17] * 4 + [16] * 4) == 17424 / 2180
    assert op.effective_experts([100, 32] + [0] * 6) == 17424 / 11024


def test_effective_experts_limits():
    """The metric equals the expert count under uniform routing and tends to
    one when a single expert carries nearly all tokens (same section)."""
    for E in (1, 2, 7, 64, 256):
        for t in (1, 3, 1000):
            assert op.effective_experts([t] * E) == float(E)
    assert op.effective_experts([5000, 0, 0, 0]) == 1.0
    assert 1.0 < op.effective_experts([10 ** 6] + [1] * 31) < 1.0001
    rng = random.Random(5)
    for _ in range(500):
        c = [rng.randint(0, 50) * (rng.random() < 0.7) for _ in range(rng.randint(1, 20))]
        p = op.plan(c, 8)
        if p.active:
            assert 1.0 - 1e-12 <= p.eff_experts <= p.active + 1e-9


def brute_force_tiles(counts, q):
    """Walk every row of every expert; open a new tile whenever the row index
    inside the expert is a multiple of q; lay segments end to end, each
    padded to whole tiles."""
    tiles = []
    offsets = [0]
    cursor = 0
    for e, t in enumerate(counts):
        start = cursor
        cur = None
        for r in range(t):
            if r % q == 0:
                cur = [e, start + r, 0]
                tiles.append(cur)
            cur[2] += 1
        ntiles = sum(1 for x in tiles if x[0] == e)
        cursor = start + ntiles * q
        offsets.append(cursor)
    return offsets, [tuple(x) for x in tiles]


def test_brute_force_all_tiny_histograms():
    """Every histogram with E <= 3 experts, counts <= 6 and q <= 5."""
    for E in (1, 2, 3):
        for counts in itertools.product(range(7), repeat=E):
            for q in range(1, 6):
                p = op.plan(list(counts), q)
                offs, tiles = brute_force_tiles(list(counts), q)
                assert p.offsets == offs
                assert p.tiles == tiles
                assert p.P == offs[-1] == sum(len([1 for x in tiles if x[0] == e]) * q for e in range(E))
                assert p.U == sum(counts)
                assert p.num_tiles == len(tiles)
                assert p.sumsq == sum(t * t for t in counts)
                assert p.active == sum(1 for t in counts if t)


def test_issue32_histogram_brute_force():
    """The issue's 32-expert histogram: the page prints no P, so P at each
    candidate block is fixed by enumeration."""
    counts = load_golden("issue32_histogram.json")["counts"]
    assert sum(counts) == 8048 and sum(1 for t in counts if t == 0) == 7
    for q in (8, 16, 32, 64, 128, 256):
        offs, tiles = brute_force_tiles(counts, q)
        p = op.plan(counts, q)
        assert p.P == offs[-1]
        assert p.tiles == tiles
    # P grows with the block and the occupancy the issue worries about falls
    Ps = [op.plan(counts, q).P for q in (8, 16, 32, 64, 128, 256)]
    assert Ps == sorted(Ps)
    assert op.plan(counts, 128).P == 10240


def test_invariants_random():
    """P is a multiple of q, U <= P < U + q*active, q = 1 gives P = U, zero
    experts add nothing (padding blog, "Calculate padded token columns")."""
    rng = random.Random(11)
    for _ in range(2000):
        E = rng.randint(1, 40)
        c = [rng.randint(0, 3000) if rng.random() < 0.8 else 0 for _ in range(E)]
        q = rng.choice([1, 2, 3, 7, 8, 16, 32, 64, 128, 256])
        p = op.plan(c, q)
        assert p.P % q == 0
        assert p.U <= p.P < p.U + q * p.active or (p.active == 0 and p.P == 0)
        assert op.plan(c, 1).P == p.U
        assert op.plan(c + [0, 0], q).P == p.P
        assert p.offsets[-1] == p.P and all(o % q == 0 for o in p.offsets)
        assert p.pad_frac == (float(p.P - p.U) / float(p.P) if p.P else 0.0)


def test_empty_and_degenerate():
    p = op.plan([0, 0, 0], 16)
    assert (p.P, p.U, p.sumsq, p.active, p.num_tiles) == (0, 0, 0, 0, 0)
    assert p.pad_frac == 0.0 and p.eff_experts == 0.0 and p.tiles == []
    p = op.plan([1], 256)
    assert p.P == 256 and p.tiles == [(0, 0, 1)] and p.eff_experts == 1.0
    # P past 2^31 (with a wide tile, so the tile list stays short)
    huge = [2 ** 31 - 1] * 3
    p = op.plan(huge, 1 << 20)
    assert p.P == 3 * (1 << 20) * math.ceil((2 ** 31 - 1) / (1 << 20)) and p.P > 2 ** 32
    assert p.num_tiles == 3 * 2048 and p.U == 3 * (2 ** 31 - 1)
    with pytest.raises(ValueError):
        op.plan([1, -1], 8)
    with pytest.raises(ValueError):
        op.plan([1], 0)


def test_m_occupancy_matches_single_expert_share():
    """"Query on performance-modeling of MoE Grouped GEMM", "Background":
    M-occupancy of one GEMM equals the useful share U/P of a one-expert plan,
    is 1 when B_M divides M, and is M/B_M for M < B_M."""
    for M in range(1, 600, 7):
        for BM in (8, 16, 64, 128, 256):
            p = op.plan([M], BM)
            assert abs(op.m_occupancy(M, BM) - p.U / p.P) < 1e-15
    assert op.m_occupancy(256, 128) == 1.0
    assert op.m_occupancy(1, 128) == 1 / 128


def test_average_assignments_per_expert():
    assert op.avg_assignments_per_expert(4096, 8, 256) == 128.0
    assert op.avg_assignments_per_expert(32768, 1, 64) == 512.0


def test_token_offsets():
    assert op.token_offsets([3, 0, 5]) == [0, 3, 3, 8]
