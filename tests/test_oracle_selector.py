"""Pins of the exemplar selector's oracle (oracle/selector.py): feature values
worked by hand, invariances of a sorted and normalised histogram, and the
choice and hysteresis rules on tiny tables."""
import itertools
import random

import pytest

from oracle import selector as osel

pytestmark = pytest.mark.cpu


def test_uniform_histograms_give_the_diagonal():
    """Equal counts: the top k/16 of the experts hold k/16 of the tokens,
    whatever the expert count (E a multiple of 16)."""
    for E in (16, 64, 256):
        lu, shares = osel.features([10] * E)
        assert shares == [4096 * k for k in range(1, 17)]


def test_worked_concentrated_example():
    """[100, 32, 0, 0, 0, 0, 0, 0] ("MoE GroupGEMM padding under expert skew",
    "Contrast a concentrated histogram"): the top expert (first two of the
    16 points, m = ceil(k*8/16) = 1) holds 100/132 of the tokens, two experts
    hold all of them."""
    lu, shares = osel.features([100, 32, 0, 0, 0, 0, 0, 0])
    assert shares[:2] == [6553600 // 132] * 2 == [49648, 49648]
    assert shares[2:] == [65536] * 14
    # U = 132 = 2^7 + 4: 16 * 7 + floor(16 * 4 / 128) = 112
    assert lu == 112


def test_single_hot_expert_and_empty():
    assert osel.features([0, 0, 7, 0])[1] == [65536] * 16
    assert osel.features([0] * 5) == (0, [0] * 16)
    assert osel.features([-3, 0]) == (0, [0] * 16)          # negative counts read as 0


def test_log_feature():
    for U, want in ((1, 0), (2, 16), (3, 24), (1024, 160), (1536, 168), (32768, 240), (32767, 239)):
        assert osel.features([U])[0] == want, U


def test_invariances():
    rng = random.Random(3)
    for _ in range(50):
        c = [rng.randrange(0, 500) for _ in range(rng.randrange(1, 40))]
        f = osel.features(c)
        rng.shuffle(c)
        assert osel.features(c) == f                          # order of experts does not matter
        if sum(c):
            lu2, s2 = osel.features([2 * x for x in c])
            assert s2 == f[1] and lu2 == f[0] + 16            # scale: same curve, log up by one
        assert all(a <= b for a, b in zip(f[1], f[1][1:]))    # cumulative shares never decrease


def test_choice_ties_and_hysteresis():
    table = [{"lu": 100, "shares": [4096 * k for k in range(1, 17)]},
             {"lu": 100, "shares": [65536] * 16},
             {"lu": 100, "shares": [4096 * k for k in range(1, 17)]}]   # a duplicate of 0
    uniform = [8] * 16                                                  # U = 128: lu = 112
    assert osel.choose(uniform, table) == 0                             # tie 0 / 2 -> lower index
    d0 = osel.distance(osel.features(uniform), table[0])
    d1 = osel.distance(osel.features(uniform), table[1])
    assert d0 == 2048 * 12 and d1 > d0
    assert osel.choose(uniform, table, prev=1, margin=d1 - d0) == 1     # within the margin: keep
    assert osel.choose(uniform, table, prev=1, margin=d1 - d0 - 1) == 0
    assert osel.choose(uniform, table, prev=7, margin=10 ** 9) == 0     # no valid history


def test_choice_brute_force():
    rng = random.Random(5)
    for _ in range(30):
        table = [{"lu": rng.randrange(0, 300), "shares": sorted(rng.randrange(0, 65537) for _ in range(16))}
                 for _ in range(rng.randrange(1, 6))]
        c = [rng.randrange(0, 50) for _ in range(rng.randrange(1, 20))]
        f = osel.features(c)
        d = [sum(abs(a - b) for a, b in zip(f[1], x["shares"])) + 2048 * abs(f[0] - x["lu"]) for x in table]
        best = min(range(len(table)), key=lambda i: (d[i], i))
        assert osel.choose(c, table) == best


def test_committed_exemplar_tables_are_consistent():
    """The tables tuned on the GPU store, per exemplar, the histogram it was
    tuned on: its features must be the oracle's, and every tactic must be one
    the GEMMs accept."""
    import glob
    import json
    import os
    from tests.conftest import ROOT
    paths = sorted(glob.glob(os.path.join(ROOT, "moe_grouped_gemm_side_gb300", "exemplars", "*.json")))
    assert paths
    for path in paths:
        with open(path) as f:
            t = json.load(f)
        assert t["exemplars"]
        for x in t["exemplars"]:
            assert (x["lu"], x["shares"]) == osel.features(x["counts"])
            assert x["tile_q"] % 16 == 0 and 16 <= x["tile_q"] <= 256 and x["blocks"] in (1, 2)
            assert f"{x['tile_q']}x{x['blocks']}" in x["times_us"]
