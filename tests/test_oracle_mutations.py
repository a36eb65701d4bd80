"""The pins are strong enough: plant plausible mistakes in the oracle (on the
CPU, by monkeypatching) and check that some pin fails for each."""
import numpy as np
import pytest

import oracle.gemm as og
import oracle.numerics as on
import oracle.plan as op
from tests import test_oracle_gemm as tg
from tests import test_oracle_numerics as tn
from tests import test_oracle_plan as tp

pytestmark = pytest.mark.cpu


def fails(fn, *args):
    try:
        fn(*args)
    except (AssertionError, ValueError, IndexError):
        return True
    return False


def test_floor_instead_of_ceil_is_caught(monkeypatch):
    monkeypatch.setattr(op, "ceil_div", lambda a, b: a // b)
    assert fails(tp.test_worked_padding_examples, tp.GOLD["padding_cases"][0])


def test_dropped_square_in_effective_experts_is_caught(monkeypatch):
    orig = op.effective_experts
    monkeypatch.setattr(op, "effective_experts", lambda c: orig(c) ** 0.5)
    assert fails(tp.test_worked_effective_experts, tp.GOLD["effective_experts_cases"][1])


def test_tile_rows_off_by_one_is_caught(monkeypatch):
    orig = op.plan

    def bad(counts, q):
        p = orig(counts, q)
        p.tiles = [(e, r, min(q, n + 1)) for e, r, n in p.tiles]
        return p
    monkeypatch.setattr(op, "plan", bad)
    assert fails(tp.test_brute_force_all_tiny_histograms)


def test_transposed_weight_is_caught(monkeypatch):
    monkeypatch.setattr(og, "expert_product", lambda a, b: np.asarray(a) @ np.asarray(b).reshape(b.shape[1], b.shape[0]))
    assert fails(tg.test_contiguous_vs_triple_loop, [3, 0, 5, 1], 4)


def test_unaligned_segments_are_caught(monkeypatch):
    orig = op.plan

    def bad(counts, q):
        p = orig(counts, 1)
        return p
    monkeypatch.setattr(og, "plan", bad)
    assert fails(tg.test_contiguous_vs_triple_loop, [3, 0, 5, 1], 4)


def test_wrong_e4m3_bias_is_caught(monkeypatch):
    orig = on.decode_e4m3
    monkeypatch.setattr(on, "decode_e4m3", lambda c: orig(c) * 2.0)
    assert fails(tn.test_e4m3_all_codes_against_torch)


def test_wrong_weight_scale_index_is_caught(monkeypatch):
    def bad(codes, sf):
        N, K = codes.shape
        scale = on.decode_ue8m0(sf).reshape(N // 128, K // 128)   # reshape, not transpose
        full = np.repeat(np.repeat(scale, 128, axis=0), 128, axis=1)
        return on.decode_e4m3(codes) * full
    monkeypatch.setattr(on, "dequant_weight", bad)
    assert fails(tn.test_dequant_weight_brute_force)
