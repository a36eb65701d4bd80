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


# --- SwiGLU / FP8 re-quantisation (oracle/epilogue.py) ---------------------
import oracle.epilogue as oe                     # noqa: E402
from tests import test_oracle_epilogue as te     # noqa: E402


def test_sigmoid_sign_flip_is_caught(monkeypatch):
    monkeypatch.setattr(oe, "silu", lambda x: np.asarray(x, float) / (1.0 + np.exp(np.asarray(x, float))))
    assert fails(te.test_silu_closed_forms)


def test_ties_away_from_zero_is_caught(monkeypatch):
    mag = oe._MAG

    def bad(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.minimum(np.abs(x), 448.0)
        hi = np.clip(np.searchsorted(mag, a, side="left"), 0, 126)
        lo = np.clip(hi - 1, 0, 126)
        code = np.where(a - mag[lo] < mag[hi] - a, lo, hi).astype(np.uint8)
        return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    monkeypatch.setattr(oe, "encode_e4m3", bad)
    assert fails(te.test_encode_rounds_to_nearest_even_and_saturates)


def test_scale_off_by_one_is_caught(monkeypatch):
    orig = oe.ue8m0_for_amax
    monkeypatch.setattr(oe, "ue8m0_for_amax", lambda a: np.where(np.asarray(a) == 0, 127, orig(a) + 1).astype(np.uint8))
    assert fails(te.test_ue8m0_boundaries)
    assert fails(te.test_quantize_blocks_bounds_and_layout)


def test_amax_bound_strictness_is_caught(monkeypatch):
    # using m >= 0.875 instead of m > 0.875 doubles the scale exactly on the bound
    def bad(amax):
        amax = np.asarray(amax, dtype=np.float64)
        m, e = np.frexp(amax)
        s = np.clip(e.astype(np.int64) + 118 + (m >= 0.875), 1, 254)
        return np.where(amax == 0, 127, s).astype(np.uint8)
    monkeypatch.setattr(oe, "ue8m0_for_amax", bad)
    assert fails(te.test_ue8m0_boundaries)


def test_swapped_gate_and_up_is_caught(monkeypatch):
    orig = oe.gate_up_halves
    monkeypatch.setattr(oe, "gate_up_halves", lambda H: orig(H)[::-1])
    assert fails(te.test_gate_up_halves_layout)



def test_e2m1_wrong_bias_is_caught(monkeypatch):
    orig = on.decode_e2m1
    monkeypatch.setattr(on, "decode_e2m1", lambda c: orig(c) * 2.0)
    assert fails(tn.test_e2m1_all_codes)


def test_mx4_nibble_swap_is_caught(monkeypatch):
    def bad(packed):
        p = np.asarray(packed, dtype=np.uint8)
        out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
        out[..., 0::2] = p >> 4
        out[..., 1::2] = p & 0xF
        return out
    monkeypatch.setattr(on, "unpack_e2m1", bad)
    assert fails(tn.test_unpack_e2m1_nibble_order)
    assert fails(tn.test_dequant_weight_mx4_brute_force)


def test_mx4_scale_granularity_is_caught(monkeypatch):
    def bad(packed, sf):
        codes = on.unpack_e2m1(packed)
        return on.decode_e2m1(codes) * np.repeat(on.decode_ue8m0(sf), 32, axis=1)[:, ::-1]
    monkeypatch.setattr(on, "dequant_weight_mx4", bad)
    assert fails(tn.test_dequant_weight_mx4_brute_force)


# --- exemplar selector (oracle/selector.py) --------------------------------
import oracle.selector as osel                   # noqa: E402
from tests import test_oracle_selector as tsel   # noqa: E402


def test_ascending_sort_is_caught(monkeypatch):
    orig = osel.features

    def bad(counts):
        lu, shares = orig(counts)
        c = sorted(max(0, int(x)) for x in counts)                  # ascending
        U = sum(c)
        if U == 0:
            return lu, shares
        E = len(c)
        return lu, [65536 * sum(c[:-(-k * E // 16)]) // U for k in range(1, 17)]
    monkeypatch.setattr(osel, "features", bad)
    assert fails(tsel.test_worked_concentrated_example)


def test_floor_expert_count_is_caught(monkeypatch):
    orig_sorted = sorted

    def bad(counts):
        c = orig_sorted((max(0, int(x)) for x in counts), reverse=True)
        U, E = sum(c), len(c)
        if U == 0:
            return 0, [0] * 16
        shares = [65536 * sum(c[:k * E // 16]) // U for k in range(1, 17)]   # floor, not ceil
        e = U.bit_length() - 1
        return 16 * e + (16 * (U - (1 << e))) // (1 << e), shares
    monkeypatch.setattr(osel, "features", bad)
    assert fails(tsel.test_worked_concentrated_example)


def test_hysteresis_inverted_is_caught(monkeypatch):
    def bad(counts, table, prev=-1, margin=0):
        feat = osel.features(counts)
        d = [osel.distance(feat, x) for x in table]
        best = min(range(len(d)), key=lambda i: (d[i], i))
        if 0 <= prev < len(table) and d[prev] - d[best] < margin:    # strict: off by one at the margin
            return prev
        return best
    monkeypatch.setattr(osel, "choose", bad)
    assert fails(tsel.test_choice_ties_and_hysteresis)


def test_kgrouped_aligned_token_segments_are_caught(monkeypatch):
    """K-grouped tokens are packed with no alignment: segments that start on
    a block boundary (the contiguous form's layout) must fail a pin."""
    monkeypatch.setattr(og, "token_offsets", lambda counts: op.plan(counts, 4).offsets)
    assert fails(tg.test_kgrouped_vs_outer_product_sum)


def test_kgrouped_segment_shifted_by_one_is_caught(monkeypatch):
    orig = op.token_offsets
    monkeypatch.setattr(og, "token_offsets", lambda counts: [0] + [o + 1 for o in orig(counts)[1:]])
    assert fails(tg.test_kgrouped_vs_outer_product_sum)


def test_masked_extra_row_is_caught(monkeypatch):
    orig = og.masked

    def bad(A, B, valid_m):
        return orig(A, B, [min(v + 1, A.shape[1]) if v else 0 for v in valid_m])
    monkeypatch.setattr(og, "masked", bad)
    assert fails(tg.test_masked_vs_triple_loop)


def test_masked_wrong_expert_weights_are_caught(monkeypatch):
    orig = og.masked
    monkeypatch.setattr(og, "masked", lambda A, B, v: orig(A, np.roll(B, 1, axis=0), v))
    assert fails(tg.test_masked_vs_triple_loop)


def test_contiguous_dropped_expert_is_caught(monkeypatch):
    orig = og.contiguous

    def bad(A, B, counts, align_q):
        c = list(counts)
        c[-1] = 0
        R, w = orig(A, B, c, align_q)
        return R, w
    monkeypatch.setattr(og, "contiguous", bad)
    assert fails(tg.test_contiguous_vs_triple_loop, [3, 0, 5, 1], 4)
