"""C ABI checks that need no GPU: the library loads, exports every function
the header declares, the host planner matches the oracle bit for bit, and
bad arguments come back as error codes before anything is launched."""
import ctypes
import os
import random
import re

import numpy as np
import pytest

from moe_grouped_gemm_side_gb300 import binding as mb
from oracle import plan as op
from tests.conftest import ROOT

pytestmark = pytest.mark.cpu

HEADER = os.path.join(ROOT, "include", "moegemm.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", src, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("moe_plan", "moe_plan_host", "mgemm_contiguous", "mgemm_masked", "kgemm_grouped", "moe_select_exemplar", "mgemm_contiguous_tactic",
              "moe_select_tile", "mg_status_str", "mgemm_contiguous_swiglu", "mgemm_masked_swiglu"):
        assert f in names
    assert set(names) == set(mb.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in mb.STATUS_NAMES.items():
        assert mb.status_str(code) == name
    assert mb.status_str(99) == "MG_ERR_UNKNOWN"


def _check_plan(counts, q):
    offs, tiles, st, code = mb.plan_host(counts, q)
    ref = op.plan(counts, q)
    assert code == 0
    assert offs.tolist() == ref.offsets
    assert [tuple(t) for t in tiles.tolist()] == ref.tiles
    assert (st.P, st.U, st.sumsq, st.active, st.num_tiles) == (ref.P, ref.U, ref.sumsq, ref.active, ref.num_tiles)
    # the two ratios are bit-identical doubles
    assert st.pad_frac.hex() == ref.pad_frac.hex()
    assert st.eff_experts.hex() == ref.eff_experts.hex()


def test_host_plan_worked_examples(lib):
    for counts in ([17, 17, 17, 17, 16, 16, 16, 16], [100, 32, 0, 0, 0, 0, 0, 0]):
        for q in (8, 16, 32):
            _check_plan(counts, q)


def test_host_plan_random_bit_exact(lib):
    rng = random.Random(21)
    for _ in range(3000):
        E = rng.randint(1, 70)
        zero = rng.random()
        c = [0 if rng.random() < zero else rng.randint(1, rng.choice([3, 40, 500, 20000])) for _ in range(E)]
        _check_plan(c, rng.choice([1, 2, 5, 8, 16, 32, 64, 128, 256]))


def test_host_plan_edges(lib):
    _check_plan([0], 8)
    _check_plan([0] * 300, 128)
    _check_plan([1], 1)
    _check_plan(list(range(1024)), 7)
    # P beyond int32: offsets and stats stay exact, the int32 tile list is refused
    huge = [2 ** 31 - 1, 2 ** 31 - 1]
    offs, tiles, st, code = mb.plan_host(huge, 1 << 20)
    ref = op.plan(huge, 1 << 20)
    assert code == 2 and offs.tolist() == ref.offsets and st.P == ref.P
    assert st.eff_experts.hex() == ref.eff_experts.hex()
    fits = [t for t in ref.tiles if t[1] <= 2 ** 31 - 1]
    assert [tuple(t) for t in tiles.tolist()][:len(fits)] == fits
    offs, _, st, code = mb.plan_host(huge, 1 << 20, max_tiles=0)
    assert code == 0 and offs.tolist() == ref.offsets
    _check_plan(list(range(1024)), 7)


# Sums of squares around 2^63: just below (exact), just above through the
# low-half carry, and far above; sumsq saturates, eff_experts stays the
# correctly rounded ratio of the exact integers.
SQ = 2 ** 31 - 1
SQUARE_SUM_EDGES = ([SQ, SQ], [SQ, SQ, 92681], [SQ, SQ, 92681, 65535], [SQ] * 3, [SQ] * 1000 + [0, 7])


def test_host_plan_square_sum_past_int64(lib):
    for counts in SQUARE_SUM_EDGES:
        offs, _, st, code = mb.plan_host(counts, 1 << 20, max_tiles=0)
        ref = op.plan(counts, 1 << 20)
        assert code == 0 and offs.tolist() == ref.offsets
        assert (st.P, st.U, st.active) == (ref.P, ref.U, ref.active)
        assert st.sumsq == min(ref.sumsq, 2 ** 63 - 1)
        assert st.pad_frac.hex() == ref.pad_frac.hex()
        assert st.eff_experts.hex() == ref.eff_experts.hex()
    assert sum(c * c for c in SQUARE_SUM_EDGES[1]) == 2 ** 63 - 166829
    assert sum(c * c for c in SQUARE_SUM_EDGES[2]) > 2 ** 63


def test_host_plan_maximum_experts(lib):
    """2^20 experts, the documented maximum, bit-exact; one more is refused."""
    rng = random.Random(5)
    c = [rng.choice([0, 0, 1, 3, 17, 40, 129]) for _ in range(1 << 20)]
    _check_plan(c, 16)
    _, _, _, code = mb.plan_host(c + [1], 16, max_tiles=0)
    assert code == 1


def test_host_plan_tile_count_saturates(lib):
    """sum_e ceil(t_e/q) past 2^31-1 reads 2^31-1 (a closed form, no list)."""
    huge = [2 ** 31 - 1, 2 ** 31 - 1]
    offs, _, st, code = mb.plan_host(huge, 1, max_tiles=0)
    assert code == 0 and st.P == 2 * (2 ** 31 - 1) and st.num_tiles == 2 ** 31 - 1
    _, _, st, code = mb.plan_host([2 ** 31 - 1], 1, max_tiles=0)
    assert code == 0 and st.num_tiles == 2 ** 31 - 1
    _, _, st, code = mb.plan_host([2 ** 31 - 2, 0], 1, max_tiles=0)
    assert code == 0 and st.num_tiles == 2 ** 31 - 2
    # the binding sizes a list from that count and refuses one that cannot exist
    _, tiles, st, code = mb.plan_host(huge, 1)
    assert code == 2 and tiles.shape == (0, 3)


def test_host_plan_sizing_call_matches_list(lib):
    """A call without a tile list reports the count the list then holds."""
    counts = [4, 1026, 0, 17, 255, 256, 257]
    for q in (1, 7, 16, 128):
        _, _, st0, code0 = mb.plan_host(counts, q, max_tiles=0)
        offs, tiles, st, code = mb.plan_host(counts, q)
        assert code0 == 0 and code == 0 and len(tiles) == st0.num_tiles == st.num_tiles
        assert [tuple(t) for t in tiles.tolist()] == op.plan(counts, q).tiles


def test_host_plan_capacity_and_errors(lib):
    offs, tiles, st, code = mb.plan_host([17] * 8, 8, max_tiles=5)
    assert code == 4 and st.P == 192 and st.num_tiles == 24 and offs[-1] == 192
    assert [tuple(t) for t in tiles.tolist()] == op.plan([17] * 8, 8).tiles[:5]
    _, _, _, code = mb.plan_host([3, -1], 8)
    assert code == 1
    _, _, _, code = mb.plan_host([3], 0)
    assert code == 1
    st = mb.PlanStats()
    off = np.zeros(2, np.int64)
    assert lib.moe_plan_host(None, 1, 8, off.ctypes.data_as(mb._c_i64p), None, 0, ctypes.byref(st)) == 1


def test_select_tile_host(lib):
    # many tokens per expert: the largest tile; bf16 and fp8 candidates differ
    big = [4096] * 64
    assert mb.select_tile_host(mb.MG_BF16, big, 4096, 7168) == 256
    assert mb.select_tile_host(mb.MG_FP8_E4M3_UE8M0, big, 4096, 7168) == 240
    for seed in range(50):
        c = [random.Random(seed).randint(0, 300) for _ in range(32)]
        q = mb.select_tile_host(mb.MG_BF16, c, 4096, 2048)
        assert q in (32, 64, 128, 256)
    assert mb.select_tile_host(mb.MG_BF16, [0] * 8, 256, 256) == 256


FAKE = ctypes.c_void_p(1 << 20)       # aligned, never dereferenced
MISALIGNED = ctypes.c_void_p((1 << 20) + 8)


def test_device_calls_reject_bad_arguments_before_launch(lib):
    L = lib
    # contiguous
    args = [mb.MG_BF16, FAKE, None, FAKE, None, FAKE, FAKE, 8, 1024, 256, 256, 16, 0, None, None]

    def contig(kw):
        a = list(args)
        for k, v in kw.items():
            a[k] = v
        return L.mgemm_contiguous(*a)
    assert contig({1: None}) == 1            # A NULL
    assert contig({0: 7}) == 1               # bad dtype
    assert contig({7: 0}) == 1               # E <= 0
    assert contig({9: 200}) == 2             # N not a multiple of 128
    assert contig({10: 192}) == 2            # K not a multiple of 128
    assert contig({11: 0}) == 1              # align_q
    assert contig({12: 24}) == 1             # tile_q not a multiple of 16
    assert contig({12: 512}) == 1            # tile_q too large
    assert contig({8: 0}) == 1               # rows_cap
    assert contig({1: MISALIGNED}) == 1      # alignment
    assert contig({7: 5000}) == 2            # too many experts
    assert contig({0: 1}) == 1               # fp8 without scales
    assert contig({0: 1, 2: FAKE, 4: FAKE, 11: 8}) == 2     # fp8 align_q % 16
    assert contig({0: 1, 2: FAKE, 4: FAKE, 12: 248}) == 1   # fp8 tile 248
    fp4 = {0: mb.MG_FP8_X_FP4_E2M1, 2: FAKE, 4: FAKE, 10: 512}
    assert contig({**fp4, 10: 640}) == 2                    # FP4 weights need K % 512
    assert contig({**fp4, 3: ctypes.c_void_p((1 << 20) + 16)}) == 1   # packed FP4 base 32-byte aligned
    assert contig({**fp4, 4: None}) == 1                    # FP4 without weight scales
    # masked
    m = [mb.MG_BF16, FAKE, None, FAKE, None, FAKE, FAKE, 8, 256, 256, 256, None, None]
    assert L.mgemm_masked(*[None if i == 6 else v for i, v in enumerate(m)]) == 1
    assert L.mgemm_masked(*[0 if i == 8 else v for i, v in enumerate(m)]) == 1
    assert L.mgemm_masked(*[1 if i == 0 else v for i, v in enumerate(m)]) == 1
    mm = list(m)
    mm[0], mm[2], mm[4], mm[8] = 1, FAKE, FAKE, 40
    assert L.mgemm_masked(*mm) == 2            # fp8 M_max % 16
    # contiguous / masked with the SwiGLU epilogue
    sw = [mb.MG_BF16, mb.MG_SWIGLU_BF16, FAKE, None, FAKE, None, FAKE, None, FAKE, 8, 1024, 512, 256, 16, 0,
          None, None]

    def swig(kw):
        a = list(sw)
        for k_, v in kw.items():
            a[k_] = v
        return L.mgemm_contiguous_swiglu(*a)
    assert swig({1: 0}) == 1                 # bad output kind
    assert swig({1: 3}) == 1
    assert swig({11: 384}) == 2              # N not whole gate/up pairs
    assert swig({1: mb.MG_SWIGLU_FP8_E4M3_UE8M0}) == 1      # E4M3 output without scales
    assert swig({6: None}) == 1              # Y NULL
    assert swig({13: 0}) == 1                # align_q (checks of the plain call)
    ms = [mb.MG_BF16, mb.MG_SWIGLU_BF16, FAKE, None, FAKE, None, FAKE, None, FAKE, 8, 64, 512, 256, None, None]
    assert L.mgemm_masked_swiglu(*[128 if i == 11 else v for i, v in enumerate(ms)]) == 2
    assert L.mgemm_masked_swiglu(*[0 if i == 10 else v for i, v in enumerate(ms)]) == 1
    assert L.mgemm_masked_swiglu(*[mb.MG_SWIGLU_FP8_E4M3_UE8M0 if i == 1 else v for i, v in enumerate(ms)]) == 1
    # k-grouped
    k = [FAKE, FAKE, FAKE, FAKE, 4, 4096, 256, 256, None, None]
    assert L.kgemm_grouped(*[None if i == 2 else v for i, v in enumerate(k)]) == 1
    assert L.kgemm_grouped(*[0 if i == 5 else v for i, v in enumerate(k)]) == 1
    assert L.kgemm_grouped(*[320 if i == 6 else v for i, v in enumerate(k)]) == 2
    # plan / select / self-test
    assert L.moe_plan(FAKE, 4, 0, FAKE, None, 0, FAKE, None, None) == 1
    assert L.moe_plan(FAKE, 4, 8, FAKE, None, 5, FAKE, None, None) == 1
    assert L.moe_select_tile(3, FAKE, 4, 256, 256, FAKE, None, None) == 1
    assert L.moe_select_tile(0, FAKE, 4, 250, 256, FAKE, None, None) == 2
    assert L.mg_wait_selftest(None, 1000, None) == 1


def test_gemm_shape_limits(lib):
    """The limits the header states for every GEMM call: 1024 experts,
    E * N < 2^31, fp8 K <= 16384; all refused before any launch."""
    L = lib
    base = [mb.MG_BF16, FAKE, None, FAKE, None, FAKE, FAKE, 8, 1024, 256, 256, 16, 0, None, None]

    def contig(**kw):
        a = list(base)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.mgemm_contiguous(*a)
    assert contig(a7=1025) == 2
    assert contig(a7=1024, a9=2 ** 21) == 2                                  # E * N = 2^31
    assert contig(a0=mb.MG_FP8_E4M3_UE8M0, a2=FAKE, a4=FAKE, a10=16384 + 128) == 2
    kg = [FAKE, FAKE, FAKE, FAKE, 8, 1024, 256, 256, None, None]
    assert L.kgemm_grouped(*[1025 if i == 4 else v for i, v in enumerate(kg)]) == 2
    assert L.kgemm_grouped(*[1024 if i == 4 else 2 ** 21 if i == 6 else v for i, v in enumerate(kg)]) == 2
    # (every case here is refused on the host: the pointers are fake)


def test_wait_limit_setting(lib):
    old = lib.mg_get_wait_limit_ns()
    try:
        lib.mg_set_wait_limit_ns(12345)
        assert lib.mg_get_wait_limit_ns() == 12345
        lib.mg_set_wait_limit_ns(0)
        assert lib.mg_get_wait_limit_ns() == 2_000_000_000
    finally:
        lib.mg_set_wait_limit_ns(old)


def test_kernel_policy_setting(lib):
    assert lib.mg_get_kernel_policy() == 0
    try:
        for v in (1, 2, 3, 4, 5, 0):
            assert lib.mg_set_kernel_policy(v) == 0 and lib.mg_get_kernel_policy() == v
        assert lib.mg_set_kernel_policy(6) == 1 and lib.mg_get_kernel_policy() == 0
        assert lib.mg_set_kernel_policy(-1) == 1 and lib.mg_get_kernel_policy() == 0
    finally:
        lib.mg_set_kernel_policy(0)


def test_exemplar_features_and_choice_match_the_oracle(lib):
    """Host features and choice (what table builders and tests use) equal the
    oracle's integer definitions bit for bit."""
    from oracle import selector as osel
    rng = random.Random(11)
    for _ in range(300):
        E = rng.choice([1, 3, 8, 16, 33, 64, 256, 1000])
        c = [rng.choice([0, 0, 1, 5, 17, 300, 9000, 40000]) * rng.randrange(0, 3) for _ in range(E)]
        assert mb.exemplar_features_host(c) == osel.features(c)
    for _ in range(200):
        n = rng.randrange(1, 12)
        entries = [{"lu": rng.randrange(0, 300), "shares": sorted(rng.randrange(0, 65537) for _ in range(16)),
                    "tile_q": 16 * rng.randrange(1, 16), "blocks": rng.choice([1, 2])} for _ in range(n)]
        table = mb.exemplar_table(entries)
        c = [rng.randrange(0, 2000) for _ in range(rng.randrange(1, 70))]
        prev = rng.randrange(-1, n)
        margin = rng.choice([0, 1000, 30000, 10 ** 6])
        assert mb.select_exemplar_host(c, table, margin, prev) == osel.choose(c, entries, prev, margin)


def test_exemplar_host_limits(lib):
    """The largest histogram the host calls accept (4096 experts, every count
    at the int32 maximum) stays exact; one expert more is refused, as on the
    device, instead of overflowing the top-share products."""
    from oracle import selector as osel
    top = [2 ** 31 - 1] * 4096
    assert mb.exemplar_features_host(top) == osel.features(top)
    skew = [2 ** 31 - 1] * 7 + [1] * 4089
    assert mb.exemplar_features_host(skew) == osel.features(skew)
    c = (ctypes.c_int32 * 4097)(*([5] * 4097))
    lu, share = ctypes.c_int32(0), (ctypes.c_int32 * 16)()
    assert lib.moe_exemplar_features_host(c, 4097, ctypes.byref(lu), share) == 2
    table = mb.exemplar_table([{"lu": 0, "shares": [0] * 16, "tile_q": 16, "blocks": 1}])
    out = ctypes.c_int32(-7)
    assert lib.moe_select_exemplar_host(c, 4097, table.ctypes.data, 1, 0, -1, ctypes.byref(out)) == 2
    assert out.value == -7


def test_exemplar_calls_reject_bad_arguments(lib):
    L = lib
    assert L.moe_select_exemplar(FAKE, 0, FAKE, 1, 0, None, FAKE, None, None) == 1        # E
    assert L.moe_select_exemplar(FAKE, 8, FAKE, 0, 0, None, FAKE, None, None) == 1        # n
    assert L.moe_select_exemplar(FAKE, 8, FAKE, 1, -1, None, FAKE, None, None) == 1       # margin
    assert L.moe_select_exemplar(FAKE, 5000, FAKE, 1, 0, None, FAKE, None, None) == 2     # E > 4096
    assert L.moe_select_exemplar(FAKE, 8, FAKE, 2000, 0, None, FAKE, None, None) == 2     # n > 1024
    assert L.moe_select_exemplar(FAKE, 8, FAKE, 1, 0, None, None, None, None) == 1        # tactic NULL
    t = [mb.MG_BF16, FAKE, None, FAKE, None, FAKE, FAKE, 8, 1024, 256, 256, 16, None, None, None]
    assert L.mgemm_contiguous_tactic(*t) == 1                                              # tactic NULL
    assert L.mgemm_masked_tactic(mb.MG_BF16, FAKE, None, FAKE, None, FAKE, FAKE, 8, 64, 256, 256, None,
                                 None, None) == 1
    m = [mb.MG_BF16, FAKE, None, FAKE, None, FAKE, FAKE, 8, 64, 256, 256]
    assert L.mgemm_masked_exemplar(*m, None, 4, None, None, None) == 1                     # table NULL
    assert L.mgemm_masked_exemplar(*m, FAKE, 0, None, None, None) == 1                     # n
    assert L.mgemm_masked_exemplar(*m, FAKE, 2000, None, None, None) == 2                  # n > 1024
    m[7] = 33
    assert L.mgemm_masked_exemplar(*m, FAKE, 4, None, None, None) == 2                     # E > 32
