"""Host-side pieces of bench.py that need no GPU: the tactic report (tile the
device prices, the pages' P at it, rows the kernel computes) against the
oracle's plan, and the binding's choice of the FP8 x FP4 dtype from operand
shapes."""
import numpy as np
import pytest
import torch

import bench
from moe_grouped_gemm_side_gb300 import binding as mb
from moe_grouped_gemm_side_gb300 import workloads as wl
from oracle import plan as op

pytestmark = pytest.mark.cpu


@pytest.mark.parametrize("counts", [wl.counts_zipf_decode(), wl.counts_uniformish(), wl.counts_issue32(),
                                    [0, 0, 0], [1, 15, 16, 17, 239, 240, 241]])
def test_tactic_report_against_the_oracle_plan(lib, counts):
    r = bench.tactic_report(mb, mb.MG_FP8_E4M3_UE8M0, counts, 4096, 7168, 1.0)
    q = r["tile_q"]
    assert q == mb.select_tile_host(mb.MG_FP8_E4M3_UE8M0, counts, 4096, 7168, 0)
    ref = op.plan(counts, q)
    assert (r["P_at_tile"], r["U"], r["active_experts"]) == (ref.P, ref.U, ref.active)
    # full tiles of q rows, the last tile of each expert trimmed to a multiple of 16
    rows = sum((t // q) * q + (-(-(t % q) // 16) * 16) for t in counts)
    assert r["rows_computed"] == rows
    assert r["U"] <= r["rows_computed"] <= r["P_at_tile"]
    # physical throughput as the pages define it (padded rows P), and of the rows computed
    assert r["physical_tflops"] == pytest.approx(2.0 * ref.P * 4096 * 7168 / 1e-3 / 1e12)
    assert r["computed_rows_tflops"] == pytest.approx(2.0 * rows * 4096 * 7168 / 1e-3 / 1e12)


def test_fp4_dtype_is_read_from_the_weight_shape():
    A = torch.zeros((32, 512), dtype=torch.uint8)
    assert mb._fwd_dtype(A, torch.zeros((2, 256, 256), dtype=torch.uint8), 512) == mb.MG_FP8_X_FP4_E2M1
    assert mb._fwd_dtype(A, torch.zeros((2, 256, 512), dtype=torch.uint8), 512) == mb.MG_FP8_E4M3_UE8M0
    assert mb._fwd_dtype(torch.zeros((32, 512), dtype=torch.bfloat16),
                         torch.zeros((2, 256, 512), dtype=torch.bfloat16), 512) == mb.MG_BF16


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the contract's keys and the GPU arm's config, on a small
    workload, without loading any part of the CUDA library."""
    import json
    import subprocess
    import sys
    from tests.conftest import ROOT
    probe = (
        "import runpy, sys\n"
        "sys.argv = ['bench.py', '--impl', 'reference', '--workload', 'contig_bf16_e8_n256_k256',"
        " '--steps', '2', '--warmup', '3']\n"
        "runpy.run_path('bench.py', run_name='__main__')\n"
        "maps = open('/proc/self/maps').read()\n"
        "print('LOADED', 'libmoegemm' in maps, 'moe_grouped_gemm_side_gb300.binding' in sys.modules)\n")
    r = subprocess.run([sys.executable, "-c", probe], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == "contig_bf16_e8_n256_k256"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"] == bench.Workload("contig_bf16_e8_n256_k256").config()
    assert "LOADED False False" in r.stdout


@pytest.mark.parametrize("name", bench.CONFIGS)
def test_host_operands_follow_the_workload_recipe(name):
    """The reference arm's host operands have the shapes and dtypes of the
    GPU arm's, and its per-expert weights are the same draws the full
    weight tensor makes (one seeded draw per expert)."""
    w = bench.Workload(name)
    spec = wl.WORKLOADS[name]
    if w.form == "kgrouped":
        w.spec = dict(spec, T=300, N=256, K=128)
        w.counts = [100, 0, 200]
        w.attach_cpu()
        dY, X = w.host["rows"][0]
        assert dY.shape == (300, 256) and X.shape == (300, 128) and dY.dtype == torch.bfloat16
        return
    e = next(i for i, t in enumerate(w.counts) if t)
    w.gemms[0].update(N=256, K=512)          # small shapes, same recipe
    w.host = {"w": {}}
    b, sfb = w._host_weight(0, e)
    full_b, full_sfb = wl.make_weights(e + 1, 256, 512, w.dtype_name, spec["seed"] + 1, "cpu",
                                       spec.get("b_std", 1.0))
    assert torch.equal(b, full_b[e])
    assert (sfb is None and full_sfb is None) or torch.equal(sfb, full_sfb[e])


def test_exemplar_tuner_guardrail():
    """The tuner keeps the default tactic unless another beats it by more
    than the margin; the default is the best geometric mean over the tuning
    sweeps; its histograms have the stated totals and respect M_max."""
    from moe_grouped_gemm_side_gb300 import tune_exemplars as te
    t = {"240x2": 100.0, "16x1": 98.0, "32x2": 101.0}
    assert te.pick_tactic(t, "240x2", 0.03) == "240x2"           # 2 % better: not enough
    assert te.pick_tactic(dict(t, **{"16x1": 96.0}), "240x2", 0.03) == "16x1"
    assert te.pick_tactic({"256x2": 10.0, "64x2": 9.0}, "256x2", 0.03) == "64x2"
    sweeps = [{"a": 1.0, "b": 2.0}, {"a": 4.0, "b": 1.0}, {"a": 1.0, "b": 1.5}]
    assert te.default_tactic(sweeps) == "b"                       # geomeans 1.59 vs 1.44
    sweeps[1]["a"] = 2.0
    assert te.default_tactic(sweeps) == "a"                       # 1.26 vs 1.44
    assert te.default_tactic([{"a": 2.0, "b": 1.0}]) == "b"
    for U in (32, 1024, 32768):
        for i, (shape, param) in enumerate(te.SHAPES):
            c = te.histogram(shape, param, 64, U, seed=2000 + 37 * i + U)
            assert len(c) == 64 and sum(c) == U and min(c) >= 0
    for held_out in (False, True):
        for label, c in te.decode_histograms(16, 256, held_out):
            assert len(c) == 16 and max(c) <= 256 and sum(1 for x in c if x == 0) >= 3
    for U in te.U_TUNE["masked"] + te.U_EVAL["masked"]:
        for i, (shape, param) in enumerate(te.SHAPES):
            c = te.histogram(shape, param, 16, U, seed=9000 + 53 * i + U, cap=256)
            assert len(c) == 16 and sum(c) == U and 0 <= min(c) and max(c) <= 256


def test_exemplar_table_only_for_masked_shapes():
    """The bench's selector record looks for a tuned table of the masked
    decode shape only; the committed one is there."""
    assert bench.exemplar_table_path(bench.Workload("prefill_fp8_e64_t32768_n4096_k7168")) is None
    assert bench.exemplar_table_path(bench.Workload("kgrouped_bf16_e32_t65536_n4096_k2048")) is None
    p = bench.exemplar_table_path(bench.Workload("masked_fp8_e16_m256_n4096_k7168"))
    assert p is not None and p.endswith("fp8_masked_e16_m256_n4096_k7168.json")
    assert bench.exemplar_table_path(bench.Workload("masked_fp8xfp4_e16_m256_n4096_k7168")) is None


PEAKS = {"hbm_gbs": 6789.6, "bf16_tflops": 1869.1, "source": "measured"}


@pytest.mark.parametrize("case", ["prefill", "masked", "kgrouped"])
def test_roofline_traffic_is_per_launch(case):
    """roofline.traffic is the ncu DRAM bytes of one launch (the step's
    launches averaged) beside the algorithmic bytes of one launch; the
    per-step figure and the launch count come with it."""
    import json
    import os
    if case == "prefill":
        name = "prefill_fp8_e64_t32768_n4096_k7168"
        r, launches, kind = bench.Workload(name).roofline([0.84, 0.48], PEAKS), 2, "fwd"
    elif case == "masked":
        name = "masked_fp8_e16_m256_n4096_k7168"
        r, launches, kind = bench.Workload(name).roofline([0.0927], PEAKS), 1, "fwd"
    else:
        name = "kgrouped_bf16_e32_t65536_n4096_k2048"
        w = bench.Workload(name)
        r, launches, kind = w.roofline([0.787], PEAKS), 1, "kg"
        assert w.bytes_alg_total() == 65536 * (4096 + 2048) * 2 + 32 * 4096 * 2048 * 4
    assert r["launches_per_step"] == launches
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f).get(name)
    if rec and rec["sources_sha256"] == bench.kernel_sources_sha(kind):
        assert rec["launches"] == launches
        assert r["traffic_per_step"] == rec["bytes_per_step"]
        assert r["traffic"] == pytest.approx(rec["bytes_per_step"] / launches)
        # operands come from DRAM about once: traffic within 20 % of the
        # algorithmic bytes (a little below them where part of the output is
        # still in the write-back L2 when the kernel ends)
        assert 0.9 <= r["traffic"] / r["algorithmic_bytes_per_launch"] < 1.2
    else:
        assert r["traffic"] is None and r["traffic_per_step"] is None


@pytest.mark.parametrize("name", bench.CONFIGS)
def test_roofline_bound_is_the_slower_of_compute_and_memory(name):
    """Every form, the masked one included, is scored against whichever of
    the useful flops at the tensor peak and the algorithmic bytes at HBM
    bandwidth takes longer, and frac = that time / the measured time."""
    w = bench.Workload(name)
    ms = 1.0
    r = w.roofline([ms / len(w.gemms)] * len(w.gemms), PEAKS)
    peak = PEAKS["bf16_tflops"] * (2.0 if w.fp8 else 1.0)
    t_c = w.flops() / (peak * 1e12)
    t_m = w.bytes_alg_total() / (PEAKS["hbm_gbs"] * 1e9)
    assert r["bound"] == ("tensor" if t_c >= t_m else "hbm")
    assert r["frac"] == pytest.approx(max(t_c, t_m) / (ms * 1e-3))


def test_masked_roofline_turns_tensor_bound_when_rows_fill_the_buffers():
    """A masked decode whose buffers are full does enough work per weight
    byte to be bound by the tensor peak, not by HBM."""
    w = bench.Workload("masked_fp8_e16_m256_n4096_k7168")
    assert w.roofline([0.1], PEAKS)["bound"] == "hbm"
    w.counts = [256] * 16
    w.U, w.active = 4096, 16
    peaks = dict(PEAKS, hbm_gbs=20000.0)
    assert w.roofline([0.1], peaks)["bound"] == "tensor"


def test_traffic_is_null_once_kernel_sources_change(monkeypatch):
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda kind: "0" * 64)
    f = bench.traffic_fields("prefill_fp8_e64_t32768_n4096_k7168", "fwd", 3.86e9, 2)
    assert f["traffic"] is None and f["traffic_per_step"] is None
    assert f["algorithmic_bytes_per_launch"] == pytest.approx(1.93e9)
