"""Offline tuning of the exemplar table, and its evaluation, on the GPU.

"MoE GroupGEMM padding under expert skew", "Padding is not the whole cost
model" and "Build a routing-shaped benchmark": candidates that share a tile
can differ by more than 10 %, so the table is measured, not derived from the
padding formula; the benchmark covers low-token decode buckets and broad and
concentrated histograms at the same token count U.

Tuning: for each histogram of a seeded set (U from 32 to 32768 assignments,
Dirichlet shares from concentrated to broad, Zipf ranks), every candidate
(token tile x weight blocks per tile) runs the contiguous grouped GEMM
through ``mgemm_contiguous_tactic``.  The histogram becomes one exemplar (its
features from ``moe_exemplar_features_host``) whose tactic is the default
(the widest tile, two blocks) unless the fastest candidate beats it by more
than ``--min-gain``: many candidates finish within the run-to-run spread of
each other, and a table of near-ties would carry that noise to neighbouring
histograms.

Evaluation, on histograms drawn with other seeds: the latency of the
exemplar choice, of the built-in cost-model choice (tile_q = 0), and of
fixed tactics, each relative to the fastest candidate for that histogram;
and, on a walk of neighbouring histograms, how often the choice switches
with and without the hysteresis margin.

Usage (writes the table and a summary):
    python -m moe_grouped_gemm_side_gb300.tune_exemplars --dtype fp8 --N 4096 --K 7168 \\
        --out moe_grouped_gemm_side_gb300/exemplars/fp8_e64_n4096_k7168.json
    python -m moe_grouped_gemm_side_gb300.tune_exemplars --evaluate TABLE.json
"""
import argparse
import json
import math
import os
import time

import numpy as np
import torch

from . import binding as mb
from . import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
TILES = {"fp8": (16, 32, 64, 128, 240), "bf16": (16, 32, 64, 128, 256)}
U_TUNE = (32, 64, 128, 256, 512, 1024, 2048, 4096, 8192, 16384, 32768)
U_EVAL = (32, 48, 64, 96, 200, 1024, 1500, 3000, 6000, 12000, 24000, 32768)
SHAPES = (("dirichlet", 0.2), ("dirichlet", 1.0), ("dirichlet", 8.0), ("zipf", 1.2), ("zipf", 0.6))


def histogram(shape, param, E, U, seed):
    if shape == "dirichlet":
        return wl.counts_dirichlet(seed=seed, E=E, total=U, alpha=param)
    return wl.counts_zipf_prefill(seed=seed, E=E, total=U, s=param)


class Bench:
    """Operands sized for the largest histogram; each call times one tactic."""

    def __init__(self, dtype, E, N, K, max_rows, dev="cuda", align=16):
        self.dtype, self.E, self.N, self.K, self.align, self.dev = dtype, E, N, K, align, dev
        self.rows_cap = (max_rows + E * align + 15) // 16 * 16
        ops = wl.make_contiguous(E, self.rows_cap, N, K, dtype, 77, dev)
        self.A, self.B, self.SFA, self.SFB = ops.A, ops.B, ops.SFA, ops.SFB
        self.D = torch.empty((self.rows_cap, N), dtype=torch.bfloat16, device=dev)
        self.tactic = torch.zeros(3, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # larger than L2

    def _time(self, fn, reps):
        for _ in range(2):
            fn()
        ts = []
        for _ in range(reps):
            self.flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        return float(np.median(ts))

    def time_tactic(self, d_counts, tq, blocks, reps=9):
        self.tactic.copy_(torch.tensor([tq, blocks, 0], dtype=torch.int32))
        return self._time(lambda: mb.mgemm_contiguous_tactic(
            self.A, self.B, self.D, d_counts, self.align, self.tactic, SFA=self.SFA, SFB=self.SFB,
            status=self.status), reps)

    def time_builtin(self, d_counts, reps=9):
        return self._time(lambda: mb.mgemm_contiguous(
            self.A, self.B, self.D, d_counts, self.align, SFA=self.SFA, SFB=self.SFB, status=self.status), reps)

    def sweep(self, counts):
        d_counts = torch.tensor(counts, dtype=torch.int32, device=self.dev)
        times = {}
        for tq in TILES[self.dtype]:
            for blocks in (1, 2):
                times[f"{tq}x{blocks}"] = self.time_tactic(d_counts, tq, blocks)
        assert int(self.status.item()) == 0
        return times, d_counts


def pick_tactic(times, dtype, min_gain):
    """The tactic an exemplar keeps: the default (widest tile, two blocks)
    unless the fastest candidate beats it by more than min_gain."""
    best = min(times, key=times.get)
    default = f"{TILES[dtype][-1]}x2"
    return best if times[best] < times[default] * (1.0 - min_gain) else default


def tune(args):
    bench = Bench(args.dtype, args.E, args.N, args.K, max(U_TUNE))
    exemplars = []
    for U in U_TUNE:
        for i, (shape, param) in enumerate(SHAPES):
            counts = histogram(shape, param, args.E, U, seed=2000 + 37 * i + U)
            times, _ = bench.sweep(counts)
            best = min(times, key=times.get)
            default = f"{TILES[args.dtype][-1]}x2"
            pick = pick_tactic(times, args.dtype, args.min_gain)
            tq, blocks = (int(x) for x in pick.split("x"))
            lu, shares = mb.exemplar_features_host(counts)
            exemplars.append({"lu": lu, "shares": shares, "tile_q": tq, "blocks": blocks, "U": U,
                              "shape": f"{shape}({param})", "counts": counts, "times_us": times})
            print(f"U={U:6d} {shape}({param}): best {best} {times[best]:.1f} us, default {times[default]:.1f} us"
                  f" -> {pick}", flush=True)
    out = {"dtype": args.dtype, "E": args.E, "N": args.N, "K": args.K, "align_q": bench.align,
           "min_gain": args.min_gain,
           "candidates": [f"{t}x{b}" for t in TILES[args.dtype] for b in (1, 2)],
           "exemplars": exemplars}
    os.makedirs(os.path.dirname(os.path.abspath(args.out)), exist_ok=True)
    with open(args.out, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", args.out)


def load_table(path):
    with open(path) as f:
        t = json.load(f)
    return t, mb.exemplar_table(t["exemplars"])


def evaluate(args):
    meta, table = load_table(args.evaluate)
    entries = meta["exemplars"]
    bench = Bench(meta["dtype"], meta["E"], meta["N"], meta["K"], max(U_EVAL))
    d_table = mb.exemplar_table_device(table)
    rows = []
    for U in U_EVAL:
        for i, (shape, param) in enumerate(SHAPES):
            counts = histogram(shape, param, meta["E"], U, seed=9000 + 53 * i + U)   # held out
            times, d_counts = bench.sweep(counts)
            best = min(times.values())
            mb.select_exemplar(d_counts, d_table, len(table), bench.tactic, status=bench.status)
            torch.cuda.synchronize()
            tq, blocks, idx = bench.tactic.cpu().tolist()
            t_ex = times[f"{tq}x{blocks}"]
            t_cm = bench.time_builtin(d_counts)
            lu, shares = mb.exemplar_features_host(counts)
            rows.append({"U": U, "shape": f"{shape}({param})", "best_us": best, "best": min(times, key=times.get),
                         "exemplar": f"{tq}x{blocks}", "exemplar_us": t_ex, "costmodel_us": t_cm,
                         "fixed_us": {k: times[k] for k in ("240x2" if meta["dtype"] == "fp8" else "256x2", "32x1")},
                         "eff_experts": (sum(counts) ** 2 / max(1, sum(c * c for c in counts)))})
            r = rows[-1]
            print(f"U={U:6d} {r['shape']:15s} best {r['best']:6s} {best:8.1f}  exemplar {r['exemplar']:6s} "
                  f"{t_ex:8.1f}  cost model {t_cm:8.1f}", flush=True)

    def geo(key):
        return math.exp(np.mean([math.log(r[key] / r["best_us"]) for r in rows]))
    fixed_keys = list(rows[0]["fixed_us"])
    summary = {"histograms": len(rows), "geomean_vs_best": {
        "exemplar": geo("exemplar_us"), "cost_model": geo("costmodel_us"),
        **{f"fixed_{k}": math.exp(np.mean([math.log(r["fixed_us"][k] / r["best_us"]) for r in rows]))
           for k in fixed_keys}}}
    # hysteresis: a walk of neighbouring histograms around two bases
    state = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(17)
    walk = {}
    for margin in (0, 30000):
        switches, prev = 0, -1
        state.fill_(-1)
        for base_U in (1024, 8192):
            base = np.array(histogram("dirichlet", 1.0, meta["E"], base_U, seed=31))
            for _ in range(40):
                c = np.maximum(0, base + rng.integers(-base.max() // 20 - 1, base.max() // 20 + 2, size=base.size))
                mb.select_exemplar(torch.tensor(c.tolist(), dtype=torch.int32, device="cuda"), d_table, len(table),
                                   bench.tactic, margin=margin, d_state=state)
                torch.cuda.synchronize()
                idx = int(bench.tactic[2].item())
                switches += idx != prev
                prev = idx
        walk[str(margin)] = switches
    summary["choice_switches_over_80_neighbouring_histograms"] = walk
    out = {"table": args.evaluate, "rows": rows, "summary": summary}
    with open(args.report, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps(summary, indent=1))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--dtype", default="fp8", choices=["fp8", "bf16"])
    ap.add_argument("--E", type=int, default=64)
    ap.add_argument("--N", type=int, default=4096)
    ap.add_argument("--K", type=int, default=7168)
    ap.add_argument("--out", default=os.path.join(HERE, "exemplars", "fp8_e64_n4096_k7168.json"))
    ap.add_argument("--min-gain", type=float, default=0.03,
                    help="a tactic other than the default must be this much faster to enter the table")
    ap.add_argument("--evaluate", default=None, help="evaluate this table instead of tuning")
    ap.add_argument("--report", default="exemplar_eval.json")
    args = ap.parse_args()
    if not torch.cuda.is_available():
        raise SystemExit("needs a GPU")
    mb.load()
    t0 = time.time()
    if args.evaluate:
        evaluate(args)
    else:
        tune(args)
    print(f"{time.time() - t0:.0f} s")


if __name__ == "__main__":
    main()
