"""Benchmark of the MoE grouped GEMM hot path on GB300.

A step is one pass of the path over one batch of synthetic input: the
device plan (padded offsets and stats at the layout alignment), the device
token-tile choice and the grouped GEMMs, all through the C ABI of
libmoegemm.so.  The headline workload is the skewed FP8 prefill: 64 experts,
32768 token-expert assignments drawn from a Zipf(1.2) law over a seeded
expert permutation, GEMM1 N=4096 K=7168 then GEMM2 N=7168 K=2048, E4M3
operands with UE8M0 per-128 block scales.

Every other workload of the benchmark set is measured in the same run and
reported under "configs": the 8-expert near-uniform example, the 32-expert
issue histogram, the masked FP8 decode, the skewed prefill in FP8 and BF16,
the K-grouped weight gradient, and the FP8 x FP4 decode and fused-SwiGLU FFN
variants.  Each config record carries its effective and physical
throughput, the padding accounting at the chosen tile, the roofline (the
slower of the useful flops at the dense tensor peak and the algorithmic
bytes at HBM bandwidth) and the CPU oracle timed on a bounded sample.

Timing: L2 is flushed between timed repetitions by writing a buffer of twice
the L2 size, outside the CUDA events that bracket each step.

Metric: effective TFLOP/s, counting only valid token rows
(2 * U * N * K per GEMM), the whole job over all ranks.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU runs are independent replicas, one per rank (torchrun).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_grouped_gemm_side_gb300 import workloads as wl  # noqa: E402

HEADLINE = "prefill_fp8_e64_t32768_n4096_k7168"
# the benchmark set reported under "configs", in order
CONFIGS = [
    "contig_bf16_e8_n256_k256",
    "contig_bf16_e32_n4096_k2048",
    "masked_fp8_e16_m256_n4096_k7168",
    "prefill_fp8_e64_t32768_n4096_k7168",
    "prefill_bf16_e64_t32768_n4096_k7168",
    "kgrouped_bf16_e32_t65536_n4096_k2048",
    "masked_fp8xfp4_e16_m256_n4096_k7168",
    "prefill_ffn_fp8_e64_t32768_n4096_k7168",
]
FP8_OVER_BF16 = 2.0   # nominal dense fp8 : bf16 tensor throughput ratio
METRIC = "effective TFLOPS (valid rows only)"
L2_NOTE = ("L2 flushed between timed reps: 2 x l2CacheSize bytes written, 2 x l2CacheSize bytes of another "
           "buffer read (the written lines go back to HBM before the rep), then a ~0.2 ms GPU spin, all outside "
           "the CUDA events")


def _binding():
    """The C-ABI binding; imported only by the GPU arm (the reference arm
    loads no part of the library)."""
    from moe_grouped_gemm_side_gb300 import binding
    return binding


# ------------------------------------------------------------------ helpers
def ptr(t):
    return None if t is None else t.data_ptr()


# DRAM bytes per step measured by ncu (dram__bytes_read.sum +
# dram__bytes_write.sum over the step's GEMM launches), valid only for the
# kernel sources they were taken with.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
KERNEL_SOURCES = {
    "fwd": ["gemm_fwd.cu", "common.cuh", "sched.cuh"],
    "kg": ["gemm_kgrouped.cu", "common.cuh"],
}


def kernel_sources_sha(kind):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "moe_grouped_gemm_side_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(workload, kind):
    """ncu DRAM bytes of one step of `workload`, or None when none were taken
    with the current kernel sources."""
    try:
        with open(TRAFFIC_FILE) as fh:
            rec = json.load(fh).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("sources_sha256") != kernel_sources_sha(kind):
        return None
    return rec.get("bytes_per_step")


def traffic_fields(workload, kind, alg_bytes_per_step, launches):
    """The dominant kernel's ncu DRAM bytes beside its algorithmic bytes, per
    launch (the step's launches averaged, like `achieved`) and per step;
    traffic is None when no capture matches the current kernel sources."""
    t = measured_traffic(workload, kind)
    return {"traffic": None if t is None else t / launches, "traffic_per_step": t,
            "algorithmic_bytes_per_launch": alg_bytes_per_step / launches,
            "launches_per_step": launches}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def roofline_record(flops, byts, ms, tensor_peak, peaks, peak_label, tr):
    """Roofline of one timed launch set: the bound is whichever of the useful
    flops at the tensor peak and the algorithmic bytes at HBM bandwidth
    takes longer; `achieved` and `frac` are in that bound's unit."""
    t_compute = flops / (tensor_peak * 1e12)
    t_mem = byts / (peaks["hbm_gbs"] * 1e9)
    common = {"flops": flops, "algorithmic_bytes": byts, "t_compute_us": t_compute * 1e6,
              "t_mem_us": t_mem * 1e6, **tr}
    if t_compute >= t_mem:
        ach = flops / (ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": tensor_peak, "unit": "TFLOP/s",
                "frac": ach / tensor_peak, **common, "peak_source": peak_label}
    ach = byts / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": ach / peaks["hbm_gbs"], **common, "peak_source": f"{peaks['source']} copy"}


class ClockSampler:
    """nvidia-smi clock / throttle samples with host timestamps."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        """Median SM clock over the samples of [t0, t1] taken under load
        (utilisation >= 50 %; all samples of the window if none was), the
        maximum clock, board power and every throttle reason seen."""
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        win = [s for (t, s) in self.samples if t0 - 0.3 <= t <= t1 + 0.3 and len(s) >= 9]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4) if s[4 + i].lower() == "active"})
        loaded = [s for s in win if (num(s[8]) or 0.0) >= 50.0]
        use = loaded or win
        sm = [v for v in (num(s[0]) for s in use) if v is not None]
        mx = [v for v in (num(s[1]) for s in win) if v is not None]
        pw = [v for v in (num(s[2]) for s in win) if v is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(win),
                "samples_under_load": len(loaded)}


def dist_setup():
    """One process per GPU (torchrun env).  The ranks are independent
    replicas; the only collectives are the timing barrier and the max of the
    timed spans (NCCL on GPUs, gloo without)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(units_per_rank, ws, ms_max):
    """Whole-job throughput: the units every rank processed over the slowest
    rank's span (per-rank work fixed as ranks are added)."""
    return ws * units_per_rank / (ms_max * 1e-3)


def operands_label(fp8, w4):
    if w4:
        return "e4m3 + ue8m0 per (row, 128 K) x e2m1 weights + ue8m0 per (row, 32 K)"
    return "e4m3 + ue8m0 per-128 scales" if fp8 else "bf16"


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


# ------------------------------------------------------------------ workloads
class Workload:
    """What a workload is (histogram, shapes, dtype), independent of where its
    operands live.  `attach_gpu` builds the device operands for the library;
    `attach_cpu` makes the host copies the oracle reads, drawn lazily per
    expert.  `oracle_sample` times the oracle on some experts either way."""

    def __init__(self, name):
        spec = wl.WORKLOADS[name]
        self.name, self.spec = name, spec
        self.form = spec["form"]
        self.dtype_name = spec["dtype"]
        self.fp8 = spec["dtype"] in ("fp8", "fp8xfp4")
        self.w4 = spec["dtype"] == "fp8xfp4"
        self.elem = 1 if self.fp8 else 2
        self.counts = spec["counts"]()
        self.E = spec["E"]
        self.U = sum(self.counts)
        self.active = sum(1 for t in self.counts if t > 0)
        self.swiglu = bool(spec.get("swiglu", False))
        shapes = [(spec["N"], spec["K"])]
        if "second" in spec:
            shapes.append((spec["second"]["N"], spec["second"]["K"]))
        self.gemms = [dict(N=N, K=K, swiglu=self.swiglu and i == 0) for i, (N, K) in enumerate(shapes)]
        self.host = None

    # ---- pure accounting
    def flops(self):
        return sum(2.0 * self.U * g["N"] * g["K"] for g in self.gemms)

    def bytes_alg(self, g):
        """Algorithmic bytes of one GEMM: weights (and scales) of active
        experts, valid activation rows (and scales), valid output rows."""
        N, K = g["N"], g["K"]
        if self.form == "kgrouped":
            return self.U * (N + K) * 2 + self.E * N * K * 4
        act = self.active
        out = self.U * (N // 2 + N // 256) if g["swiglu"] else self.U * N * 2   # E4M3 Y + scales, or bf16 D
        w = act * (N * K // 2 + N * K // 32) if self.w4 else act * N * K * self.elem
        b = w + self.U * K * self.elem + out
        if self.fp8:
            b += self.U * (K // 128) + (0 if self.w4 else act * (K // 128) * (N // 128))
        return b

    def bytes_alg_total(self):
        return sum(self.bytes_alg(g) for g in self.gemms)

    def launches_per_step(self):
        return (1 if self.form == "contiguous" else 0) + len(self.gemms)

    def tensor_peak(self, peaks):
        return peaks["bf16_tflops"] * (FP8_OVER_BF16 if self.fp8 else 1.0)

    def roofline(self, per_gemm_ms, peaks):
        kind = "kg" if self.form == "kgrouped" else "fwd"
        byts = self.bytes_alg_total()
        tr = traffic_fields(self.name, kind, byts, len(self.gemms))
        label = f"{peaks['source']} bf16 burst x{FP8_OVER_BF16 if self.fp8 else 1.0:g}"
        return roofline_record(self.flops(), byts, sum(per_gemm_ms), self.tensor_peak(peaks), peaks, label, tr)

    def config(self):
        """The workload's description; identical in both arms."""
        d = {"workload": self.name, "form": self.form, "experts": self.E,
             "operands": operands_label(self.fp8, self.w4) if self.form != "kgrouped" else "bf16 in, fp32 dW",
             "l2": L2_NOTE}
        if self.form == "contiguous":
            d.update(assignments=self.U, align_q=self.spec["align_q"], tile_q="device-selected",
                     gemms=[f"N={g['N']},K={g['K']}" for g in self.gemms])
        elif self.form == "masked":
            d.update(M_max=self.spec["M_max"], valid_rows=self.U, N=self.spec["N"], K=self.spec["K"],
                     tile_q="device-selected")
        else:
            d.update(tokens=self.U, N=self.spec["N"], K=self.spec["K"])
        if self.swiglu:
            d["epilogue"] = "GEMM1: SwiGLU of interleaved gate/up blocks, re-quantised to e4m3 + ue8m0; feeds GEMM2"
        return d

    # ---- device operands (GPU arm)
    def attach_gpu(self, mb, dev):
        self.mb = mb
        spec = self.spec
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.d_counts = torch.tensor(self.counts, dtype=torch.int32, device=dev)
        self.dtype = (mb.MG_FP8_X_FP4_E2M1 if self.w4 else mb.MG_FP8_E4M3_UE8M0) if self.fp8 else mb.MG_BF16
        if self.form == "contiguous":
            self.align = spec["align_q"]
            _, _, st, code = mb.plan_host(self.counts, self.align, max_tiles=0)
            assert code == 0
            self.rows_cap = (st.P + 15) // 16 * 16
            for i, g in enumerate(self.gemms):
                seed = spec["seed"] + 100 * i
                ops = wl.make_contiguous(self.E, self.rows_cap, g["N"], g["K"], spec["dtype"], seed, dev,
                                         spec["a_std"] if i == 0 else 1.0, spec["b_std"] if i == 0 else 1.0)
                A, SFA = ops.A, ops.SFA
                if self.swiglu and i == 1:
                    A, SFA = self.gemms[0]["D"], self.gemms[0]["SFD"]      # GEMM1's output
                if g["swiglu"]:
                    D = torch.empty((self.rows_cap, g["N"] // 2), dtype=torch.uint8, device=dev)
                    SFD = torch.empty((g["N"] // 256, self.rows_cap), dtype=torch.uint8, device=dev)
                else:
                    D, SFD = torch.empty((self.rows_cap, g["N"]), dtype=torch.bfloat16, device=dev), None
                g.update(A=A, B=ops.B, SFA=SFA, SFB=ops.SFB, D=D, SFD=SFD)
            self.offsets = torch.empty(self.E + 1, dtype=torch.int64, device=dev)
            self.stats = torch.empty(48, dtype=torch.uint8, device=dev)
        elif self.form == "masked":
            M, N, K = spec["M_max"], spec["N"], spec["K"]
            ops = wl.make_masked(self.E, M, N, K, spec["dtype"], spec["seed"], dev)
            self.gemms[0].update(A=ops.A, B=ops.B, SFA=ops.SFA, SFB=ops.SFB,
                                 D=torch.empty((self.E, M, N), dtype=torch.bfloat16, device=dev))
        else:
            N, K, T = spec["N"], spec["K"], spec["T"]
            dY, X = wl.make_kgrouped(T, N, K, spec["seed"], dev)
            self.gemms[0].update(dY=dY, X=X, dW=torch.empty((self.E, N, K), dtype=torch.float32, device=dev))
        return self

    def step(self, lib, stream, ev=None):
        """One pass: (contiguous) the device plan, then each GEMM; ev[i] =
        (start, end) events around GEMM i."""
        import ctypes
        s = ctypes.c_void_p(stream.cuda_stream)
        mb = self.mb
        if self.form == "contiguous":
            rc = lib.moe_plan(ptr(self.d_counts), self.E, self.align, ptr(self.offsets), None, 0,
                              ptr(self.stats), ptr(self.status), s)
            assert rc == 0, rc
        for i, g in enumerate(self.gemms):
            if ev is not None:
                ev[i][0].record(stream)
            if self.form == "kgrouped":
                rc = lib.kgemm_grouped(ptr(g["dY"]), ptr(g["X"]), ptr(g["dW"]), ptr(self.d_counts), self.E,
                                       self.spec["T"], g["N"], g["K"], ptr(self.status), s)
            elif self.form == "masked":
                rc = lib.mgemm_masked(self.dtype, ptr(g["A"]), ptr(g["SFA"]), ptr(g["B"]), ptr(g["SFB"]),
                                      ptr(g["D"]), ptr(self.d_counts), self.E, self.spec["M_max"], g["N"], g["K"],
                                      ptr(self.status), s)
            elif g["swiglu"]:
                rc = lib.mgemm_contiguous_swiglu(self.dtype, mb.MG_SWIGLU_FP8_E4M3_UE8M0, ptr(g["A"]),
                                                 ptr(g["SFA"]), ptr(g["B"]), ptr(g["SFB"]), ptr(g["D"]),
                                                 ptr(g["SFD"]), ptr(self.d_counts), self.E, self.rows_cap,
                                                 g["N"], g["K"], self.align, 0, ptr(self.status), s)
            else:
                rc = lib.mgemm_contiguous(self.dtype, ptr(g["A"]), ptr(g["SFA"]), ptr(g["B"]), ptr(g["SFB"]),
                                          ptr(g["D"]), ptr(self.d_counts), self.E, self.rows_cap, g["N"], g["K"],
                                          self.align, 0, ptr(self.status), s)
            assert rc == 0, rc
            if ev is not None:
                ev[i][1].record(stream)

    def check_status(self):
        code = int(self.status.item())
        if code != 0:
            raise RuntimeError(f"{self.name}: device status " + self.mb.status_str(code))

    # end-to-end: inputs from pinned host memory, outputs back to pinned host
    def e2e_setup(self):
        self.h_in = [(self.d_counts, self.d_counts.cpu().pin_memory())]
        keys = ("dY", "X") if self.form == "kgrouped" else ("A", "SFA")
        for i, g in enumerate(self.gemms):
            if self.swiglu and i == 1:
                continue                      # produced on the device by GEMM1
            for k in keys:
                if g.get(k) is not None:
                    self.h_in.append((g[k], g[k].cpu().pin_memory()))
        out_key = "dW" if self.form == "kgrouped" else "D"
        outs = [self.gemms[-1]] if self.swiglu else self.gemms
        self.h_out = [(g[out_key], torch.empty(g[out_key].shape, dtype=g[out_key].dtype).pin_memory())
                      for g in outs]
        return (sum(h.numel() * h.element_size() for _, h in self.h_in),
                sum(h.numel() * h.element_size() for _, h in self.h_out))

    def e2e_step(self, lib, stream):
        for d, h in self.h_in:
            d.copy_(h, non_blocking=True)
        self.step(lib, stream)
        for d, h in self.h_out:
            h.copy_(d, non_blocking=True)

    def tactics(self, per_gemm_ms):
        if self.form == "kgrouped":
            return None
        return [tactic_report(self.mb, self.dtype, self.counts, g["N"], g["K"], t)
                for g, t in zip(self.gemms, per_gemm_ms)]

    # ---- host operands for the oracle
    def attach_cpu(self):
        """Host operands drawn with the workload's own seeded generators on
        the CPU: activations whole, weights one expert at a time on first
        use.  (Draws on the CPU and on the GPU follow the same recipe but not
        the same random stream.)"""
        from oracle import plan as op
        spec = self.spec
        self.host = {"w": {}}
        if self.form == "contiguous":
            rows_cap = (op.plan(self.counts, spec["align_q"]).P + 15) // 16 * 16
            self.host["rows"] = []
            for i, g in enumerate(self.gemms):
                if self.swiglu and i == 1:
                    self.host["rows"].append(None)       # GEMM1's output, made by the oracle
                    continue
                A, SFA = wl.make_rows(rows_cap, g["K"], "bf16" if not self.fp8 else "fp8",
                                      spec["seed"] + 100 * i, "cpu", spec["a_std"] if i == 0 else 1.0)
                self.host["rows"].append((A, SFA))
        elif self.form == "masked":
            M, K = spec["M_max"], spec["K"]
            A2, SFA2 = wl.make_rows(self.E * M, K, "fp8" if self.fp8 else "bf16", spec["seed"], "cpu")
            SFA = None if SFA2 is None else SFA2.reshape(K // 128, self.E, M).permute(1, 0, 2).contiguous()
            self.host["rows"] = [(A2.reshape(self.E, M, K), SFA)]
        else:
            self.host["rows"] = [wl.make_kgrouped(spec["T"], spec["N"], spec["K"], spec["seed"], "cpu")]
        return self

    def _host_weight(self, i, e):
        key = (i, e)
        if key not in self.host["w"]:
            g, spec = self.gemms[i], self.spec
            seed = (spec["seed"] + 100 * i if self.form == "contiguous" else spec["seed"]) + 1
            std = spec.get("b_std", 1.0) if i == 0 else 1.0
            self.host["w"][key] = wl.expert_weight(e, g["N"], g["K"], self.dtype_name, seed, "cpu", std)
        return self.host["w"][key]

    def _rows(self, i, e, lo, hi):
        """Activation rows [lo, hi) of GEMM i (expert e for the masked form)
        and their scale columns, on the host."""
        if self.host is not None:
            A, SFA = self.host["rows"][i]
        else:
            g = self.gemms[i]
            A, SFA = g["A"], g["SFA"]
        if self.form == "masked":
            a = A[e, lo:hi]
            sf = None if SFA is None else SFA[e][:, lo:hi]
        else:
            a = A[lo:hi]
            sf = None if SFA is None else SFA[:, lo:hi]
        return a.cpu(), (None if sf is None else sf.cpu())

    def _weight(self, i, e):
        if self.host is not None:
            return self._host_weight(i, e)
        g = self.gemms[i]
        return g["B"][e].cpu(), (None if g["SFB"] is None else g["SFB"][e].cpu())

    def oracle_sample(self, experts):
        """The oracle (plan + fp64 dequantisation + per-expert GEMMs) on the
        given experts; returns (useful flops, seconds).  Operand copies to
        the host are made before the clock starts."""
        from oracle import epilogue as oe
        from oracle import gemm as og
        from oracle import numerics as on
        from oracle import plan as op
        if self.form == "kgrouped":
            return self._oracle_sample_kg(experts)
        align = self.spec.get("align_q", 1)
        offs = op.plan(self.counts, align).offsets if self.form == "contiguous" else None
        # host copies first (not timed)
        staged = []
        for e in experts:
            t = self.counts[e]
            if t == 0:
                continue
            lo = offs[e] if offs is not None else 0
            per = []
            for i in range(len(self.gemms)):
                rows = None if (self.swiglu and i == 1) else self._rows(i, e, lo, lo + t)
                per.append((rows, self._weight(i, e)))
            staged.append((e, t, per))
        t0 = time.perf_counter()
        if self.form == "contiguous":
            op.plan(self.counts, align)
        useful = 0.0
        for e, t, per in staged:
            prev = None
            for g, (rows, (b, sfb)) in zip(self.gemms, per):
                if prev is not None:
                    a = prev                    # GEMM2 reads GEMM1's re-quantised SwiGLU output
                elif self.fp8:
                    a = on.dequant_rows(rows[0].numpy(), rows[1].numpy())
                else:
                    a = on.decode_bf16(rows[0].view(torch.int16).numpy().view(np.uint16))
                if self.fp8:
                    deq_w = on.dequant_weight_mx4 if self.w4 else on.dequant_weight
                    bw = deq_w(b.numpy(), sfb.numpy())
                else:
                    bw = on.decode_bf16(b.view(torch.int16).numpy().view(np.uint16))
                r = og.expert_product(a, bw)
                if g["swiglu"]:
                    codes, sf = oe.quantize_blocks(oe.swiglu(*oe.gate_up_halves(r)))
                    prev = on.dequant_rows(codes, sf)
                useful += 2.0 * t * g["N"] * g["K"]
        return useful, time.perf_counter() - t0

    def _oracle_sample_kg(self, experts):
        from oracle import gemm as og
        from oracle import numerics as on
        off = np.concatenate([[0], np.cumsum(self.counts)])
        if self.host is not None:
            dY, X = self.host["rows"][0]
        else:
            dY, X = self.gemms[0]["dY"], self.gemms[0]["X"]
        staged = []
        for e in experts:
            a, b = int(off[e]), int(off[e + 1])
            if b > a:
                staged.append((dY[a:b].cpu(), X[a:b].cpu()))
        t0 = time.perf_counter()
        useful = 0.0
        for dy, x in staged:
            n = dy.shape[0]
            og.kgrouped(on.decode_bf16(dy.view(torch.int16).numpy().view(np.uint16)),
                        on.decode_bf16(x.view(torch.int16).numpy().view(np.uint16)), [n])
            useful += 2.0 * n * self.spec["N"] * self.spec["K"]
        return useful, time.perf_counter() - t0

    def sample_steps(self):
        if self.swiglu:
            return "plan + fp64 dequantise + per-expert GEMM1, SwiGLU, E4M3 re-quantisation, GEMM2"
        if self.form == "kgrouped":
            return "fp64 decode + per-expert dY^T X"
        return "plan + fp64 dequantise + per-expert GEMMs" if self.form == "contiguous" else \
            "fp64 dequantise + per-expert GEMMs"


def tactic_report(mb, dtype, counts, N, K, ms):
    """The token tile the kernel picks on the device for this histogram (the
    same pricing on the host), the pages' padded rows P at that tile, the rows
    the kernel actually computes (each expert's last tile trimmed to a
    multiple of 16) and the physical throughput they imply: the pages'
    (2 P N K / t) and the computed rows' (2 R N K / t)."""
    q = mb.select_tile_host(dtype, counts, N, K, 0)
    offs, _, st, code = mb.plan_host(counts, q, max_tiles=0)
    assert code == 0
    computed = 0
    for t in counts:
        if t > 0:
            full, last = divmod(t, q)
            computed += full * q + (-(-last // 16) * 16 if last else 0)
    return {"N": N, "K": K, "tile_q": q, "P_at_tile": st.P, "U": st.U, "pad_frac_at_tile": st.pad_frac,
            "rows_computed": computed, "active_experts": st.active, "effective_experts": st.eff_experts,
            "physical_tflops": 2.0 * st.P * N * K / (ms * 1e-3) / 1e12,
            "computed_rows_tflops": 2.0 * computed * N * K / (ms * 1e-3) / 1e12}


def oracle_sample_bounded(w, budget_s):
    """The oracle on a bounded sample: active experts in index order, one at
    a time, until about `budget_s` seconds of CPU work have been spent.
    Returns (experts, useful flops, seconds)."""
    experts, useful, secs = [], 0.0, 0.0
    for e, t in enumerate(w.counts):
        if not t:
            continue
        u, s = w.oracle_sample([e])
        experts.append(e)
        useful += u
        secs += s
        if secs >= budget_s:
            break
    return experts, useful, secs


def cpu_baseline(w, budget_s):
    experts, useful, secs = oracle_sample_bounded(w, budget_s)
    return {"value": useful / secs / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"experts {experts} of {w.name}: {w.sample_steps()}, "
                      f"{useful / 1e9:.2f} useful GFLOP in {secs:.2f} s"}


class E2EPipeline:
    """End-to-end steps through the C ABI with host buffers, two sets of
    device inputs and outputs in flight: step i's inputs are copied in
    (pinned host -> device) on one stream while step i-1's GEMMs run, and step
    i-1's outputs are copied out on a third stream while step i's GEMMs run.
    Every step still moves all of its own inputs in and all of its results
    out, inside the timed region.  (Splitting the copies over four streams
    per direction measured no faster: the device-to-host copies run at
    ~175 GB/s either way.)"""

    def __init__(self, w, compute_stream):
        self.w, self.cs = w, compute_stream
        self.bi, self.bo = w.e2e_setup()
        self.ins, self.outs = torch.cuda.Stream(), torch.cuda.Stream()
        # set 0: the workload's own device tensors; set 1: copies of the ones
        # the transfers touch (inputs and results), weights shared
        m1 = {}
        for d, _ in w.h_in + w.h_out:
            if id(d) not in m1:
                m1[id(d)] = d.clone()   # rows a call never writes match set 0's
        self.sets = []
        for m in (None, m1):
            sub = (lambda t: t) if m is None else (lambda t: m.get(id(t), t) if t is not None else t)
            gemms = [{k: (sub(v) if isinstance(v, torch.Tensor) else v) for k, v in g.items()} for g in w.gemms]
            self.sets.append({"gemms": gemms, "counts": sub(w.d_counts),
                              "h_in": [(sub(d), h) for d, h in w.h_in],
                              "h_out": [(sub(d), h) for d, h in w.h_out]})
        self.base = (w.gemms, w.d_counts)
        self.ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "comp", "out")}
        self.used = [False, False]
        self.i = 0

    def begin(self):
        """Orders the copy streams after everything queued on the compute
        stream so far (e.g. the start event)."""
        e = torch.cuda.Event()
        e.record(self.cs)
        self.ins.wait_event(e)
        self.outs.wait_event(e)

    def step(self, lib):
        s = self.i & 1
        st = self.sets[s]
        if self.used[s]:
            self.ins.wait_event(self.ev["comp"][s])      # step i-2 has read this set's inputs
        with torch.cuda.stream(self.ins):
            for d, h in st["h_in"]:
                d.copy_(h, non_blocking=True)
        self.ev["in"][s].record(self.ins)
        self.cs.wait_event(self.ev["in"][s])
        if self.used[s]:
            self.cs.wait_event(self.ev["out"][s])        # step i-2's results have left this set
        self.w.gemms, self.w.d_counts = st["gemms"], st["counts"]
        self.w.step(lib, self.cs)
        self.ev["comp"][s].record(self.cs)
        self.outs.wait_event(self.ev["comp"][s])
        with torch.cuda.stream(self.outs):
            for d, h in st["h_out"]:
                h.copy_(d, non_blocking=True)
        self.ev["out"][s].record(self.outs)
        self.used[s] = True
        self.i += 1

    def end(self):
        """The compute stream waits for every copy still in flight."""
        for s in (0, 1):
            if self.used[s]:
                self.cs.wait_event(self.ev["out"][s])

    def close(self):
        self.w.gemms, self.w.d_counts = self.base
        self.w.h_in = self.w.h_out = None
        self.sets = None


class L2Flush:
    """Between timed repetitions: writes 2 x l2CacheSize bytes, so every rep
    reads its operands from HBM; then reads 2 x l2CacheSize bytes of a second
    buffer, so the written lines are written back to HBM here rather than
    while the next rep runs (the write-back of the flush's own dirty lines is
    not the GEMM's cost); then the GPU spins ~0.2 ms, so the host has queued
    the next start event and launch before the GPU reaches them (a short
    GEMM's host-side preparation otherwise lands inside its events)."""

    SETTLE_CYCLES = 400_000

    def __init__(self, dev):
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.bytes = 2 * int(l2)
        self.buf = torch.empty(self.bytes, dtype=torch.uint8, device=dev)
        self.clean = torch.ones(self.bytes // 4, dtype=torch.int32, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self):
        self.buf.fill_(1)
        torch.sum(self.clean, dim=0, out=self.sink)
        torch.cuda._sleep(self.SETTLE_CYCLES)


def timed_reps(w, lib, stream, flush, reps):
    """`reps` steps, each after an L2 flush, each GEMM bracketed by CUDA
    events; returns per-rep lists of per-GEMM milliseconds."""
    n_g = len(w.gemms)
    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(n_g)]
           for _ in range(reps)]
    for i in range(reps):
        flush()
        w.step(lib, stream, evs[i])
    torch.cuda.synchronize()
    return [[evs[i][g][0].elapsed_time(evs[i][g][1]) for g in range(n_g)] for i in range(reps)]


def exemplar_table_path(w):
    """The tuned exemplar table of a masked workload's shape, if there is one."""
    sp = w.spec
    if sp.get("form") != "masked":
        return None
    name = f"{sp['dtype']}_masked_e{w.E}_m{sp['M_max']}_n{sp['N']}_k{sp['K']}.json"
    path = os.path.join(ROOT, "moe_grouped_gemm_side_gb300", "exemplars", name)
    return path if os.path.exists(path) else None


def selector_record(w, stream, flush, reps):
    """Masked decode: the exemplar selector's choice (select kernel + tactic
    GEMM, both timed) next to every fixed tactic; the built-in cost model's
    time is the record's own ms_per_step."""
    path = exemplar_table_path(w)
    if path is None:
        return None
    mb = w.mb
    with open(path) as f:
        meta = json.load(f)
    table = mb.exemplar_table(meta["exemplars"])
    dev = w.d_counts.device
    d_table = mb.exemplar_table_device(table, device=dev)
    g = w.gemms[0]
    tactic = torch.zeros(3, dtype=torch.int32, device=dev)

    def run_tactic():
        mb.mgemm_masked_tactic(g["A"], g["B"], g["D"], w.d_counts, tactic, SFA=g["SFA"], SFB=g["SFB"],
                               status=w.status, stream=stream)

    def run_selected():
        mb.select_exemplar(w.d_counts, d_table, len(table), tactic, status=w.status, stream=stream)
        run_tactic()

    fused_tactic = torch.zeros(3, dtype=torch.int32, device=dev)

    def run_fused():
        mb.mgemm_masked_exemplar(g["A"], g["B"], g["D"], w.d_counts, d_table, len(table), SFA=g["SFA"],
                                 SFB=g["SFB"], tactic_out=fused_tactic, status=w.status, stream=stream)

    def median_ms(fn):
        for _ in range(3):
            flush()
            fn()
        ts = []
        for _ in range(reps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return sorted(ts)[len(ts) // 2]

    ex_ms = median_ms(run_selected)
    chosen = tactic.cpu().tolist()
    fused_ms = median_ms(run_fused) if w.E <= 32 else None
    fused = fused_tactic.cpu().tolist()
    fixed = {}
    for cand in meta["candidates"]:
        tq, blocks = (int(x) for x in cand.split("x"))
        tactic.copy_(torch.tensor([tq, blocks, 0], dtype=torch.int32))
        fixed[cand] = median_ms(run_tactic)
    w.check_status()
    best = min(fixed, key=fixed.get)
    return {"table": os.path.relpath(path, ROOT), "table_default": meta.get("default"),
            "exemplar": {"tactic": f"{chosen[0]}x{chosen[1]}", "index": chosen[2], "ms": ex_ms,
                         "path": "select kernel + tactic GEMM"},
            "exemplar_in_gemm": None if fused_ms is None else {
                "tactic": f"{fused[0]}x{fused[1]}", "index": fused[2], "ms": fused_ms,
                "path": "mgemm_masked_exemplar (choice in the GEMM prologue)"},
            "fixed_ms": fixed, "best_fixed": best,
            "exemplar_vs_best_fixed": (fused_ms if fused_ms is not None else ex_ms) / fixed[best]}


def config_record(w, lib, stream, flush, peaks, args, cpu=None):
    """One entry of "configs": warm-up, then the median of `reps` L2-flushed
    steps (each GEMM between its own events), with the roofline, the tactic
    and padding accounting, and the oracle's CPU baseline."""
    for _ in range(5):
        flush()
        w.step(lib, stream)
    torch.cuda.synchronize()
    w.check_status()
    per_rep = timed_reps(w, lib, stream, flush, args.reps)
    w.check_status()
    tot = [sum(r) for r in per_rep]
    med_i = sorted(range(len(tot)), key=lambda i: tot[i])[len(tot) // 2]
    per_gemm = per_rep[med_i]
    ms = tot[med_i]
    tac = w.tactics(per_gemm)
    rec = {"value": w.flops() / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
           "ms_mean": sum(tot) / len(tot), "ms_min": min(tot), "reps": args.reps,
           "per_gemm_ms": per_gemm, "useful_flops": w.flops(), "U": w.U,
           "active_experts": w.active, "config": w.config(), "l2": L2_NOTE,
           "roofline": w.roofline(per_gemm, peaks), "tactics": tac}
    if tac:
        rec["physical_tflops"] = sum(2.0 * t["P_at_tile"] * t["N"] * t["K"] for t in tac) / (ms * 1e-3) / 1e12
        rec["computed_rows_tflops"] = sum(2.0 * t["rows_computed"] * t["N"] * t["K"] for t in tac) / (ms * 1e-3) / 1e12
        rec["P_at_tile"] = [t["P_at_tile"] for t in tac]
        rec["pad_frac_at_tile"] = [t["pad_frac_at_tile"] for t in tac]
        rec["effective_experts"] = tac[0]["effective_experts"]
    sel = selector_record(w, stream, flush, args.reps)
    if sel is not None:
        sel["cost_model_ms"] = ms
        rec["selector"] = sel
    if cpu is None and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.config_cpu_budget)
    rec["cpu_baseline"] = cpu
    return rec


# ------------------------------------------------------------------ arms
def run_ours(args):
    ws, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    mb = _binding()
    lib = mb.load()
    mb.set_kernel_policy(mb.POLICIES[args.kernel_policy])
    w = Workload(args.workload).attach_gpu(mb, dev)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    flush = L2Flush(dev)

    for _ in range(args.warmup):
        flush()
        w.step(lib, stream)
    torch.cuda.synchronize()
    w.check_status()

    n_g = len(w.gemms)
    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(n_g)]
           for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.6)
    # soak: the same steps back to back for `--soak` seconds right before the
    # timed region, so the clock record holds samples taken under this load
    t_soak0 = time.time()
    while True:
        for _ in range(max(3, args.warmup)):
            flush()
            w.step(lib, stream)
        torch.cuda.synchronize()
        if time.time() - t_soak0 >= args.soak:
            break
    barrier(ws)
    torch.cuda.synchronize()
    t_host0 = time.time()
    for i in range(args.steps):
        flush()
        w.step(lib, stream, evs[i])
    torch.cuda.synchronize()
    t_host1 = time.time()
    barrier(ws)
    per_step = [sum(evs[i][g][0].elapsed_time(evs[i][g][1]) for g in range(n_g)) for i in range(args.steps)]
    ms = sum(per_step)
    ms_max = max_over_ranks(ms, ws)
    per_gemm = [sum(evs[i][g][0].elapsed_time(evs[i][g][1]) for i in range(args.steps)) / args.steps
                for g in range(n_g)]
    w.check_status()
    value = weak_scaling_value(w.flops() * args.steps, ws, ms_max) / 1e12

    # end to end: host buffers in, results back to host, same step count
    e2e = None
    if not args.no_e2e:
        pipe = E2EPipeline(w, stream)
        pipe.begin()
        for _ in range(2):
            pipe.step(lib)
        pipe.end()
        barrier(ws)
        torch.cuda.synchronize()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n2 = max(3, min(args.steps, 20))
        s2.record(stream)
        pipe.begin()
        for _ in range(n2):
            pipe.step(lib)
        pipe.end()
        e2.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        w.check_status()
        ms2 = max_over_ranks(s2.elapsed_time(e2), ws)
        e2e = {"value": weak_scaling_value(w.flops() * n2, ws, ms2) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": pipe.bi, "d2h_bytes_per_step": pipe.bo, "steps": n2,
               "ms_per_step": ms2 / n2,
               "pipelining": "two buffer sets: step i's host->device copies and step i-1's device->host "
                             "copies on their own streams, overlapping the GEMMs"}
        pipe.close()

    roof = w.roofline(per_gemm, peaks)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_budget)

    configs, t_cfg0, t_cfg1 = None, None, None
    if rank == 0 and not args.no_configs:
        configs = {}
        t_cfg0 = time.time()
        for name in CONFIGS:
            if name == w.name:
                cw = w
            else:
                cw = Workload(name).attach_gpu(mb, dev)
            configs[name] = config_record(cw, lib, stream, flush, peaks, args,
                                          cpu=cpu if cw is w else None)
            if cw is not w:
                del cw
                torch.cuda.empty_cache()
        t_cfg1 = time.time()
    time.sleep(0.3)
    sampler.stop()
    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ("e4m3xe2m1" if w.w4 else "e4m3") if w.fp8 else "bf16",
        "data": "synthetic",
        "config": w.config(),
        "kernel_policy": args.kernel_policy,
        "per_gemm_ms": per_gemm,
        "tactics": w.tactics(per_gemm),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": w.launches_per_step() * args.steps,
        "clocks": dict(sampler.summary(t_soak0, t_host1), window="soak of the same steps + timed region",
                       soak_s=round(t_host0 - t_soak0, 2), timed_s=round(t_host1 - t_host0, 3)),
    }
    if configs is not None:
        line["configs"] = configs
        line["clocks_configs"] = sampler.summary(t_cfg0, t_cfg1)
    print(json.dumps(line))


def run_reference(args):
    """The oracle on the host cores, one rotating active expert per step of
    the same workload and config as the GPU arm; loads no part of the
    CUDA library."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = Workload(args.workload).attach_cpu()
    active = [e for e, t in enumerate(w.counts) if t]
    total_u, total_s = 0.0, 0.0
    for i in range(args.warmup + args.steps):
        u, s = w.oracle_sample([active[i % len(active)]])
        if i >= args.warmup:
            total_u += u
            total_s += s
    value = total_u / total_s / 1e12
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_s * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": w.config(),
        "kernel_policy": args.kernel_policy,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"one active expert per step (rotating) of {args.workload}: "
                                   f"{w.sample_steps()}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config records")
    ap.add_argument("--reps", type=int, default=20, help="timed L2-flushed reps per config record")
    ap.add_argument("--soak", type=float, default=1.0,
                    help="seconds of back-to-back steps right before the timed region (clock record)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--config-cpu-budget", type=float, default=5.0,
                    help="seconds of oracle work for each config record's cpu_baseline")
    ap.add_argument("--kernel-policy", choices=["auto", "single", "dual", "pair", "pair_dual"], default="auto",
                    help="grouped GEMM kernel family (auto: the library's default per shape)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
