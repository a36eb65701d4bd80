"""Benchmark of the MoE grouped GEMM hot path on GB300.

A step is one pass of the path over one batch of synthetic input: the
device plan (padded offsets and stats at the layout alignment), the device
token-tile choice and the grouped GEMMs, all through the C ABI of
libmoegemm.so.  The headline workload is the skewed FP8 prefill: 64 experts,
32768 token-expert assignments drawn from a Zipf(1.2) law over a seeded
expert permutation, GEMM1 N=4096 K=7168 then GEMM2 N=7168 K=2048, E4M3
operands with UE8M0 per-128 block scales.  Other workloads (--workload) are
parity cases that can be measured the same way.

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

from moe_grouped_gemm_side_gb300 import binding as mb  # noqa: E402
from moe_grouped_gemm_side_gb300 import workloads as wl  # noqa: E402

HEADLINE = "prefill_fp8_e64_t32768_n4096_k7168"
FP8_OVER_BF16 = 2.0   # nominal dense fp8 : bf16 tensor throughput ratio


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


class ClockSampler:
    """nvidia-smi clock / throttle samples with host timestamps."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

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
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        win = [s for (t, s) in self.samples if t0 - 0.3 <= t <= t1 + 0.3 and len(s) >= 8]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4) if s[4 + i].lower() == "active"})
        sm = [v for v in (num(s[0]) for s in win) if v is not None]
        mx = [v for v in (num(s[1]) for s in win) if v is not None]
        pw = [v for v in (num(s[2]) for s in win) if v is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(win)}


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


# ------------------------------------------------------------------ workloads
class Contiguous:
    """Plan + one or two contiguous grouped GEMMs over the same histogram."""

    def __init__(self, name, dev):
        spec = wl.WORKLOADS[name]
        self.name, self.spec, self.dev = name, spec, dev
        self.fp8 = spec["dtype"] in ("fp8", "fp8xfp4")
        self.w4 = spec["dtype"] == "fp8xfp4"      # E2M1 weights, one scale per (row, 32 K)
        self.counts = spec["counts"]()
        self.E = spec["E"]
        self.align = spec["align_q"]
        offs, _, st, code = mb.plan_host(self.counts, self.align, max_tiles=0)
        assert code == 0
        self.U = st.U
        self.rows_cap = (st.P + 15) // 16 * 16
        shapes = [(spec["N"], spec["K"])]
        if "second" in spec:
            shapes.append((spec["second"]["N"], spec["second"]["K"]))
        # swiglu: GEMM1's epilogue applies SwiGLU to interleaved gate/up blocks and
        # re-quantises (E4M3 + UE8M0), and GEMM2 consumes that output (K = N1/2)
        self.swiglu = bool(spec.get("swiglu", False))
        self.gemms = []
        for i, (N, K) in enumerate(shapes):
            seed = spec["seed"] + 100 * i
            ops = wl.make_contiguous(self.E, self.rows_cap, N, K, spec["dtype"], seed, dev,
                                     spec["a_std"] if i == 0 else 1.0, spec["b_std"] if i == 0 else 1.0)
            A, SFA = ops.A, ops.SFA
            if self.swiglu and i == 1:
                A, SFA = self.gemms[0]["D"], self.gemms[0]["SFD"]      # GEMM1's output
            if self.swiglu and i == 0:
                D = torch.empty((self.rows_cap, N // 2), dtype=torch.uint8, device=dev)
                SFD = torch.empty((N // 256, self.rows_cap), dtype=torch.uint8, device=dev)
            else:
                D, SFD = torch.empty((self.rows_cap, N), dtype=torch.bfloat16, device=dev), None
            self.gemms.append(dict(N=N, K=K, A=A, B=ops.B, SFA=SFA, SFB=ops.SFB, D=D, SFD=SFD,
                                   swiglu=self.swiglu and i == 0))
        self.d_counts = torch.tensor(self.counts, dtype=torch.int32, device=dev)
        self.offsets = torch.empty(self.E + 1, dtype=torch.int64, device=dev)
        self.stats = torch.empty(48, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.dtype = mb.MG_FP8_X_FP4_E2M1 if self.w4 else (mb.MG_FP8_E4M3_UE8M0 if self.fp8 else mb.MG_BF16)
        self.elem = 1 if self.fp8 else 2

    def flops(self):
        return sum(2.0 * self.U * g["N"] * g["K"] for g in self.gemms)

    def bytes_alg(self, g):
        """Algorithmic bytes of one GEMM: weights of active experts (+scales),
        valid activation rows (+scales), valid output rows."""
        act = sum(1 for t in self.counts if t > 0)
        N, K = g["N"], g["K"]
        out = self.U * (N // 2 + N // 256) if g["swiglu"] else self.U * N * 2   # E4M3 Y + scales, or bf16 D
        w = act * (N * K // 2 + N * K // 32) if self.w4 else act * N * K * self.elem
        b = w + self.U * K * self.elem + out
        if self.fp8:
            b += self.U * (K // 128) + (0 if self.w4 else act * (K // 128) * (N // 128))
        return b

    def launches_per_step(self):
        return 1 + len(self.gemms)

    def step(self, lib, stream, ev=None):
        s = ctypes_stream(stream)
        rc = lib.moe_plan(ptr(self.d_counts), self.E, self.align, ptr(self.offsets), None, 0,
                          ptr(self.stats), ptr(self.status), s)
        assert rc == 0, rc
        for i, g in enumerate(self.gemms):
            if ev is not None:
                ev[i][0].record(stream)
            if g["swiglu"]:
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

    # end-to-end: inputs from pinned host memory, outputs back to pinned host
    def e2e_setup(self):
        self.h_in = [(self.d_counts, self.d_counts.cpu().pin_memory())]
        for i, g in enumerate(self.gemms):
            if self.swiglu and i == 1:
                continue                      # produced on the device by GEMM1
            for k in ("A", "SFA"):
                if g[k] is not None:
                    self.h_in.append((g[k], g[k].cpu().pin_memory()))
        outs = [self.gemms[-1]] if self.swiglu else self.gemms
        self.h_out = [(g["D"], torch.empty(g["D"].shape, dtype=g["D"].dtype).pin_memory()) for g in outs]
        return (sum(h.numel() * h.element_size() for _, h in self.h_in),
                sum(h.numel() * h.element_size() for _, h in self.h_out))

    def e2e_step(self, lib, stream):
        for d, h in self.h_in:
            d.copy_(h, non_blocking=True)
        self.step(lib, stream)
        for d, h in self.h_out:
            h.copy_(d, non_blocking=True)

    def roofline(self, per_gemm_ms, peaks):
        flops = sum(2.0 * self.U * g["N"] * g["K"] for g in self.gemms)
        ms = sum(per_gemm_ms)
        byts = sum(self.bytes_alg(g) for g in self.gemms)
        tensor_peak = peaks["bf16_tflops"] * (FP8_OVER_BF16 if self.fp8 else 1.0)
        t_compute = flops / (tensor_peak * 1e12)
        t_mem = byts / (peaks["hbm_gbs"] * 1e9)
        tr = traffic_fields(self.name, "fwd", byts, len(self.gemms))
        if t_compute >= t_mem:
            ach = flops / (ms * 1e-3) / 1e12
            return {"bound": "tensor", "achieved": ach, "peak": tensor_peak, "unit": "TFLOP/s",
                    "frac": ach / tensor_peak, **tr,
                    "peak_source": f"{peaks['source']} bf16 burst x{FP8_OVER_BF16 if self.fp8 else 1.0:g}"}
        ach = byts / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], **tr, "peak_source": f"{peaks['source']} copy"}

    def config(self):
        d = {"workload": self.name, "form": "contiguous", "experts": self.E, "assignments": self.U,
             "align_q": self.align, "rows_cap": self.rows_cap, "tile_q": "device-selected",
             "gemms": [f"N={g['N']},K={g['K']}" for g in self.gemms],
             "operands": operands_label(self.fp8, self.w4),
             "l2": "inputs larger than L2 (no flush)"}
        if self.swiglu:
            d["epilogue"] = "GEMM1: SwiGLU of interleaved gate/up blocks, re-quantised to e4m3 + ue8m0; feeds GEMM2"
        return d

    # ---- CPU oracle on a bounded sample (experts given by index)
    def oracle_sample(self, experts):
        from oracle import gemm as og
        from oracle import numerics as on
        from oracle import plan as op
        from oracle import epilogue as oe
        host = []
        for g in self.gemms:
            host.append({k: (g[k].cpu() if g[k] is not None else None) for k in ("A", "SFA")})
        t0 = time.perf_counter()
        p = op.plan(self.counts, self.align)
        useful = 0.0
        for e in experts:
            t = self.counts[e]
            if t == 0:
                continue
            o = p.offsets[e]
            prev = None
            for g, h in zip(self.gemms, host):
                if prev is not None:
                    a = prev                    # GEMM2 reads GEMM1's re-quantised SwiGLU output
                elif self.fp8:
                    a = on.dequant_rows(h["A"][o:o + t].numpy(), h["SFA"][:, o:o + t].numpy())
                else:
                    a = on.decode_bf16(h["A"][o:o + t].view(torch.int16).numpy().view(np.uint16))
                if self.fp8:
                    deq_w = on.dequant_weight_mx4 if self.w4 else on.dequant_weight
                    b = deq_w(g["B"][e].cpu().numpy(), g["SFB"][e].cpu().numpy())
                else:
                    b = on.decode_bf16(g["B"][e].cpu().view(torch.int16).numpy().view(np.uint16))
                r = og.expert_product(a, b)
                if g["swiglu"]:
                    codes, sf = oe.quantize_blocks(oe.swiglu(*oe.gate_up_halves(r)))
                    prev = on.dequant_rows(codes, sf)
                useful += 2.0 * t * g["N"] * g["K"]
        return useful, time.perf_counter() - t0


class Masked:
    def __init__(self, name, dev):
        spec = wl.WORKLOADS[name]
        self.name, self.spec = name, spec
        self.fp8 = spec["dtype"] in ("fp8", "fp8xfp4")
        self.w4 = spec["dtype"] == "fp8xfp4"      # E2M1 weights, one scale per (row, 32 K)
        self.E, self.M, self.N, self.K = spec["E"], spec["M_max"], spec["N"], spec["K"]
        self.counts = spec["counts"]()
        self.U = sum(self.counts)
        ops = wl.make_masked(self.E, self.M, self.N, self.K, spec["dtype"], spec["seed"], dev)
        self.A, self.B, self.SFA, self.SFB = ops.A, ops.B, ops.SFA, ops.SFB
        self.D = torch.empty((self.E, self.M, self.N), dtype=torch.bfloat16, device=dev)
        self.d_counts = torch.tensor(self.counts, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.dtype = mb.MG_FP8_X_FP4_E2M1 if self.w4 else (mb.MG_FP8_E4M3_UE8M0 if self.fp8 else mb.MG_BF16)
        self.elem = 1 if self.fp8 else 2
        self.gemms = [dict(N=self.N, K=self.K)]

    def flops(self):
        return 2.0 * self.U * self.N * self.K

    def launches_per_step(self):
        return 1

    def bytes_alg(self):
        act = sum(1 for t in self.counts if t > 0)
        N, K = self.N, self.K
        w = act * (N * K // 2 + N * K // 32) if self.w4 else act * N * K * self.elem
        b = w + self.U * K * self.elem + self.U * N * 2
        if self.fp8:
            b += self.U * (K // 128) + (0 if self.w4 else act * (K // 128) * (N // 128))
        return b

    def step(self, lib, stream, ev=None):
        if ev is not None:
            ev[0][0].record(stream)
        rc = lib.mgemm_masked(self.dtype, ptr(self.A), ptr(self.SFA), ptr(self.B), ptr(self.SFB), ptr(self.D),
                              ptr(self.d_counts), self.E, self.M, self.N, self.K, ptr(self.status),
                              ctypes_stream(stream))
        assert rc == 0, rc
        if ev is not None:
            ev[0][1].record(stream)

    def e2e_setup(self):
        self.h_in = [(self.d_counts, self.d_counts.cpu().pin_memory()), (self.A, self.A.cpu().pin_memory())]
        if self.SFA is not None:
            self.h_in.append((self.SFA, self.SFA.cpu().pin_memory()))
        self.h_out = [(self.D, torch.empty(self.D.shape, dtype=self.D.dtype).pin_memory())]
        return (sum(h.numel() * h.element_size() for _, h in self.h_in),
                sum(h.numel() * h.element_size() for _, h in self.h_out))

    def e2e_step(self, lib, stream):
        for d, h in self.h_in:
            d.copy_(h, non_blocking=True)
        self.step(lib, stream)
        for d, h in self.h_out:
            h.copy_(d, non_blocking=True)

    def roofline(self, per_gemm_ms, peaks):
        ms = sum(per_gemm_ms)
        ach = self.bytes_alg() / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], **traffic_fields(self.name, "fwd", self.bytes_alg(), 1),
                "peak_source": f"{peaks['source']} copy"}

    def config(self):
        return {"workload": self.name, "form": "masked", "experts": self.E, "M_max": self.M,
                "valid_rows": self.U, "N": self.N, "K": self.K,
                "operands": operands_label(self.fp8, self.w4),
                "l2": "inputs larger than L2 (no flush)"}

    def oracle_sample(self, experts):
        from oracle import gemm as og
        from oracle import numerics as on
        t0 = time.perf_counter()
        useful = 0.0
        for e in experts:
            v = self.counts[e]
            if v == 0:
                continue
            if self.fp8:
                a = on.dequant_rows(self.A[e, :v].cpu().numpy(), self.SFA[e][:, :v].cpu().numpy())
                deq_w = on.dequant_weight_mx4 if self.w4 else on.dequant_weight
                b = deq_w(self.B[e].cpu().numpy(), self.SFB[e].cpu().numpy())
            else:
                a = on.decode_bf16(self.A[e, :v].cpu().view(torch.int16).numpy().view(np.uint16))
                b = on.decode_bf16(self.B[e].cpu().view(torch.int16).numpy().view(np.uint16))
            og.expert_product(a, b)
            useful += 2.0 * v * self.N * self.K
        return useful, time.perf_counter() - t0


class KGrouped:
    def __init__(self, name, dev):
        spec = wl.WORKLOADS[name]
        self.name = name
        self.E, self.N, self.K, self.T = spec["E"], spec["N"], spec["K"], spec["T"]
        self.counts = spec["counts"]()
        self.U = sum(self.counts)
        self.dY, self.X = wl.make_kgrouped(self.T, self.N, self.K, spec["seed"], dev)
        self.dW = torch.empty((self.E, self.N, self.K), dtype=torch.float32, device=dev)
        self.d_counts = torch.tensor(self.counts, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.fp8 = False
        self.gemms = [dict(N=self.N, K=self.K)]

    def flops(self):
        return 2.0 * self.U * self.N * self.K

    def launches_per_step(self):
        return 1

    def step(self, lib, stream, ev=None):
        if ev is not None:
            ev[0][0].record(stream)
        rc = lib.kgemm_grouped(ptr(self.dY), ptr(self.X), ptr(self.dW), ptr(self.d_counts), self.E, self.T,
                               self.N, self.K, ptr(self.status), ctypes_stream(stream))
        assert rc == 0, rc
        if ev is not None:
            ev[0][1].record(stream)

    def e2e_setup(self):
        self.h_in = [(self.d_counts, self.d_counts.cpu().pin_memory()), (self.dY, self.dY.cpu().pin_memory()),
                     (self.X, self.X.cpu().pin_memory())]
        self.h_out = [(self.dW, torch.empty(self.dW.shape, dtype=self.dW.dtype).pin_memory())]
        return (sum(h.numel() * h.element_size() for _, h in self.h_in),
                sum(h.numel() * h.element_size() for _, h in self.h_out))

    def e2e_step(self, lib, stream):
        for d, h in self.h_in:
            d.copy_(h, non_blocking=True)
        self.step(lib, stream)
        for d, h in self.h_out:
            h.copy_(d, non_blocking=True)

    def bytes_alg(self):
        """Valid dY and X rows read once, every expert's fp32 dW written once."""
        return self.U * (self.N + self.K) * 2 + self.E * self.N * self.K * 4

    def roofline(self, per_gemm_ms, peaks):
        ach = self.flops() / (sum(per_gemm_ms) * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops"], **traffic_fields(self.name, "kg", self.bytes_alg(), 1),
                "peak_source": f"{peaks['source']} bf16 burst"}

    def config(self):
        return {"workload": self.name, "form": "kgrouped", "experts": self.E, "tokens": self.U,
                "N": self.N, "K": self.K, "operands": "bf16 in, fp32 dW",
                "l2": "inputs larger than L2 (no flush)"}

    def oracle_sample(self, experts):
        from oracle import gemm as og
        from oracle import numerics as on
        off = np.concatenate([[0], np.cumsum(self.counts)])
        t0 = time.perf_counter()
        useful = 0.0
        for e in experts:
            a, b = int(off[e]), int(off[e + 1])
            if b == a:
                continue
            cnt = [0] * self.E
            cnt[e] = b - a
            dy = on.decode_bf16(self.dY[a:b].cpu().view(torch.int16).numpy().view(np.uint16))
            x = on.decode_bf16(self.X[a:b].cpu().view(torch.int16).numpy().view(np.uint16))
            og.kgrouped(dy, x, [b - a])
            useful += 2.0 * (b - a) * self.N * self.K
        return useful, time.perf_counter() - t0


def make_workload(name, dev):
    form = wl.WORKLOADS[name]["form"]
    return {"contiguous": Contiguous, "masked": Masked, "kgrouped": KGrouped}[form](name, dev)


def ctypes_stream(stream):
    import ctypes
    return ctypes.c_void_p(stream.cuda_stream)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def tactic_report(dtype, counts, N, K, ms):
    """The token tile the kernel picks on the device for this histogram (the
    same pricing on the host), the pages' padded rows P at that tile, the rows
    the kernel actually computes (each expert's last tile trimmed to a
    multiple of 16) and the physical throughput they imply."""
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
            "physical_tflops": 2.0 * computed * N * K / (ms * 1e-3) / 1e12}


def operands_label(fp8, w4):
    if w4:
        return "e4m3 + ue8m0 per (row, 128 K) x e2m1 weights + ue8m0 per (row, 32 K)"
    return "e4m3 + ue8m0 per-128 scales" if fp8 else "bf16"


def sample_steps(w):
    if getattr(w, "swiglu", False):
        return "plan + fp64 dequantise + per-expert GEMM1, SwiGLU, E4M3 re-quantisation, GEMM2"
    return "plan + fp64 dequantise + per-expert GEMMs"


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


# ------------------------------------------------------------------ arms
def run_ours(args):
    ws, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    lib = mb.load()
    mb.set_kernel_policy(mb.POLICIES[args.kernel_policy])
    w = make_workload(args.workload, dev)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()

    for _ in range(args.warmup):
        w.step(lib, stream)
    torch.cuda.synchronize()
    if int(w.status.item()) != 0:
        raise RuntimeError("device status " + mb.status_str(int(w.status.item())))

    n_g = len(w.gemms)
    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(n_g)]
           for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.6)
    for _ in range(max(3, args.warmup)):
        w.step(lib, stream)
    barrier(ws)
    torch.cuda.synchronize()
    t_host0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        w.step(lib, stream, evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    barrier(ws)
    time.sleep(0.3)
    sampler.stop()
    ms = start.elapsed_time(end)
    ms_max = max_over_ranks(ms, ws)
    per_gemm = [sum(evs[i][g][0].elapsed_time(evs[i][g][1]) for i in range(args.steps)) / args.steps
                for g in range(n_g)]
    if int(w.status.item()) != 0:
        raise RuntimeError("device status " + mb.status_str(int(w.status.item())))
    value = weak_scaling_value(w.flops() * args.steps, ws, ms_max) / 1e12

    # end to end: host buffers in, results back to host, same step count
    e2e = None
    if not args.no_e2e:
        bi, bo = w.e2e_setup()
        for _ in range(2):
            w.e2e_step(lib, stream)
        barrier(ws)
        torch.cuda.synchronize()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n2 = max(3, min(args.steps, 20))
        s2.record(stream)
        for _ in range(n2):
            w.e2e_step(lib, stream)
        e2.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        ms2 = max_over_ranks(s2.elapsed_time(e2), ws)
        e2e = {"value": weak_scaling_value(w.flops() * n2, ws, ms2) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": n2,
               "ms_per_step": ms2 / n2}

    roof = w.roofline(per_gemm, peaks)
    if rank != 0:
        return
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        experts, useful, secs = oracle_sample_bounded(w, args.cpu_budget)
        cpu = {"value": useful / secs / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "sample": f"experts {experts} of {args.workload}: {sample_steps(w)}, "
                         f"{useful / 1e9:.1f} useful GFLOP in {secs:.1f} s"}
    line = {
        "metric": "effective TFLOPS (valid rows only)",
        "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ("e4m3xe2m1" if getattr(w, "w4", False) else "e4m3") if w.fp8 else "bf16",
        "data": "synthetic",
        "config": dict(w.config(), kernel_policy=args.kernel_policy),
        "per_gemm_ms": per_gemm,
        "tactics": ([tactic_report(w.dtype, w.counts, g["N"], g["K"], t) for g, t in zip(w.gemms, per_gemm)]
                    if hasattr(w, "dtype") else None),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": w.launches_per_step() * args.steps,
        "clocks": sampler.summary(t_host0, t_host1),
    }
    print(json.dumps(line))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    w = make_workload(args.workload, dev)
    active = [e for e, t in enumerate(w.counts) if t]
    total_u, total_s = 0.0, 0.0
    per_step = 1
    for i in range(args.warmup + args.steps):
        experts = [active[(i * per_step + j) % len(active)] for j in range(per_step)]
        u, s = w.oracle_sample(experts)
        if i >= args.warmup:
            total_u += u
            total_s += s
    value = total_u / total_s / 1e12
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": "effective TFLOPS (valid rows only)", "value": value, "unit": "TFLOP/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_s * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": w.config(),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"one active expert per step (rotating) of {args.workload}: "
                                   f"{sample_steps(w)}"},
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
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--kernel-policy", choices=["auto", "single", "dual", "pair", "pair_dual"], default="auto",
                    help="grouped GEMM kernel family (auto: two 128-row weight blocks per SM when N %% 256 == 0)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
