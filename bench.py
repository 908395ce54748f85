#!/usr/bin/env python
"""Benchmark of the block-scaled FP4 hot path on GB300.

A step is one call of the hot path on one batch of synthetic input. The
headline (the JSON line's value) is the largest of the five workloads the
library targets, --workload compute:
  compute           mxfp4_quant_gemm_fused, A bf16 [8192, 8192] x MXFP4 B [8192, 8192]
                    (dynamic quantization of A, then the CTA-pair GEMM), bf16 C
The same run measures every workload into the line's "configs" object (the
five targets) and "extra" object (the grouped MXFP4, NVFP4 decode, grouped
NVFP4 from bf16 and RMSNorm + MXFP4 calls):
  tiny / decode / medium   mxfp4_quant_gemm_fused at M = 8 / 16 / 256
  nvfp4_grouped     nvfp4_group_gemm over 8 groups (M_g 64..1024, N 4096, K 7168)
  mxfp4_grouped     mxfp4_group_gemm over the same groups with MXFP4 operands
  nvfp4_decode      nvfp4_quant_gemm_fused on the decode shape (NVFP4 operands, fp16 C)
  nvfp4_grouped_bf16  nvfp4_group_quant_gemm: the nvfp4_grouped shapes with bf16 A_g,
                    quantized inside every call (grouped quantization + grouped GEMM)
  rmsnorm_decode / rmsnorm_prefill  mxfp4_rmsnorm_quantize on bf16 X [16 | 4096, 7168]
Weights are pre-quantized once, untimed, by the library's own quantizer.

`value` is microseconds per call over the whole job (all ranks), lower is
better. Each timed region holds exactly its steps (--steps for the headline)
between a barrier + synchronize on both sides, replayed from CUDA graphs so
that host launch cost does not pad the timing; HBM-bound shapes rotate over
enough copies of their inputs to exceed twice the L2 size. Every workload
reports the roofline of its dominant kernel (FP4 tensor peak = measured bf16
burst x 13.5/2.25, also given against the nominal 13.5 PFLOP/s and the
measured sustained rate; HBM = measured copy bandwidth) and the call's
fraction of the slower of the FP4-tensor and HBM time of the whole call.

--impl reference times the CPU oracle (the pages' method restated in plain C,
fp64) on all host cores, on a bounded sample of the same workload, scaled to
one full call.
"""
import argparse
import concurrent.futures as cf
import ctypes
import functools
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_scaled_fp4_mxfp4_gb300 import workloads as wl  # noqa: E402

METRIC = "µs/call & TFLOP/s, MXFP4 quant+GEMM; % of FP4-tensor/HBM roofline (1 GB300)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP4_OVER_BF16 = 13.5 / 2.25        # nominal dense FP4 : BF16 tensor ratio
NOMINAL_FP4_TFLOPS = 13500.0       # GB300 dense FP4, nominal
NOMINAL_HBM_GBS = 8000.0           # GB300 HBM3e, nominal (~8 TB/s)
L2_BYTES = 129 << 20               # GB300 L2, for the input rotation count

WORKLOADS = {
    "decode": wl.DECODE,
    "tiny": wl.TINY,
    "medium": wl.MEDIUM,
    "compute": wl.COMPUTE,
    "nvfp4_grouped": wl.NVFP4_GROUPED,
    "mxfp4_grouped": wl.MXFP4_GROUPED,
    "nvfp4_decode": wl.NVFP4_DECODE,
    "nvfp4_grouped_bf16": wl.NVFP4_GROUPED_BF16,
    "rmsnorm_decode": wl.RMSNORM_DECODE,
    "rmsnorm_prefill": wl.RMSNORM_PREFILL,
}
HEADLINE = "compute"
TARGETS = ["tiny", "decode", "medium", "compute", "nvfp4_grouped"]
EXTRAS = ["mxfp4_grouped", "nvfp4_decode", "nvfp4_grouped_bf16", "rmsnorm_decode", "rmsnorm_prefill"]
DEFAULT_STEPS = {"decode": 2000, "tiny": 2000, "medium": 2000, "compute": 50, "nvfp4_grouped": 200,
                 "mxfp4_grouped": 200, "nvfp4_decode": 2000, "nvfp4_grouped_bf16": 200,
                 "rmsnorm_decode": 2000, "rmsnorm_prefill": 200}


def grouped(name):
    """Whether a workload is a grouped GEMM (NVFP4 or MXFP4)."""
    return isinstance(WORKLOADS[name], wl.NVWorkload)


def rmsnorm(name):
    """Whether a workload is the fused RMSNorm + MXFP4 quantization."""
    return isinstance(WORKLOADS[name], wl.RMSWorkload)


def max_over_ranks(value, world, device):
    """The largest of every rank's value: a job's time is its slowest rank's."""
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_call(elapsed_ms, steps, world):
    """Whole-job microseconds per call: `world` replicas each made `steps` calls
    within elapsed_ms (the slowest rank's time)."""
    return elapsed_ms * 1000.0 / (steps * world)


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None, help="timed steps of the headline workload")
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    p.add_argument("--configs", choices=["all", "targets", "none"], default="all",
                   help="which other workloads to measure into the same line")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    return p.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "block_scaled_fp4_mxfp4_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "fused_quant_gemm_kernel": ["fused.cu", "ptx.cuh", "quant_math.cuh"],
    "bs_gemm_kernel": ["gemm.cu", "gemm_common.cuh", "ptx.cuh"],
    "bs_gemm_pair_kernel": ["gemm_pair.cu", "gemm_common.cuh", "ptx.cuh"],
    "rmsnorm_mx_quant_kernel": ["rmsnorm_quant.cu", "quant_math.cuh", "ptx.cuh"],
}


def kernel_of(plan, kind):
    """(label, source files) of the GEMM kernel a call's plan launches."""
    name = plan["kernel"]
    if name == "fused_quant_gemm_kernel":
        label = f"{name}<{plan['tile_m']}> x{plan['tiles']} tiles, {plan['splits']}-CTA K-split clusters"
    else:
        label = (f"{name}<{kind}> {plan['tile_m']}x{plan['tile_n']} tiles x{plan['tiles']}"
                 + (f", {plan['splits']} K-splits" if plan["splits"] > 1 else ""))
    return label, KERNEL_SOURCES[name]


def ncu_traffic(workload, kernel_files):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary table, or None if that kernel's source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(kernel_files)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == want:
                return int(parts[2])
    return None


def rotation_copies(name):
    """Copies of the per-call inputs rotated through so that consecutive calls
    never find them in L2 (their total exceeds twice the L2)."""
    w = WORKLOADS[name]
    if grouped(name):
        return 1                      # ~170 MB of operands per call already exceed twice the L2
    per = w.alg_bytes
    return max(1, min(64, math.ceil(2 * L2_BYTES / per)))


def config_of(name, world):
    """The line's `config` (identical for both arms)."""
    w = WORKLOADS[name]
    rot = rotation_copies(name)
    per = w.alg_bytes
    return {"workload": w.name, "parallelism": f"replicas x{world}",
            "l2": (f"rotating {rot} copies of the inputs ({rot * per / 1e6:.0f} MB > 2x L2)"
                   if rot > 1 else "inputs larger than 2x L2 per call"),
            "timing": "CUDA graph replay of the timed steps, CUDA events"}


@functools.lru_cache(maxsize=8)
def _nv_group_bits(seed, g, m, n, k):
    w = wl.NVWorkload("cache", [0] * g + [m], n, k, seed=seed)
    return wl.gen_nv_group(w, g)


def nv_group_bits(w, g):
    """bf16 bits of group g's (A_g, B_g); shared by the grouped workloads, which
    draw the same seeded streams."""
    return _nv_group_bits(w.seed, g, w.Ms[g], w.N, w.K)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        top = max(r[0] for r in rows)
        loaded = [r for r in rows if r[0] >= 0.5 * top] or rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in loaded:
            for name, v in zip(names, r[2:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(loaded)}


# ----------------------------------------------------------------- GPU arm --

class MXCase:
    """One quant+GEMM workload resident on the device, with L2 rotation: MXFP4
    (mxfp4_quant_gemm_fused), or NVFP4 (nvfp4_quant_gemm_fused) when w.vec == 16."""

    def __init__(self, name, w, dev, mx, torch):
        self.w, self.mx, self.torch = w, mx, torch
        self.nv = w.vec == 16
        a_bits, b_bits = wl.gen_a(w), wl.gen_b(w)
        to = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
        A0 = to(a_bits)
        quant = mx.nvfp4_quantize if self.nv else mx.mxfp4_quantize
        Bq0, Bsf0 = quant(to(b_bits))   # weight pre-quantization (untimed)
        torch.cuda.synchronize()
        self.a_host_bits = a_bits
        per = w.alg_bytes
        self.rot = rotation_copies(name)
        self.A = [A0] + [A0.clone() for _ in range(self.rot - 1)]
        self.Bq = [Bq0.contiguous()] + [Bq0.contiguous().clone() for _ in range(self.rot - 1)]
        self.Bsf = [Bsf0] + [Bsf0.clone() for _ in range(self.rot - 1)]
        self.C = torch.empty((w.M, w.N), dtype=torch.float16 if self.nv else torch.bfloat16, device=dev)
        self.ws = mx.new_workspace(w.M, w.N, w.K, dev)
        self.fused = w.M <= 64      # the library's fused small-M path (one launch)
        self.launches_per_step = 1 if self.fused else 2
        plan = mx.gemm_plan(w.M, w.N, w.K, fused=True, nvfp4=self.nv)
        self.kernel_label, self.kernel_files = kernel_of(plan, "mxf4nvf4" if self.nv else "mxf4")
        self.rot_bytes = per * self.rot

    def step(self, i):
        j = i % self.rot
        if self.nv:
            self.mx.nvfp4_quant_gemm_fused(self.A[j], self.Bq[j], self.Bsf[j], self.C)
        else:
            self.mx.mxfp4_quant_gemm_fused(self.A[j], self.Bq[j], self.Bsf[j], self.C, self.ws)

    def prepare_gemm_only(self):
        """Pre-quantized A for timing the GEMM kernel of the two-kernel path alone."""
        self._aq, self._asf = self.mx.mxfp4_quantize(self.A[0])

    def step_gemm_only(self, i):
        j = i % self.rot
        self.mx.mxfp4_gemm_a4w4(self._aq, self._asf, self.Bq[j], self.Bsf[j], self.w.K, self.C, self.ws)

    def alg_bytes(self):
        return self.w.alg_bytes

    def gemm_alg_bytes(self):
        """Bytes the GEMM kernel of the two-kernel path must move: packed A and B,
        both scale sets and bf16 C."""
        w = self.w
        return w.M * w.K // 2 + w.M * w.K // 32 + w.N * w.K // 2 + w.N * w.K // 32 + 2 * w.M * w.N

    def e2e(self, steps, torch):
        """Host buffers: per step copy A in from pinned memory, call the C ABI,
        copy C out to pinned memory. Consecutive calls are independent jobs and
        rotate over three streams (own device buffers each), so one call's
        copies overlap another call's kernel; the copies are cudaMemcpyAsync
        calls and the call goes straight to the C entry point, so that host
        overhead does not set the rate."""
        w, mx = self.w, self.mx
        L = mx.lib()
        a_pin = torch.from_numpy(self.a_host_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
        nA, nC = a_pin.numel() * 2, w.M * w.N * 2
        memcpy = _cuda_memcpy_async()
        lanes = []
        for _ in range(3):
            st = torch.cuda.Stream()
            A_dev = torch.empty_like(self.A[0])
            cdt = torch.float16 if self.nv else torch.bfloat16
            C = torch.empty((w.M, w.N), dtype=cdt, device=A_dev.device)
            c_pin = torch.empty((w.M, w.N), dtype=cdt).pin_memory()
            ws = mx.new_workspace(w.M, w.N, w.K, A_dev.device)
            sp = ctypes.c_void_p(st.cuda_stream)
            lanes.append((st, A_dev, C, c_pin, ws, sp))

        def one(i):
            st, A_dev, C, c_pin, ws, sp = lanes[i % 3]
            j = i % self.rot
            if memcpy:
                memcpy(A_dev.data_ptr(), a_pin.data_ptr(), nA, 1, sp)
            else:
                with torch.cuda.stream(st):
                    A_dev.copy_(a_pin, non_blocking=True)
            if self.nv:
                status = L.nvfp4_quant_gemm_fused(A_dev.data_ptr(), A_dev.stride(0), self.Bq[j].data_ptr(),
                                                  self.Bq[j].stride(0), self.Bsf[j].data_ptr(), C.data_ptr(),
                                                  C.stride(0), w.M, w.N, w.K, sp)
            else:
                status = L.mxfp4_quant_gemm_fused(A_dev.data_ptr(), A_dev.stride(0), self.Bq[j].data_ptr(),
                                                  self.Bq[j].stride(0), self.Bsf[j].data_ptr(), C.data_ptr(),
                                                  C.stride(0), w.M, w.N, w.K, ws.data_ptr(), ws.numel(), sp)
            if status != 0:
                raise RuntimeError(f"quant+GEMM call returned {status}")
            if memcpy:
                memcpy(c_pin.data_ptr(), C.data_ptr(), nC, 2, sp)
            else:
                with torch.cuda.stream(st):
                    c_pin.copy_(C, non_blocking=True)

        for i in range(6):
            one(i)
        torch.cuda.synchronize()
        main = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        for st, *_ in lanes:
            st.wait_event(e0)
        for i in range(steps):
            one(i)
        for st, *_ in lanes:
            main.wait_stream(st)
        e1.record(main)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1000.0 / steps, nA, nC


def _cuda_memcpy_async():
    """cudaMemcpyAsync from the CUDA runtime next to PyTorch's or in the
    toolkit, or None (bench.py then copies through PyTorch)."""
    import glob
    import torch
    cands = sorted(glob.glob(os.path.join(os.path.dirname(torch.__file__), "lib", "libcudart.so*")))
    cands += sorted(glob.glob("/usr/local/cuda/lib64/libcudart.so*"))
    for c in cands:
        try:
            rt = ctypes.CDLL(c)
            fn = rt.cudaMemcpyAsync
        except OSError:
            continue
        fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
        fn.restype = ctypes.c_int
        return fn
    return None


class NVCase:
    """Grouped workload (NVFP4, or MXFP4 when w.vec == 32): operands quantized
    once (untimed) by nvfp4_quantize / mxfp4_quantize; with w.bf16_a the A_g stay
    bf16 and nvfp4_group_quant_gemm quantizes them inside every call."""

    def __init__(self, name, w, dev, mx, torch):
        self.w, self.mx, self.torch = w, mx, torch
        nv = w.vec == 16
        quant = mx.nvfp4_quantize if nv else mx.mxfp4_quantize
        to = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
        self.groups = []     # pre-quantized operands (the grouped GEMM's own inputs)
        self.act = []        # bf16 activations (w.bf16_a)
        for g in range(len(w.Ms)):
            a_bits, b_bits = nv_group_bits(w, g)
            a16 = to(a_bits)
            qa, sfa = quant(a16)
            qb, sfb = quant(to(b_bits))
            c = torch.empty((w.Ms[g], w.N), dtype=torch.float16 if nv else torch.bfloat16, device=dev)
            self.groups.append(dict(a=qa, sfa=sfa, b=qb, sfb=sfb, c=c, k=w.K))
            if w.bf16_a:
                self.act.append(dict(a=a16, b=qb, sfb=sfb, c=c))
        torch.cuda.synchronize()
        if nv:
            self.problems = mx.make_nv_problems(self.groups)
            self.call = mx.nvfp4_group_gemm
            plan = mx.nvfp4_group_gemm_plan(self.problems)
        else:
            self.problems = mx.make_mx_problems(self.groups)
            self.call = mx.mxfp4_group_gemm
            plan = mx.mxfp4_group_gemm_plan(self.problems)
        self.launches_per_step = 1
        if w.bf16_a:
            self.act_problems = mx.make_nv_act_problems(self.act)
            self.ws = torch.empty(mx.nvfp4_group_quant_gemm_workspace_bytes(self.act_problems),
                                  dtype=torch.uint8, device=dev)
            self.launches_per_step = 2       # grouped quantization + grouped GEMM
        self.rot = 1                # ~170 MB of operands per call already exceed twice the L2
        self.kernel_label, self.kernel_files = kernel_of(plan, "mxf4nvf4" if nv else "mxf4")
        self.rot_bytes = w.alg_bytes

    def step(self, i):
        if self.w.bf16_a:
            self.mx.nvfp4_group_quant_gemm(self.act, self.act_problems, workspace=self.ws)
        else:
            self.call(self.groups, self.problems)

    def prepare_gemm_only(self):
        """The grouped GEMM alone runs on the operands quantized at set-up."""

    def step_gemm_only(self, i):
        self.call(self.groups, self.problems)

    def alg_bytes(self):
        return self.w.alg_bytes

    def gemm_alg_bytes(self):
        return self.w.gemm_alg_bytes

    def e2e(self, steps, torch):
        """Host buffers: per step copy every A_g in (packed codes + scales, or bf16
        with w.bf16_a), call, copy every C_g out."""
        if self.w.bf16_a:
            ins = [[g["a"]] for g in self.act]
        else:
            ins = [[g["a"], g["sfa"]] for g in self.groups]
        pins_in = [[t.cpu().pin_memory() for t in ts] for ts in ins]
        pins_out = [torch.empty_like(g["c"], device="cpu").pin_memory() for g in self.groups]
        s = torch.cuda.current_stream()

        def one():
            for ps, ts in zip(pins_in, ins):
                for p_, t in zip(ps, ts):
                    t.copy_(p_, non_blocking=True)
            self.step(0)
            for po, g in zip(pins_out, self.groups):
                po.copy_(g["c"], non_blocking=True)

        for _ in range(2):
            one()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            one()
        e1.record(s)
        torch.cuda.synchronize()
        h2d = sum(p_.numel() * p_.element_size() for ps in pins_in for p_ in ps)
        d2h = sum(po.numel() * 2 for po in pins_out)
        return e0.elapsed_time(e1) * 1000.0 / steps, h2d, d2h


class RMSCase:
    """Fused RMSNorm + MXFP4 quantization of resident bf16 activations
    (mxfp4_rmsnorm_quantize), rotating over copies of X to defeat the L2."""

    def __init__(self, name, w, dev, mx, torch):
        self.w, self.mx, self.torch = w, mx, torch
        x_bits, g_bits = wl.gen_rms(w)
        to = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
        X0 = to(x_bits)
        self.weight = to(g_bits)
        per = w.alg_bytes
        self.rot = rotation_copies(name)
        self.X = [X0] + [X0.clone() for _ in range(self.rot - 1)]
        self.Aq, self.sf = mx.mxfp4_rmsnorm_quantize(X0, self.weight, w.eps)
        torch.cuda.synchronize()
        self.launches_per_step = 1
        rows = (w.M + 127) // 128 * 128
        self.kernel_label = f"rmsnorm_mx_quant_kernel x{rows} rows (one CTA per row)"
        self.kernel_files = KERNEL_SOURCES["rmsnorm_mx_quant_kernel"]
        self.rot_bytes = per * self.rot

    def step(self, i):
        self.mx.mxfp4_rmsnorm_quantize(self.X[i % self.rot], self.weight, self.w.eps, self.Aq, self.sf)

    def alg_bytes(self):
        return self.w.alg_bytes

    def e2e(self, steps, torch):
        """Host buffers: per step copy X in, call, copy the codes and scales out."""
        pin_x = self.X[0].cpu().pin_memory()
        pin_q = torch.empty_like(self.Aq, device="cpu").pin_memory()
        pin_s = torch.empty_like(self.sf, device="cpu").pin_memory()
        s = torch.cuda.current_stream()

        def one():
            self.X[0].copy_(pin_x, non_blocking=True)
            self.step(0)
            pin_q.copy_(self.Aq, non_blocking=True)
            pin_s.copy_(self.sf, non_blocking=True)

        for _ in range(3):
            one()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            one()
        e1.record(s)
        torch.cuda.synchronize()
        return (e0.elapsed_time(e1) * 1000.0 / steps, pin_x.numel() * 2,
                pin_q.numel() + pin_s.numel())


# ------------------------------------------------------------ measurement --

def roofline_of(name, case, kernel_us, peaks, peak_src):
    """Roofline of the dominant kernel (the GEMM of a two-launch call, else the
    call's one kernel): algorithmic FLOPs or bytes per launch / its time."""
    w = WORKLOADS[name]
    if name == "compute":
        burst = peaks["bf16_tflops"] * FP4_OVER_BF16
        ach = w.flops / (kernel_us * 1e-6) / 1e12
        return {"bound": "tensor", "achieved": round(ach, 1), "peak": round(burst, 1), "unit": "TFLOP/s",
                "frac": round(ach / burst, 4),
                "frac_of_nominal_fp4": round(ach / NOMINAL_FP4_TFLOPS, 4),
                "frac_of_sustained_fp4": round(ach / (peaks["bf16_tflops_sustained"] * FP4_OVER_BF16), 4),
                "peak_source": f"{peak_src} bf16 burst x {FP4_OVER_BF16:g} (nominal FP4:BF16); the kernel "
                               f"is timed alone over its steps"}
    nbytes = case.gemm_alg_bytes() if case.launches_per_step > 1 else case.alg_bytes()
    ach = nbytes / (kernel_us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / peaks["hbm_gbs"], 4), "bytes_per_launch": int(nbytes),
            "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"}


def call_roofline(name, us_per_call, peaks):
    """The whole call against the slower of its FLOPs at the FP4 tensor peak and
    its algorithmic bytes at the HBM peak: with the nominal GB300 figures
    (13.5 PFLOP/s, 8 TB/s) and with the measured ones."""
    w = WORKLOADS[name]
    if rmsnorm(name):
        flops = 0
    else:
        flops = w.flops
    nb = w.alg_bytes
    out = {}
    for tag, p_fp4, bw in (("nominal", NOMINAL_FP4_TFLOPS, NOMINAL_HBM_GBS),
                           ("measured", peaks["bf16_tflops"] * FP4_OVER_BF16, peaks["hbm_gbs"])):
        t_tc = flops / (p_fp4 * 1e12) * 1e6
        t_hbm = nb / (bw * 1e9) * 1e6
        out[tag] = {"roofline_us": round(max(t_tc, t_hbm), 4), "bound": "tensor" if t_tc > t_hbm else "hbm",
                    "frac": round(max(t_tc, t_hbm) / us_per_call, 4)}
    return out


def measure(args, name, steps, warmup, world, dev, e2e=True):
    """Time one workload: its call, its dominant kernel alone (two-launch calls),
    clocks during the timed region and, unless disabled, the end-to-end call
    from host buffers."""
    import torch
    from block_scaled_fp4_mxfp4_gb300 import mxfp4 as mx

    w = WORKLOADS[name]
    if rmsnorm(name):
        case = RMSCase(name, w, dev, mx, torch)
    else:
        case = NVCase(name, w, dev, mx, torch) if grouped(name) else MXCase(name, w, dev, mx, torch)

    for i in range(max(warmup, case.rot)):  # warm-up (also encodes every TMA descriptor once)
        case.step(i)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    cap_stream = torch.cuda.Stream()

    def capture(fn, count):
        """CUDA graphs holding exactly `count` calls of fn(i), in chunks of G."""
        G = case.rot * max(1, min(1000, count) // case.rot)
        graphs = []
        for c in ([G] * (count // G)) + ([count % G] if count % G else []):
            if graphs and c == graphs[0][1]:
                graphs.append(graphs[0])     # replay the same chunk again
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap_stream):
                for i in range(c):
                    fn(i)
            graphs.append((g, c))
        return graphs

    def timed(graphs, settle_s):
        s = torch.cuda.current_stream()
        t_end = time.time() + settle_s      # untimed replays so clocks settle
        while time.time() < t_end:
            graphs[0][0].replay()
            torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for g, _ in graphs:
            g.replay()
        e1.record(s)
        barrier()
        return e0.elapsed_time(e1)

    step_graphs = capture(case.step, steps)
    with ClockSampler(dev.index or 0) as clk:
        elapsed_ms = timed(step_graphs, 0.5)
    del step_graphs
    kernel_timing = "per step (one launch per step)"
    per_kernel_us = elapsed_ms * 1000.0 / steps
    split = None
    if case.launches_per_step > 1:
        # the dominant kernel (the GEMM) timed alone on the same rotation
        case.prepare_gemm_only()
        gemm_graphs = capture(case.step_gemm_only, steps)
        gemm_ms = timed(gemm_graphs, 0.1)
        del gemm_graphs
        per_kernel_us = max_over_ranks(gemm_ms, world, dev) * 1000.0 / steps
        split = {"gemm_us": round(per_kernel_us, 3), "step_us": round(elapsed_ms * 1000.0 / steps, 3)}
        kernel_timing = "GEMM kernel timed alone: CUDA-graph replay of the same number of launches"

    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    us_per_call = job_us_per_call(elapsed_ms, steps, world)
    peaks, peak_src = load_peaks()
    roof = roofline_of(name, case, per_kernel_us, peaks, peak_src)
    roof["traffic"] = ncu_traffic(name, case.kernel_files)
    roof["kernel"] = case.kernel_label
    roof["kernel_us"] = round(per_kernel_us, 3)
    roof["kernel_timing"] = kernel_timing
    out = {"workload": w.name, "us_per_call": round(us_per_call, 4), "steps": steps, "warmup": warmup,
           "ms_per_step": round(elapsed_ms / steps, 6),
           "tflops": round(w.flops * steps * world / (elapsed_ms * 1e-3) / 1e12, 3),
           "roofline": roof, "call_roofline": call_roofline(name, us_per_call, peaks),
           "gpu_launches": steps * case.launches_per_step, "clocks": clk.summary(),
           "config": config_of(name, world)}
    if split:
        out["kernels_us"] = split
    if e2e and not args.no_e2e:
        short = case.launches_per_step == 1 and not grouped(name)
        e2e_steps = max(10, min(steps, 2000 if short else 20))
        e_us, h2d, d2h = case.e2e(e2e_steps, torch)
        e_us = max_over_ranks(e_us, world, dev) / world
        out["e2e"] = {"value": round(e_us, 4), "unit": "us/call", "h2d_bytes_per_step": int(h2d),
                      "d2h_bytes_per_step": int(d2h), "steps": e2e_steps}
    del case
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def run_ours(args, name, rank, world, local_rank):
    import torch

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[name]
    warmup = args.warmup if args.warmup is not None else max(3, min(100, steps // 10))
    head = measure(args, name, steps, warmup, world, dev)

    line = {
        "metric": METRIC, "value": head["us_per_call"], "unit": "us/call", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "fp4 e2m1 (fp32 accumulate)",
        "data": "synthetic (seeded SplitMix64/Box-Muller; weights pre-quantized untimed)",
        "config": head["config"], "tflops": head["tflops"], "roofline": head["roofline"],
        "call_roofline": head["call_roofline"], "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
    }
    if "kernels_us" in head:
        line["kernels_us"] = head["kernels_us"]
    if "e2e" in head:
        line["e2e"] = head["e2e"]

    others = []
    if args.configs in ("all", "targets"):
        others += TARGETS
    if args.configs == "all":
        others += EXTRAS
    configs, extra = {}, {}
    for other in others:
        if other == name:
            entry = {k: v for k, v in head.items() if k != "config"}
        else:
            o_steps = DEFAULT_STEPS[other]
            entry = measure(args, other, o_steps, max(3, min(100, o_steps // 10)), world, dev)
            entry.pop("config", None)
        (configs if other in TARGETS else extra)[other] = entry
    if configs:
        line["configs"] = configs
    if extra:
        line["extra"] = extra

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(name)
    return line


# ------------------------------------------------------------- oracle arm --

_ORACLE_PREP = {}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_prep(name):
    """Untimed oracle-side inputs: bf16 activations (at most 4096 rows, more than
    any bounded sample uses) and the pre-quantized weights."""
    import oracle
    if name in _ORACLE_PREP:
        return _ORACLE_PREP[name]
    w = WORKLOADS[name]
    if rmsnorm(name):
        prep = wl.gen_rms(w)
    elif grouped(name):
        quant = oracle.nv_quantize if w.vec == 16 else oracle.mx_quantize
        prep = []
        for g in range(len(w.Ms)):
            a_bits, b_bits = nv_group_bits(w, g)
            qa, sfa = quant(a_bits)
            qb, sfb = quant(b_bits)
            prep.append((a_bits, qa, sfa, qb, sfb))
    else:
        a_bits = wl.gen_a(w) if w.M <= 4096 else wl.gen_a(w, M=4096)
        qb, sfb = (oracle.nv_quantize if w.vec == 16 else oracle.mx_quantize)(wl.gen_b(w))
        prep = (a_bits, qb, sfb)
    _ORACLE_PREP[name] = prep
    return prep


def _run_split(threads, jobs):
    """Run the thunks in `jobs` on `threads` host threads (the oracle's C loops
    release the GIL); return the wall time in seconds."""
    t0 = time.perf_counter()
    if threads == 1:
        for j in jobs:
            j()
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda j: j(), jobs))
    return time.perf_counter() - t0


def _chunks(n, parts):
    parts = max(1, min(parts, n))
    edges = [n * i // parts for i in range(parts + 1)]
    return [(edges[i], edges[i + 1]) for i in range(parts) if edges[i + 1] > edges[i]]


def oracle_timing(name, threads, budget_s):
    """The oracle (as it stands) on a bounded sample of one call of `name`,
    split over `threads` host threads by rows: quantization of A and the
    dequantize-then-fp64 GEMM timed separately, each scaled to the full call.
    Returns a dict with quant_us, gemm_us, call_us (microseconds), threads and
    the sample's description."""
    import oracle
    w = WORKLOADS[name]
    if rmsnorm(name):
        x_bits, g_bits = _oracle_prep(name)
        t0 = time.perf_counter()
        oracle.rmsnorm_mx_quantize(x_bits[:1], g_bits, w.eps)
        per_row = max(1e-6, time.perf_counter() - t0)
        r = max(1, min(w.M, int(budget_s / per_row)))
        dt = _run_split(1, [lambda: oracle.rmsnorm_mx_quantize(x_bits[:r], g_bits, w.eps)])
        us = dt / r * w.M * 1e6
        return {"quant_us": round(us, 1), "gemm_us": None, "call_us": round(us, 1), "threads": 1,
                "sample": f"rows 0..{r - 1} of {w.M} (exact sum of squares, fp32 y, OCP MX blocks; "
                          f"Python-level loops, one thread), scaled by rows"}
    quant_budget, gemm_budget = 0.35 * budget_s, 0.65 * budget_s
    if grouped(name):
        prep = _oracle_prep(name)
        quant = oracle.nv_quantize if w.vec == 16 else oracle.mx_quantize
        total = sum(w.Ms)
        a0, qa0, sfa0, qb0, sfb0 = prep[0]
        t0 = time.perf_counter()
        quant(a0[:8])
        q_row = max(1e-7, (time.perf_counter() - t0) / 8)
        t0 = time.perf_counter()
        oracle.gemm_sampled(qa0, sfa0, qb0, sfb0, w.K, w.vec, np.zeros(w.N // 8, np.int64), np.arange(w.N // 8))
        g_row = max(1e-6, (time.perf_counter() - t0) * 8)
        quant_us = None
        if w.bf16_a:
            rq = max(1, min(min(w.Ms), int(quant_budget * threads / q_row / len(w.Ms))))
            jobs = [functools.partial(quant, a[lo:hi]) for a, *_ in prep for lo, hi in _chunks(rq, threads)]
            quant_us = _run_split(threads, jobs) / (rq * len(w.Ms)) * total * 1e6
        rg = max(1, min(min(w.Ms), int(gemm_budget * threads / g_row / len(w.Ms))))
        jobs = []
        for a, qa, sfa, qb, sfb in prep:
            for lo, hi in _chunks(rg, threads):
                rows = np.repeat(np.arange(lo, hi), w.N)
                cols = np.tile(np.arange(w.N), hi - lo)
                jobs.append(functools.partial(oracle.gemm_sampled, qa, sfa, qb, sfb, w.K, w.vec, rows, cols))
        gemm_us = _run_split(threads, jobs) / (rg * len(w.Ms)) * total * 1e6
        call = gemm_us + (quant_us or 0.0)
        return {"quant_us": None if quant_us is None else round(quant_us, 1), "gemm_us": round(gemm_us, 1),
                "call_us": round(call, 1), "threads": threads,
                "sample": (f"first {rg} rows of each group x all {w.N} columns (GEMM)"
                           + (f", first {rq} rows of each group (quantization)" if w.bf16_a else "")
                           + ", scaled by rows")}
    a_bits, qb, sfb = _oracle_prep(name)
    quant = oracle.nv_quantize if w.vec == 16 else oracle.mx_quantize
    avail = a_bits.shape[0]
    t0 = time.perf_counter()
    quant(a_bits[:min(8, avail)])
    q_row = max(1e-7, (time.perf_counter() - t0) / min(8, avail))
    rq = max(1, min(w.M, avail, int(quant_budget * threads / q_row)))
    qa_s, sfa_s = quant(a_bits[:rq])            # the GEMM's A sample (untimed)
    quant_us = _run_split(threads, [functools.partial(quant, a_bits[lo:hi]) for lo, hi in _chunks(rq, threads)]) \
        / rq * w.M * 1e6
    n_probe = max(1, w.N // 16)
    t0 = time.perf_counter()
    oracle.gemm_sampled(qa_s, sfa_s, qb, sfb, w.K, w.vec, np.zeros(n_probe, np.int64), np.arange(n_probe))
    g_row = max(1e-6, (time.perf_counter() - t0) * w.N / n_probe)
    rg = max(1, min(rq, int(gemm_budget * threads / g_row)))
    jobs = []
    for lo, hi in _chunks(rg, threads):
        rows = np.repeat(np.arange(lo, hi), w.N)
        cols = np.tile(np.arange(w.N), hi - lo)
        jobs.append(functools.partial(oracle.gemm_sampled, qa_s, sfa_s, qb, sfb, w.K, w.vec, rows, cols))
    gemm_us = _run_split(threads, jobs) / rg * w.M * 1e6
    full = "all rows" if rg == w.M else f"rows 0..{rg - 1} of {w.M}"
    return {"quant_us": round(quant_us, 1), "gemm_us": round(gemm_us, 1), "call_us": round(quant_us + gemm_us, 1),
            "threads": threads,
            "sample": (f"quantization of rows 0..{rq - 1} of {w.M}; GEMM of {full} x all {w.N} columns "
                       f"(dequantize-then-fp64 per output); each scaled by rows")}


def cpu_baseline(name):
    """The oracle on one host core and on all of them, quantization and GEMM
    timed separately; `value` is the all-core call."""
    cores = host_cores()
    one = oracle_timing(name, 1, 8.0)
    allc = oracle_timing(name, cores, 8.0) if cores > 1 and not rmsnorm(name) else one
    return {"value": allc["call_us"], "unit": "us/call", "cores": allc["threads"], "kind": "oracle",
            "sample": allc["sample"],
            "single_core": {k: one[k] for k in ("quant_us", "gemm_us", "call_us", "sample")},
            "all_cores": {k: allc[k] for k in ("quant_us", "gemm_us", "call_us", "threads")}}


def run_reference(args, name):
    w = WORKLOADS[name]
    steps = args.steps if args.steps is not None else 5
    warmup = args.warmup if args.warmup is not None else 1
    budget = max(0.5, min(20.0, 150.0 / max(1, steps + warmup)))
    cores = host_cores() if not rmsnorm(name) else 1
    for _ in range(warmup):
        oracle_timing(name, cores, budget)
    vals, last = [], None
    for _ in range(steps):
        last = oracle_timing(name, cores, budget)
        vals.append(last["call_us"])
    us = statistics.mean(vals) if vals else 0.0
    return {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/call", "n_gpus": 1,
        "steps": steps, "warmup": warmup, "ms_per_step": round(us / 1000.0, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(name, 1),
        "cpu_baseline": {"value": round(us, 1), "unit": "us/call", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {last['sample'] if last else ''}",
                         "quant_us": last["quant_us"] if last else None,
                         "gemm_us": last["gemm_us"] if last else None},
        "e2e": {"value": round(us, 1), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, args.workload)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, args.workload, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
