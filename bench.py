#!/usr/bin/env python
"""Benchmark of the block-scaled FP4 hot path on GB300.

A step is one call of the hot path on one batch of synthetic input:
  decode (default)  mxfp4_quant_gemm_fused, A bf16 [16, 7168] x MXFP4 B [2112, 7168]
  tiny / medium / compute   the other MXFP4 quant+GEMM shapes
  nvfp4_grouped     nvfp4_group_gemm over 8 groups (M_g 64..1024, N 4096, K 7168)
  mxfp4_grouped     mxfp4_group_gemm over the same groups with MXFP4 operands
  nvfp4_decode      nvfp4_quant_gemm_fused on the decode shape (NVFP4 operands, fp16 C)
  nvfp4_grouped_bf16  nvfp4_group_quant_gemm: the nvfp4_grouped shapes with bf16 A_g,
                    quantized inside every call (grouped quantization + grouped GEMM)
  rmsnorm_decode / rmsnorm_prefill  mxfp4_rmsnorm_quantize on bf16 X [16 | 4096, 7168]
Weights are pre-quantized once, untimed, by the library's own quantizer.

Prints one JSON line (rank 0). `value` is microseconds per call over the whole
job (all ranks), lower is better. The timed region holds exactly --steps steps
between a barrier + synchronize on both sides; HBM-bound shapes rotate over
enough copies of their inputs to exceed twice the L2 size. The timed steps are
replayed from CUDA graphs so host launch cost does not pad the timing.

--impl reference times the CPU oracle (the pages' method restated in plain C,
fp64) on a bounded sample of the same workload, scaled to one full call.
"""
import argparse
import ctypes
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
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 : BF16 tensor ratio

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
DEFAULT_STEPS = {"decode": 20000, "tiny": 20000, "medium": 10000, "compute": 50, "nvfp4_grouped": 500,
                 "mxfp4_grouped": 500, "nvfp4_decode": 20000, "nvfp4_grouped_bf16": 500,
                 "rmsnorm_decode": 20000, "rmsnorm_prefill": 1000}


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


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    return p.parse_args()


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

    def __init__(self, w, dev, mx, torch):
        self.w, self.mx, self.torch = w, mx, torch
        self.nv = w.vec == 16
        a_bits, b_bits = wl.gen_a(w), wl.gen_b(w)
        to = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
        A0 = to(a_bits)
        quant = mx.nvfp4_quantize if self.nv else mx.mxfp4_quantize
        Bq0, Bsf0 = quant(to(b_bits))   # weight pre-quantization (untimed)
        torch.cuda.synchronize()
        self.a_host_bits = a_bits
        per = A0.numel() * 2 + Bq0.numel() + Bsf0.numel() + w.M * w.N * 2
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20)
        self.rot = max(1, min(64, math.ceil(2 * l2 / per)))
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

    def __init__(self, w, dev, mx, torch):
        self.w, self.mx, self.torch = w, mx, torch
        nv = w.vec == 16
        quant = mx.nvfp4_quantize if nv else mx.mxfp4_quantize
        to = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
        self.groups = []     # pre-quantized operands (the grouped GEMM's own inputs)
        self.act = []        # bf16 activations (w.bf16_a)
        for g in range(len(w.Ms)):
            a_bits, b_bits = wl.gen_nv_group(w, g)
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

    def __init__(self, w, dev, mx, torch):
        self.w, self.mx, self.torch = w, mx, torch
        x_bits, g_bits = wl.gen_rms(w)
        to = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
        X0 = to(x_bits)
        self.weight = to(g_bits)
        per = w.alg_bytes
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20)
        self.rot = max(1, min(64, math.ceil(2 * l2 / per)))
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


def run_ours(args, name, rank, world, local_rank):
    import torch
    from block_scaled_fp4_mxfp4_gb300 import mxfp4 as mx

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = WORKLOADS[name]
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[name]
    warmup = args.warmup if args.warmup is not None else max(3, min(100, steps // 10))
    if rmsnorm(name):
        case = RMSCase(w, dev, mx, torch)
    else:
        case = NVCase(w, dev, mx, torch) if grouped(name) else MXCase(w, dev, mx, torch)

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
    with ClockSampler(local_rank) as clk:
        elapsed_ms = timed(step_graphs, 0.5)
    del step_graphs
    kernel_timing = "per step (one launch per step)"
    per_kernel_us = elapsed_ms * 1000.0 / steps
    split_times = None
    if case.launches_per_step > 1:
        # the dominant kernel (the GEMM) timed alone on the same rotation
        case.prepare_gemm_only()
        gemm_graphs = capture(case.step_gemm_only, steps)
        gemm_ms = timed(gemm_graphs, 0.1)
        del gemm_graphs
        per_kernel_us = gemm_ms * 1000.0 / steps
        split_times = {"gemm_us": per_kernel_us, "step_us": elapsed_ms * 1000.0 / steps}
        kernel_timing = "GEMM kernel timed alone: CUDA-graph replay of --steps launches"

    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    us_per_call = job_us_per_call(elapsed_ms, steps, world)
    tflops = w.flops * steps * world / (elapsed_ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    clocks = clk.summary()

    # roofline of the dominant kernel
    if name == "compute":
        fp4_peak = peaks["bf16_tflops_sustained"] * FP4_OVER_BF16
        ach = w.flops / (per_kernel_us * 1e-6) / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                "frac": round(ach / fp4_peak, 4),
                "peak_source": f"{peak_src} bf16 sustained x {FP4_OVER_BF16:g} (nominal FP4:BF16)"}
    else:
        nbytes = case.gemm_alg_bytes() if case.launches_per_step > 1 else case.alg_bytes()
        ach = nbytes / (per_kernel_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "peak_source": f"{peak_src} hbm_gbs"}
    roof["traffic"] = ncu_traffic(name, case.kernel_files)
    roof["kernel"] = case.kernel_label
    roof["kernel_us"] = round(per_kernel_us, 3)
    roof["kernel_timing"] = kernel_timing

    line = {
        "metric": METRIC, "value": round(us_per_call, 4), "unit": "us/call", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(elapsed_ms / steps, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "fp4 e2m1 (fp32 accumulate)",
        "data": "synthetic (seeded SplitMix64/Box-Muller; weights pre-quantized untimed)",
        "config": {"workload": w.name, "parallelism": f"replicas x{world}",
                   "l2": (f"rotating {case.rot} copies of inputs ({case.rot_bytes / 1e6:.0f} MB > 2x L2)"
                          if case.rot > 1 else "inputs larger than 2x L2 per call"),
                   "timing": "CUDA graph replay of the timed steps"},
        "tflops": round(tflops, 3),
        "roofline": roof,
        "gpu_launches": steps * case.launches_per_step,
        "clocks": clocks,
    }
    if split_times:
        line["kernels_us"] = {k: round(v, 3) for k, v in split_times.items()}

    if not args.no_e2e:
        short = case.launches_per_step == 1 and not grouped(name)
        e2e_steps = max(10, min(steps, 2000 if short else 20))
        e_us, h2d, d2h = case.e2e(e2e_steps, torch)
        e_us = max_over_ranks(e_us, world, dev) / world
        line["e2e"] = {"value": round(e_us, 4), "unit": "us/call",
                       "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(name, budget_s=12.0)
    return line


# ------------------------------------------------------------- oracle arm --

_ORACLE_PREP = {}


def _oracle_prep(name):
    """Untimed oracle-side inputs: bf16 activations and the pre-quantized weights."""
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
            a_bits, b_bits = wl.gen_nv_group(w, g)
            qb, sfb = quant(b_bits)
            prep.append((a_bits, qb, sfb))
    else:
        a_bits = wl.gen_a(w) if w.M <= 4096 else wl.gen_a(w, M=64)
        qb, sfb = (oracle.nv_quantize if w.vec == 16 else oracle.mx_quantize)(wl.gen_b(w))
        prep = (a_bits, qb, sfb)
    _ORACLE_PREP[name] = prep
    return prep


def oracle_call_sampled(name, budget_s):
    """Time the oracle on a bounded sample of one call; return (us per full call, sample text)."""
    import oracle
    w = WORKLOADS[name]
    if rmsnorm(name):
        x_bits, g_bits = _oracle_prep(name)
        t0 = time.perf_counter()
        oracle.rmsnorm_mx_quantize(x_bits[:1], g_bits, w.eps)
        per_row = time.perf_counter() - t0
        r = max(1, min(w.M, int(budget_s / per_row)))
        t0 = time.perf_counter()
        oracle.rmsnorm_mx_quantize(x_bits[:r], g_bits, w.eps)
        dt = time.perf_counter() - t0
        full = "the full call" if r == w.M else f"rows 0..{r - 1} of {w.M}, scaled by rows"
        return dt / r * w.M * 1e6, f"{full} (exact sum of squares, fp32 y, OCP MX blocks)"
    if grouped(name):
        # sample: the first r rows of every group, all N columns
        quant = oracle.nv_quantize if w.vec == 16 else oracle.mx_quantize
        prep = _oracle_prep(name)
        t0 = time.perf_counter()
        a_bits, qb, sfb = prep[0]
        qa, sfa = quant(a_bits[:1])
        oracle.gemm_sampled(qa, sfa, qb, sfb, w.K, w.vec, np.zeros(w.N, np.int64), np.arange(w.N))
        per_row = time.perf_counter() - t0
        total_rows = sum(w.Ms)
        r = max(1, min(max(w.Ms), int(budget_s / per_row / len(w.Ms))))
        t0 = time.perf_counter()
        done_rows = 0
        for a_bits, qb, sfb in prep:
            rr = min(r, a_bits.shape[0])
            qa, sfa = quant(a_bits[:rr])
            rows = np.repeat(np.arange(rr), w.N)
            cols = np.tile(np.arange(w.N), rr)
            oracle.gemm_sampled(qa, sfa, qb, sfb, w.K, w.vec, rows, cols)
            done_rows += rr
        dt = time.perf_counter() - t0
        return (dt / done_rows * total_rows * 1e6,
                f"first {r} rows of each group x all {w.N} columns (quantize + GEMM), scaled by rows")
    a_bits, qb, sfb = _oracle_prep(name)
    quant = oracle.nv_quantize if w.vec == 16 else oracle.mx_quantize
    t0 = time.perf_counter()
    qa, sfa = quant(a_bits[:1])
    oracle.gemm_sampled(qa, sfa, qb, sfb, w.K, w.vec, np.zeros(w.N, np.int64), np.arange(w.N))
    per_row = time.perf_counter() - t0
    r = max(1, min(w.M, a_bits.shape[0], int(budget_s / per_row)))
    t0 = time.perf_counter()
    qa, sfa = quant(a_bits[:r])
    if r == w.M:
        oracle.gemm_full(qa, sfa, qb, sfb, w.K, w.vec)
    else:
        oracle.gemm_sampled(qa, sfa, qb, sfb, w.K, w.vec, np.repeat(np.arange(r), w.N), np.tile(np.arange(w.N), r))
    dt = time.perf_counter() - t0
    full = "the full call" if r == w.M else f"rows 0..{r - 1} of {w.M} x all {w.N} columns, scaled by rows"
    return dt / r * w.M * 1e6, f"{full} (quantize A + dequantize-then-fp64 GEMM)"


def cpu_baseline(name, budget_s):
    us, sample = oracle_call_sampled(name, budget_s)
    return {"value": round(us, 1), "unit": "us/call", "cores": 1, "kind": "oracle", "sample": sample}


def run_reference(args, name):
    w = WORKLOADS[name]
    steps = args.steps if args.steps is not None else 5
    warmup = args.warmup if args.warmup is not None else 1
    budget = max(0.5, min(20.0, 150.0 / (steps + warmup)))
    for _ in range(warmup):
        oracle_call_sampled(name, budget)
    vals = []
    sample = ""
    for _ in range(steps):
        us, sample = oracle_call_sampled(name, budget)
        vals.append(us)
    us = statistics.mean(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/call", "n_gpus": 1,
        "steps": steps, "warmup": warmup, "ms_per_step": round(us / 1000.0, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "parallelism": "single host thread"},
        "cpu_baseline": {"value": round(us, 1), "unit": "us/call", "cores": 1, "kind": "oracle",
                         "sample": f"per step: {sample}"},
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
