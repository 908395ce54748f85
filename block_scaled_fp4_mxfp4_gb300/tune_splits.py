"""Measure the K-splits of the split-K paths and write the planner's table.

For every shape of a regime (the small-M decode and prefill GEMMs: M from 4
to 256, N in {512, 2112, 4096, 7168}, K from 512 to 7168) and every K-split
count the kernel can run, this times the call on the current GPU and keeps
the fastest count. The result is written as csrc/split_table.inc, which the
library's planner consults before its shape-derived rule; rebuild the library
afterwards. Paths:
  fused      mxfp4_quant_gemm_fused at M <= 64 (fused small-M kernel, K-split
             clusters of 1..8 CTAs), buckets by MMA width 16 / 32 / 64
  fused_nv   nvfp4_quant_gemm_fused, the same buckets
  gemm       mxfp4_gemm_a4w4 on the single-CTA kernel (the GEMM of the
             two-kernel path at M > 64), buckets by 128-row tiles of M
Timing: CUDA-graph replay of repeated calls with the weights rotated over
enough copies to exceed twice the L2, best of three replays.

Usage: python tune_splits.py [--out PATH] [--paths fused,fused_nv,gemm] [--quick]
"""
import argparse
import math
import os
import sys
import time

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

from block_scaled_fp4_mxfp4_gb300 import mxfp4 as mx  # noqa: E402
from block_scaled_fp4_mxfp4_gb300 import workloads as wl  # noqa: E402

NS = [512, 2112, 4096, 7168]
KS = [512, 1024, 2048, 4096, 7168]
BUCKET_M = {"fused": [16, 32, 64], "fused_nv": [16, 32, 64], "gemm": [128, 256]}
CANDIDATES = {"fused": list(range(1, 9)), "fused_nv": list(range(1, 9)), "gemm": [1, 2, 3, 4, 6, 8, 12, 16]}
L2_BYTES = 129 << 20


def to_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def graph_time_us(fn, calls, reps=3):
    s = torch.cuda.Stream()
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(calls):
            fn(i)
    best = float("inf")
    for _ in range(reps):
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1000.0 / calls)
    del g
    return best


def plan_splits(path, M, N, K):
    p = mx.gemm_plan(M, N, K, fused=path != "gemm", nvfp4=path == "fused_nv")
    return p["splits"], p["kernel"]


_B_CACHE = {}


def weights(N, K):
    """bf16 weights [N, K] on the device (seeded, N(0, 0.02)), generated once per shape."""
    if (N, K) not in _B_CACHE:
        _B_CACHE[(N, K)] = to_dev(wl.gen_bf16(7, 1000 + N + K, N, K, "normal", 0.02))
    return _B_CACHE[(N, K)]


def sweep_shape(path, M, N, K, seed):
    nv = path == "fused_nv"
    quant = mx.nvfp4_quantize if nv else mx.mxfp4_quantize
    a = to_dev(wl.gen_bf16(seed, 1, M, K))
    b = weights(N, K)
    per = N * K // 2 + N * K // (16 if nv else 32)
    rot = max(1, min(64, math.ceil(2 * L2_BYTES / per)))
    Bs = [quant(b) for _ in range(rot)]
    C = torch.empty((M, N), dtype=torch.float16 if nv else torch.bfloat16, device="cuda")
    if path == "gemm":
        aq, asf = mx.mxfp4_quantize(a)
    calls = max(rot, 64)
    results = {}
    formula = None
    mx.set_split_override(path, 0)
    formula, kernel = plan_splits(path, M, N, K)
    for want in CANDIDATES[path]:
        mx.set_split_override(path, want)
        got, kernel = plan_splits(path, M, N, K)
        if got in results:
            continue
        if path == "gemm" and kernel != "bs_gemm_kernel":
            break
        ws = mx.new_workspace(M, N, K)
        if path == "gemm":
            fn = lambda i: mx.mxfp4_gemm_a4w4(aq, asf, Bs[i % rot][0], Bs[i % rot][1], K, C, ws)
        elif nv:
            fn = lambda i: mx.nvfp4_quant_gemm_fused(a, Bs[i % rot][0], Bs[i % rot][1], C)
        else:
            fn = lambda i: mx.mxfp4_quant_gemm_fused(a, Bs[i % rot][0], Bs[i % rot][1], C, ws)
        results[got] = graph_time_us(fn, calls)
        del ws
    mx.set_split_override(path, 0)
    if mx.get_device_error() != 0:
        raise RuntimeError(f"device error during {path} {M}x{N}x{K}")
    del Bs
    torch.cuda.empty_cache()
    return formula, results


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=os.path.join(HERE, "csrc", "split_table.inc"))
    ap.add_argument("--paths", default="fused,fused_nv,gemm")
    ap.add_argument("--quick", action="store_true", help="N in {2112, 7168}, K in {2048, 7168} only")
    args = ap.parse_args()
    ns, ks = (NS, KS) if not args.quick else ([2112, 7168], [2048, 7168])
    entries, lines = [], []
    t0 = time.time()
    for path in args.paths.split(","):
        which = mx.SPLIT_PATHS[path]
        for M in BUCKET_M[path]:
            bucket = (M + 127) // 128 if path == "gemm" else (16 if M <= 16 else 32 if M <= 32 else 64)
            for N in ns:
                for K in ks:
                    formula, res = sweep_shape(path, M, N, K, seed=len(entries) + 1)
                    if not res:
                        continue
                    best = min(res, key=res.get)
                    entries.append((which, bucket, N, K, best))
                    gain = res[formula] / res[best] if formula in res else float("nan")
                    lines.append(f"    {{{which}, {bucket}, {N}, {K}, {best}}},   // {path} M={M}: rule {formula} "
                                 f"{res.get(formula, float('nan')):.2f} us, best {res[best]:.2f} us "
                                 f"(x{gain:.3f}); " + " ".join(f"{s}:{t:.2f}" for s, t in sorted(res.items())))
                    print(lines[-1].strip(), flush=True)
    dev = torch.cuda.get_device_name()
    with open(args.out, "w") as f:
        f.write("// Measured split-K table, consulted by the planner before its shape-derived\n"
                "// rule. Written by block_scaled_fp4_mxfp4_gb300/tune_splits.py; every entry is\n"
                "// checked for parity by tests/test_gpu_split_table.py.\n"
                "// {which, bucket, N, K, splits}: which 0 = two-kernel GEMM path (bucket =\n"
                "// 128-row tiles of M), 1 = fused MXFP4, 2 = fused NVFP4 (bucket = MMA width).\n"
                f"// Measured on {dev}: CUDA-graph replay, weights rotated past twice the L2;\n"
                "// each line gives the rule's K-splits and time, the best, and every count timed.\n"
                "static const mxfp4::SplitEntry kSplitTable[] = {\n")
        for line in lines:
            f.write(line + "\n")
        f.write("    {-1, 0, 0, 0, 0},   // end\n};\n")
    print(f"wrote {len(entries)} entries to {args.out} in {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main()
