"""Stream order of back-to-back calls under programmatic dependent launch.

The GEMM kernels request their first weight stages before their dependency
wait, and the quantization of a quant -> GEMM call lets its GEMM start early.
The header promises that weights written by this library's quantization calls
are still read in stream order. Here every step re-quantizes new weights into
the SAME buffers and runs the GEMM right after, on one stream with no
synchronization in between; each step's C must equal, bit for bit, the same
step run alone with the device synchronized around every call. A GEMM that
read the previous step's weights (or a quantization that read A early) would
produce the previous step's product."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")

STEPS = 6

# (label, M, N, K, kernel the plan must name): the fused small-M kernel, the
# single-CTA GEMM and the CTA-pair GEMM, each through the quant -> GEMM call
# and through the GEMM on pre-quantized A.
CASES = [
    ("fused", 16, 2112, 7168, "fused_quant_gemm_kernel"),
    ("single", 256, 1024, 2048, "bs_gemm_kernel"),
    ("pair", 2560, 2048, 512, "bs_gemm_pair_kernel"),
]


def inputs(M, N, K, seed):
    a = [dev_bf16(wl.gen_bf16(seed + s, 1, M, K)) for s in range(STEPS)]
    b = [dev_bf16(wl.gen_bf16(seed + s, 2, N, K, "normal", 0.05)) for s in range(STEPS)]
    return a, b


@pytest.mark.parametrize("label,M,N,K,kernel", CASES)
@pytest.mark.parametrize("path", ["quant_gemm", "gemm"])
def test_requantized_weights_are_read_in_stream_order(label, M, N, K, kernel, path):
    plan = mx.gemm_plan(M, N, K, fused=path == "quant_gemm")
    if path == "gemm" and kernel == "fused_quant_gemm_kernel":
        kernel = "bs_gemm_kernel"   # the plain GEMM has no fused path
    assert plan["kernel"] == kernel, plan
    a, b = inputs(M, N, K, 900 + M)
    Bq, Bsf = mx.mxfp4_quantize(b[0])           # the shared weight buffers
    Aq, Asf = mx.mxfp4_quantize(a[0])           # shared quantized-A buffers (gemm path)
    ws = mx.new_workspace(M, N, K)
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(STEPS)]

    def step(s):
        mx.mxfp4_quantize(b[s], Bq, Bsf)
        if path == "quant_gemm":
            mx.mxfp4_quant_gemm_fused(a[s], Bq, Bsf, outs[s], ws)
        else:
            mx.mxfp4_quantize(a[s], Aq, Asf)
            mx.mxfp4_gemm_a4w4(Aq, Asf, Bq, Bsf, K, outs[s], ws)

    torch.cuda.synchronize()
    for s in range(STEPS):        # back to back on one stream
        step(s)
    torch.cuda.synchronize()
    assert mx.get_device_error() == 0
    got = [o.clone() for o in outs]
    for s in range(STEPS):        # each step alone
        torch.cuda.synchronize()
        step(s)
        torch.cuda.synchronize()
        assert torch.equal(got[s].view(torch.int16), outs[s].view(torch.int16)), \
            f"{label}/{path}: step {s} differs from the same step run alone"
    # the steps really differ, so a stale read could not pass unseen
    assert not torch.equal(got[0], got[1])
    assert mx.get_device_error() == 0


def test_requantized_grouped_weights_are_read_in_stream_order():
    """The grouped NVFP4 GEMM (CTA pairs) with weights re-quantized before
    every call into the same buffers."""
    shapes = [(512, 2048, 1024), (1024, 2048, 1024), (768, 2048, 1024), (256, 2048, 1024)]
    groups = []
    for g, (m, n, k) in enumerate(shapes):
        qa, sfa = mx.nvfp4_quantize(dev_bf16(wl.gen_bf16(70 + g, 1, m, k)))
        qb, sfb = mx.nvfp4_quantize(dev_bf16(wl.gen_bf16(80 + g, 2, n, k)))
        groups.append(dict(a=qa, sfa=sfa, b=qb, sfb=sfb, c=torch.empty((m, n), dtype=torch.float16, device="cuda"),
                           k=k))
    bsrc = [[dev_bf16(wl.gen_bf16(90 + 10 * s + g, 2, n, k)) for g, (m, n, k) in enumerate(shapes)]
            for s in range(STEPS)]
    problems = mx.make_nv_problems(groups)
    assert mx.nvfp4_group_gemm_plan(problems)["kernel"] == "bs_gemm_pair_kernel"

    def step(s):
        for g, grp in enumerate(groups):
            mx.nvfp4_quantize(bsrc[s][g], grp["b"], grp["sfb"])
        mx.nvfp4_group_gemm(groups, problems)
        return [grp["c"].clone() for grp in groups]

    torch.cuda.synchronize()
    got = [step(s) for s in range(STEPS)]     # clones are stream-ordered copies
    torch.cuda.synchronize()
    for s in range(STEPS):
        torch.cuda.synchronize()
        want = step(s)
        torch.cuda.synchronize()
        for g in range(len(groups)):
            assert torch.equal(got[s][g].view(torch.int16), want[g].view(torch.int16)), \
                f"grouped: step {s} group {g} differs from the same step run alone"
    assert mx.get_device_error() == 0
