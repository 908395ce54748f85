"""The kernels' bounded waits, made to run out on purpose.

Every wait of a kernel on an mbarrier (a TMA stage landing, the MMAs freeing a
stage, the accumulator being complete, the other CTA of a pair) gives up after
a limit, records a code in the library's device error word and lets the kernel
leave cleanly: it waits (with the default 2 s limit) for every copy and MMA it
issued, frees its TMEM and exits, so the context stays usable. With the limit
set to 1 ns no operand can arrive in time, so the waits give up on their own
(nothing is broken, no wait is endless). The test checks that the timeout is
reported and that the next call, with the default limit, is bit-identical to
the same call made before: TMEM was returned and nothing was left in flight."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")

# (call, M, N, K, kernel the plan must name, range of the recorded code); the
# split-K case forces 4 K-splits through the planner's override. The
# fused shapes give each CTA more K-stages than its weight ring has slots, so
# that its producer must wait for MMAs: a wait long enough for the GPU's
# timer to see the limit pass (the fused kernel's other waits can all end
# within one tick of that timer).
CASES = {
    "gemm": ("gemm", 256, 512, 2048, "bs_gemm_kernel", (1, 15)),
    "gemm_splitk": ("gemm", 16, 640, 4096, "bs_gemm_kernel", (1, 15)),
    "fused_mxfp4": ("fused", 16, 8192, 7168, "fused_quant_gemm_kernel", (17, 31)),
    "fused_nvfp4": ("fused_nv", 16, 8192, 7168, "fused_quant_gemm_kernel", (17, 31)),
    "pair": ("gemm", 2560, 2048, 512, "bs_gemm_pair_kernel", (33, 47)),
}


def make_call(kind, M, N, K):
    a = wl.gen_bf16(500 + M, 1, M, K)
    b = wl.gen_bf16(500 + M, 2, N, K, "normal", 0.02)
    A, B = dev_bf16(a), dev_bf16(b)
    if kind == "fused_nv":
        qb, sfb = mx.nvfp4_quantize(B)

        def call():
            return mx.nvfp4_quant_gemm_fused(A, qb, sfb)
        return call
    qb, sfb = mx.mxfp4_quantize(B)
    if kind == "fused":
        def call():
            return mx.mxfp4_quant_gemm_fused(A, qb, sfb, workspace=mx.new_workspace(M, N, K))
        return call
    qa, sfa = mx.mxfp4_quantize(A)

    def call():
        return mx.mxfp4_gemm_a4w4(qa, sfa, qb, sfb, K, workspace=mx.new_workspace(M, N, K))
    return call


@pytest.mark.parametrize("name", list(CASES))
def test_short_wait_limit_gives_up_cleanly_and_recovers(name):
    old = mx.set_split_override("gemm", 4 if name == "gemm_splitk" else 0)
    try:
        wait_limit_case(name)
    finally:
        mx.set_split_override("gemm", old)


def wait_limit_case(name):
    kind, M, N, K, kernel, (lo, hi) = CASES[name]
    plan = mx.gemm_plan(M, N, K, fused=kind != "gemm", nvfp4=kind == "fused_nv")
    assert plan["kernel"] == kernel, plan
    if name == "gemm_splitk":
        assert plan["splits"] > 1, plan
    call = make_call(kind, M, N, K)
    before = call()
    torch.cuda.synchronize()
    assert mx.get_device_error() == 0
    want = before.view(torch.int16).cpu().numpy()
    timeouts = 0
    for attempt in range(4):
        old = mx.set_wait_limit_ns(1)
        try:
            call()
        finally:
            mx.set_wait_limit_ns(0)
        code = mx.get_device_error()          # synchronizes the device
        assert code == 0 or lo <= code <= hi, f"{name} attempt {attempt}: device error code {code}"
        timeouts += code != 0
        after = call()
        torch.cuda.synchronize()
        assert mx.get_device_error() == 0, f"{name} attempt {attempt}: the default-limit call also gave up"
        got = after.view(torch.int16).cpu().numpy()
        assert np.array_equal(got, want), f"{name} attempt {attempt}: the call after the timeout differs"
    assert old == 2_000_000_000
    assert timeouts >= 2, f"{name}: only {timeouts} of 4 calls with a 1 ns limit gave up"
