"""GPU fused NVFP4 quant + GEMM (nvfp4_quant_gemm_fused, M <= 64) vs the oracle:
A is quantized on chip (E4M3 per 16, the oracle's nvfp4 rule); B is quantized
by nvfp4_quantize (bytes compared with the oracle's); C (fp16) is checked
element by element against the oracle's dequantize-then-double GEMM of the
oracle's own quantization of A and B."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import assert_bytes_equal, assert_within_tolerance, c_f64, dev_bf16, host

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")

SHAPES = [
    (1, 128, 256), (8, 512, 1024), (16, 2112, 7168), (16, 200, 96), (5, 130, 4128), (17, 384, 768),
    (32, 256, 2048), (33, 300, 512), (64, 640, 1024), (3, 96, 16),
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_nvfp4_fused(M, N, K):
    a = wl.gen_bf16(200 + M, 1, M, K)
    b = wl.gen_bf16(200 + M, 2, N, K, "normal", 0.02)
    qb, sfb = mx.nvfp4_quantize(dev_bf16(b))
    qb_r, sfb_r = oracle.nv_quantize(b)
    assert_bytes_equal(host(qb), qb_r, "B codes")
    assert_bytes_equal(host(sfb), sfb_r, "B scales")
    qa_r, sfa_r = oracle.nv_quantize(a)
    c_ref, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, K, 16)
    A = dev_bf16(a)
    for _ in range(2):   # the second call reuses the same buffers
        C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        mx.nvfp4_quant_gemm_fused(A, qb, sfb, C)
        torch.cuda.synchronize()
        assert_within_tolerance(c_f64(C), c_ref, s, f"nvfp4 fused {M}x{N}x{K}")
    assert mx.get_device_error() == 0


def test_fused_agrees_with_quantize_then_group_gemm():
    """On-chip quantization gives the same A as nvfp4_quantize: the fused call
    and nvfp4_quantize + nvfp4_group_gemm agree to accumulation order."""
    M, N, K = 16, 1024, 4096
    a = wl.gen_bf16(210, 1, M, K)
    b = wl.gen_bf16(210, 2, N, K, "normal", 0.02)
    A = dev_bf16(a)
    qb, sfb = mx.nvfp4_quantize(dev_bf16(b))
    fused = mx.nvfp4_quant_gemm_fused(A, qb, sfb)
    qa, sfa = mx.nvfp4_quantize(A)
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    mx.nvfp4_group_gemm([dict(a=qa, sfa=sfa, b=qb, sfb=sfb, c=c, k=K)])
    torch.cuda.synchronize()
    d = (fused.float() - c.float()).abs()
    assert float(d.max()) <= 2.0 ** -8 * float(c.float().abs().max()) + 1e-3


def test_decode_shape_workload_full():
    """The benchmarked NVFP4 decode call on the workload's own inputs."""
    w = wl.NVFP4_DECODE
    a_bits, b_bits = wl.gen_a(w), wl.gen_b(w)
    qb, sfb = mx.nvfp4_quantize(dev_bf16(b_bits))
    C = mx.nvfp4_quant_gemm_fused(dev_bf16(a_bits), qb, sfb)
    torch.cuda.synchronize()
    qa_r, sfa_r = oracle.nv_quantize(a_bits)
    qb_r, sfb_r = oracle.nv_quantize(b_bits)
    assert_bytes_equal(host(sfb), sfb_r, "B scales")
    c_ref, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, w.K, 16)
    assert_within_tolerance(c_f64(C), c_ref, s, w.name)
    assert mx.get_device_error() == 0
