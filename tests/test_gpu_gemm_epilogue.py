"""mxfp4_gemm_a4w4_ex: the GEMM epilogue extras (alpha, beta, bias) on every
GEMM kernel path (single CTA with 128- and 256-wide tiles, split-K, CTA pairs)
against the oracle's fp64 product and epilogue, within
2^-8 * (|alpha| * sum|a b| + |beta * C_in| + |bias|) + 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import assert_within_tolerance, c_f64, dev_bf16

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")

SHAPES = [
    ((130, 300, 96), "bs_gemm_kernel", 1),          # 128-wide tiles, ragged
    ((16, 640, 4096), "bs_gemm_kernel", 4),         # 4 K-splits (forced): epilogue in the final reduction
    ((1300, 1900, 320), "bs_gemm_kernel", 1),       # 256-wide tiles
    ((2100, 2100, 96), "bs_gemm_pair_kernel", 1),   # CTA pairs, ragged
]


def quant_pair(M, N, K, seed):
    a = wl.gen_bf16(seed, 1, M, K)
    b = wl.gen_bf16(seed, 2, N, K)
    qa, sfa = mx.mxfp4_quantize(dev_bf16(a))
    qb, sfb = mx.mxfp4_quantize(dev_bf16(b))
    qa_r, sfa_r = oracle.mx_quantize(a)
    qb_r, sfb_r = oracle.mx_quantize(b)
    return (qa, sfa, qb, sfb), (qa_r, sfa_r, qb_r, sfb_r)


@pytest.mark.parametrize("shape,kernel,splits", SHAPES)
@pytest.mark.parametrize("alpha,beta,use_bias", [(0.5, -1.25, True), (2.0, 0.0, False), (1.0, 1.0, True)])
def test_epilogue_matches_oracle(shape, kernel, splits, alpha, beta, use_bias):
    old = mx.set_split_override("gemm", splits if splits > 1 else 0)
    try:
        epilogue_case(shape, kernel, splits, alpha, beta, use_bias)
    finally:
        mx.set_split_override("gemm", old)


def epilogue_case(shape, kernel, splits, alpha, beta, use_bias):
    M, N, K = shape
    plan = mx.gemm_plan(M, N, K)
    assert plan["kernel"] == kernel and plan["splits"] == splits, plan
    (qa, sfa, qb, sfb), (qa_r, sfa_r, qb_r, sfb_r) = quant_pair(M, N, K, 90 + M)
    c_in_bits = wl.gen_bf16(91 + M, 3, M, N)
    bias_bits = wl.gen_bf16(92 + M, 4, 1, N).reshape(N)
    C = dev_bf16(c_in_bits).clone()
    bias = dev_bf16(bias_bits.reshape(1, N)).reshape(N) if use_bias else None
    mx.mxfp4_gemm_a4w4_ex(qa, sfa, qb, sfb, K, C, alpha=alpha, beta=beta, bias=bias)
    torch.cuda.synchronize()
    c_acc, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, K, 32)
    c_in = wl.bf16_bits_to_float(c_in_bits).astype(np.float64)
    b = wl.bf16_bits_to_float(bias_bits).astype(np.float64) if use_bias else None
    c_ref, S = oracle.gemm_epilogue(c_acc, s, alpha, beta, c_in, b)
    assert_within_tolerance(c_f64(C), c_ref, S, f"epilogue {M}x{N}x{K} a={alpha} b={beta} bias={use_bias}")
    assert mx.get_device_error() == 0


def test_identity_epilogue_is_the_plain_gemm_bitwise():
    M, N, K = 130, 300, 96
    (qa, sfa, qb, sfb), _ = quant_pair(M, N, K, 93)
    plain = mx.mxfp4_gemm_a4w4(qa, sfa, qb, sfb, K)
    ex = mx.mxfp4_gemm_a4w4_ex(qa, sfa, qb, sfb, K, alpha=1.0, beta=0.0, bias=None)
    torch.cuda.synchronize()
    assert torch.equal(plain, ex)
