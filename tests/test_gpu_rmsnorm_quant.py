"""GPU fused RMSNorm + MXFP4 quantization (mxfp4_rmsnorm_quantize) vs the
oracle's reading of it: codes and E8M0 scale bytes bit-exact on ragged shapes,
strided rows, several eps values, zero rows and rows whose norm is a power of
two; the output also feeds the MXFP4 GEMM like mxfp4_quantize's does."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import assert_bytes_equal, assert_within_tolerance, c_f64, dev_bf16, host

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")


def check(X_bits, w_bits, eps, pad_cols=0, what=""):
    X = dev_bf16(X_bits, pad_cols=pad_cols)
    w = dev_bf16(w_bits[None, :])[0].contiguous()
    q, sf = mx.mxfp4_rmsnorm_quantize(X, w, eps)
    torch.cuda.synchronize()
    q_ref, sf_ref = oracle.rmsnorm_mx_quantize(X_bits, w_bits, eps)
    assert_bytes_equal(host(q), q_ref, f"codes {what}")
    assert_bytes_equal(host(sf)[:sf_ref.size], sf_ref, f"scales {what}")
    return q, sf


@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (37, 256), (130, 288), (16, 7168), (200, 2048)])
def test_shapes(M, K):
    X = wl.gen_bf16(11, 1, M, K)
    w = wl.gen_bf16(11, 2, 1, K)[0]
    check(X, w, 1e-6, what=f"{M}x{K}")


def test_strided_rows_and_eps_values():
    X = wl.gen_bf16(12, 1, 70, 160, dist="uniform", scale=3.0)
    w = wl.gen_bf16(12, 2, 1, 160)[0]
    for eps in (0.0, 1e-5, 0.5, 100.0):
        check(X, w, eps, pad_cols=8, what=f"eps={eps}")


def test_zero_rows_power_of_two_rows_and_wide_range():
    K = 128
    rows = [np.zeros(K), np.full(K, 2.0 ** -30), np.full(K, -(2.0 ** 40)),
            np.where(np.arange(K) % 3 == 0, 1e-9, 7.5),      # magnitudes 2^33 apart: still exact
            np.where(np.arange(K) % 5 == 0, 3e4, -2e-5)]
    X = wl.to_bf16_bits(np.array(rows))
    X[0, 5] = 0x8000                                           # a -0 in the zero row
    w = wl.gen_bf16(13, 2, 1, K)[0]
    for eps in (0.0, 1e-6):
        check(X, w, eps, what=f"special rows eps={eps}")


def test_feeds_the_gemm():
    M, N, K = 64, 256, 1024
    X = wl.gen_bf16(14, 1, M, K)
    w = wl.gen_bf16(14, 2, 1, K)[0]
    B = wl.gen_bf16(14, 3, N, K)
    qa, sfa = check(X, w, 1e-6, what="gemm operand")
    qb, sfb = mx.mxfp4_quantize(dev_bf16(B))
    C = mx.mxfp4_gemm_a4w4(qa, sfa, qb, sfb, K)
    torch.cuda.synchronize()
    qa_r, sfa_r = oracle.rmsnorm_mx_quantize(X, w, 1e-6)
    qb_r, sfb_r = oracle.mx_quantize(B)
    c_ref, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, K, 32)
    assert_within_tolerance(c_f64(C), c_ref, s, "rmsnorm-quantized GEMM")
    assert mx.get_device_error() == 0
