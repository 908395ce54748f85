"""The no-allocation MXFP4 GEMM (mxfp4_gemm_a4w4_noalloc) against the regular
entry point (mxfp4_gemm_a4w4, which takes a caller-allocated workspace).

The variant exists for callers that cannot allocate device memory themselves,
such as a plugin inside an engine that owns all device allocations, or a
program whose memory plan is fixed at start-up: its split-K scratch lives in a
fixed device array inside the library. Called twice in a row on each shape,
its result must match the regular entry point's and the oracle within the
tolerance the other tests use. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import assert_within_tolerance, c_f64, dev_bf16

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")


@pytest.mark.parametrize("M,N,K,splits", [(16, 640, 4096, 0),    # one split: tickets only
                                          (16, 640, 4096, 3),    # split-K: partials + tickets in the array
                                          (130, 300, 96, 0),     # ragged, no split
                                          (64, 1000, 1536, 0)])
def test_noalloc_gemm_matches_regular_entry_point_twice(M, N, K, splits):
    old = mx.set_split_override("gemm", splits)
    try:
        run_noalloc_twice(M, N, K)
    finally:
        mx.set_split_override("gemm", old)


def run_noalloc_twice(M, N, K):
    a = wl.gen_bf16(300 + M, 1, M, K)
    b = wl.gen_bf16(300 + M, 2, N, K)
    qa, sfa = mx.mxfp4_quantize(dev_bf16(a))
    qb, sfb = mx.mxfp4_quantize(dev_bf16(b))
    C_regular = mx.mxfp4_gemm_a4w4(qa, sfa, qb, sfb, K)
    qa_r, sfa_r = oracle.mx_quantize(a)
    qb_r, sfb_r = oracle.mx_quantize(b)
    c_ref, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, K, 32)
    torch.cuda.synchronize()
    regular = c_f64(C_regular)
    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        status = mx.lib().mxfp4_gemm_a4w4_noalloc(
            qa.data_ptr(), qa.stride(0), sfa.data_ptr(), qb.data_ptr(), qb.stride(0), sfb.data_ptr(),
            C.data_ptr(), C.stride(0), M, N, K, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert status == 0, mx.STATUS.get(status, status)
        torch.cuda.synchronize()
        got = c_f64(C)
        assert_within_tolerance(got, regular, s, f"noalloc vs regular {M}x{N}x{K} call {call}")
        assert_within_tolerance(got, c_ref, s, f"noalloc vs oracle {M}x{N}x{K} call {call}")
    assert mx.get_device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """M=128, N=8192, K=16384 with 3 K-splits (forced by the override) plans
    12.6 MB of partials > the 8 MiB array; the call is rejected on the host
    (the plan is checked before the pointers are used)."""
    assert mx.lib().mxfp4_noalloc_scratch_bytes() == 8 << 20
    M, N, K = 128, 8192, 16384
    old = mx.set_split_override("gemm", 3)
    try:
        plan = mx.gemm_plan(M, N, K)
        assert plan["splits"] == 3, plan
        aq = torch.zeros(16, dtype=torch.uint8, device="cuda")
        status = mx.lib().mxfp4_gemm_a4w4_noalloc(aq.data_ptr(), K // 2, aq.data_ptr(), aq.data_ptr(), K // 2,
                                                  aq.data_ptr(), aq.data_ptr(), N, M, N, K, None)
    finally:
        mx.set_split_override("gemm", old)
    assert status == 4  # MXFP4_ERR_WORKSPACE_TOO_SMALL, nothing enqueued
