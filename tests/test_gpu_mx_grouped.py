"""GPU grouped MXFP4 GEMM (tcgen05 kind::mxf4, E8M0 per 32, bf16 C) vs the
oracle: each group's operands are quantized on both sides (bytes compared
bit-exactly), then every C_g is checked element by element against the
oracle's dequantize-then-double GEMM within 2^-8 * sum|a b| + 1e-3."""
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import assert_bytes_equal, assert_within_tolerance, c_f64, dev_bf16, host

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")


def mx_both(bits):
    q, sf = mx.mxfp4_quantize(dev_bf16(bits))
    q_ref, sf_ref = oracle.mx_quantize(bits)
    assert_bytes_equal(host(q), q_ref, "mx codes")
    assert_bytes_equal(host(sf), sf_ref, "mx scales")
    return q, sf, q_ref, sf_ref


def run_groups(shapes, seed, kernel=None):
    groups, refs = [], []
    for i, (m, n, k) in enumerate(shapes):
        a = wl.gen_bf16(seed, 10 + 2 * i, m, k)
        b = wl.gen_bf16(seed, 11 + 2 * i, n, k)
        qa, sfa, qa_r, sfa_r = mx_both(a)
        qb, sfb, qb_r, sfb_r = mx_both(b)
        c = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        groups.append(dict(a=qa, sfa=sfa, b=qb, sfb=sfb, c=c, k=k))
        refs.append((qa_r, sfa_r, qb_r, sfb_r, k))
    problems = mx.make_mx_problems(groups)
    if kernel is not None:
        assert mx.mxfp4_group_gemm_plan(problems)["kernel"] == kernel
    mx.mxfp4_group_gemm(groups, problems)
    torch.cuda.synchronize()
    for (m, n, k), g, (qa_r, sfa_r, qb_r, sfb_r, _) in zip(shapes, groups, refs):
        c_ref, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, k, 32)
        assert_within_tolerance(c_f64(g["c"]), c_ref, s, f"mxfp4 group {m}x{n}x{k}")
    assert mx.get_device_error() == 0


def test_single_group():
    run_groups([(128, 256, 256)], 1, "bs_gemm_kernel")


def test_groups_ragged_m_n_k():
    run_groups([(64, 256, 512), (1, 130, 32), (130, 300, 288), (257, 512, 1024), (200, 64, 64)], 2,
               "bs_gemm_kernel")


def test_groups_on_cta_pairs_ragged():
    # 110 tiles of 256 x 256: the CTA-pair kernel; ragged M, N and K
    run_groups([(100, 2600, 288), (700, 2600, 512), (1300, 2600, 96)], 3, "bs_gemm_pair_kernel")


def test_sixteen_groups_max():
    shapes = [(16 + 8 * i, 128 + 64 * (i % 3), 128 + 32 * (i % 4)) for i in range(16)]
    run_groups(shapes, 4)


def test_matches_the_single_problem_gemm():
    """A one-group call and mxfp4_gemm_a4w4 on the same operands agree."""
    M, N, K = 300, 520, 1024
    a = wl.gen_bf16(5, 1, M, K)
    b = wl.gen_bf16(5, 2, N, K)
    qa, sfa = mx.mxfp4_quantize(dev_bf16(a))
    qb, sfb = mx.mxfp4_quantize(dev_bf16(b))
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    mx.mxfp4_group_gemm([dict(a=qa, sfa=sfa, b=qb, sfb=sfb, c=c, k=K)])
    ref = mx.mxfp4_gemm_a4w4(qa, sfa, qb, sfb, K)
    torch.cuda.synchronize()
    d = (c.float() - ref.float()).abs()
    assert float(d.max()) <= 2.0 ** -7 * float(ref.float().abs().max()) + 1e-3


def test_forty_groups_device_table():
    """More than 16 MXFP4 problems through the device problem table."""
    shapes = [(2 + 11 * i, 64 + 64 * (i % 4), 64 + 32 * (i % 5)) for i in range(40)]
    run_groups(shapes, 9, "bs_gemm_kernel")


def test_groups_on_cta_pairs_device_table():
    shapes = [(256 + 5 * (i % 4), 1024, 128 + 64 * (i % 2)) for i in range(20)]
    run_groups(shapes, 10, "bs_gemm_pair_kernel")
