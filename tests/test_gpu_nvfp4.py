"""GPU grouped NVFP4 GEMM (tcgen05 kind::mxf4nvf4, E4M3 per 16, fp16 C) vs the
oracle. Operands are quantized from seeded bf16 on each side (bytes compared
bit-exactly), then every C_g is checked against the double-precision GEMM."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import assert_bytes_equal, assert_within_tolerance, c_f64, dev_bf16, host

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")


def nv_both(bits):
    q, sf = mx.nvfp4_quantize(dev_bf16(bits))
    q_ref, sf_ref = oracle.nv_quantize(bits)
    assert_bytes_equal(host(q), q_ref, "nv codes")
    assert_bytes_equal(host(sf), sf_ref, "nv scales")
    return q, sf, q_ref, sf_ref


def run_groups(shapes, seed):
    groups, refs = [], []
    for i, (m, n, k) in enumerate(shapes):
        a = wl.gen_bf16(seed, 10 + 2 * i, m, k)
        b = wl.gen_bf16(seed, 11 + 2 * i, n, k)
        qa, sfa, qa_r, sfa_r = nv_both(a)
        qb, sfb, qb_r, sfb_r = nv_both(b)
        c = torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
        groups.append(dict(a=qa, sfa=sfa, b=qb, sfb=sfb, c=c, k=k))
        refs.append((qa_r, sfa_r, qb_r, sfb_r, k))
    mx.nvfp4_group_gemm(groups)
    torch.cuda.synchronize()
    for (m, n, k), g, (qa_r, sfa_r, qb_r, sfb_r, _) in zip(shapes, groups, refs):
        c_ref, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, k, 16)
        assert_within_tolerance(c_f64(g["c"]), c_ref, s, f"nvfp4 group {m}x{n}x{k}")
    assert mx.get_device_error() == 0


def test_single_group_small():
    run_groups([(128, 256, 256)], 1)


def test_groups_ragged_m_n_k():
    run_groups([(64, 256, 512), (1, 130, 16), (130, 300, 272), (257, 512, 1024), (200, 64, 48)], 2)


def test_eight_groups_small_k():
    shapes = [(m, 512, 256) for m in (64, 128, 256, 384, 512, 640, 768, 1024)]
    run_groups(shapes, 3)


def test_groups_on_cta_pairs_ragged():
    # 110 tiles of 256 x 256 in total: the CTA-pair kernel; ragged M, N and K
    run_groups([(100, 2600, 272), (700, 2600, 512), (1300, 2600, 96)], 3)


def test_sixteen_groups_max():
    shapes = [(16 + 8 * i, 128 + 64 * (i % 3), 128 + 32 * (i % 4)) for i in range(16)]
    run_groups(shapes, 4)


def test_probe_single_nonzero():
    m_, n_, k_ = 130, 260, 512
    for (m, n, k) in [(0, 0, 0), (129, 259, 511), (40, 140, 17), (3, 200, 300)]:
        a = np.zeros((m_, k_)); a[m, k] = 1.5
        b = np.zeros((n_, k_)); b[n, k] = -1.5
        qa, sfa, _, _ = nv_both(wl.to_bf16_bits(a))
        qb, sfb, _, _ = nv_both(wl.to_bf16_bits(b))
        c = torch.zeros((m_, n_), dtype=torch.float16, device="cuda")
        mx.nvfp4_group_gemm([dict(a=qa, sfa=sfa, b=qb, sfb=sfb, c=c, k=k_)])
        C = c_f64(c)
        want = np.zeros((m_, n_)); want[m, n] = -2.25
        assert np.array_equal(C, want), (m, n, k, np.argwhere(C != want)[:5])


def test_sixty_four_groups_device_table():
    """More than 16 problems: the problem table goes into the workspace and one
    GEMM launch covers all of them (single-CTA kernel, ragged shapes)."""
    shapes = [(1 + 9 * i, 64 + 64 * (i % 5), 64 + 64 * (i % 3)) for i in range(64)]
    run_groups(shapes, 5)


def test_groups_on_cta_pairs_device_table():
    """24 problems with 96 tiles of 256 x 256 in total: the CTA-pair kernel
    reading its problems from the device table."""
    shapes = [(256 + 7 * (i % 3), 1024 - 48 * (i % 2), 128 + 64 * (i % 4)) for i in range(24)]
    groups = [dict(a=torch.zeros((m, k // 2), dtype=torch.uint8, device="cuda"),
                   sfa=torch.zeros(mx.sf_bytes(m, k, 16), dtype=torch.uint8, device="cuda"),
                   b=torch.zeros((n, k // 2), dtype=torch.uint8, device="cuda"),
                   sfb=torch.zeros(mx.sf_bytes(n, k, 16), dtype=torch.uint8, device="cuda"),
                   c=torch.zeros((m, n), dtype=torch.float16, device="cuda"), k=k) for (m, n, k) in shapes]
    assert mx.nvfp4_group_gemm_plan(mx.make_nv_problems(groups))["kernel"] == "bs_gemm_pair_kernel"
    del groups
    run_groups(shapes, 6)


def test_device_table_is_rewritten_between_calls():
    """Two different long problem lists through one workspace, each checked."""
    ws = mx.group_workspace(40)
    for rnd, seed in enumerate((7, 8)):
        shapes = [(3 + 5 * i + rnd, 128 + 64 * ((i + rnd) % 3), 128) for i in range(40 - 10 * rnd)]
        groups, refs = [], []
        for i, (m, n, k) in enumerate(shapes):
            a = wl.gen_bf16(seed, 10 + 2 * i, m, k)
            b = wl.gen_bf16(seed, 11 + 2 * i, n, k)
            qa, sfa, qa_r, sfa_r = nv_both(a)
            qb, sfb, qb_r, sfb_r = nv_both(b)
            c = torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
            groups.append(dict(a=qa, sfa=sfa, b=qb, sfb=sfb, c=c, k=k))
            refs.append((qa_r, sfa_r, qb_r, sfb_r, k))
        mx.nvfp4_group_gemm(groups, workspace=ws)
        torch.cuda.synchronize()
        for (m, n, k), g, (qa_r, sfa_r, qb_r, sfb_r, _) in zip(shapes, groups, refs):
            c_ref, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, k, 16)
            assert_within_tolerance(c_f64(g["c"]), c_ref, s, f"round {rnd} group {m}x{n}x{k}")
    assert mx.get_device_error() == 0
