"""Parity at the benchmark's full workload sizes, through the same calls and the
same seeded generators bench.py times.

Small workloads are compared element by element; large ones on sampled outputs
(random (m, n) pairs plus whole rows and columns), each computed by the oracle
one by one from its own quantization of the same bf16 inputs. Quantized bytes
and scales are compared bit-exactly in full."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import (assert_bytes_equal, assert_within_tolerance, c_f64, dev_bf16, gemm_sampled_parallel, host,
                      sample_pairs)

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")


def run_mx_workload(w, sampled):
    a_bits, b_bits = wl.gen_a(w), wl.gen_b(w)
    A = dev_bf16(a_bits)
    Bq, Bsf = mx.mxfp4_quantize(dev_bf16(b_bits))
    C = torch.full((w.M, w.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = mx.new_workspace(w.M, w.N, w.K)
    mx.mxfp4_quant_gemm_fused(A, Bq, Bsf, C, ws)          # the call bench.py times
    Aq, Asf = mx.mxfp4_quantize(A)                       # A's bytes, for the bit-exact check
    torch.cuda.synchronize()
    qb_r, sfb_r = oracle.mx_quantize(b_bits)
    assert_bytes_equal(host(Bq), qb_r, f"{w.name} B codes")
    assert_bytes_equal(host(Bsf), sfb_r, f"{w.name} B scales")
    qa_r, sfa_r = oracle.mx_quantize(a_bits)
    assert_bytes_equal(host(Aq), qa_r, f"{w.name} A codes")
    assert_bytes_equal(host(Asf), sfa_r, f"{w.name} A scales")
    if not sampled:
        c_ref, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, w.K, 32)
        assert_within_tolerance(c_f64(C), c_ref, s, w.name)
    else:
        rows, cols = sample_pairs(w.M, w.N, *sampled, seed=17)
        c_ref, s = gemm_sampled_parallel(qa_r, sfa_r, qb_r, sfb_r, w.K, 32, rows, cols)
        got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].float().cpu().numpy()
        assert_within_tolerance(got.astype(np.float64), c_ref, s, w.name + " (sampled)")
    assert mx.get_device_error() == 0


def test_tiny_full():
    run_mx_workload(wl.TINY, None)


def test_decode_full():
    run_mx_workload(wl.DECODE, None)


def test_medium_heavy_tail_sampled():
    run_mx_workload(wl.MEDIUM, (16384, 2, 2))


def test_compute_8192_sampled():
    # 65,536 random outputs plus 16 whole rows and 16 whole columns
    run_mx_workload(wl.COMPUTE, (65536, 16, 16))


def test_nvfp4_grouped_sampled():
    w = wl.NVFP4_GROUPED
    groups, refs = [], []
    for g in range(len(w.Ms)):
        a_bits, b_bits = wl.gen_nv_group(w, g)
        qa, sfa = mx.nvfp4_quantize(dev_bf16(a_bits))
        qb, sfb = mx.nvfp4_quantize(dev_bf16(b_bits))
        c = torch.full((w.Ms[g], w.N), float("nan"), dtype=torch.float16, device="cuda")
        groups.append(dict(a=qa, sfa=sfa, b=qb, sfb=sfb, c=c, k=w.K))
        refs.append((a_bits, b_bits, qa, sfa, qb, sfb))
    mx.nvfp4_group_gemm(groups)                          # the call bench.py times
    torch.cuda.synchronize()
    for g, (gd, (a_bits, b_bits, qa, sfa, qb, sfb)) in enumerate(zip(groups, refs)):
        qa_r, sfa_r = oracle.nv_quantize(a_bits)
        qb_r, sfb_r = oracle.nv_quantize(b_bits)
        assert_bytes_equal(host(qa), qa_r, f"group {g} A codes")
        assert_bytes_equal(host(sfa), sfa_r, f"group {g} A scales")
        assert_bytes_equal(host(qb), qb_r, f"group {g} B codes")
        assert_bytes_equal(host(sfb), sfb_r, f"group {g} B scales")
        rows, cols = sample_pairs(w.Ms[g], w.N, 2048, 1, 1, seed=40 + g)
        c_ref, s = oracle.gemm_sampled(qa_r, sfa_r, qb_r, sfb_r, w.K, 16, rows, cols)
        got = gd["c"][torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].float().cpu().numpy()
        assert_within_tolerance(got.astype(np.float64), c_ref, s, f"nvfp4 group {g} (sampled)")
    assert mx.get_device_error() == 0


def test_plans_of_the_benchmarked_calls():
    """The kernel each benchmarked call launches (what bench.py reports)."""
    p = mx.gemm_plan(wl.DECODE.M, wl.DECODE.N, wl.DECODE.K, fused=True)
    assert p["kernel"] == "fused_quant_gemm_kernel" and p["tile_m"] == 16 and p["tiles"] == 17
    assert 1 <= p["splits"] <= 8 and not p["quant_launch"]
    p = mx.gemm_plan(wl.MEDIUM.M, wl.MEDIUM.N, wl.MEDIUM.K, fused=True)
    assert p["kernel"] == "bs_gemm_kernel" and (p["tile_m"], p["tile_n"]) == (128, 128) and p["quant_launch"]
    p = mx.gemm_plan(wl.COMPUTE.M, wl.COMPUTE.N, wl.COMPUTE.K)
    assert p["kernel"] == "bs_gemm_pair_kernel" and p["tiles"] == 32 * 32 and p["splits"] == 1
    w = wl.NVFP4_GROUPED
    groups = []
    for m in w.Ms:
        groups.append(dict(a=torch.zeros((m, w.K // 2), dtype=torch.uint8, device="cuda"),
                           sfa=torch.zeros(mx.sf_bytes(m, w.K, 16), dtype=torch.uint8, device="cuda"),
                           b=torch.zeros((w.N, w.K // 2), dtype=torch.uint8, device="cuda"),
                           sfb=torch.zeros(mx.sf_bytes(w.N, w.K, 16), dtype=torch.uint8, device="cuda"),
                           c=torch.zeros((m, w.N), dtype=torch.float16, device="cuda"), k=w.K))
    p = mx.nvfp4_group_gemm_plan(mx.make_nv_problems(groups))
    assert p["kernel"] == "bs_gemm_pair_kernel"
    assert p["tiles"] == sum((m + 255) // 256 for m in w.Ms) * (w.N // 256)


def test_mxfp4_grouped_sampled():
    w = wl.MXFP4_GROUPED
    groups, refs = [], []
    for g in range(len(w.Ms)):
        a_bits, b_bits = wl.gen_nv_group(w, g)
        qa, sfa = mx.mxfp4_quantize(dev_bf16(a_bits))
        qb, sfb = mx.mxfp4_quantize(dev_bf16(b_bits))
        c = torch.full((w.Ms[g], w.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        groups.append(dict(a=qa, sfa=sfa, b=qb, sfb=sfb, c=c, k=w.K))
        refs.append((a_bits, b_bits))
    problems = mx.make_mx_problems(groups)
    assert mx.mxfp4_group_gemm_plan(problems)["kernel"] == "bs_gemm_pair_kernel"
    mx.mxfp4_group_gemm(groups, problems)                 # the call bench.py times
    torch.cuda.synchronize()
    for g, (gd, (a_bits, b_bits)) in enumerate(zip(groups, refs)):
        qa_r, sfa_r = oracle.mx_quantize(a_bits)
        qb_r, sfb_r = oracle.mx_quantize(b_bits)
        assert_bytes_equal(host(gd["a"]), qa_r, f"group {g} A codes")
        assert_bytes_equal(host(gd["sfb"]), sfb_r, f"group {g} B scales")
        rows, cols = sample_pairs(w.Ms[g], w.N, 2048, 1, 1, seed=60 + g)
        c_ref, s = oracle.gemm_sampled(qa_r, sfa_r, qb_r, sfb_r, w.K, 32, rows, cols)
        got = gd["c"][torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].float().cpu().numpy()
        assert_within_tolerance(got.astype(np.float64), c_ref, s, f"mxfp4 group {g} (sampled)")
    assert mx.get_device_error() == 0


def test_nvfp4_grouped_bf16_sampled():
    """The bf16-activation grouped call bench.py times: C_g sampled against the
    oracle, which quantizes the same bf16 A_g itself."""
    w = wl.NVFP4_GROUPED_BF16
    groups, refs = [], []
    for g in range(len(w.Ms)):
        a_bits, b_bits = wl.gen_nv_group(w, g)
        qb, sfb = mx.nvfp4_quantize(dev_bf16(b_bits))
        c = torch.full((w.Ms[g], w.N), float("nan"), dtype=torch.float16, device="cuda")
        groups.append(dict(a=dev_bf16(a_bits), b=qb, sfb=sfb, c=c))
        refs.append((a_bits, b_bits))
    problems = mx.make_nv_act_problems(groups)
    mx.nvfp4_group_quant_gemm(groups, problems)
    torch.cuda.synchronize()
    for g, (gd, (a_bits, b_bits)) in enumerate(zip(groups, refs)):
        qa_r, sfa_r = oracle.nv_quantize(a_bits)
        qb_r, sfb_r = oracle.nv_quantize(b_bits)
        assert_bytes_equal(host(gd["b"]), qb_r, f"group {g} B codes")
        rows, cols = sample_pairs(w.Ms[g], w.N, 2048, 1, 1, seed=80 + g)
        c_ref, s = oracle.gemm_sampled(qa_r, sfa_r, qb_r, sfb_r, w.K, 16, rows, cols)
        got = gd["c"][torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].float().cpu().numpy()
        assert_within_tolerance(got.astype(np.float64), c_ref, s, f"nvfp4 bf16-A group {g} (sampled)")
    assert mx.get_device_error() == 0
