"""GPU grouped NVFP4 GEMM from bf16 activations (nvfp4_group_quant_gemm: every
A_g quantized in the call, then the grouped GEMM) vs the oracle: the oracle
quantizes the same seeded bf16 A_g with its own NVFP4 rule and computes each C_g
in double precision. Each C_g must also equal, bit for bit, what the standalone
nvfp4_quantize + nvfp4_group_gemm pair produces (same quantized operands, same
GEMM kernel), and the workspace's quantized A_g must equal the oracle's bytes."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import assert_bytes_equal, assert_within_tolerance, c_f64, dev_bf16, host

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")


def up(x, a):
    return (x + a - 1) // a * a


def run(shapes, seed, a_pad_cols=0):
    groups, refs, plain = [], [], []
    for i, (m, n, k) in enumerate(shapes):
        a_bits = wl.gen_bf16(seed, 20 + 2 * i, m, k)
        b_bits = wl.gen_bf16(seed, 21 + 2 * i, n, k)
        a = dev_bf16(a_bits, pad_cols=a_pad_cols)
        qb, sfb = mx.nvfp4_quantize(dev_bf16(b_bits))
        qb_r, sfb_r = oracle.nv_quantize(b_bits)
        assert_bytes_equal(host(qb), qb_r, "B codes")
        c = torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
        groups.append(dict(a=a, b=qb, sfb=sfb, c=c))
        refs.append((oracle.nv_quantize(a_bits), qb_r, sfb_r, k))
        qa, sfa = mx.nvfp4_quantize(a)
        plain.append(dict(a=qa, sfa=sfa, b=qb, sfb=sfb, k=k,
                          c=torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")))
    problems = mx.make_nv_act_problems(groups)
    ws_bytes = mx.nvfp4_group_quant_gemm_workspace_bytes(problems)
    ws = torch.full((ws_bytes,), 0xA5, dtype=torch.uint8, device="cuda")   # not zero: no reliance on it
    mx.nvfp4_group_quant_gemm(groups, problems, workspace=ws)
    mx.nvfp4_group_gemm(plain)
    torch.cuda.synchronize()
    off = 0
    w = host(ws)
    for (m, n, k), g, p, ((qa_r, sfa_r), qb_r, sfb_r, _) in zip(shapes, groups, plain, refs):
        ldq = up(k // 2, 16)
        got_q = w[off:off + m * ldq].reshape(m, ldq)[:, :k // 2]
        off += up(m * ldq, 256)
        nsf = mx.sf_bytes(m, k, 16)
        got_sf = w[off:off + nsf]
        off += up(nsf, 256)
        assert_bytes_equal(got_q, qa_r, f"workspace A codes {m}x{k}")
        assert_bytes_equal(got_sf, sfa_r, f"workspace A scales {m}x{k}")
        c_ref, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, k, 16)
        assert_within_tolerance(c_f64(g["c"]), c_ref, s, f"group {m}x{n}x{k}")
        assert torch.equal(g["c"], p["c"]), f"group {m}x{n}x{k} differs from quantize + group GEMM"
    assert mx.get_device_error() == 0


def test_single_group():
    run([(128, 256, 256)], 1)


def test_ragged_groups_single_cta_kernel():
    run([(64, 256, 512), (1, 130, 16), (130, 300, 272), (257, 512, 1024), (200, 64, 48)], 2)


def test_ragged_groups_cta_pairs_strided_a():
    # 110 pair tiles: the CTA-pair GEMM; A rows carry 8 extra columns
    run([(100, 2600, 272), (700, 2600, 512), (1300, 2600, 96)], 3, a_pad_cols=8)


def test_sixteen_groups():
    run([(8 + 40 * i, 128 + 64 * (i % 3), 64 + 48 * (i % 4)) for i in range(16)], 4)


def test_thirty_five_groups():
    """More than 16 groups: the quantization runs in launches of 16 groups and
    the GEMM reads its problems from the table after the quantized A_g."""
    run([(3 + 17 * i, 64 + 64 * (i % 4), 64 + 32 * (i % 5)) for i in range(35)], 5)
