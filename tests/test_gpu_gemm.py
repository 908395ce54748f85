"""GPU MXFP4 GEMM (tcgen05 kind::mxf4) and the fused quant+GEMM vs the oracle.

Both sides start from the same seeded bf16 A and B; each side quantizes them
itself (the quantized bytes are compared bit-exactly on the way) and C is
checked element by element against the oracle's dequantize-then-double GEMM:
|C_gpu - C_ref| <= 2^-8 * sum_k |a_k b_k| + 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import assert_bytes_equal, assert_within_tolerance, c_f64, dev_bf16, host

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")


def quant_both(bits):
    q, sf = mx.mxfp4_quantize(dev_bf16(bits))
    q_ref, sf_ref = oracle.mx_quantize(bits)
    assert_bytes_equal(host(q), q_ref, "codes")
    assert_bytes_equal(host(sf), sf_ref, "scales")
    return q, sf, q_ref, sf_ref


def inputs(M, N, K, seed, a_scale=1.0, b_scale=1.0):
    a = wl.gen_bf16(seed, 1, M, K, "normal", a_scale)
    b = wl.gen_bf16(seed, 2, N, K, "normal", b_scale)
    return a, b


GEMM_SHAPES = [
    (1, 1, 32), (8, 512, 1024), (128, 256, 256), (130, 300, 96), (256, 512, 512),
    (200, 384, 2080), (16, 512, 4096), (16, 640, 4096), (64, 1000, 1536), (300, 130, 64), (129, 257, 288),
    # enough tiles for 256-wide tiles: ragged second half-tile, a partial last K stage
    (1300, 1900, 320),
    # at least one 256 x 256 tile per SM pair: the CTA-pair kernel. 80 tiles (some
    # pairs take a second tile); then ragged M (the second CTA of the last tile row
    # has no rows), ragged N (no second B half) and K = 96 (half an MMA step of zeros)
    (2560, 2048, 128), (2100, 2100, 96),
    # 81 pair tiles = 76 + 5: a second wave of five tiles on the ragged last tile
    # row (its last tile 152 columns wide, the second CTA with 124 rows), K of
    # five stages, the last one partial
    (2300, 2200, 1056),
]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_a4w4(M, N, K):
    a, b = inputs(M, N, K, 100 + M + N + K)
    qa, sfa, qa_r, sfa_r = quant_both(a)
    qb, sfb, qb_r, sfb_r = quant_both(b)
    C = mx.mxfp4_gemm_a4w4(qa, sfa, qb, sfb, K)
    torch.cuda.synchronize()
    c_ref, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, K, 32)
    assert_within_tolerance(c_f64(C), c_ref, s, f"gemm {M}x{N}x{K}")
    assert mx.get_device_error() == 0


FUSED_SHAPES = [
    (1, 128, 256), (8, 512, 1024), (16, 2112, 7168), (16, 200, 96), (5, 130, 4128),
    (17, 384, 768), (32, 256, 2048), (33, 300, 512), (64, 640, 1024),      # fused small-M path
    (65, 256, 512), (130, 300, 96), (256, 512, 2048),                       # quant -> GEMM path
    (2300, 2200, 1056),                                                     # ... on CTA pairs, ragged edges
]


@pytest.mark.parametrize("M,N,K", FUSED_SHAPES)
def test_quant_gemm_fused(M, N, K):
    a, b = inputs(M, N, K, 200 + M + N + K, b_scale=0.02)
    qb, sfb, qb_r, sfb_r = quant_both(b)
    ws = mx.new_workspace(M, N, K)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    qa_r, sfa_r = oracle.mx_quantize(a)
    c_ref, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, K, 32)
    for i in range(2):  # the second call checks the workspace was left reusable
        C.fill_(float("nan"))
        mx.mxfp4_quant_gemm_fused(dev_bf16(a), qb, sfb, C, ws)
        torch.cuda.synchronize()
        assert_within_tolerance(c_f64(C), c_ref, s, f"fused {M}x{N}x{K} call {i}")
    assert mx.get_device_error() == 0


def test_fused_matches_two_kernel_path_bitwise_on_quant():
    """The fused path's on-chip quantization equals the standalone kernel's: its
    C equals the GEMM of the standalone-quantized A up to accumulation order."""
    M, N, K = 16, 512, 2048
    a, b = inputs(M, N, K, 7, a_scale=3.0)
    qb, sfb, _, _ = quant_both(b)
    A = dev_bf16(a)
    C1 = mx.mxfp4_quant_gemm_fused(A, qb, sfb)
    qa, sfa = mx.mxfp4_quantize(A)
    C2 = mx.mxfp4_gemm_a4w4(qa, sfa, qb, sfb, K)
    torch.cuda.synchronize()
    d = (C1.float() - C2.float()).abs()
    assert float(d.max()) <= 2.0 ** -7 * float(C2.float().abs().max()) + 1e-3


def test_single_nonzero_probe_pins_nibble_and_scale_placement():
    """One nonzero element in A and B: C is nonzero in exactly one place, with
    the product of the two dequantized values."""
    M, N, K = 130, 260, 512
    for (m, n, k) in [(0, 0, 0), (1, 2, 1), (129, 259, 511), (37, 140, 200), (64, 7, 33)]:
        a = np.zeros((M, K)); a[m, k] = 3.0
        b = np.zeros((N, K)); b[n, k] = -0.75
        qa, sfa, _, _ = quant_both(wl.to_bf16_bits(a))
        qb, sfb, _, _ = quant_both(wl.to_bf16_bits(b))
        C = c_f64(mx.mxfp4_gemm_a4w4(qa, sfa, qb, sfb, K))
        want = np.zeros((M, N)); want[m, n] = -2.25
        assert np.array_equal(C, want), (m, n, k, np.argwhere(C != want)[:5])


def test_gemm_rejects_bad_arguments_without_launching():
    qa = torch.zeros((8, 512), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    C = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.mxfp4_gemm_a4w4(qa, sf, qa[:, :512], sf, 1024, C[:, :8], ws)
    assert e.value.status == 4  # workspace too small
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.mxfp4_gemm_a4w4(qa, sf, qa, sf, 1000, C, mx.new_workspace(8, 8, 1024))
    assert e.value.status == 2


@pytest.mark.parametrize("M,N,K,S", [(16, 640, 4096, 3), (200, 384, 2080, 6)])
def test_gemm_workspace_split_k(M, N, K, S):
    """K-splits (forced by the override; the planner picks one split unless its
    table says otherwise) write fp32 partials to the workspace and the last
    split to arrive sums them; with and without the epilogue extras."""
    a, b = inputs(M, N, K, 400 + M + N + K)
    qa, sfa, qa_r, sfa_r = quant_both(a)
    qb, sfb, qb_r, sfb_r = quant_both(b)
    c_in_bits = wl.gen_bf16(401 + M, 3, M, N)
    old = mx.set_split_override("gemm", S)
    try:
        plan = mx.gemm_plan(M, N, K)
        assert plan["kernel"] == "bs_gemm_kernel" and plan["splits"] == S, plan
        C = mx.mxfp4_gemm_a4w4(qa, sfa, qb, sfb, K)
        Ce = dev_bf16(c_in_bits).clone()
        mx.mxfp4_gemm_a4w4_ex(qa, sfa, qb, sfb, K, Ce, alpha=0.5, beta=-1.0)
        torch.cuda.synchronize()
    finally:
        mx.set_split_override("gemm", old)
    c_ref, s = oracle.gemm_full(qa_r, sfa_r, qb_r, sfb_r, K, 32)
    assert_within_tolerance(c_f64(C), c_ref, s, f"workspace split-K {S}: {M}x{N}x{K}")
    c_in = wl.bf16_bits_to_float(c_in_bits).astype(np.float64)
    ce_ref, se = oracle.gemm_epilogue(c_ref, s, 0.5, -1.0, c_in, None)
    assert_within_tolerance(c_f64(Ce), ce_ref, se, f"workspace split-K {S} with epilogue")
    assert mx.get_device_error() == 0
