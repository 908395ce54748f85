"""GPU quantization kernels vs the oracle: packed codes and every byte of the
blocked scale buffer (pads included) must match bit-exactly."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import assert_bytes_equal, dev_bf16, host

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")


def finite_bf16_bits() -> np.ndarray:
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return bits[((bits >> 7) & 0xFF) != 0xFF]


def anchored_blocks(vec: int) -> np.ndarray:
    """Every finite bf16 value at several block scales: each block's first
    element is an anchor magnitude, the rest are all values not above it."""
    vals = finite_bf16_bits()
    mag = wl.bf16_bits_to_float(vals).astype(np.float64)
    anchors = [2.0 ** -130, 2.0 ** -126, 1e-20, 0.75, 1.0, 5.0, 6.0, 7.9375, 2.0 ** 60, 3.0e38]
    rows = []
    for i, a in enumerate(anchors):
        ab = wl.to_bf16_bits(np.array([a if i % 2 == 0 else -a]))[0]
        amag = abs(wl.bf16_bits_to_float(np.array([ab]))[0])
        pool = vals[np.abs(mag) <= amag]
        per = vec - 1
        nblk = -(-pool.size // per)
        pool = np.concatenate([pool, np.zeros(nblk * per - pool.size, np.uint16)])
        blk = np.empty((nblk, vec), np.uint16)
        blk[:, 0] = ab
        blk[:, 1:] = pool.reshape(nblk, per)
        rows.append(blk.reshape(-1))
    flat = np.concatenate(rows)
    K = 1024
    flat = np.concatenate([flat, np.zeros((-flat.size) % K, np.uint16)])
    return flat.reshape(-1, K)


def run_both(bits: np.ndarray, vec: int, pad_cols: int = 0, ldq_pad: int = 0):
    M, K = bits.shape
    A = dev_bf16(bits, pad_cols)
    Aq = torch.full((M, K // 2 + ldq_pad), 0xAB, dtype=torch.uint8, device="cuda")[:, :K // 2]
    sf = torch.full((mx.sf_bytes(M, K, vec),), 0xCD, dtype=torch.uint8, device="cuda")
    fn = mx.mxfp4_quantize if vec == 32 else mx.nvfp4_quantize
    fn(A, Aq, sf)
    torch.cuda.synchronize()
    q_ref, sf_ref = (oracle.mx_quantize if vec == 32 else oracle.nv_quantize)(bits)
    assert_bytes_equal(host(Aq), q_ref, f"codes vec={vec} {M}x{K}")
    assert_bytes_equal(host(sf), sf_ref, f"scales vec={vec} {M}x{K}")


@pytest.mark.parametrize("vec", [32, 16])
def test_every_finite_bf16_natural_blocks(vec):
    bits = finite_bf16_bits().reshape(255, 256)
    run_both(bits, vec)


@pytest.mark.parametrize("vec", [32, 16])
def test_every_finite_bf16_at_anchored_scales(vec):
    run_both(anchored_blocks(vec), vec)


@pytest.mark.parametrize("vec", [32, 16])
@pytest.mark.parametrize("M,K", [(1, 32), (1, 16 * 3), (7, 96), (130, 96), (257, 288), (128, 256),
                                 (3, 4096), (200, 160)])
def test_ragged_shapes(vec, M, K):
    if K % vec:
        pytest.skip("K not a multiple of the block")
    bits = wl.gen_bf16(40, M * 7 + K, M, K, "normal", 3.0)
    run_both(bits, vec)


@pytest.mark.parametrize("vec", [32, 16])
def test_strided_rows(vec):
    bits = wl.gen_bf16(41, 1, 37, 512)
    run_both(bits, vec, pad_cols=64, ldq_pad=48)


@pytest.mark.parametrize("name", ["mxfp4_tiny_M8_N512_K1024", "mxfp4_decode_M16_N2112_K7168",
                                  "mxfp4_medium_heavytail_M256_N7168_K2048"])
def test_workload_activations(name):
    w = wl.MX_WORKLOADS[name]
    run_both(wl.gen_a(w), 32)


def test_zero_blocks_and_signed_zeros():
    bits = np.zeros((4, 64), np.uint16)
    bits[1, :] = 0x8000                   # all -0
    bits[2, 5] = 0x8001                   # one negative subnormal
    bits[3, :32] = wl.to_bf16_bits(np.linspace(-6, 6, 32))
    run_both(bits, 32)
    run_both(bits, 16)
