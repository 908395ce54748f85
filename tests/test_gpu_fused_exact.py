"""Bit-exact check of the quantization the fused kernels do on chip.

mxfp4_quant_gemm_fused and nvfp4_quant_gemm_fused quantize bf16 A inside the
GEMM (kernelbot-amd-mxfp4-mm-517169, "Optimization 5": the quantized A never
reaches global memory), so their codes and scales can only be seen through C.
C's contract tolerance (2^-8 * sum |a b| + 1e-3) is far too loose to see one
wrong code, a lost sign or a scale byte off by one. Here B is a permutation
matrix scaled by a power of two (MXFP4) or by 6 (NVFP4): weight row n holds one
nonzero, at column k = (n + off) % K, whose quantization is exact. Then every
output is one dequantized A element times that constant,
    C[m, n] = A_hat[m, (n + off) % K] * b_hat,
exactly representable in C's type, and every other product is an exact zero.
C is compared for equality with the oracle's own dequantized A (only the sign
of zero is ignored), so every code and every scale of every nonzero block that
the fused kernel formed on chip is checked bit for bit.

The rows come from every finite bf16 value placed in blocks under anchors that
span the whole exponent range, from zero and signed-zero blocks, bf16
subnormals, block maxima in [6, 8) and the heavy-tailed medium activations, at
M = 1, 16, 33 and the full row set (MMA widths 16, 32 and 64)."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import assert_bytes_equal, dev_bf16, host

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")

K = 2048
# block maxima over the whole bf16 range: E8M0 scales from 2^-127 to 2^125,
# E4M3 scales that round to zero, subnormal E4M3 scales (0.01 .. 0.05), normal
# ones, and the saturated 448
ANCHORS = [2.0 ** -130, 2.0 ** -126, 2.0 ** -125, 1e-20, 0.01, 0.03, 0.05, 0.25, 0.75, 1.0, 5.0, 6.0,
           7.9375, 100.0, 2.0 ** 60, 3.0e38]


def finite_bf16_bits() -> np.ndarray:
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return bits[((bits >> 7) & 0xFF) != 0xFF]


def anchored_rows(anchor: float, vec: int, rows: int = 64) -> np.ndarray:
    """rows x K bf16 bits: every block starts with +-anchor (alternating sign)
    and holds further finite values of magnitude <= anchor, cycling through all
    of them (a fresh permutation per pass), so each appears at least once."""
    vals = finite_bf16_bits()
    mag = np.abs(wl.bf16_bits_to_float(vals).astype(np.float64))
    ab = wl.to_bf16_bits(np.array([anchor]))[0]
    amag = float(wl.bf16_bits_to_float(np.array([ab]))[0])
    pool = vals[mag <= amag]
    nblk = rows * K // vec
    need = nblk * (vec - 1)
    rng = np.random.default_rng(int(ab) * 7 + vec)
    reps = -(-need // pool.size)
    body = np.concatenate([rng.permutation(pool) for _ in range(reps)])[:need]
    blk = np.empty((nblk, vec), np.uint16)
    blk[:, 0] = np.where(np.arange(nblk) % 2 == 0, ab, ab | 0x8000)
    blk[:, 1:] = body.reshape(nblk, vec - 1)
    # the anchor moves around inside its block
    shift = np.arange(nblk) % vec
    idx = (np.arange(vec)[None, :] - shift[:, None]) % vec
    blk = np.take_along_axis(blk, idx, axis=1)
    return blk.reshape(rows, K)


def edge_rows(vec: int, tiny: bool) -> np.ndarray:
    """tiny=False: zero and signed-zero blocks, block maxima in [6, 8) and a
    single nonzero per block, mixed with ordinary N(0, 4) blocks.
    tiny=True: zero and signed-zero blocks and blocks of bf16 subnormals (kept
    apart so that one power-of-two B keeps every output of the call normal)."""
    rows = 64
    x = wl.gen_bf16(71 + tiny, 3, rows, K, "normal", 2.0).copy()
    nb = K // vec
    for r in range(rows):
        for b in range(nb):
            sl = slice(b * vec, (b + 1) * vec)
            kind = (r * nb + b) % (4 if tiny else 7)
            if kind == 0:
                x[r, sl] = 0                                  # all +0
            elif kind == 1:
                x[r, sl] = 0x8000                             # all -0
            elif tiny and kind == 2:
                x[r, sl] = np.where(np.arange(vec) % 2, 0x8000, 0)
                x[r, b * vec + (r % vec)] = 0x8001 if r % 2 else 0x0001   # one subnormal
            elif tiny:
                sub = (np.arange(vec, dtype=np.uint16) * 3 + r) & 0x7F
                x[r, sl] = sub | np.where(np.arange(vec) % 3 == 0, 0x8000, 0).astype(np.uint16)
            elif kind == 2:
                amax = [6.0, 6.5, 7.0, 7.5, 7.9375][(r + b) % 5]
                x[r, sl] = wl.to_bf16_bits(np.linspace(-amax, amax, vec))
            elif kind == 3:
                x[r, sl] = 0
                x[r, b * vec + (b % vec)] = wl.to_bf16_bits(np.array([-3.0 * (1 + r % 4)]))[0]
            # kinds 4-6: the N(0, 4) values stay
    return x


def heavy_rows() -> np.ndarray:
    """The medium workload's heavy-tailed activations (outliers x50, zeros,
    zeroed blocks), its first 64 rows and first K columns."""
    return np.ascontiguousarray(wl.gen_a(wl.MEDIUM, M=64)[:, :K])


def b_value(vec: int, a_bits: np.ndarray) -> float:
    """The nonzero of B. NVFP4: 6 (E4M3 scale 1.0, code 6: exact), so C = 6 A_hat
    stays inside fp16 for every A. MXFP4: 2^j with j = -e of the largest block
    exponent, so every A_hat * 2^j is a normal float that bf16 holds exactly."""
    if vec == 16:
        return 6.0
    amax = np.max(np.abs(wl.bf16_bits_to_float(a_bits).astype(np.float64)))
    if amax == 0.0 or amax < 2.0 ** -126:
        return 2.0 ** 125
    e = max(-127, int(np.floor(np.log2(amax))) - 2)
    return 2.0 ** max(-125, min(125, -e))


_B_CACHE = {}


def identity_b(vec: int, bval: float, off: int):
    """Device (codes, scales) of the scaled permutation B and its dequantized
    nonzero, checked against the oracle's quantization of the same B."""
    key = (vec, bval, off, K)
    if key not in _B_CACHE:
        N = K
        b = np.zeros((N, K))
        b[np.arange(N), (np.arange(N) + off) % K] = bval
        b_bits = wl.to_bf16_bits(b)
        quant = mx.mxfp4_quantize if vec == 32 else mx.nvfp4_quantize
        oquant = oracle.mx_quantize if vec == 32 else oracle.nv_quantize
        qb, sfb = quant(dev_bf16(b_bits))
        qb_r, sfb_r = oquant(b_bits)
        torch.cuda.synchronize()
        assert_bytes_equal(host(qb), qb_r, "B codes")
        assert_bytes_equal(host(sfb), sfb_r, "B scales")
        bhat = oracle.dequant(qb_r, sfb_r, K, vec)
        assert np.all(bhat[np.arange(N), (np.arange(N) + off) % K] == bval), "B's nonzero must quantize exactly"
        assert np.count_nonzero(bhat) == N
        _B_CACHE.clear()
        _B_CACHE[key] = (qb, sfb)
    return _B_CACHE[key]


def run_identity(a_bits: np.ndarray, vec: int, off: int, what: str):
    M = a_bits.shape[0]
    N = K
    bval = b_value(vec, a_bits)
    qb, sfb = identity_b(vec, bval, off)
    oquant = oracle.mx_quantize if vec == 32 else oracle.nv_quantize
    plan = mx.gemm_plan(M, N, K, fused=True, nvfp4=(vec == 16))
    assert plan["kernel"] == "fused_quant_gemm_kernel", plan
    A = dev_bf16(a_bits)
    if vec == 32:
        C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        mx.mxfp4_quant_gemm_fused(A, qb, sfb, C)
    else:
        C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        mx.nvfp4_quant_gemm_fused(A, qb, sfb, C)
    torch.cuda.synchronize()
    qa_r, sfa_r = oquant(a_bits)
    ahat = oracle.dequant(qa_r, sfa_r, K, vec)
    want = ahat[:, (np.arange(N) + off) % K] * bval
    got = C.double().cpu().numpy()
    bad = np.argwhere(~(got == want))
    if bad.size:
        m, n = bad[0]
        k = (n + off) % K
        raise AssertionError(
            f"{what}: {len(bad)} of {M * N} outputs differ; first C[{m},{n}] = {got[m, n]!r}, "
            f"want {want[m, n]!r} (A[{m},{k}] bf16 0x{int(a_bits[m, k]):04x}, block {k // vec})")
    assert mx.get_device_error() == 0


def row_sets(vec):
    sets = [(f"anchor {a:g}", anchored_rows(a, vec)) for a in ANCHORS]
    sets.append(("edge blocks", edge_rows(vec, False)))
    sets.append(("subnormal blocks", edge_rows(vec, True)))
    sets.append(("medium heavy-tail rows", heavy_rows()))
    return sets


@pytest.mark.parametrize("vec", [32, 16], ids=["mxfp4", "nvfp4"])
def test_fused_on_chip_quantization_is_bit_exact(vec):
    for name, rows in row_sets(vec):
        for M in (64, 33, 16, 1):
            a = np.ascontiguousarray(rows[:M])
            for off in (0, 37 * 32 + 5):
                run_identity(a, vec, off, f"{'MXFP4' if vec == 32 else 'NVFP4'} {name}, M={M}, off={off}")


@pytest.mark.parametrize("vec", [32, 16], ids=["mxfp4", "nvfp4"])
def test_fused_identity_decode_depth(vec):
    """K = 7168 (the decode depth): several K-stages per CTA of each K-split
    cluster, all of them checked through the same exact identity."""
    global K
    saved = K
    K = 7168
    try:
        a = np.concatenate([wl.gen_a(wl.DECODE), edge_rows(vec, False)[:16]])[:32]
        a = np.ascontiguousarray(a)
        for M in (16, 32):
            run_identity(np.ascontiguousarray(a[:M]), vec, 3 * 32 + 1, f"decode depth M={M}")
    finally:
        K = saved
