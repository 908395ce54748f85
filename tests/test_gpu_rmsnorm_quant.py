"""GPU fused RMSNorm + MXFP4 quantization (mxfp4_rmsnorm_quantize) vs the
oracle's reading of it: codes and E8M0 scale bytes bit-exact on ragged shapes,
strided rows, several eps values, zero rows and rows whose norm is a power of
two; the output also feeds the MXFP4 GEMM like mxfp4_quantize's does."""
import math

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


# ------------------------------------------------------- exact sum of squares
def bf16_row(values, K):
    """Row of K bf16 values (the given ones first, then zeros); every value
    must be exactly representable in bf16."""
    row = np.zeros(K)
    row[:len(values)] = values
    bits = wl.to_bf16_bits(row[None, :])[0]
    assert np.array_equal(oracle._bf16_bits_to_f64(bits), row), "value not representable in bf16"
    return bits


def exact_sumsq(bits):
    x = oracle._bf16_bits_to_f64(bits)
    return math.fsum((x * x).tolist())   # each square is exact in fp64; fsum rounds the exact total once


def check_stats(X_bits, w_bits, eps, what):
    X = dev_bf16(X_bits)
    w = dev_bf16(w_bits[None, :])[0].contiguous()
    q, sf, rstd, ss = mx.mxfp4_rmsnorm_quantize(X, w, eps, stats=True)
    torch.cuda.synchronize()
    M, K = X_bits.shape
    ss_ref = np.array([exact_sumsq(X_bits[m]) for m in range(M)])
    got = host(ss)
    bad = np.flatnonzero(got.view(np.int64) != ss_ref.view(np.int64))
    assert bad.size == 0, f"{what}: rows {bad[:5]} sum of squares {got[bad[:5]]!r} != {ss_ref[bad[:5]]!r}"
    e = float(np.float32(eps))
    r_ref = np.array([np.float32(0.0 if s / K + e == 0.0 else 1.0 / math.sqrt(s / K + e)) for s in ss_ref],
                     dtype=np.float32)
    assert np.array_equal(host(rstd).view(np.int32), r_ref.view(np.int32)), f"{what}: rstd"
    q_ref, sf_ref = oracle.rmsnorm_mx_quantize(X_bits, w_bits, eps)
    assert_bytes_equal(host(q), q_ref, f"codes {what}")
    assert_bytes_equal(host(sf)[:sf_ref.size], sf_ref, f"scales {what}")
    return got


def tie_rows():
    """Rows whose squares at most 2^80 below the largest square sum to an exact
    fp64 tie (or just below one), and whose squares further below decide the
    rounding. Returns (values, what the retained squares alone round to)."""
    rows = []
    # 1 + 2^-54 + 2^-54 is the midpoint of 1 and 1 + 2^-52; one square of
    # 2^-122 (|x| = 2^-61, 2^61 below the largest) breaks the tie upwards
    rows.append([1.0, 2.0 ** -27, 2.0 ** -27, 2.0 ** -61])
    # the same tie alone rounds to even (1.0)
    rows.append([1.0, 2.0 ** -27, 2.0 ** -27])
    # 2^40 + (2^-13 - 2^-40) lies 2^-40 below the midpoint of 2^40 and
    # 2^40 + 2^-12; 256 squares of 2^-42 (2^41 below the largest |x|) add 2^-34,
    # more than one unit of a 2^-80-relative window, and carry it over
    vals = [2.0 ** 20]
    for i in range(14, 41):
        vals += [2.0 ** (-i / 2)] if i % 2 == 0 else [2.0 ** (-(i + 1) / 2)] * 2
    rows.append(vals + [2.0 ** -21] * 256)
    rows.append(vals)                      # without them: rounds down
    # the largest bf16 exponent with subnormal squares below it (a 2^260 span)
    rows.append([1.5 * 2.0 ** 127, -(2.0 ** -133), 3 * 2.0 ** -133, 2.0 ** 100, -(2.0 ** -60)])
    return rows


def test_sum_of_squares_is_exact_across_any_range():
    K = 384
    rows = tie_rows()
    X = np.stack([bf16_row(v, K) for v in rows])
    # pins on the construction: the squares far below decide the rounding
    s = [exact_sumsq(X[i]) for i in range(len(rows))]
    assert s[0] == 1.0 + 2.0 ** -52 and s[1] == 1.0
    assert s[2] == 2.0 ** 40 + 2.0 ** -12 and s[3] == 2.0 ** 40
    w = wl.gen_bf16(15, 2, 1, K)[0]
    for eps in (0.0, 1e-6):
        check_stats(X, w, eps, f"tie rows eps={eps}")


def test_sum_of_squares_exponent_boundaries():
    """Values at exactly 16, 17, 40 and 41 binades below the largest (the
    limits of the 64-bit, 128-bit and limb paths), all-subnormal rows and rows
    whose largest value is tiny (every square takes the 128-bit path)."""
    K = 64
    rows = []
    for top in (0.0, -60.0, 90.0, 127.0):
        big = 2.0 ** top * 1.75
        rows.append([big] + [1.5 * 2.0 ** (top - d) for d in (15, 16, 17, 39, 40, 41, 42)])
    rows.append([3 * 2.0 ** -133, 2.0 ** -133, 127 * 2.0 ** -133])          # subnormals only
    rows.append([2.0 ** -110, 2.0 ** -111, 2.0 ** -126, 5 * 2.0 ** -133])   # largest field 17 / 16
    rows.append([2.0 ** -112, 2.0 ** -120, 2.0 ** -133])
    rows.append([])                                                         # zeros
    X = np.stack([bf16_row(v, K) for v in rows])
    check_stats(X, wl.gen_bf16(16, 2, 1, K)[0], 1e-6, "boundaries")
    # with eps = 0 the all-subnormal row has r = 2^129, beyond fp32 (outside
    # the documented domain: every |y| finite); the others keep a finite r
    keep = [i for i in range(len(rows)) if i != 4]
    assert exact_sumsq(X[4]) / K < 2.0 ** -256
    check_stats(X[keep], wl.gen_bf16(16, 2, 1, K)[0], 0.0, "boundaries eps=0")


def test_sum_of_squares_random_wide_rows():
    """Random rows whose magnitudes span up to 2^200 (every path, shared
    atomics from many threads), several row lengths including chunked rows."""
    rng = np.random.default_rng(17)
    for M, K in ((9, 7168), (4, 2048), (3, 139264)):
        e = rng.integers(-100, 100, size=(M, K))
        x = np.ldexp(rng.uniform(1.0, 2.0, size=(M, K)), e) * rng.choice([-1.0, 1.0], size=(M, K))
        x[rng.random((M, K)) < 0.1] = 0.0
        X = wl.to_bf16_bits(x)
        check_stats(X, wl.gen_bf16(18, 2, 1, K)[0], 1e-6, f"wide {M}x{K}")


def test_sum_of_squares_gaussian_rows_match_fsum():
    """Ordinary activations (the fast path) and the 4096 x 7168 shape."""
    X = wl.gen_bf16(19, 1, 64, 7168)
    check_stats(X, wl.gen_bf16(19, 2, 1, 7168)[0], 1e-6, "gaussian 64x7168")


# ---------------------------------------------------------------- r decided
def near_midpoint_rows(count, eps, seed=23, n=1 << 20):
    """Rows of 32 values m * 2^-7 (|m| <= 255, exact in bf16; their sum of
    squares is exact in fp64) whose r64 = 1 / sqrt(ss / 32 + eps) lies closest
    to an fp32 rounding midpoint, found among n random rows; with n = 2^20 the
    closest lie within ~2^-44 (relative) of a midpoint, well inside the band
    where the kernel must fall back to the fp64 sequence."""
    rng = np.random.default_rng(seed)
    m = rng.integers(-255, 256, size=(n, 32), dtype=np.int32)
    ss = (m * m).sum(axis=1).astype(np.float64) * 2.0 ** -14
    e = float(np.float32(eps))
    r64 = 1.0 / np.sqrt(ss / 32 + e)
    c = r64.astype(np.float32)
    up = np.nextafter(c, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(c, np.float32(0)).astype(np.float64)
    c64 = c.astype(np.float64)
    dist = np.minimum(np.abs(r64 - (c64 + up) / 2), np.abs(r64 - (c64 + dn) / 2)) / r64
    pick = np.argsort(dist)[:count]
    return m[pick].astype(np.float64) * 2.0 ** -7, dist[pick]


@pytest.mark.parametrize("eps", [1e-6, 0.0, 3.0])
def test_rstd_near_fp32_rounding_midpoints(eps):
    """r equals RN32 of the fp64 sequence also when that value lies within
    2^-38 of an fp32 rounding midpoint (the float-float estimate cannot decide
    it there and the kernel takes the fp64 sequence)."""
    x, dist = near_midpoint_rows(192, eps)
    assert dist[0] < 2.0 ** -40 and (dist < 2.0 ** -37).sum() >= 16   # the band is exercised
    X = wl.to_bf16_bits(x)
    assert np.array_equal(oracle._bf16_bits_to_f64(X), x)
    check_stats(X, wl.gen_bf16(24, 2, 1, 32)[0], eps, f"near midpoints eps={eps}")


def test_rstd_extreme_scales():
    """r across the fp32 range: rows near the bf16 maximum (r subnormal in
    fp32, decided by the fp64 sequence), tiny rows with eps = 0 (r near
    2^100), and eps dominating the row."""
    K = 64
    rows = [[1.5 * 2.0 ** 127] * 64, [1.0 * 2.0 ** 126] * 3, [2.0 ** 100, 3.0 * 2.0 ** 90],
            [2.0 ** -90, -(2.0 ** -95)], [1.0, 2.0, 3.0], [2.0 ** -20] * 64]
    X = np.stack([bf16_row(v, K) for v in rows])
    for eps in (0.0, 1e-6, 1e30):
        got = check_stats(X, wl.gen_bf16(25, 2, 1, K)[0], eps, f"extreme eps={eps}")
        assert np.isfinite(got).all()


def test_rstd_very_long_rows():
    """K = 2^24: the estimate needs K < 2^24, so r comes from the fp64
    sequence; the rows are taken in chunks of 8192 vectors."""
    K = 1 << 24
    x = wl.gen_bf16(26, 1, 2, K)
    X = dev_bf16(x)
    w = dev_bf16(wl.gen_bf16(26, 2, 1, K))[0].contiguous()
    _, _, rstd, ss = mx.mxfp4_rmsnorm_quantize(X, w, 1e-6, stats=True)
    torch.cuda.synchronize()
    ss_ref = np.array([exact_sumsq(x[m]) for m in range(2)])
    assert np.array_equal(host(ss).view(np.int64), ss_ref.view(np.int64))
    e = float(np.float32(1e-6))
    r_ref = np.array([np.float32(1.0 / math.sqrt(s / K + e)) for s in ss_ref], dtype=np.float32)
    assert np.array_equal(host(rstd).view(np.int32), r_ref.view(np.int32))
