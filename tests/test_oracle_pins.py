"""Pins the CPU oracle to what the pages and the mathematics fix (no GPU).

Each test checks the oracle against something other than itself: values the
pages print (tests/golden/), closed forms, brute force, invariants, or a library
routine on independently decoded operands.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from conftest import read_golden

LEVELS = {int(c): float(v) for c, v in read_golden("e2m1_levels.txt")}
MAGS = np.array([LEVELS[i] for i in range(8)])


def nearest_e2m1(v: float) -> int:
    """Brute force: the level nearest |v| among all eight, a tie going to the even
    code index; the sign bit copied from v."""
    a = min(abs(v), 8.0)
    d = np.abs(MAGS - a)
    best = np.flatnonzero(d == d.min())
    idx = int(best[0]) if best.size == 1 else int([i for i in best if i % 2 == 0][0])
    return (8 if math.copysign(1.0, v) < 0 else 0) | idx


def nearest_e2m1_vec(v: np.ndarray) -> np.ndarray:
    # every magnitude >= 6 is nearest to 6; clipping at 8 keeps the double
    # distances below exact without changing which level is nearest
    a = np.minimum(np.abs(v), 8.0)
    d = np.abs(a[:, None] - MAGS[None, :])
    dmin = d.min(axis=1, keepdims=True)
    cand = d == dmin
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    idx = np.where(even.any(axis=1), np.argmax(even, axis=1), np.argmax(cand, axis=1))
    return np.where(np.signbit(v), 8, 0) | idx


def all_finite_bf16() -> np.ndarray:
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    return bits[exp != 0xFF]


# ----------------------------------------------------------------- E2M1 ----

def test_e2m1_decode_matches_printed_levels():
    for code in range(16):
        got = oracle.e2m1_decode(code)
        assert got == LEVELS[code]
        assert math.copysign(1.0, got) == math.copysign(1.0, LEVELS[code])


def test_e2m1_code_roundtrip_all_16_codes():
    for code in range(16):
        assert oracle.e2m1_encode(oracle.e2m1_decode(code)) == code


def test_e2m1_midpoint_ties_follow_round_half_even():
    for mid, page_code, ocp_code in read_golden("e2m1_midpoints.txt"):
        v = float(mid)
        assert oracle.e2m1_encode(v) == int(ocp_code), mid
        assert oracle.e2m1_encode(-v) == 8 | int(ocp_code), mid
        # just above / below a midpoint the two rules agree
        assert oracle.e2m1_encode(np.nextafter(v, 10)) == int(page_code)
        assert oracle.e2m1_encode(np.nextafter(v, -10)) == int(page_code) - 1


@pytest.mark.parametrize("e", [-127, -10, -2, 0, 3, 125])
def test_e2m1_encoder_brute_force_every_bf16(e):
    """Every finite bf16 x at scale 2^e: oracle == nearest-of-8 with ties to even."""
    bits = all_finite_bf16()
    x = wl.bf16_bits_to_float(bits).astype(np.float64)
    v = np.ldexp(x, -e)
    want = nearest_e2m1_vec(v)
    got = np.array([oracle.e2m1_encode(float(t)) for t in v])
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, (v[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_e2m1_saturates_and_keeps_sign_of_zero():
    assert oracle.e2m1_encode(6.0) == 7
    assert oracle.e2m1_encode(7.999) == 7
    assert oracle.e2m1_encode(1e30) == 7
    assert oracle.e2m1_encode(-7.5) == 15
    assert oracle.e2m1_encode(0.0) == 0
    assert oracle.e2m1_encode(-0.0) == 8
    assert oracle.e2m1_encode(-1e-30) == 8


# ----------------------------------------------------------------- E8M0 ----

def test_e8m0_unit_and_bias_match_page():
    for b, v in read_golden("e8m0_unit.txt"):
        assert oracle.e8m0_decode(int(b)) == float(v)
    assert math.isnan(oracle.e8m0_decode(255))


def test_shared_exponent_closed_forms():
    # amax = 6 -> exponent 0 (byte 127); amax = 1 -> -2 (byte 125)
    assert oracle.mx_shared_exponent(6.0) == 0
    assert oracle.mx_shared_exponent(1.0) == -2
    assert oracle.mx_shared_exponent(2.0 ** -130) == -127  # clamp at the bottom
    assert oracle.mx_shared_exponent(0.0) == -127
    assert oracle.mx_shared_exponent(7.99) == 0
    assert oracle.mx_shared_exponent(8.0) == 1


def test_shared_exponent_matches_frexp_for_every_positive_bf16():
    bits = all_finite_bf16()
    x = wl.bf16_bits_to_float(bits).astype(np.float64)
    x = np.unique(np.abs(x[x != 0]))
    for v in x:
        _, ex = math.frexp(float(v))  # v = m * 2^ex, 0.5 <= m < 1
        want = max(-127, min(127, (ex - 1) - 2))
        assert oracle.mx_shared_exponent(float(v)) == want, v


# ------------------------------------------------------- MX block quant ----

def test_block_closed_forms():
    x = np.zeros(32)
    x[:8] = [6.0, -4.0, 3.0, -2.0, 1.5, 1.0, 0.5, -0.0]
    sb, codes = oracle.mx_quantize_block(x)
    assert sb == 127
    assert list(codes[:8]) == [7, 14, 5, 12, 3, 2, 1, 8]
    assert all(c == 0 for c in codes[8:])

    x = np.zeros(32)
    x[0], x[1], x[2] = 1.0, 0.5, -0.375
    sb, codes = oracle.mx_quantize_block(x)
    assert sb == 125  # s = 1/4
    assert list(codes[:3]) == [6, 4, 8 | 3]  # 4.0, 2.0, -1.5

    sb, codes = oracle.mx_quantize_block(np.zeros(32))
    assert sb == 0 and not codes.any()

    x = np.zeros(32)
    x[3] = 2.0 ** -130  # bf16 subnormal
    sb, codes = oracle.mx_quantize_block(x)
    assert sb == 0 and not codes.any()  # 2^-130 * 2^127 = 1/8 rounds to 0


def test_scale_rule_variants_differ_from_ocp():
    """A block with amax = 5: OCP gives s = 1 and 5 -> 4 (tie to even);
    the floor rule of _e8m0_scale gives s = 1/2 and 10 saturates to 6 (3.0);
    the docstring's round rule gives s = 1 and the strict-< thresholds send 5 to 6."""
    x = np.zeros(32)
    x[0] = 5.0
    sb, codes = oracle.mx_quantize_block(x)
    assert sb == 127 and codes[0] == 6
    e1, c1 = oracle.mx_block_variant(x, 1)
    assert e1 == -1 and c1[0] == 7
    e2, c2 = oracle.mx_block_variant(x, 2)
    assert e2 == 0 and c2[0] == 7
    deq = [oracle.e2m1_decode(codes[0]) * 2.0 ** (sb - 127),
           oracle.e2m1_decode(c1[0]) * 2.0 ** e1,
           oracle.e2m1_decode(c2[0]) * 2.0 ** e2]
    assert deq == [4.0, 3.0, 6.0]


@pytest.mark.parametrize("dist", ["normal", "heavy"])
def test_block_invariants(dist):
    rng_bits = wl.gen_bf16(7, 1, 64, 32 * 64)
    x = wl.bf16_bits_to_float(rng_bits).astype(np.float64)
    if dist == "heavy":
        x[:, ::37] *= 50.0
        x[::5, :32] = 0.0
    for row in x.reshape(-1, 32)[:2000]:
        sb, codes = oracle.mx_quantize_block(row)
        assert 0 <= sb < 255
        s = 2.0 ** (sb - 127)
        deq = np.array([oracle.e2m1_decode(c) for c in codes]) * s
        assert np.all(np.abs(deq) <= 6.0 * s)
        amax = np.abs(row).max()
        if amax == 0:
            assert sb == 0
            continue
        r = amax / s
        assert 4.0 <= r < 8.0
        i = int(np.argmax(np.abs(row)))
        assert abs(oracle.e2m1_decode(codes[i])) >= 4.0
        for xv, dv in zip(row, deq):
            a = abs(xv) / s
            if a >= 6.0:
                assert abs(dv) == 6.0 * s
                continue
            half = 0.25 if a < 2 else (0.5 if a < 4 else 1.0)
            assert abs(dv - xv) <= half * s * (1 + 1e-12)


# -------------------------------------------------------- scale layout ----

def page_blocked(lin: np.ndarray, pad: int) -> np.ndarray:
    """The blocked layout built the way the page describes it: fill a
    [32, 4, rest_m, 4, rest_k] tensor by the index map, then permute (2,4,0,1,3)."""
    spec = dict(read_golden("blocked_layout.txt"))
    assert spec["permute"] == "2,4,0,1,3" and spec["block_bytes"] == "512"
    R, C = lin.shape
    rest_m, rest_k = -(-R // 128), -(-C // 4)
    t = np.full((32, 4, rest_m, 4, rest_k), pad, dtype=np.uint8)
    i, j = np.meshgrid(np.arange(R), np.arange(C), indexing="ij")
    t[i % 32, (i % 128) // 32, i // 128, j % 4, j // 4] = lin
    return np.ascontiguousarray(t.transpose(2, 4, 0, 1, 3)).ravel()


@pytest.mark.parametrize("R,C", [(128, 4), (256, 56), (200, 7), (16, 224), (8, 32), (1, 1)])
def test_blocked_layout_matches_page(R, C):
    lin = (np.arange(R * C) * 2654435761 % 251).astype(np.uint8).reshape(R, C)
    want = page_blocked(lin, 0x7F)
    got = oracle.sf_pack(lin, 0x7F)
    assert got.size == oracle.sf_bytes(R, C) == want.size
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.sf_unpack(got, R, C), lin)


def test_worked_sizes_from_pages():
    s = dict(read_golden("worked_sizes.txt"))
    M, K = int(s["decode_M"]), int(s["decode_K"])
    a = wl.gen_bf16(0, 1, M, K)
    q, sf = oracle.mx_quantize(a)
    assert q.nbytes == int(s["decode_aq_bytes"])
    assert 2 * q.nbytes == int(s["decode_aq_roundtrip_bytes"])
    # NVFP4: 256-wide K step, 16 scales per row = rep_k groups of 4 blocked columns
    assert int(s["nv_block_k"]) // int(s["nv_vec"]) // 4 == int(s["nv_rep_k"])
    assert oracle.sf_bytes(128, int(s["nv_block_k"]) // int(s["nv_vec"])) == int(s["nv_rep_k"]) * 512


def test_matrix_quantize_packs_low_nibble_first():
    """[MM-517169] docstring: of two packed values the first sits in the low nibble."""
    x = np.zeros((1, 32))
    x[0, :4] = [6.0, -1.0, 0.5, 4.0]
    q, sf = oracle.mx_quantize(wl.to_bf16_bits(x))
    assert q.shape == (1, 16)
    assert q[0, 0] == (7 | (10 << 4))
    assert q[0, 1] == (1 | (6 << 4))
    assert sf[oracle.sf_offset(0, 0, 1)] == 127
    # pad cells of the blocked buffer hold 127
    mask = np.ones(sf.size, bool)
    mask[oracle.sf_offset(0, 0, 1)] = False
    assert np.all(sf[mask] == 0x7F)


def test_matrix_quantize_equals_per_block_rule():
    a = wl.gen_bf16(3, 2, 5, 96, "uniform", 3.0)
    q, sf = oracle.mx_quantize(a)
    x = wl.bf16_bits_to_float(a).astype(np.float64)
    for r in range(5):
        for b in range(3):
            sb, codes = oracle.mx_quantize_block(x[r, 32 * b:32 * b + 32])
            assert sf[oracle.sf_offset(r, b, 3)] == sb
            packed = (codes[0::2] & 15) | ((codes[1::2] & 15) << 4)
            assert np.array_equal(q[r, 16 * b:16 * b + 16], packed.astype(np.uint8))


# ----------------------------------------------------------------- E4M3 ----

def test_e4m3_decode_matches_torch_float8_all_bytes():
    t = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    want = t.to(torch.float64).numpy()
    for b in range(256):
        got = oracle.e4m3_decode(b)
        if math.isnan(want[b]):
            assert math.isnan(got)
        else:
            assert got == want[b] and math.copysign(1, got) == math.copysign(1, want[b])


def test_e4m3_encode_matches_torch_rne():
    vals = [oracle.e4m3_decode(b) for b in range(0x7F)]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    rnd = wl.uniform01(wl.stream_key(5, 9), 20000) * 464.0
    small = wl.uniform01(wl.stream_key(5, 10), 5000) * 2.0 ** -5
    f = np.concatenate([vals, mids, rnd, small, [464.0]]).astype(np.float32)
    want = torch.from_numpy(f).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode_satfinite(float(v)) for v in f])
    assert np.array_equal(got, want)
    assert oracle.e4m3_encode_satfinite(1e6) == 0x7E  # saturates instead of NaN


# ------------------------------------------------------------ NV quant ----

def test_nv_quantize_scale_is_nearest_e4m3_and_codes_nearest_level():
    a = wl.gen_bf16(11, 3, 6, 64)
    a[0, :16] = 0  # all-zero block
    q, sf = oracle.nv_quantize(a)
    x = wl.bf16_bits_to_float(a)
    for r in range(6):
        for b in range(4):
            blk = x[r, 16 * b:16 * b + 16]
            amax = np.float32(np.abs(blk).max())
            ratio = np.float32(amax / np.float32(6.0))
            want_sb = int(torch.tensor([ratio]).to(torch.float8_e4m3fn).view(torch.uint8)[0])
            sb = int(sf[oracle.sf_offset(r, b, 4)])
            assert sb == want_sb
            s = np.float32(oracle.e4m3_decode(sb))
            for i in range(16):
                byte = q[r, 8 * b + i // 2]
                code = (byte & 15) if i % 2 == 0 else (byte >> 4)
                if s == 0:
                    assert code & 7 == 0
                else:
                    assert code == nearest_e2m1(float(np.float32(blk[i] / s)))


# ----------------------------------------------------------------- GEMM ----

def decode_np(q: np.ndarray, sf: np.ndarray, K: int, vec: int) -> np.ndarray:
    """Independent decode: golden level table, E8M0 by 2^(b-127) or E4M3 via
    torch float8, blocked offsets by the page's construction."""
    R = q.shape[0]
    lo, hi = q & 15, q >> 4
    codes = np.empty((R, K), dtype=np.int64)
    codes[:, 0::2], codes[:, 1::2] = lo, hi
    table = np.array([LEVELS[c] for c in range(16)])
    vals = table[codes]
    C = K // vec
    lin = sf[page_blocked_positions(R, C)]
    if vec == 32:
        s = np.ldexp(1.0, lin.astype(np.int64) - 127)
    else:
        s = torch.from_numpy(lin.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return vals * np.repeat(s, vec, axis=1)


def page_blocked_positions(R: int, C: int) -> np.ndarray:
    """For each logical (r, c) the flat byte position in the page's blocked buffer."""
    rest_m, rest_k = -(-R // 128), -(-C // 4)
    pos = np.arange(32 * 4 * rest_m * 4 * rest_k, dtype=np.int64)
    # invert the page's permutation: flat index of permuted tensor -> coordinates
    t = pos.reshape(rest_m, rest_k, 32, 4, 4)  # contiguous order after the permute
    back = t.transpose(2, 3, 0, 4, 1)  # -> [32, 4, rest_m, 4, rest_k]
    i, j = np.meshgrid(np.arange(R), np.arange(C), indexing="ij")
    return back[i % 32, (i % 128) // 32, i // 128, j % 4, j // 4]


@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (4, 3, 64), (3, 4, 128), (2, 5, 96)])
def test_mx_gemm_tiny_vs_numpy(M, N, K):
    a = wl.gen_bf16(21, 1, M, K, "uniform", 4.0)
    b = wl.gen_bf16(21, 2, N, K)
    qa, sfa = oracle.mx_quantize(a)
    qb, sfb = oracle.mx_quantize(b)
    c, s = oracle.gemm_full(qa, sfa, qb, sfb, K, 32)
    A = decode_np(qa, sfa, K, 32)
    B = decode_np(qb, sfb, K, 32)
    assert np.allclose(c, A @ B.T, rtol=0, atol=1e-12 * (np.abs(A) @ np.abs(B).T).max())
    assert np.allclose(s, np.abs(A) @ np.abs(B).T)
    assert np.array_equal(oracle.dequant(qa, sfa, K, 32), A)


@pytest.mark.parametrize("M,N,K", [(2, 3, 16), (4, 4, 64), (3, 2, 48)])
def test_nv_gemm_tiny_vs_numpy(M, N, K):
    a = wl.gen_bf16(22, 1, M, K)
    b = wl.gen_bf16(22, 2, N, K)
    qa, sfa = oracle.nv_quantize(a)
    qb, sfb = oracle.nv_quantize(b)
    c, s = oracle.gemm_full(qa, sfa, qb, sfb, K, 16)
    A = decode_np(qa, sfa, K, 16)
    B = decode_np(qb, sfb, K, 16)
    assert np.allclose(c, A @ B.T, rtol=1e-12, atol=1e-12)
    assert np.array_equal(oracle.dequant(qb, sfb, K, 16), B)


def test_gemm_identity_like_b_gathers_columns():
    """B with a single 1.0 per row (row n at k = n) gives C[:, n] = A_hat[:, n]."""
    M, N, K = 3, 8, 64
    a = wl.gen_bf16(23, 1, M, K)
    qa, sfa = oracle.mx_quantize(a)
    bx = np.zeros((N, K))
    for n in range(N):
        bx[n, n] = 1.0
    qb, sfb = oracle.mx_quantize(wl.to_bf16_bits(bx))
    c, _ = oracle.gemm_full(qa, sfa, qb, sfb, K, 32)
    A = oracle.dequant(qa, sfa, K, 32)
    assert np.array_equal(c, A[:, :N])


def test_gemm_all_ones_closed_form():
    M, N, K = 2, 3, 256
    ones = np.full((M, K), 0x22, dtype=np.uint8)  # code 2 = 1.0 in both nibbles
    onesb = np.full((N, K), 0x22, dtype=np.uint8)
    sfa = np.full(oracle.sf_bytes(M, K // 32), 127, dtype=np.uint8)
    sfb = np.full(oracle.sf_bytes(N, K // 32), 128, dtype=np.uint8)  # scale 2
    c, s = oracle.gemm_full(ones[:, :K // 2], sfa, onesb[:, :K // 2], sfb, K, 32)
    assert np.all(c == 2.0 * K) and np.all(s == 2.0 * K)


def test_sampled_gemm_equals_full():
    M, N, K = 5, 7, 128
    qa, sfa = oracle.mx_quantize(wl.gen_bf16(24, 1, M, K))
    qb, sfb = oracle.mx_quantize(wl.gen_bf16(24, 2, N, K))
    c, s = oracle.gemm_full(qa, sfa, qb, sfb, K, 32)
    rows = np.array([0, 4, 2, 3])
    cols = np.array([6, 0, 3, 3])
    cs, ss = oracle.gemm_sampled(qa, sfa, qb, sfb, K, 32, rows, cols)
    assert np.array_equal(cs, c[rows, cols]) and np.array_equal(ss, s[rows, cols])


def test_tolerance_checker_bound():
    ref = np.array([1.0, -2.0, 0.0])
    s = np.array([256.0, 512.0, 0.0])  # bounds 1 + 1e-3, 2 + 1e-3, 1e-3
    assert oracle.check_tolerance(ref + [1.0, -2.0, 0.0009], ref, s)[0] == 0
    n, worst = oracle.check_tolerance(ref + [1.01, 0, 0], ref, s)
    assert n == 1 and worst > 1.0
    assert oracle.check_tolerance(ref + [np.nan, 0, 0], ref, s)[0] == 1


# ------------------------------------------------------------ GEMM epilogue
def _small_gemm(seed, M=5, N=7, K=64):
    a = wl.gen_bf16(seed, 1, M, K)
    b = wl.gen_bf16(seed, 2, N, K)
    qa, sfa = oracle.mx_quantize(a)
    qb, sfb = oracle.mx_quantize(b)
    return oracle.gemm_full(qa, sfa, qb, sfb, K, 32)


def test_epilogue_identity_is_the_plain_gemm():
    c, s = _small_gemm(70)
    c2, s2 = oracle.gemm_epilogue(c, s, 1.0, 0.0)
    assert np.array_equal(c, c2) and np.array_equal(s, s2)


def test_epilogue_with_zero_product_is_beta_c_plus_bias():
    """A = 0: every code and scale is zero, the product vanishes and C is the
    closed form beta * C_in + bias."""
    M, N, K = 4, 6, 64
    qa, sfa = oracle.mx_quantize(np.zeros((M, K), dtype=np.uint16))
    qb, sfb = oracle.mx_quantize(wl.gen_bf16(71, 2, N, K))
    c, s = oracle.gemm_full(qa, sfa, qb, sfb, K, 32)
    assert np.all(c == 0.0)
    c_in = np.arange(M * N, dtype=np.float64).reshape(M, N) - 7.5
    bias = np.linspace(-2.0, 3.0, N)
    out, S = oracle.gemm_epilogue(c, s, 3.0, -0.5, c_in, bias)
    assert np.array_equal(out, -0.5 * c_in + bias[None, :])
    assert np.array_equal(S, np.abs(0.5 * c_in) + np.abs(bias)[None, :])


def test_epilogue_is_linear_in_alpha_and_beta():
    c, s = _small_gemm(72)
    c_in = wl.bf16_bits_to_float(wl.gen_bf16(72, 3, *c.shape)).astype(np.float64)
    one, _ = oracle.gemm_epilogue(c, s, 1.0, 0.0)
    two, _ = oracle.gemm_epilogue(c, s, 2.0, 0.0)
    assert np.array_equal(two, 2.0 * one)
    with_c, _ = oracle.gemm_epilogue(c, s, 1.0, 0.25, c_in)
    assert np.allclose(with_c - one, 0.25 * c_in, rtol=0, atol=1e-12)


# ------------------------------------------------- RMSNorm + MXFP4 (reading) --

def _bits(x):
    return wl.to_bf16_bits(np.asarray(x, dtype=np.float64))


def test_rmsnorm_on_power_of_two_rows_is_the_plain_quantizer_of_w():
    # rows of +-2^j: sum x^2 / K = 4^j exactly, r = 2^-j, y = sign(x) * w exactly,
    # so the fused output must equal the plain MXFP4 quantizer applied to sign(x) * w
    K = 96
    w = wl.gen_bf16(7, 1, 1, K)[0]
    wv = oracle._bf16_bits_to_f64(w)
    rng = np.random.default_rng(3)
    rows, want_rows = [], []
    for j in (-20, -3, 0, 1, 9, 60):
        sign = np.where(rng.random(K) < 0.5, -1.0, 1.0)
        rows.append(sign * 2.0 ** j)
        want_rows.append(sign * wv)
    q, sf = oracle.rmsnorm_mx_quantize(_bits(rows), w, 0.0)
    q_ref, sf_ref = oracle.mx_quantize(_bits(want_rows))
    assert np.array_equal(q, q_ref) and np.array_equal(sf, sf_ref)


def test_rmsnorm_is_scale_invariant_without_eps():
    X = wl.gen_bf16(8, 2, 5, 128)
    w = wl.gen_bf16(8, 3, 1, 128)[0]
    q1, s1 = oracle.rmsnorm_mx_quantize(X, w, 0.0)
    X4 = _bits(oracle._bf16_bits_to_f64(X) * 4.0)      # exact in bf16
    q2, s2 = oracle.rmsnorm_mx_quantize(X4, w, 0.0)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
    # a bias in the mean (dividing by K - 1, say) or a dropped square root breaks this pin
    y = oracle.rmsnorm_y(X, w, 0.0)
    assert not np.array_equal(y, oracle.rmsnorm_y(X4, w, 0.0) * 0.5)


def test_rmsnorm_constant_rows_closed_form():
    # x = c = 2^j everywhere, w = 1, eps tiny: r = 2^-j, y = 1, amax 1 -> scale
    # 2^-2 (byte 125), every code 4.0 (index 6); -c gives 0xE
    K = 64
    w = _bits(np.ones(K))
    X = _bits([np.full(K, 2.0 ** 5), np.full(K, -(2.0 ** -7))])
    q, sf = oracle.rmsnorm_mx_quantize(X, w, 1e-30)
    assert np.all(q[0] == 0x66) and np.all(q[1] == 0xEE)
    lin = oracle.sf_unpack(sf, 2, K // 32)
    assert np.all(lin == 125)


def test_rmsnorm_zero_row_without_eps_gives_signed_zeros():
    K = 32
    X = np.zeros((1, K), dtype=np.uint16)
    X[0, 3] = 0x8000                                     # -0
    w = _bits(np.where(np.arange(K) % 2 == 0, 1.0, -1.0))
    q, sf = oracle.rmsnorm_mx_quantize(X, w, 0.0)
    codes = np.stack([q[0] & 15, q[0] >> 4], axis=1).ravel()
    # y = (x * 0) * w: +0 * w has w's sign, -0 * w the opposite
    want = np.where(np.arange(K) % 2 == 0, 0, 8)
    want[3] ^= 8
    assert np.array_equal(codes, want)
    assert oracle.sf_unpack(sf, 1, 1)[0, 0] == 0


def test_rmsnorm_y_matches_a_high_precision_evaluation():
    # three fp32 roundings (r, x*r, *w) bound the error of y by ~3 ulp
    from decimal import Decimal, getcontext
    getcontext().prec = 60
    X = wl.gen_bf16(9, 4, 4, 160)
    w = wl.gen_bf16(9, 5, 1, 160)[0]
    for eps in (0.0, 1e-6, 0.75):
        y = oracle.rmsnorm_y(X, w, eps)
        Xd = oracle._bf16_bits_to_f64(X)
        wd = oracle._bf16_bits_to_f64(w)
        e = Decimal(float(np.float32(eps)))
        for m in range(X.shape[0]):
            ms = sum(Decimal(float(v)) ** 2 for v in Xd[m]) / Decimal(X.shape[1]) + e
            r = 1 / ms.sqrt()
            for k in range(X.shape[1]):
                exact = Decimal(float(Xd[m, k])) * r * Decimal(float(wd[k]))
                err = abs(Decimal(float(y[m, k])) - exact)
                assert err <= Decimal(3.01) * Decimal(2) ** -24 * abs(exact), (eps, m, k)
