"""Exactness of the division-free NVFP4 encoding (codes and scale bytes) used by
the kernels.

The NVFP4 quantizers compute each element's code as E2M1_RNE_sat(fp32(x / s))
for a bf16 x and a decoded E4M3 scale s (the reading of the NVFP4 producer rule
the oracle follows: [NV-496271], input generation of custom_kernel). The CUDA
kernels take no division: they multiply by r = fp32(1/s), move the product onto
the grid of multiples of 2^-12 (adding and subtracting 3072), put x's sign back
and convert that.
This test models that arithmetic in numpy float32 (IEEE round-to-nearest-even,
subnormals kept, as the kernels compile) and checks, over EVERY finite bf16 x and
EVERY finite non-negative E4M3 scale, that it gives the same code as the
correctly rounded quotient. The numpy E2M1 encoder it uses is first checked
against the oracle's encoder at every midpoint, its neighbours and random values.
The scale byte E4M3(fp32(amax) / 6) is likewise formed as E4M3(amax * fp32(1/6)),
checked over every bf16 amax. No GPU, no CUDA code: these pin the argument, the
GPU parity tests pin the kernels.
"""
import numpy as np

import oracle

MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def e2m1_rne_sat(v: np.ndarray) -> np.ndarray:
    """Sign-magnitude E2M1 code of float32 values: nearest of 0, .5, 1, 1.5, 2,
    3, 4, 6 with ties to the even code, saturating at 6."""
    a = np.abs(v.astype(np.float64))
    mag = ((a > 0.25).astype(np.int64) + (a >= 0.75) + (a > 1.25) + (a >= 1.75)
           + (a > 2.5) + (a >= 3.5) + (a > 5.0))
    return mag | (np.signbit(v).astype(np.int64) << 3)


def kernel_model(x: np.ndarray, r: np.float32) -> np.ndarray:
    q = (x * r).astype(np.float32)
    big = np.float32(3072.0)                      # fp32 spacing 2^-12 below 4096
    q = ((q + big).astype(np.float32) - big).astype(np.float32)
    u = q.view(np.uint32) | (x.view(np.uint32) & np.uint32(0x80000000))
    return e2m1_rne_sat(u.astype(np.uint32).view(np.float32))


def test_numpy_encoder_matches_oracle():
    pts = []
    for m in MIDPOINTS:
        f = np.float32(m)
        pts += [f, np.nextafter(f, np.float32(0)), np.nextafter(f, np.float32(10))]
    pts += [np.float32(v) for v in (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 6.5, 1e30, 1e-30)]
    rng = np.random.default_rng(7)
    pts += list(rng.uniform(0, 8, 400).astype(np.float32))
    pts = np.array(pts, dtype=np.float32)
    pts = np.concatenate([pts, -pts])
    got = e2m1_rne_sat(pts)
    want = np.array([oracle.e2m1_encode(float(v)) for v in pts])
    assert np.array_equal(got, want)


def test_division_free_encoding_is_exact_for_all_bf16_and_e4m3():
    bits = np.arange(1 << 16, dtype=np.uint32)
    finite = (bits & 0x7F80) != 0x7F80
    x = (bits[finite] << 16).view(np.float32)
    for sb in range(0x7F):   # 0x00 (zero) .. 0x7E (448); 0x7F is NaN
        s = np.float32(oracle.e4m3_decode(sb))
        if s == 0:
            want = (np.signbit(x).astype(np.int64) << 3)
            r = np.float32(0)
        else:
            with np.errstate(over="ignore"):
                want = e2m1_rne_sat((x / s).astype(np.float32))
            r = np.float32(1) / s
        with np.errstate(over="ignore"):
            got = kernel_model(x, r)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (sb, float(s), float(x[bad[0]]), int(got[bad[0]]), int(want[bad[0]]))


def test_midpoint_ties_are_reached():
    # the exhaustive sweep above must include exact midpoints (else the snap
    # would be untested): x = t * s is a bf16 for many (t, s)
    hits = 0
    for sb in range(1, 0x7F):
        s = oracle.e4m3_decode(sb)
        for t in MIDPOINTS:
            v = np.float32(t * s)
            if float(v) == t * s and (v.view(np.uint32) & 0xFFFF) == 0:
                hits += 1
    assert hits > 100


def test_scale_byte_without_division_for_all_bf16_amax():
    # the kernels form the E4M3 scale byte as E4M3(amax * fp32(1/6)); the
    # oracle's reading is E4M3(fp32(amax) / 6), correctly rounded
    bits = np.arange(1 << 15, dtype=np.uint32)
    bits = bits[((bits & 0x7F80) != 0x7F80) | (bits == 0x7F80)]   # finite and +inf
    a = (bits << 16).view(np.float32)
    sixth = np.uint32(0x3E2AAAAB).view(np.float32)
    assert sixth == np.float32(1) / np.float32(6)
    with np.errstate(over="ignore"):
        want = [oracle.e4m3_encode_satfinite(float(v)) for v in (a / np.float32(6)).astype(np.float32)]
        got = [oracle.e4m3_encode_satfinite(float(v)) for v in (a * sixth).astype(np.float32)]
    assert got == want
