"""CPU oracle for block-scaled FP4 (MXFP4 / NVFP4) quantization and GEMM.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``. The product path never imports it.

A thin numpy wrapper around the plain C loops in ``mxfp4_oracle.c`` (fp64,
single-threaded). The C file states, per function, which passage of the pages
it restates. Parity pins:

* E2M1 level set, code order and sign bit, E8M0 unit, the blocked scale layout
  index map and the worked A_q size are pinned to values the pages print
  (``tests/golden/``).
* The E2M1 encoder is pinned by brute force (nearest of the 8 levels, ties to
  the even code) over every bf16 pattern at several scales; the E4M3 codec
  against PyTorch's float8_e4m3fn conversion; the OCP shared exponent against
  ``math.frexp``; the GEMM against numpy matmul of independently decoded
  operands and against closed-form special cases.
* The NVFP4 *quantization* rule (E4M3 scale = RNE(amax/6)) is a reading: the
  pages consume NVFP4 operands but do not print the producer's rule. Its
  codecs are pinned; the rule as a whole is "parity unpinned" beyond them.
* The fused RMSNorm + MXFP4 quantization (``rmsnorm_y``,
  ``rmsnorm_mx_quantize``) is a reading too (the pages name the fused
  operation, not its arithmetic); it is pinned by its reduction to the plain
  MXFP4 quantizer on rows whose norm is a power of two, by scale invariance,
  by closed forms and by a high-precision evaluation of y.
"""
import math
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_int]
        L.orc_e2m1_encode.restype = ctypes.c_int
        L.orc_e2m1_encode.argtypes = [ctypes.c_double]
        L.orc_e8m0_decode.restype = ctypes.c_double
        L.orc_e8m0_decode.argtypes = [ctypes.c_int]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_int]
        L.orc_e4m3_encode_satfinite.restype = ctypes.c_int
        L.orc_e4m3_encode_satfinite.argtypes = [ctypes.c_double]
        L.orc_bf16_to_double.restype = ctypes.c_double
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_sf_offset.restype = _i64
        L.orc_sf_offset.argtypes = [_i64, _i64, _i64]
        L.orc_sf_bytes.restype = _i64
        L.orc_sf_bytes.argtypes = [_i64, _i64]
        L.orc_sf_pack.restype = None
        L.orc_sf_pack.argtypes = [_p, _i64, _i64, ctypes.c_uint8, _p]
        L.orc_sf_unpack.restype = None
        L.orc_sf_unpack.argtypes = [_p, _i64, _i64, _p]
        L.orc_mx_shared_exponent.restype = ctypes.c_int
        L.orc_mx_shared_exponent.argtypes = [ctypes.c_double]
        L.orc_mx_quantize_block.restype = None
        L.orc_mx_quantize_block.argtypes = [_p, _p, _p]
        L.orc_mx_block_variant.restype = None
        L.orc_mx_block_variant.argtypes = [_p, ctypes.c_int, _p, _p]
        L.orc_mx_quantize.restype = ctypes.c_int
        L.orc_mx_quantize.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p]
        L.orc_nv_quantize.restype = ctypes.c_int
        L.orc_nv_quantize.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p]
        L.orc_dequant.restype = None
        L.orc_dequant.argtypes = [_p, _i64, _p, _i64, _i64, ctypes.c_int, _p]
        L.orc_gemm_full.restype = None
        L.orc_gemm_full.argtypes = [_p, _i64, _p, _p, _i64, _p, _i64, _i64, _i64,
                                    ctypes.c_int, _p, _p]
        L.orc_gemm_sampled.restype = None
        L.orc_gemm_sampled.argtypes = [_p, _i64, _p, _p, _i64, _p, _i64, ctypes.c_int,
                                       _p, _p, _i64, _p, _p]
        L.orc_check_tolerance.restype = _i64
        L.orc_check_tolerance.argtypes = [_p, _p, _p, _i64, _p]
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ codecs --

def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code))


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(float(v))


def e8m0_decode(b: int) -> float:
    return lib().orc_e8m0_decode(int(b))


def e4m3_decode(b: int) -> float:
    return lib().orc_e4m3_decode(int(b))


def e4m3_encode_satfinite(f: float) -> int:
    return lib().orc_e4m3_encode_satfinite(float(f))


def bf16_to_double(h: int) -> float:
    return lib().orc_bf16_to_double(int(h))


def mx_shared_exponent(amax: float) -> int:
    return lib().orc_mx_shared_exponent(float(amax))


# ------------------------------------------------------------- scale layout --

def sf_offset(r: int, c: int, C: int) -> int:
    return lib().orc_sf_offset(r, c, C)


def sf_bytes(R: int, C: int) -> int:
    return lib().orc_sf_bytes(R, C)


def sf_pack(lin: np.ndarray, pad: int) -> np.ndarray:
    lin = np.ascontiguousarray(lin, dtype=np.uint8)
    R, C = lin.shape
    out = np.empty(sf_bytes(R, C), dtype=np.uint8)
    lib().orc_sf_pack(_ptr(lin), R, C, pad, _ptr(out))
    return out


def sf_unpack(blk: np.ndarray, R: int, C: int) -> np.ndarray:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size >= sf_bytes(R, C)
    out = np.empty((R, C), dtype=np.uint8)
    lib().orc_sf_unpack(_ptr(blk), R, C, _ptr(out))
    return out


# ---------------------------------------------------------------- quantize --

def mx_quantize_block(x) -> tuple:
    """OCP MX quantization of one 32-value block: (scale byte, 32 codes)."""
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    assert xa.shape == (32,)
    sb = np.zeros(1, dtype=np.int32)
    codes = np.zeros(32, dtype=np.int32)
    lib().orc_mx_quantize_block(_ptr(xa), _ptr(sb), _ptr(codes))
    return int(sb[0]), codes


def mx_block_variant(x, variant: int) -> tuple:
    """The pages' differing rules (1: floor of log2(amax/6), 2: round): (exponent, codes)."""
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    e = np.zeros(1, dtype=np.int32)
    codes = np.zeros(32, dtype=np.int32)
    lib().orc_mx_block_variant(_ptr(xa), int(variant), _ptr(e), _ptr(codes))
    return int(e[0]), codes


def _quantize(fn, A_bits: np.ndarray, vec: int):
    A_bits = np.ascontiguousarray(A_bits, dtype=np.uint16)
    M, K = A_bits.shape
    if K % vec:
        raise ValueError(f"K={K} is not a multiple of {vec}")
    q = np.empty((M, K // 2), dtype=np.uint8)
    sf = np.empty(sf_bytes(M, K // vec), dtype=np.uint8)
    rc = fn(_ptr(A_bits), M, K, K, _ptr(q), K // 2, _ptr(sf))
    assert rc == 0
    return q, sf


def mx_quantize(A_bits: np.ndarray):
    """bf16 bits [M, K] -> (packed codes [M, K/2] u8, blocked E8M0 scales)."""
    return _quantize(lib().orc_mx_quantize, A_bits, 32)


def nv_quantize(A_bits: np.ndarray):
    """bf16 bits [M, K] -> (packed codes [M, K/2] u8, blocked E4M3 scales)."""
    return _quantize(lib().orc_nv_quantize, A_bits, 16)


def dequant(q: np.ndarray, sf: np.ndarray, K: int, vec: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    R = q.shape[0]
    out = np.empty((R, K), dtype=np.float64)
    lib().orc_dequant(_ptr(q), q.shape[1], _ptr(sf), R, K, vec, _ptr(out))
    return out


# -------------------------------------------------------------------- GEMM --

def gemm_full(qa, sfa, qb, sfb, K: int, vec: int):
    """Reference C [M, N] and S = sum_k |a_k b_k| [M, N], both float64."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    sfa = np.ascontiguousarray(sfa, dtype=np.uint8)
    sfb = np.ascontiguousarray(sfb, dtype=np.uint8)
    M, N = qa.shape[0], qb.shape[0]
    c = np.empty((M, N), dtype=np.float64)
    s = np.empty((M, N), dtype=np.float64)
    lib().orc_gemm_full(_ptr(qa), qa.shape[1], _ptr(sfa), _ptr(qb), qb.shape[1], _ptr(sfb),
                        M, N, K, vec, _ptr(c), _ptr(s))
    return c, s


def gemm_sampled(qa, sfa, qb, sfb, K: int, vec: int, rows, cols):
    """Reference C and S at the (rows[i], cols[i]) pairs."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    sfa = np.ascontiguousarray(sfa, dtype=np.uint8)
    sfb = np.ascontiguousarray(sfb, dtype=np.uint8)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    n = rows.size
    c = np.empty(n, dtype=np.float64)
    s = np.empty(n, dtype=np.float64)
    lib().orc_gemm_sampled(_ptr(qa), qa.shape[1], _ptr(sfa), _ptr(qb), qb.shape[1], _ptr(sfb),
                           K, vec, _ptr(rows), _ptr(cols), n, _ptr(c), _ptr(s))
    return c, s


def gemm_epilogue(c_acc, s_abs, alpha: float, beta: float, c_in=None, bias=None):
    """The GEMM call's epilogue extras (kernelbot-amd-mxfp4-mm-683203, the
    hot-path "Launch 2" call passes bias, alpha and beta, there None, 1.0 and
    0.0; the page gives no formula). Reading, the usual GEMM epilogue:
        C[m, n] = alpha * acc[m, n] + beta * C_in[m, n] + bias[n]
    in fp64 on the exact product `c_acc` (from gemm_full / gemm_sampled).
    Returns (C_ref, S) for check_tolerance, with S = |alpha| * sum|a b| +
    |beta * C_in| + |bias|: the contract's 2^-8 * S term grows by the terms the
    epilogue adds to the value that is rounded to bf16.
    c_in and bias are float arrays (bias broadcast over rows), or None."""
    c = alpha * np.asarray(c_acc, dtype=np.float64)
    S = abs(alpha) * np.asarray(s_abs, dtype=np.float64)
    if beta != 0.0:
        cin = np.asarray(c_in, dtype=np.float64)
        c = c + beta * cin
        S = S + np.abs(beta * cin)
    if bias is not None:
        b = np.asarray(bias, dtype=np.float64)
        c = c + b
        S = S + np.abs(b)
    return c, S


def check_tolerance(c_gpu, c_ref, s_abs):
    """Contract: |C_gpu - C_ref| <= 2^-8 * S + 1e-3 per element -> (n_bad, worst ratio)."""
    cg = np.ascontiguousarray(c_gpu, dtype=np.float64).ravel()
    cr = np.ascontiguousarray(c_ref, dtype=np.float64).ravel()
    sa = np.ascontiguousarray(s_abs, dtype=np.float64).ravel()
    worst = np.zeros(1, dtype=np.float64)
    bad = lib().orc_check_tolerance(_ptr(cg), _ptr(cr), _ptr(sa), cg.size, _ptr(worst))
    return int(bad), float(worst[0])


# ------------------------------------------------ RMSNorm + MXFP4 quantize --

def _bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rmsnorm_y(X_bits: np.ndarray, w_bits: np.ndarray, eps: float) -> np.ndarray:
    """Normalized rows y [M, K] (float32) of the fused RMSNorm + MXFP4
    quantization. The source pages (kernelbot-amd-mxfp4-mm-683203, the fused
    RMSNorm + MXFP4 quantization kernel its activation path cites) name the
    operation without its arithmetic; the reading taken, for bf16 x [K] and a
    bf16 weight w [K]:
      ss  = sum_k x_k^2, the exact sum (each square is exact in fp64; math.fsum
            rounds the exact total once)
      r64 = 1 / sqrt(ss / K + eps) in fp64, or 0 when ss / K + eps == 0
      r   = fp32(r64)
      y_k = fp32(fp32(x_k * r) * w_k)
    with eps the caller's fp32 value."""
    X = _bf16_bits_to_f64(X_bits)
    w32 = _bf16_bits_to_f64(w_bits).astype(np.float32)
    M, K = X.shape
    assert w32.shape == (K,)
    e = float(np.float32(eps))
    y = np.empty((M, K), dtype=np.float32)
    for m in range(M):
        row = X[m]
        ss = math.fsum((row * row).tolist())
        d = ss / K + e
        r = np.float32(0.0 if d == 0.0 else 1.0 / math.sqrt(d))
        y[m] = (row.astype(np.float32) * r).astype(np.float32) * w32
    return y


def rmsnorm_mx_quantize(X_bits: np.ndarray, w_bits: np.ndarray, eps: float):
    """bf16 X [M, K], bf16 w [K] -> (packed E2M1 codes [M, K/2], blocked E8M0
    scales) of y = rmsnorm_y(X, w, eps), each 32-value block of y quantized by
    the OCP MX rule exactly as mx_quantize_block does (scale pad 0x7F)."""
    y = rmsnorm_y(X_bits, w_bits, eps)
    M, K = y.shape
    if K % 32:
        raise ValueError(f"K={K} is not a multiple of 32")
    C = K // 32
    q = np.zeros((M, K // 2), dtype=np.uint8)
    lin = np.zeros((M, C), dtype=np.uint8)
    for m in range(M):
        for b in range(C):
            sb, codes = mx_quantize_block(y[m, 32 * b:32 * b + 32].astype(np.float64))
            lin[m, b] = sb
            c = np.asarray(codes, dtype=np.uint8) & 15
            q[m, 16 * b:16 * b + 16] = c[0::2] | (c[1::2] << 4)
    return q, sf_pack(lin, 127)
