"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds only random-number generation and the shapes of the five
workloads; it contains none of the quantization or GEMM arithmetic, so the CUDA
path and the CPU oracle can both consume what it produces without sharing any
of the method's code.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", 2014) evaluated counter-style, value i of a stream being
mix(key + (i + 1) * 0x9E3779B97F4A7C15); uniforms take the top 53 bits; normals
use the Box-Muller transform on consecutive pairs. Samples are rounded to
float32 and then to bf16 with round-to-nearest-even. Values are returned as
uint16 bf16 bit patterns so neither side reinterprets floats differently.
"""
from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor_id: int) -> int:
    """A 64-bit stream key for (seed, tensor) built from one SplitMix64 step."""
    z = np.array([(seed * 0x100000001B3 + tensor_id * 0x632BE59BD9B4E019) & (2**64 - 1)],
                 dtype=np.uint64)
    with np.errstate(over="ignore"):
        return int(_mix(z + _GOLDEN)[0])


def uniform01(key: int, n: int, offset: int = 0) -> np.ndarray:
    """n doubles in [0, 1) from stream `key`, starting at counter `offset`."""
    out = np.empty(n, dtype=np.float64)
    k = np.uint64(key)
    with np.errstate(over="ignore"):
        for s in range(0, n, _CHUNK):
            e = min(n, s + _CHUNK)
            i = np.arange(offset + s + 1, offset + e + 1, dtype=np.uint64)
            z = _mix(k + i * _GOLDEN)
            out[s:e] = (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return out


def normal(key: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """n N(0, sigma^2) doubles by Box-Muller over consecutive uniform pairs."""
    m = (n + 1) // 2
    out = np.empty(2 * m, dtype=np.float64)
    for s in range(0, m, _CHUNK):
        e = min(m, s + _CHUNK)
        u = uniform01(key, 2 * (e - s), offset=2 * s)
        u1 = 1.0 - u[0::2]  # (0, 1]
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1)) * sigma
        out[2 * s:2 * e:2] = r * np.cos(2.0 * np.pi * u2)
        out[2 * s + 1:2 * e:2] = r * np.sin(2.0 * np.pi * u2)
    return out[:n]


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round doubles to float32 then to bf16 (nearest-even); return uint16 bit patterns."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ------------------------------------------------------------------ workloads --

@dataclass
class MXWorkload:
    """Quant+GEMM problem: bf16 A [M, K] (dynamic), bf16 B [N, K] (pre-quantized);
    MXFP4 (E8M0 per 32, bf16 C), or NVFP4 (E4M3 per 16, fp16 C) when vec == 16."""
    name: str
    M: int
    N: int
    K: int
    a_dist: str = "normal"      # "normal", "uniform4", "heavy"
    a_sigma: float = 1.0
    b_sigma: float = 1.0
    seed: int = 0
    vec: int = 32

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def alg_bytes(self) -> int:
        """bf16 A + packed B + B's scales + 16-bit C (quantized A is not counted)."""
        return 2 * self.M * self.K + self.N * self.K // 2 + self.N * self.K // self.vec + 2 * self.M * self.N


@dataclass
class NVWorkload:
    """Grouped GEMM: per group g, A_g [M_g, K] and B_g [N, K] E2M1 with a scale per
    `vec` elements (16: E4M3, NVFP4, fp16 C; 32: E8M0, MXFP4, bf16 C)."""
    name: str
    Ms: list = field(default_factory=list)
    N: int = 0
    K: int = 0
    seed: int = 0
    vec: int = 16
    bf16_a: bool = False    # A_g arrives as bf16 and is quantized inside the call

    @property
    def flops(self) -> int:
        return sum(2 * m * self.N * self.K for m in self.Ms)

    @property
    def gemm_alg_bytes(self) -> int:
        """Packed A and B + their scales + 16-bit C, summed over groups."""
        t = 0
        for m in self.Ms:
            t += (m + self.N) * self.K // 2 + (m + self.N) * self.K // self.vec + 2 * m * self.N
        return t

    @property
    def alg_bytes(self) -> int:
        """What one call must move: gemm_alg_bytes, or with bf16 A, the bf16 A_g in
        place of their packed codes and scales (the quantized A_g are not counted)."""
        if not self.bf16_a:
            return self.gemm_alg_bytes
        return sum(2 * m * self.K + self.N * self.K // 2 + self.N * self.K // self.vec + 2 * m * self.N
                   for m in self.Ms)


TINY = MXWorkload("mxfp4_tiny_M8_N512_K1024", 8, 512, 1024, "normal", 1.0, 1.0)
DECODE = MXWorkload("mxfp4_decode_M16_N2112_K7168", 16, 2112, 7168, "normal", 1.0, 0.02)
MEDIUM = MXWorkload("mxfp4_medium_heavytail_M256_N7168_K2048", 256, 7168, 2048, "heavy", 1.0, 0.02)
COMPUTE = MXWorkload("mxfp4_compute_M8192_N8192_K8192", 8192, 8192, 8192, "uniform4", 1.0, 1.0)
NVFP4_GROUPED = NVWorkload("nvfp4_grouped_8x_N4096_K7168",
                           [64, 128, 256, 384, 512, 640, 768, 1024], 4096, 7168)
# The same grouped shapes with MXFP4 operands (E8M0 per 32, bf16 C): the grouped
# MXFP4 (mixture-of-experts) GEMM beyond the pages' single-problem MXFP4 call.
MXFP4_GROUPED = NVWorkload("mxfp4_grouped_8x_N4096_K7168",
                           [64, 128, 256, 384, 512, 640, 768, 1024], 4096, 7168, vec=32)

# The grouped NVFP4 shapes with bf16 activations, quantized inside the call
# (nvfp4_group_quant_gemm): dynamic NVFP4 quantization fused with the grouped GEMM.
NVFP4_GROUPED_BF16 = NVWorkload("nvfp4_grouped_bf16a_8x_N4096_K7168",
                                [64, 128, 256, 384, 512, 640, 768, 1024], 4096, 7168, bf16_a=True)

# The decode shape with NVFP4 operands: the fused NVFP4 quant + GEMM (the NVFP4
# twin of the fused MXFP4 path).
NVFP4_DECODE = MXWorkload("nvfp4_decode_M16_N2112_K7168", 16, 2112, 7168, "normal", 1.0, 0.02, vec=16)



@dataclass
class RMSWorkload:
    """Fused RMSNorm + MXFP4 quantization: bf16 X [M, K] (N(0, 1)), bf16 weight
    [K] (1 + N(0, 0.1)), eps."""
    name: str
    M: int
    K: int
    eps: float = 1e-6
    seed: int = 0

    @property
    def flops(self) -> int:
        return 4 * self.M * self.K      # square, add, two products per element

    @property
    def alg_bytes(self) -> int:
        """bf16 X + bf16 weight + packed codes + E8M0 scales."""
        return 2 * self.M * self.K + 2 * self.K + self.M * self.K // 2 + self.M * self.K // 32


def gen_rms(w: "RMSWorkload"):
    """bf16 bits of (X [M, K], weight [K])."""
    x = normal(stream_key(w.seed, 40), w.M * w.K)
    g = 1.0 + 0.1 * normal(stream_key(w.seed, 41), w.K)
    return to_bf16_bits(x).reshape(w.M, w.K), to_bf16_bits(g)


# The activation rows of the decode GEMM (16 x 7168) and a prefill-sized batch,
# normalized and quantized in one call ahead of the MXFP4 GEMM.
RMSNORM_DECODE = RMSWorkload("mxfp4_rmsnorm_quant_M16_K7168", 16, 7168)
RMSNORM_PREFILL = RMSWorkload("mxfp4_rmsnorm_quant_M4096_K7168", 4096, 7168)

MX_WORKLOADS = {w.name: w for w in (TINY, DECODE, MEDIUM, COMPUTE)}

# tensor ids inside a workload's seed
_ID_A, _ID_B, _ID_OUTLIER_IDX, _ID_ZERO_IDX = 1, 2, 3, 4


def gen_a(w: MXWorkload, M: int = None) -> np.ndarray:
    """bf16 bits of A [M, K] for an MXFP4 workload (first M rows when M is given)."""
    M = w.M if M is None else M
    n = M * w.K
    key = stream_key(w.seed, _ID_A)
    if w.a_dist == "uniform4":
        x = uniform01(key, n) * 8.0 - 4.0
    else:
        x = normal(key, n, w.a_sigma)
    if w.a_dist == "heavy":
        x = _heavy_tail(w, x.reshape(M, w.K)).ravel()
    return to_bf16_bits(x).reshape(M, w.K)


def _heavy_tail(w: MXWorkload, x: np.ndarray) -> np.ndarray:
    """Outliers and zeros: 1% of entries (uniform random index) scaled by 50, then
    1% set to +0, then every 32-block whose linear index (m * K/32 + kb) is a
    multiple of 101 zeroed whole."""
    x = x.copy()
    M, K = x.shape
    n = w.M * w.K
    k_out = max(1, n // 100)
    idx_o = (uniform01(stream_key(w.seed, _ID_OUTLIER_IDX), k_out) * n).astype(np.int64)
    idx_z = (uniform01(stream_key(w.seed, _ID_ZERO_IDX), k_out) * n).astype(np.int64)
    flat = x.reshape(-1)
    lim = M * K
    io = idx_o[idx_o < lim]
    iz = idx_z[idx_z < lim]
    flat[io] *= 50.0
    flat[iz] = 0.0
    kb = K // 32
    blk = np.arange(M * kb, dtype=np.int64)
    zb = blk[blk % 101 == 0]
    for b in zb:
        m, j = divmod(int(b), kb)
        x[m, j * 32:(j + 1) * 32] = 0.0
    return x


def gen_b(w: MXWorkload, N: int = None) -> np.ndarray:
    """bf16 bits of the weight B [N, K] before its (untimed) MXFP4 pre-quantization."""
    N = w.N if N is None else N
    x = normal(stream_key(w.seed, _ID_B), N * w.K, w.b_sigma)
    return to_bf16_bits(x).reshape(N, w.K)


def gen_nv_group(w: NVWorkload, g: int):
    """bf16 bits of (A_g [M_g, K], B_g [N, K]) for group g, both N(0, 1)."""
    a = normal(stream_key(w.seed, 16 + 2 * g), w.Ms[g] * w.K)
    b = normal(stream_key(w.seed, 17 + 2 * g), w.N * w.K)
    return to_bf16_bits(a).reshape(w.Ms[g], w.K), to_bf16_bits(b).reshape(w.N, w.K)


def gen_bf16(seed: int, tensor_id: int, rows: int, cols: int, dist: str = "normal",
             scale: float = 1.0) -> np.ndarray:
    """Generic seeded bf16 matrix for tests (normal or uniform(-scale, scale))."""
    key = stream_key(seed, tensor_id)
    n = rows * cols
    if dist == "uniform":
        x = (uniform01(key, n) * 2.0 - 1.0) * scale
    else:
        x = normal(key, n, scale)
    return to_bf16_bits(x).reshape(rows, cols)
