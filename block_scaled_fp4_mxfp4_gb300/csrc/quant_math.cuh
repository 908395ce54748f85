// Per-element FP4 encoding math shared by the standalone quant kernels and the
// fused quant+GEMM kernel: both must produce bit-identical codes and scales.
#pragma once

#include "ptx.cuh"

namespace mxfp4 {

__device__ __forceinline__ uint4 ld_nc_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// E2M1 codes of 8 values packed into 32 bits, x0 in the low nibble of byte 0
// and x7 in the high nibble of byte 3 (round to nearest even, saturating, sign
// kept); the four converted bytes are packed by one vector move.
__device__ __forceinline__ uint32_t e2m1x8_rn_sat(float x0, float x1, float x2, float x3, float x4, float x5,
                                                  float x6, float x7)
{
    uint32_t r;
    asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c3, %8, %7;\n\t"
        "mov.b32 %0, {c0, c1, c2, c3};\n\t}"
        : "=r"(r)
        : "f"(x0), "f"(x1), "f"(x2), "f"(x3), "f"(x4), "f"(x5), "f"(x6), "f"(x7));
    return r;
}

// Lane-wise unsigned 16-bit max of two packed pairs.
__device__ __forceinline__ uint32_t umax16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Lane-wise unsigned 16-bit min of two packed pairs.
__device__ __forceinline__ uint32_t umin16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Packed (two-lane) maximum bf16 magnitude of 8 values; bf16 magnitudes
// compare like unsigned integers once the sign bit is cleared.
__device__ __forceinline__ uint32_t max_abs_pair8(const uint4 &v)
{
    return umax16x2(umax16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                    umax16x2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
}

__device__ __forceinline__ uint32_t max_abs_bits8(const uint4 &v)
{
    const uint32_t m = max_abs_pair8(v);
    return max(m & 0xFFFFu, m >> 16);
}

// Lane-wise bf16 maximum of |a| and |b| (the sign bit of each result lane is
// not meaningful: mask it off). Finite inputs only.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// bf16 bits of the largest magnitude among the 8 * N values of v[0 .. N).
template <int N>
__device__ __forceinline__ uint32_t block_amax_bits(const uint4 *v)
{
    uint32_t m = absmax_bf16x2(absmax_bf16x2(v[0].x, v[0].y), absmax_bf16x2(v[0].z, v[0].w));
#pragma unroll
    for (int i = 1; i < N; ++i)
        m = absmax_bf16x2(m, absmax_bf16x2(absmax_bf16x2(v[i].x, v[i].y), absmax_bf16x2(v[i].z, v[i].w)));
    return max(m & 0x7FFFu, (m >> 16) & 0x7FFFu);
}

// E8M0 byte of a block whose largest magnitude has bf16 bits `amax_bits`:
// floor(log2 amax) = E - 127 for a normal bf16 with exponent field E, so the
// byte is E - 2; zero, subnormal and E = 1 all clamp to byte 0 (2^-127).
__device__ __forceinline__ uint32_t e8m0_byte_from_amax(uint32_t amax_bits)
{
    const uint32_t E = amax_bits >> 7;
    return E >= 2 ? E - 2 : 0;
}

// Codes of 8 bf16 values scaled by 2^(127 - sbyte) (exact power-of-two
// scale). The conversion takes the signed values, so a negative value that
// rounds to zero keeps its sign (code 0x8), as -0 does.
__device__ __forceinline__ uint32_t mx_codes8(const uint4 &v, uint32_t sbyte)
{
    const float mult = __uint_as_float((254u - sbyte) << 23);  // 2^-e, e = sbyte - 127
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16) * mult;
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u) * mult;
    }
    return e2m1x8_rn_sat(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
}

// NVFP4 scale byte of a 16-element group whose largest magnitude has bf16 bits
// amax_bits: E4M3_RNE_satfinite(fp32(amax) / 6). The product amax * fp32(1/6)
// (0x3E2AAAAB) converts to the same byte as the correctly rounded quotient for
// every finite bf16 amax and for infinity, so no division is taken.
__device__ __forceinline__ uint32_t nv_scale_byte(uint32_t amax_bits)
{
    return e4m3_rn_sat(__uint_as_float(amax_bits << 16) * __uint_as_float(0x3E2AAAABu));
}

// Reciprocal of the decoded E4M3 scale byte for nv_codes8: 1/s rounded to
// fp32, or 0 for s == 0 (whose codes are signed zeros).
__device__ __forceinline__ float nv_recip(uint32_t sbyte)
{
    const float s = e4m3_value(sbyte);
    return s > 0.0f ? __frcp_rn(s) : 0.0f;
}

// x * (1/s) rounded onto the grid of multiples of 2^-12 by adding and
// subtracting 3072 (= 1.5 * 2^11, whose fp32 spacing is 2^-12; the product is
// below 1024 in magnitude wherever the code is not saturated), with x's sign
// put back so that a negative value that rounds to zero stays -0. For a bf16 x
// and an E4M3 s, the exact quotient x / s is either one of E2M1's rounding
// midpoints (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) or at least 2^-8 (relative)
// away from every one, while x * (1/s) is within 2^-23 of it: the grid puts a
// midpoint back exactly on itself and moves no other value across one, so the
// E2M1 conversion of the result takes the same decision as the conversion of
// the correctly rounded fp32 quotient. The _rn intrinsics keep the compiler
// from fusing the multiply and the add.
__device__ __forceinline__ float nv_snap_scaled(float x, float r)
{
    const float q = __fsub_rn(__fadd_rn(__fmul_rn(x, r), 3072.0f), 3072.0f);
    return __uint_as_float(__float_as_uint(q) | (__float_as_uint(x) & 0x80000000u));
}

// Codes of 8 bf16 values divided by the decoded E4M3 scale s, given
// r = nv_recip(scale byte): the codes of the fp32 quotients x / s rounded to
// nearest even (see nv_snap_scaled), without a division; r == 0 (s == 0)
// leaves signed zeros.
__device__ __forceinline__ uint32_t nv_codes8(const uint4 &v, float r)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = nv_snap_scaled(__uint_as_float(w[i] << 16), r);
        f[2 * i + 1] = nv_snap_scaled(__uint_as_float(w[i] & 0xFFFF0000u), r);
    }
    return e2m1x8_rn_sat(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
}

}  // namespace mxfp4
