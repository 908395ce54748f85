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

__device__ __forceinline__ uint32_t max_abs_bits8(const uint4 &v)
{
    // bf16 magnitudes compare like unsigned integers
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m = max(m, w[i] & 0x7FFFu);
        m = max(m, (w[i] >> 16) & 0x7FFFu);
    }
    return m;
}

// E8M0 byte of a block whose largest magnitude has bf16 bits `amax_bits`:
// floor(log2 amax) = E - 127 for a normal bf16 with exponent field E, so the
// byte is E - 2; zero, subnormal and E = 1 all clamp to byte 0 (2^-127).
__device__ __forceinline__ uint32_t e8m0_byte_from_amax(uint32_t amax_bits)
{
    const uint32_t E = amax_bits >> 7;
    return E >= 2 ? E - 2 : 0;
}

// Codes of 8 bf16 values scaled by 2^(127 - sbyte) (exact power-of-two scale).
__device__ __forceinline__ uint32_t mx_codes8(const uint4 &v, uint32_t sbyte)
{
    const float mult = __uint_as_float((254u - sbyte) << 23);  // 2^-e, e = sbyte - 127
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = w[i] & 0xFFFFu, hi = w[i] >> 16;
        const float flo = __uint_as_float((lo & 0x7FFFu) << 16) * mult;
        const float fhi = __uint_as_float((hi & 0x7FFFu) << 16) * mult;
        uint32_t byte = e2m1x2_rn_sat(flo, fhi);
        byte |= ((lo >> 15) << 3) | ((hi >> 15) << 7);
        out |= byte << (8 * i);
    }
    return out;
}

__device__ __forceinline__ uint32_t nv_codes8(const uint4 &v, float s)
{
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = w[i] & 0xFFFFu, hi = w[i] >> 16;
        float flo = 0.0f, fhi = 0.0f;
        if (s > 0.0f) {
            flo = __fdiv_rn(__uint_as_float((lo & 0x7FFFu) << 16), s);
            fhi = __fdiv_rn(__uint_as_float((hi & 0x7FFFu) << 16), s);
        }
        uint32_t byte = e2m1x2_rn_sat(flo, fhi);
        byte |= ((lo >> 15) << 3) | ((hi >> 15) << 7);
        out |= byte << (8 * i);
    }
    return out;
}

}  // namespace mxfp4
