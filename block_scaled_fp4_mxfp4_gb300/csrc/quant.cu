// Dynamic FP4 quantization kernels (HBM-bound): bf16 [M, K] -> packed E2M1
// codes [M, K/2] plus scales written straight into the 128x4 blocked layout.
//
// MXFP4 (kernelbot-amd-mxfp4-mm-517169 module docstring; the OCP MX rule):
//   per 32-element K-block, e = clamp(floor(log2 amax) - 2, -127, 127),
//   E8M0 byte e + 127, codes E2M1_RNE_sat(x * 2^-e).
// NVFP4 (operand format of kernelbot-nvfp4-group-gemm-496271; scale rule is
// this library's reading): per 16-element block, s = E4M3_RNE_sat(amax / 6),
//   codes E2M1_RNE_sat(x / s), s == 0 -> zero magnitudes.
// Both kernels keep the IEEE sign of every element in code bit 3.
//
// Work unit: one warp x one 256-element K segment of one row. Each lane loads
// one 16-byte vector (8 bf16) -- a warp load covers 512 contiguous bytes -- and
// stores one 32-bit word of codes (128 contiguous bytes per warp). Scale bytes
// are gathered with shuffles into 32-bit words (4 consecutive K-blocks of one
// row, which are contiguous in the blocked layout). Rows past M up to the
// next multiple of 128 and K-blocks past K inside a written word get the pad
// byte (0x7F for E8M0 = 1.0, 0x00 for E4M3).
#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mxfp4 {
namespace {

constexpr int kQuantThreads = 256;

// Byte offset of the 32-bit scale word holding columns [4*word, 4*word+4) of
// row r in a blocked buffer with `cblocks` column blocks.
__device__ __forceinline__ size_t sf_word_offset(int64_t r, int64_t word, int64_t cblocks)
{
    return (static_cast<size_t>(r / 128) * cblocks + word) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4;
}

// VEC = 32 (MXFP4) or 16 (NVFP4). Lanes per block = VEC / 8.
template <int VEC>
__global__ void __launch_bounds__(kQuantThreads) quant_kernel(const uint16_t *__restrict__ A,
                                                              int64_t M, int64_t K, int64_t lda,
                                                              uint8_t *__restrict__ Aq, int64_t ldq,
                                                              uint8_t *__restrict__ sf)
{
    constexpr int LPB = VEC / 8;            // lanes per scale block
    constexpr int BPS = 256 / VEC;          // blocks per 256-element segment (8 or 16)
    constexpr uint32_t PAD = VEC == 32 ? 0x7Fu : 0x00u;
    const int lane = threadIdx.x & 31;
    const int64_t C = K / VEC;                       // scale columns
    const int64_t cblocks = (C + 3) / 4;
    const int64_t nseg = (K + 255) / 256;
    const int64_t m_pad = (M + 127) / 128 * 128;
    const int64_t items = m_pad * nseg;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

    for (int64_t item = warp0; item < items; item += nwarps) {
        const int64_t r = item / nseg;
        const int64_t seg = item - r * nseg;
        const int64_t blk = seg * BPS + lane / LPB;       // scale column of this lane
        const int64_t k = blk * VEC + (lane % LPB) * 8;   // first element of this lane
        const bool row_ok = r < M;
        const bool blk_ok = blk < C;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row_ok && blk_ok) v = ld_nc_v4(A + r * lda + k);

        uint32_t amax = max_abs_bits8(v);
#pragma unroll
        for (int o = 1; o < LPB; o <<= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));

        uint32_t sbyte;
        uint32_t codes;
        if (VEC == 32) {
            sbyte = e8m0_byte_from_amax(amax);
            codes = mx_codes8(v, sbyte);
        } else {
            const float ratio = __fdiv_rn(__uint_as_float(amax << 16), 6.0f);
            sbyte = e4m3_rn_sat(ratio);
            codes = nv_codes8(v, e4m3_value(sbyte));
        }
        if (row_ok && blk_ok) {
            *reinterpret_cast<uint32_t *>(Aq + r * ldq + k / 2) = codes;
        }
        // scale words: 4 consecutive blocks -> lanes base + j * LPB
        const uint32_t mine = (row_ok && blk_ok) ? sbyte : PAD;
        constexpr int LANES_PER_WORD = 4 * LPB;      // 16 (MX) or 8 (NV)
        const int base = lane & ~(LANES_PER_WORD - 1);
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) word |= __shfl_sync(0xffffffffu, mine, base + j * LPB) << (8 * j);
        const int64_t widx = seg * (BPS / 4) + lane / LANES_PER_WORD;
        if ((lane & (LANES_PER_WORD - 1)) == 0 && widx < cblocks) {
            *reinterpret_cast<uint32_t *>(sf + sf_word_offset(r, widx, cblocks)) = word;
        }
    }
}

template <int VEC>
cudaError_t launch_quant(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq, int64_t ldq,
                         void *sf, int num_sms, cudaStream_t stream)
{
    const int64_t items = (M + 127) / 128 * 128 * ((K + 255) / 256);
    const int64_t warps_per_block = kQuantThreads / 32;
    int64_t blocks = (items + warps_per_block - 1) / warps_per_block;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quant_kernel<VEC><<<static_cast<unsigned>(blocks), kQuantThreads, 0, stream>>>(
        static_cast<const uint16_t *>(A), M, K, lda, static_cast<uint8_t *>(Aq), ldq,
        static_cast<uint8_t *>(sf));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_mx(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq,
                            int64_t ldq, void *sf, int num_sms, cudaStream_t stream)
{
    return launch_quant<32>(A, M, K, lda, Aq, ldq, sf, num_sms, stream);
}

cudaError_t launch_quant_nv(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq,
                            int64_t ldq, void *sf, int num_sms, cudaStream_t stream)
{
    return launch_quant<16>(A, M, K, lda, Aq, ldq, sf, num_sms, stream);
}

}  // namespace mxfp4
