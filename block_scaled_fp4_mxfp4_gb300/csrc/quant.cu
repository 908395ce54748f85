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
// Work unit: one warp x up to four consecutive 256-element K segments of one
// row (fewer when that would leave the grid too small to fill the GPU). For each segment a lane loads one 16-byte vector (8 bf16) -- a warp
// load covers 512 contiguous bytes -- and stores one 32-bit word of codes (128
// contiguous bytes per warp); the unit's loads are all issued before any
// segment is encoded. Scale bytes are gathered with shuffles into 32-bit words
// (4 consecutive K-blocks of one row, which are contiguous in the blocked
// layout). Rows past M up to the next multiple of 128 and K-blocks past K
// inside a written word get the pad byte (0x7F for E8M0 = 1.0, 0x00 for E4M3).
// One launch may quantize up to kMaxGroups matrices (the grouped path); a
// single matrix is a table of one.
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mxfp4 {
namespace {

constexpr int kQuantThreads = 256;

constexpr int kQuantUnroll = 4;     // most segments per work unit, loaded together
// resident blocks per SM: <= 48 registers a thread for MXFP4, <= 64 for NVFP4
// (its reciprocal and scale conversions need more)
template <int VEC>
constexpr int kQuantMinBlocks = VEC == 32 ? 5 : 4;

// The matrices of one launch: the work units of matrix g are the global
// units [first[g], first[g + 1]), row-major over (padded row, chunk of
// `chunk` <= kQuantUnroll segments).
struct QuantGroupsDev {
    const uint16_t *A[kMaxGroups];
    uint8_t *Aq[kMaxGroups];
    uint8_t *sf[kMaxGroups];
    int64_t lda[kMaxGroups], ldq[kMaxGroups];
    int64_t first[kMaxGroups + 1];
    int M[kMaxGroups], K[kMaxGroups], nchunk[kMaxGroups];
    int count;
    int chunk;
};

// Encode segment seg of a row (8 elements per lane in v; the row's codes at
// qrow, its scale words at sfrow + word * 512). VEC = 32 (MXFP4) or 16
// (NVFP4); lanes per scale block = VEC / 8.
template <int VEC>
__device__ __forceinline__ void encode_segment(uint4 v, bool row_ok, int seg, int C, int cblocks, uint8_t *qrow,
                                               uint8_t *sfrow, int lane)
{
    constexpr int LPB = VEC / 8;            // lanes per scale block
    constexpr int BPS = 256 / VEC;          // blocks per 256-element segment (8 or 16)
    constexpr uint32_t PAD = VEC == 32 ? 0x7Fu : 0x00u;
    const int blk = seg * BPS + lane / LPB;           // scale column of this lane
    const int k = blk * VEC + (lane % LPB) * 8;       // first element of this lane
    const bool ok = row_ok && blk < C;

    uint32_t amax = max_abs_bits8(v);
#pragma unroll
    for (int o = 1; o < LPB; o <<= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));

    uint32_t sbyte;
    uint32_t codes;
    if (VEC == 32) {
        sbyte = e8m0_byte_from_amax(amax);
        codes = mx_codes8(v, sbyte);
    } else {
        sbyte = nv_scale_byte(amax);
        codes = nv_codes8(v, nv_recip(sbyte));
    }
    if (ok) *reinterpret_cast<uint32_t *>(qrow + k / 2) = codes;
    // scale words: 4 consecutive blocks -> lanes base + j * LPB
    const uint32_t mine = ok ? sbyte : PAD;
    constexpr int LANES_PER_WORD = 4 * LPB;      // 16 (MX) or 8 (NV)
    const int base = lane & ~(LANES_PER_WORD - 1);
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) word |= __shfl_sync(0xffffffffu, mine, base + j * LPB) << (8 * j);
    const int widx = seg * (BPS / 4) + lane / LANES_PER_WORD;
    if ((lane & (LANES_PER_WORD - 1)) == 0 && widx < cblocks)
        *reinterpret_cast<uint32_t *>(sfrow + static_cast<size_t>(widx) * 512) = word;
}

// Warp w takes the units w, w + W, w + 2W, ... (W warps in the grid).
template <int VEC>
__global__ void __launch_bounds__(kQuantThreads, kQuantMinBlocks<VEC>) quant_kernel(const __grid_constant__ QuantGroupsDev q)
{
    constexpr int U = kQuantUnroll;
    constexpr int LPB = VEC / 8;
    constexpr int BPS = 256 / VEC;
    const int lane = threadIdx.x & 31;
    const int64_t units = q.first[q.count];
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    int g = 0;
    for (int64_t unit = warp0; unit < units; unit += nwarps) {
        while (unit >= q.first[g + 1]) ++g;     // units only grow along the loop
        const int64_t local = unit - q.first[g];
        const int64_t r = local / q.nchunk[g];
        const int seg0 = static_cast<int>(local - r * q.nchunk[g]) * q.chunk;
        const int K = q.K[g];
        const int C = K / VEC;
        const int cblocks = (C + 3) / 4;
        const int nseg = (K + 255) / 256;
        const bool row_ok = r < q.M[g];
        const uint16_t *arow = q.A[g] + r * q.lda[g];
        uint4 v[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int blk = (seg0 + j) * BPS + lane / LPB;
            const int k = blk * VEC + (lane % LPB) * 8;
            v[j] = make_uint4(0, 0, 0, 0);
            if (j < q.chunk && row_ok && blk < C) v[j] = ld_nc_v4(arow + k);
        }
        uint8_t *qrow = q.Aq[g] + r * q.ldq[g];
        // the row's first scale word: 128-row chunk, row within a 32-row group, group
        uint8_t *sfrow = q.sf[g] + (static_cast<size_t>(r >> 7) * cblocks) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
#pragma unroll
        for (int j = 0; j < U; ++j)
            if (j < q.chunk && seg0 + j < nseg) encode_segment<VEC>(v[j], row_ok, seg0 + j, C, cblocks, qrow, sfrow, lane);
    }
}

template <int VEC>
cudaError_t launch_quant(const QuantGroupHost *groups, int count, int num_sms, cudaStream_t stream)
{
    if (count < 1 || count > kMaxGroups) return cudaErrorInvalidValue;
    QuantGroupsDev q;
    memset(&q, 0, sizeof(q));
    q.count = count;
    for (int g = 0; g < count; ++g) {
        const QuantGroupHost &h = groups[g];
        if (h.M < 1 || h.K < 1 || h.M > 0x7fffffff || h.K > 0x7fffffff) return cudaErrorInvalidValue;
        q.A[g] = static_cast<const uint16_t *>(h.A);
        q.Aq[g] = static_cast<uint8_t *>(h.Aq);
        q.sf[g] = static_cast<uint8_t *>(h.sf);
        q.M[g] = static_cast<int>(h.M);
        q.K[g] = static_cast<int>(h.K);
        q.lda[g] = h.lda;
        q.ldq[g] = h.ldq;
    }
    // the longest chunk that still gives every SM a resident wave of warps
    // (small matrices fall back to one segment per unit, all loads in flight)
    const int64_t want_units = static_cast<int64_t>(num_sms) * kQuantMinBlocks<VEC> * (kQuantThreads / 32);
    for (int chunk = kQuantUnroll; chunk >= 1; chunk /= 2) {
        q.chunk = chunk;
        q.first[0] = 0;
        for (int g = 0; g < count; ++g) {
            q.nchunk[g] = static_cast<int>(((q.K[g] + 255) / 256 + chunk - 1) / chunk);
            q.first[g + 1] = q.first[g] + (static_cast<int64_t>(q.M[g]) + 127) / 128 * 128 * q.nchunk[g];
        }
        if (q.first[count] >= want_units) break;
    }
    for (int g = count + 1; g <= kMaxGroups; ++g) q.first[g] = q.first[count];
    const int64_t units = q.first[count];
    const int64_t per_block = kQuantThreads / 32;
    int64_t blocks = (units + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(num_sms) * kQuantMinBlocks<VEC>;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quant_kernel<VEC><<<static_cast<unsigned>(blocks), kQuantThreads, 0, stream>>>(q);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_nv_grouped(const QuantGroupHost *groups, int count, int num_sms, cudaStream_t stream)
{
    return launch_quant<16>(groups, count, num_sms, stream);
}

cudaError_t launch_quant_mx(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq,
                            int64_t ldq, void *sf, int num_sms, cudaStream_t stream)
{
    const QuantGroupHost one{A, M, K, lda, Aq, ldq, sf};
    return launch_quant<32>(&one, 1, num_sms, stream);
}

cudaError_t launch_quant_nv(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq,
                            int64_t ldq, void *sf, int num_sms, cudaStream_t stream)
{
    const QuantGroupHost one{A, M, K, lda, Aq, ldq, sf};
    return launch_quant<16>(&one, 1, num_sms, stream);
}

}  // namespace mxfp4
