// Types and helpers shared by the single-CTA (gemm.cu) and CTA-pair
// (gemm_pair.cu) block-scaled GEMM kernels. Device-side only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace mxfp4 {
namespace gemm_detail {

struct GemmProblemDev {
    const uint8_t *sfa;
    const uint8_t *sfb;
    void *c;
    int64_t ldc;
    int m, n, k;
    int m_tiles, n_tiles;
    int tile_start;
    int sf_cblocks;   // column blocks of 4 scales per 128-row chunk
    int epi;          // nonzero: C = alpha * acc + beta * C + bias[col]
    float alpha, beta;
    const uint16_t *bias;   // [n] in C's type, or null
    int c_tma;        // single-CTA kernel: store C tiles by TMA (tmc of the params)
};

static_assert(sizeof(GemmProblemDev) <= kTableProblemBytes, "problem record of the device table");

// The problems of a launch in kernel parameters (up to MAXG of them).
template <int MAXG>
struct GemmParams {
    CUtensorMap tma[MAXG];
    CUtensorMap tmb[MAXG];
    CUtensorMap tmc[MAXG];
    GemmProblemDev prob[MAXG];
    int num_groups;
    int total_tiles;
    int splits;
    int pad_;
    float *partials;
    int *tickets;
    uint64_t wait_ns;   // limit of the waits that guard work
    static constexpr bool kTable = false;
    __device__ __forceinline__ const CUtensorMap *map_a(int g) const { return &tma[g]; }
    __device__ __forceinline__ const CUtensorMap *map_b(int g) const { return &tmb[g]; }
    __device__ __forceinline__ const CUtensorMap *map_c(int g) const { return &tmc[g]; }
    __device__ __forceinline__ const GemmProblemDev &problem(int g) const { return prob[g]; }
};

// The problems of a launch in a table in global memory (any number of them):
// per group four tensor maps (A, B, C) then its problem record, laid out as
// group_table_bytes() describes.
struct GemmParamsTable {
    const CUtensorMap *maps;      // [num_groups][kTableMaps]
    const uint8_t *probs;         // [num_groups][kTableProblemBytes]
    int num_groups;
    int total_tiles;
    int splits;
    int pad_;
    float *partials;
    int *tickets;
    uint64_t wait_ns;
    static constexpr bool kTable = true;
    __device__ __forceinline__ const CUtensorMap *map_a(int g) const { return maps + g * kTableMaps; }
    __device__ __forceinline__ const CUtensorMap *map_b(int g) const { return maps + g * kTableMaps + 1; }
    __device__ __forceinline__ const CUtensorMap *map_c(int g) const { return maps + g * kTableMaps + 2; }
    __device__ __forceinline__ const GemmProblemDev &problem(int g) const
    {
        return *reinterpret_cast<const GemmProblemDev *>(probs + static_cast<size_t>(g) * kTableProblemBytes);
    }
};

// Group of linear tile `tile`: the last problem whose first tile is <= tile
// (first tiles strictly increase). A short scan for parameter tables, a
// binary search for device tables of any length.
template <class P>
__device__ __forceinline__ int group_of_tile(const P &p, int tile)
{
    if constexpr (!P::kTable) {
        int g = 0;
#pragma unroll 1
        while (g + 1 < p.num_groups && tile >= p.problem(g + 1).tile_start) ++g;
        return g;
    } else {
        int lo = 0, hi = p.num_groups - 1;
#pragma unroll 1
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.problem(mid).tile_start <= tile)
                lo = mid;
            else
                hi = mid - 1;
        }
        return lo;
    }
}

__host__ __device__ constexpr uint32_t pow2_cols(uint32_t n)
{
    return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 512;
}

template <int KIND, int BN, int STAGES>
struct GemmCfg {
    static constexpr bool MX = KIND == 0;
    static constexpr int SF_BLK = MX ? 2 : 4;   // 512-B scale blocks per 128 rows per stage
    static constexpr int NCH = BN / 128;        // 128-row chunks of the B tile
    static constexpr uint32_t A_BYTES = 128 * 128;
    static constexpr uint32_t B_BYTES = BN * 128;
    static constexpr uint32_t SFA_BYTES = SF_BLK * 512;
    static constexpr uint32_t SFB_BYTES = NCH * SF_BLK * 512;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr uint32_t SF_COLS_A = SF_BLK * 4;
    static constexpr uint32_t SF_COLS_B = NCH * SF_BLK * 4;
    static constexpr uint32_t SF_COLS = SF_COLS_A + SF_COLS_B;
    static constexpr uint32_t TMEM_COLS = pow2_cols(BN + STAGES * SF_COLS);
    static constexpr uint32_t BAR_BYTES = 512;
    // epilogue staging for TMA stores of C: two 2 KB buffers (32 x 32 16-bit
    // values) per epilogue warp, where the stages leave room for them
    static constexpr uint32_t EPI_BYTES = 4 * 2 * 2048;
    static constexpr bool TMA_EPI = STAGES * STAGE_BYTES + BAR_BYTES + 1024 + EPI_BYTES <= 232448;
    static constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + (TMA_EPI ? EPI_BYTES : 0) + BAR_BYTES + 1024;
    static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
    static_assert(BN + STAGES * SF_COLS <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    // full, empty, sf_full, sf_data per stage; accf, acc_empty, two drain
    // barriers; TMEM address and flags
    static_assert((4 * STAGES + 4) * 8 + 16 <= BAR_BYTES, "barrier area");
};

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    if constexpr (F16) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

template <bool F16>
__device__ __forceinline__ float c_to_float(uint16_t v)
{
    if constexpr (F16)
        return __half2float(__ushort_as_half(v));
    else
        return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

// Output value of element (row, col) under the epilogue of pr: in fp32,
// ((alpha * acc) + beta * C[row, col]) + bias[col], C read before it is
// overwritten; beta = 0 leaves C unread and a null bias adds nothing.
template <bool F16>
__device__ __forceinline__ float epilogue_value(const GemmProblemDev &pr, float acc, int row, int col)
{
    float t = pr.alpha * acc;
    if (pr.beta != 0.0f)
        t += pr.beta * c_to_float<F16>(static_cast<const uint16_t *>(pr.c)[static_cast<int64_t>(row) * pr.ldc + col]);
    if (pr.bias) t += c_to_float<F16>(pr.bias[col]);
    return t;
}

// Stores 32 consecutive 16-bit C values of one row (16 packed pairs) at
// (row, col0), clipped at column n; 16-byte vector stores when aligned.
__device__ __forceinline__ void store_packed32(void *c, int64_t ldc, int row, int col0, int n, const uint32_t (&w)[16])
{
    uint16_t *p = static_cast<uint16_t *>(c) + static_cast<int64_t>(row) * ldc + col0;
    if (col0 + 32 <= n && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
        uint4 *q = reinterpret_cast<uint4 *>(p);
#pragma unroll
        for (int k = 0; k < 4; ++k) q[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (col0 + j < n) p[j] = static_cast<uint16_t>((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu));
    }
}

}  // namespace gemm_detail
}  // namespace mxfp4
