// Block-scaled FP4 GEMM on the 5th-generation tensor cores (tcgen05), shared by
// the MXFP4 GEMM (kind::mxf4, E8M0 per 32, bf16 C) and the grouped NVFP4 GEMM
// (kind::mxf4nvf4 scale_vec::4X, E4M3 per 16, fp16 C).
//
// What it computes: kernelbot-amd-mxfp4-mm-517169 docstring steps 3-4 and the
// gemm_a4w4 call (C = A_q . B_q^T with fp32 accumulation, bf16 out);
// kernelbot-nvfp4-group-gemm-496271 nvfp4_gemm_kernel (dot_scaled of e2m1 with
// per-16 scales, 128x128x256 tiles with a 4-stage TMA pipeline, fp16 out) and
// its custom_kernel loop over problems, here replaced by one launch whose
// blocks map a linear tile id to (problem, m-tile, n-tile) by prefix sums.
//
// One CTA computes one 128 x BN output tile (optionally one K-split of it):
//   warp 0 lane 0  TMA producer: A/B 128-byte-swizzled K-major tiles (256 FP4
//                  per row = 128 bytes per stage) and the stage's 512-byte
//                  scale blocks (1-D bulk copies straight from the blocked
//                  layout: consecutive K-blocks of 128 rows are contiguous).
//   warp 1         allocates TMEM; lane 0 issues tcgen05.cp (scales smem ->
//                  TMEM, one TMEM slot per pipeline stage) and four MMAs of
//                  K = 64 per stage, then commits the stage's "empty" barrier.
//   warps 0-3      epilogue: tcgen05.ld of the fp32 accumulator (warp w owns
//                  TMEM lanes 32w..32w+31 = output rows), convert, store.
// Split-K (splits > 1): each split writes fp32 partials to the workspace; the
// last split to arrive (atomic ticket) sums them in split order and writes C,
// then resets its ticket so the workspace stays zeroed.
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace mxfp4 {

__device__ int g_gemm_error;

namespace {

struct GemmProblemDev {
    const uint8_t *sfa;
    const uint8_t *sfb;
    void *c;
    int64_t ldc;
    int m, n, k;
    int m_tiles, n_tiles;
    int tile_start;
    int sf_cblocks;   // column blocks of 4 scales per 128-row chunk
    int pad_;
};

template <int MAXG>
struct GemmParams {
    CUtensorMap tma[MAXG];
    CUtensorMap tmb[MAXG];
    GemmProblemDev prob[MAXG];
    int num_groups;
    int total_tiles;
    int splits;
    int pad_;
    float *partials;
    int *tickets;
};

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
    static constexpr uint32_t BAR_BYTES = 256;
    static constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
    static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
    static_assert(BN + STAGES * SF_COLS <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <bool F16>
__device__ __forceinline__ void store_row32(void *c, int64_t ldc, int row, int col0, int n,
                                            const float (&f)[32])
{
    if constexpr (F16) {
        __half *p = static_cast<__half *>(c) + static_cast<int64_t>(row) * ldc + col0;
        if (col0 + 32 <= n && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 w;
                __half2 h0 = __floats2half2_rn(f[8 * q + 0], f[8 * q + 1]);
                __half2 h1 = __floats2half2_rn(f[8 * q + 2], f[8 * q + 3]);
                __half2 h2 = __floats2half2_rn(f[8 * q + 4], f[8 * q + 5]);
                __half2 h3 = __floats2half2_rn(f[8 * q + 6], f[8 * q + 7]);
                w.x = *reinterpret_cast<uint32_t *>(&h0);
                w.y = *reinterpret_cast<uint32_t *>(&h1);
                w.z = *reinterpret_cast<uint32_t *>(&h2);
                w.w = *reinterpret_cast<uint32_t *>(&h3);
                reinterpret_cast<uint4 *>(p)[q] = w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < n) p[j] = __float2half_rn(f[j]);
        }
    } else {
        __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(c) + static_cast<int64_t>(row) * ldc + col0;
        if (col0 + 32 <= n && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 w;
                __nv_bfloat162 h0 = __floats2bfloat162_rn(f[8 * q + 0], f[8 * q + 1]);
                __nv_bfloat162 h1 = __floats2bfloat162_rn(f[8 * q + 2], f[8 * q + 3]);
                __nv_bfloat162 h2 = __floats2bfloat162_rn(f[8 * q + 4], f[8 * q + 5]);
                __nv_bfloat162 h3 = __floats2bfloat162_rn(f[8 * q + 6], f[8 * q + 7]);
                w.x = *reinterpret_cast<uint32_t *>(&h0);
                w.y = *reinterpret_cast<uint32_t *>(&h1);
                w.z = *reinterpret_cast<uint32_t *>(&h2);
                w.w = *reinterpret_cast<uint32_t *>(&h3);
                reinterpret_cast<uint4 *>(p)[q] = w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < n) p[j] = __float2bfloat16_rn(f[j]);
        }
    }
}

template <int KIND, int BN, int STAGES, int MAXG, bool F16>
__global__ void __launch_bounds__(128, 1) bs_gemm_kernel(const __grid_constant__ GemmParams<MAXG> p)
{
    using Cfg = GemmCfg<KIND, BN, STAGES>;
    constexpr bool MX = Cfg::MX;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * Cfg::STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *sf_full = empty + STAGES;   // [STAGES] the stage's scales are in TMEM
    uint64_t *accf = sf_full + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accf + 1);
    int *last_flag = reinterpret_cast<int *>(tmem_slot + 1);
    int *abort_flag = last_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- tile decode: group by prefix sums, then m fastest within an n-tile
    const int tile = blockIdx.x;
    int g = 0;
#pragma unroll 1
    while (g + 1 < p.num_groups && tile >= p.prob[g + 1].tile_start) ++g;
    const GemmProblemDev &pr = p.prob[g];
    const int local = tile - pr.tile_start;
    const int m_tile = local % pr.m_tiles;
    const int n_tile = local / pr.m_tiles;
    const int k_stages = (pr.k + 255) / 256;
    const int split = blockIdx.y;
    const int s_begin = static_cast<int>(static_cast<int64_t>(k_stages) * split / p.splits);
    const int s_end = static_cast<int>(static_cast<int64_t>(k_stages) * (split + 1) / p.splits);
    const int nst = s_end - s_begin;
    const int k_steps_total = (pr.k + 63) / 64;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
            mbar_init(sf_full + s, 1);
        }
        mbar_init(accf, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&p.tma[g]);
        tma_prefetch_desc(&p.tmb[g]);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_acc = tmem;
    const uint32_t tmem_sf = tmem + BN;
    int issued = 0;  // stages armed by the producer (warp 0 lane 0 only)

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------ TMA producer
        const uint64_t pol = policy_evict_last();
        int nch_valid = 0;
#pragma unroll
        for (int j = 0; j < Cfg::NCH; ++j)
            if ((n_tile * Cfg::NCH + j) * 128 < pr.n) ++nch_valid;
        for (int i = 0; i < nst; ++i) {
            const int slot = i % STAGES;
            if (i >= STAGES && !mbar_wait(empty + slot, ((i / STAGES) - 1) & 1, &g_gemm_error, kErrWaitEmpty)) {
                *abort_flag = 1;
                break;
            }
            const int ks = s_begin + i;
            uint8_t *st = smem + slot * Cfg::STAGE_BYTES;
            const int blk0 = ks * Cfg::SF_BLK;
            const int nblk = min(Cfg::SF_BLK, pr.sf_cblocks - blk0);
            const uint32_t bytes = Cfg::A_BYTES + Cfg::B_BYTES + (1 + nch_valid) * nblk * 512;
            mbar_arrive_expect_tx(full + slot, bytes);
            tma_load_2d(st, &p.tma[g], ks * 128, m_tile * 128, full + slot, pol);
            tma_load_2d(st + Cfg::A_BYTES, &p.tmb[g], ks * 128, n_tile * BN, full + slot, pol);
            bulk_load(st + Cfg::A_BYTES + Cfg::B_BYTES,
                      pr.sfa + (static_cast<size_t>(m_tile) * pr.sf_cblocks + blk0) * 512, nblk * 512,
                      full + slot, pol);
            for (int j = 0; j < nch_valid; ++j)
                bulk_load(st + Cfg::A_BYTES + Cfg::B_BYTES + Cfg::SFA_BYTES + j * Cfg::SF_BLK * 512,
                          pr.sfb + (static_cast<size_t>(n_tile * Cfg::NCH + j) * pr.sf_cblocks + blk0) * 512,
                          nblk * 512, full + slot, pol);
            issued = i + 1;
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------- MMA issuer
        // Only MMAs are issued here (each tcgen05 instruction costs tens of
        // cycles to issue); warp 2 stages the scale factors into TMEM.
        constexpr uint32_t IDESC = idesc_block_scaled(BN, MX);
        for (int i = 0; i < nst; ++i) {
            const int slot = i % STAGES;
            if (!mbar_wait(full + slot, (i / STAGES) & 1, &g_gemm_error, kErrWaitFull) ||
                !mbar_wait(sf_full + slot, (i / STAGES) & 1, &g_gemm_error, kErrWaitFull)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            uint8_t *st = smem + slot * Cfg::STAGE_BYTES;
            const uint32_t a_base = smem_u32(st);
            const uint32_t b_base = smem_u32(st + Cfg::A_BYTES);
            const uint32_t tsfa = tmem_sf + slot * Cfg::SF_COLS;
            const uint32_t tsfb = tsfa + Cfg::SF_COLS_A;
            const int ks = s_begin + i;
            const int ksteps = min(4, k_steps_total - ks * 4);
            for (int kk = 0; kk < ksteps; ++kk) {
                const uint64_t ad = sdesc_sw128(a_base + kk * 32);
                const uint64_t bd = sdesc_sw128(b_base + kk * 32);
                const int blk = MX ? kk / 2 : kk;
                const uint32_t sfid = MX ? static_cast<uint32_t>(kk & 1) * 2u : 0u;
                const uint32_t idesc = idesc_with_sf_ids(IDESC, sfid, sfid);
                const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                if constexpr (MX)
                    mma_mxf4(tmem_acc, ad, bd, idesc, tsfa + blk * 4, tsfb + blk * Cfg::NCH * 4, acc);
                else
                    mma_nvf4(tmem_acc, ad, bd, idesc, tsfa + blk * 4, tsfb + blk * Cfg::NCH * 4, acc);
            }
            tc_commit(empty + slot);
        }
        // arrives once every MMA issued above has completed (also on abort)
        tc_commit(accf);
    } else if (warp == 2 && lane == 0) {
        // ------------------------------------- scale staging, smem -> TMEM
        // A stage's TMEM scale slot is rewritten only after the stage that
        // used it has been consumed: its smem slot was refilled, which needed
        // the MMAs' "empty" commit, so the full wait below orders the copies.
        for (int i = 0; i < nst; ++i) {
            const int slot = i % STAGES;
            if (!mbar_wait(full + slot, (i / STAGES) & 1, &g_gemm_error, kErrWaitFull)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            uint8_t *st = smem + slot * Cfg::STAGE_BYTES;
            const uint32_t sfa_s = smem_u32(st + Cfg::A_BYTES + Cfg::B_BYTES);
            const uint32_t sfb_s = sfa_s + Cfg::SFA_BYTES;
            const uint32_t tsfa = tmem_sf + slot * Cfg::SF_COLS;
            const uint32_t tsfb = tsfa + Cfg::SF_COLS_A;
            const int ks = s_begin + i;
            const int ksteps = min(4, k_steps_total - ks * 4);
            const int nblk = MX ? (ksteps + 1) / 2 : ksteps;
            for (int b = 0; b < nblk; ++b) {
                tc_cp_scale_block(tsfa + b * 4, sdesc_scale(sfa_s + b * 512));
#pragma unroll
                for (int j = 0; j < Cfg::NCH; ++j)
                    tc_cp_scale_block(tsfb + (b * Cfg::NCH + j) * 4,
                                      sdesc_scale(sfb_s + (j * Cfg::SF_BLK + b) * 512));
            }
            tc_commit(sf_full + slot);
        }
    }
    __syncwarp();

    // ----------------------------------------------------------- epilogue
    const bool acc_ok = mbar_wait(accf, 0, &g_gemm_error, kErrWaitAccum);
    tc_fence_after();
    __syncthreads();
    const bool run = acc_ok && (*abort_flag == 0);
    const int row_in_tile = warp * 32 + lane;
    const int row = m_tile * 128 + row_in_tile;
    const uint32_t t_row = tmem_acc + (static_cast<uint32_t>(warp * 32) << 16);

    if (run && p.splits == 1) {
        for (int c0 = 0; c0 < BN; c0 += 32) {
            const int col0 = n_tile * BN + c0;
            if (col0 >= pr.n) break;
            uint32_t v[32];
            tmem_ld32(t_row + c0, v);
            tmem_ld_wait();
            float f[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
            if (row < pr.m) store_row32<F16>(pr.c, pr.ldc, row, col0, pr.n, f);
        }
    } else if (run) {
        // partials: [split][n_tile][BN columns][M rows] fp32 (only rows < M),
        // consecutive lanes = consecutive rows, so stores and loads coalesce
        const size_t col_stride = static_cast<size_t>(pr.m);
        float *part = p.partials + (static_cast<size_t>(split) * pr.n_tiles + n_tile) * BN * col_stride;
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(t_row + c0, v);
            tmem_ld_wait();
            if (row < pr.m) {
#pragma unroll
                for (int j = 0; j < 32; ++j) part[(c0 + j) * col_stride + row] = __uint_as_float(v[j]);
            }
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const int old = atomicAdd(p.tickets + tile, 1);
            *last_flag = (old == p.splits - 1);
        }
        __syncthreads();
        if (*last_flag) {
            __threadfence();
            for (int c0 = 0; c0 < BN; c0 += 32) {
                const int col0 = n_tile * BN + c0;
                if (col0 >= pr.n || row >= pr.m) break;
                float f[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) f[j] = 0.0f;
                for (int sp = 0; sp < p.splits; ++sp) {
                    const float *q = p.partials + (static_cast<size_t>(sp) * pr.n_tiles + n_tile) * BN * col_stride;
#pragma unroll
                    for (int j = 0; j < 32; ++j) f[j] += __ldcg(q + (c0 + j) * col_stride + row);
                }
                store_row32<F16>(pr.c, pr.ldc, row, col0, pr.n, f);
            }
            if (threadIdx.x == 0) p.tickets[tile] = 0;
        }
    }

    // ----------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0) {
        // copies still in flight (only after an abort) must land before exit
        for (int i = max(0, issued - STAGES); i < issued; ++i)
            mbar_wait(full + (i % STAGES), (i / STAGES) & 1, &g_gemm_error, kErrWaitDrain);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

template <int KIND, int BN, int STAGES, int MAXG, bool F16>
cudaError_t launch_bs_gemm(const GemmParams<MAXG> &params, int splits, cudaStream_t stream)
{
    using Cfg = GemmCfg<KIND, BN, STAGES>;
    auto kern = bs_gemm_kernel<KIND, BN, STAGES, MAXG, F16>;
    static uint64_t configured = 0;  // one bit per device; setting it twice is harmless
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!(configured & (1ull << (dev & 63)))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured |= 1ull << (dev & 63);
    }
    dim3 grid(params.total_tiles, splits, 1);
    kern<<<grid, 128, Cfg::SMEM_BYTES, stream>>>(params);
    return cudaGetLastError();
}

constexpr int kMxBN = 256, kMxStages = 4;
constexpr int kNvBN = 256, kNvStages = 4;

template <int MAXG>
void fill_problem(GemmParams<MAXG> &P, int g, const GemmProblemHost &h, int bn, int vec, int &tiles)
{
    P.tma[g] = h.tma;
    P.tmb[g] = h.tmb;
    GemmProblemDev &d = P.prob[g];
    d.sfa = h.sfa;
    d.sfb = h.sfb;
    d.c = h.c;
    d.ldc = h.ldc;
    d.m = h.m;
    d.n = h.n;
    d.k = h.k;
    d.m_tiles = (h.m + 127) / 128;
    d.n_tiles = (h.n + bn - 1) / bn;
    d.tile_start = tiles;
    d.sf_cblocks = (h.k / vec + 3) / 4;
    d.pad_ = 0;
    tiles += d.m_tiles * d.n_tiles;
}

}  // namespace

int gemm_block_n(bool nvfp4) { return nvfp4 ? kNvBN : kMxBN; }

cudaError_t launch_gemm_mx(const GemmProblemHost &prob, int splits, float *partials, int *tickets,
                           cudaStream_t stream)
{
    GemmParams<1> P;
    memset(&P, 0, sizeof(P));
    int tiles = 0;
    fill_problem(P, 0, prob, kMxBN, 32, tiles);
    P.num_groups = 1;
    P.total_tiles = tiles;
    P.splits = splits;
    P.partials = partials;
    P.tickets = tickets;
    return launch_bs_gemm<0, kMxBN, kMxStages, 1, false>(P, splits, stream);
}

cudaError_t launch_gemm_nv_grouped(const GemmProblemHost *probs, int num_groups, cudaStream_t stream)
{
    GemmParams<kMaxGroups> P;
    memset(&P, 0, sizeof(P));
    int tiles = 0;
    for (int g = 0; g < num_groups; ++g) fill_problem(P, g, probs[g], kNvBN, 16, tiles);
    P.num_groups = num_groups;
    P.total_tiles = tiles;
    P.splits = 1;
    P.partials = nullptr;
    P.tickets = nullptr;
    return launch_bs_gemm<1, kNvBN, kNvStages, kMaxGroups, true>(P, 1, stream);
}

int read_and_clear_gemm_error()
{
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(int)) != cudaSuccess) return -1;
    cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(int));
    return v;
}

}  // namespace mxfp4
