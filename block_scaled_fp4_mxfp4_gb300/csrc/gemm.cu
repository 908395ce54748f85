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
// Single-CTA kernel, for problems too small to give every SM pair a 256 x 256
// tile (larger ones go to the CTA-pair kernel in gemm_pair.cu). Persistent:
// one CTA per SM walks the 128 x BN output tiles (BN = 256, or 128 when
// 256-wide tiles would leave most SMs idle), optionally split along K:
//   warp 0 lane 0  TMA producer: A/B 128-byte-swizzled K-major tiles (256 FP4
//                  per row = 128 bytes per stage) and, first and on their own
//                  barrier, the stage's 512-byte scale blocks (1-D bulk copies
//                  straight from the blocked layout: consecutive K-blocks of
//                  128 rows are contiguous). The weights of the first tile's
//                  first ring of stages are requested before the grid-
//                  dependency wait.
//   warp 1         allocates TMEM; lane 0 issues the four K = 64 MMAs of each
//                  stage and commits the stage's "empty" barrier.
//   warps 2, 3     lane 0 of each copies half of every stage's scale blocks
//                  smem -> TMEM (one TMEM slot per pipeline stage).
//   warps 4-7      epilogue: tcgen05.ld of the fp32 accumulator (TMEM lane
//                  quadrant = warp % 4 = output rows), convert, store, while
//                  the next tile's mainloop runs.
// Split-K (splits > 1): each split writes fp32 partials to the workspace; the
// last split to arrive (atomic ticket) sums them in split order and writes C,
// then resets its ticket so the workspace stays zeroed.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mxfp4 {

__device__ int g_gemm_error;

namespace {

using namespace gemm_detail;

__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// 128-row chunks of the B tile n_tile that hold rows below N.
template <class Cfg>
__device__ __forceinline__ int valid_chunks(const GemmProblemDev &pr, int n_tile)
{
    int n = 0;
#pragma unroll
    for (int j = 0; j < Cfg::NCH; ++j)
        if ((n_tile * Cfg::NCH + j) * 128 < pr.n) ++n;
    return n;
}

// Bulk loads of one stage's B scale blocks (nblk blocks from blk0 of each
// valid 128-row chunk) into the stage at st, completing on bar.
template <class Cfg>
__device__ __forceinline__ void load_b_scales(uint8_t *st, const GemmProblemDev &pr, int n_tile, int nch_valid, int blk0,
                                              int nblk, uint64_t *bar, uint64_t pol)
{
    for (int j = 0; j < nch_valid; ++j)
        bulk_load(st + Cfg::A_BYTES + Cfg::B_BYTES + Cfg::SFA_BYTES + j * Cfg::SF_BLK * 512,
                  pr.sfb + (static_cast<size_t>(n_tile * Cfg::NCH + j) * pr.sf_cblocks + blk0) * 512, nblk * 512,
                  bar, pol);
}

// One unit of work: an output tile, or one K-split of it.
struct Unit {
    int g, tile, m_tile, n_tile, split, s_begin, nst;
};

template <class P>
__device__ __forceinline__ Unit decode_unit(const P &p, int u)
{
    Unit w;
    w.tile = u % p.total_tiles;
    w.split = u / p.total_tiles;
    const int g = group_of_tile(p, w.tile);
    w.g = g;
    const GemmProblemDev &pr = p.problem(g);
    const int local = w.tile - pr.tile_start;
    w.m_tile = local % pr.m_tiles;
    w.n_tile = local / pr.m_tiles;
    const int k_stages = (pr.k + 255) / 256;
    w.s_begin = static_cast<int>(static_cast<int64_t>(k_stages) * w.split / p.splits);
    w.nst = static_cast<int>(static_cast<int64_t>(k_stages) * (w.split + 1) / p.splits) - w.s_begin;
    return w;
}

// Persistent block-scaled GEMM: each CTA loops over units blockIdx.x,
// blockIdx.x + gridDim.x, ... Warp roles:
//   warp 0 lane 0  TMA producer (stage ring shared by all units of the CTA)
//   warp 1         TMEM owner; lane 0 issues the MMAs of every unit
//   warps 2, 3     lane 0 of each copies half of each stage's scale blocks
//                  smem -> TMEM
//   warps 4-7      epilogue: drain the accumulator rows of a finished unit
//                  into registers, hand TMEM back to the MMA issuer, then
//                  write C while the next unit's mainloop runs
// EPI: the variant with the alpha / beta / bias epilogue (mxfp4_gemm_a4w4_ex);
// the plain variant keeps its registers for the common case.
// P: GemmParams<MAXG> (problems in kernel parameters) or GemmParamsTable
// (problems in a device table).
template <int KIND, int BN, int STAGES, class P, bool F16, bool EPI = false>
__global__ void __launch_bounds__(256, 1) bs_gemm_kernel(const __grid_constant__ P p)
{
    using Cfg = GemmCfg<KIND, BN, STAGES>;
    constexpr bool MX = Cfg::MX;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *epi_buf = smem + STAGES * Cfg::STAGE_BYTES;   // [epilogue warp][2][2 KB] when Cfg::TMA_EPI
    uint64_t *full = reinterpret_cast<uint64_t *>(epi_buf + (Cfg::TMA_EPI ? Cfg::EPI_BYTES : 0));
    uint64_t *empty = full + STAGES;
    uint64_t *sf_full = empty + STAGES;   // [STAGES] the stage's scales are in TMEM
    uint64_t *sf_data = sf_full + STAGES; // [STAGES] the stage's scale bytes are in smem
    uint64_t *accf = sf_data + STAGES;    // a unit's accumulator is complete
    uint64_t *acc_empty = accf + 1;       // the epilogue has drained the accumulator
    uint64_t *cp_done = acc_empty + 1;    // [2] every scale copy of warp 2 / 3 has completed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(cp_done + 2);
    int *last_flag = reinterpret_cast<int *>(tmem_slot + 1);
    volatile int *abort_flag = last_flag + 1;
    volatile int *epi_go = last_flag + 2;   // [2] per-unit decision of the epilogue warps

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int units = p.total_tiles * p.splits;
    // stages of this CTA's first unit whose weights thread 0 requested before
    // the grid-dependency wait (thread 0 is also the TMA producer)
    int pre = 0;
    const uint64_t pol_w = threadIdx.x == 0 ? policy_evict_last() : 0;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
            mbar_init(sf_full + s, 2);   // one commit from each scale-copy thread
            mbar_init(sf_data + s, 1);
        }
        mbar_init(accf, 1);
        mbar_init(acc_empty, 128);
        mbar_init(cp_done, 1);
        mbar_init(cp_done + 1, 1);
        *abort_flag = 0;
        fence_mbar_init();
        // a device table's maps are fetched when first used, below
        for (int g = 0; g < (P::kTable ? 0 : p.num_groups); ++g) {
            tma_prefetch_desc(p.map_a(g));
            tma_prefetch_desc(p.map_b(g));
            if (Cfg::TMA_EPI && p.problem(g).c_tma) tma_prefetch_desc(p.map_c(g));
        }
        // Weights (B and its scales) are read-only inputs that no kernel of
        // this library writes, so the first unit's first ring of weight
        // stages is requested before the grid-dependency wait: under
        // programmatic dependent launch it streams while the preceding grid
        // (the quantization of A, in a quant -> GEMM call) finishes. Each
        // stage's barriers are armed here for the whole stage; A and its
        // scales follow once that grid has completed. Problems in a device
        // table are read only after the wait.
        if constexpr (!P::kTable) {
            if (static_cast<int>(blockIdx.x) < units) {
                const Unit w = decode_unit(p, blockIdx.x);
                const GemmProblemDev &pr = p.problem(w.g);
                const int nch_valid = valid_chunks<Cfg>(pr, w.n_tile);
                pre = min(STAGES, w.nst);
                for (int i = 0; i < pre; ++i) {
                    const int ks = w.s_begin + i;
                    const int blk0 = ks * Cfg::SF_BLK;
                    const int nblk = min(Cfg::SF_BLK, pr.sf_cblocks - blk0);
                    uint8_t *st = smem + i * Cfg::STAGE_BYTES;
                    mbar_arrive_expect_tx(sf_data + i, (1 + nch_valid) * nblk * 512);
                    load_b_scales<Cfg>(st, pr, w.n_tile, nch_valid, blk0, nblk, sf_data + i, pol_w);
                    mbar_arrive_expect_tx(full + i, Cfg::A_BYTES + Cfg::B_BYTES);
                    tma_load_2d(st + Cfg::A_BYTES, p.map_b(w.g), ks * 128, w.n_tile * BN, full + i, pol_w);
                }
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    // every other global access waits for the preceding grid in the stream
    grid_dependency_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_launch_dependents();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_acc = tmem;
    const uint32_t tmem_sf = tmem + BN;
    int issued = 0;   // stages armed by the producer (warp 0 lane 0 only)

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------ TMA producer
            const uint64_t pol = pol_w;
            int gs = 0, g_seen = -1;
            // the first unit always runs: its stages below `pre` have weights
            // in flight on armed barriers, which complete only once A follows
            for (int u = blockIdx.x; u < units && (u == static_cast<int>(blockIdx.x) || !*abort_flag);
                 u += gridDim.x) {
                const Unit w = decode_unit(p, u);
                const GemmProblemDev &pr = p.problem(w.g);
                if (P::kTable && w.g != g_seen) {
                    tma_desc_acquire(p.map_a(w.g));
                    tma_desc_acquire(p.map_b(w.g));
                    g_seen = w.g;
                }
                const int nch_valid = valid_chunks<Cfg>(pr, w.n_tile);
                for (int i = 0; i < w.nst; ++i, ++gs) {
                    const int slot = gs % STAGES;
                    if (gs >= STAGES &&
                        !mbar_wait(empty + slot, ((gs / STAGES) - 1) & 1, &g_gemm_error, kErrWaitEmpty, p.wait_ns)) {
                        *abort_flag = 1;
                        break;
                    }
                    const int ks = w.s_begin + i;
                    uint8_t *st = smem + slot * Cfg::STAGE_BYTES;
                    const int blk0 = ks * Cfg::SF_BLK;
                    const int nblk = min(Cfg::SF_BLK, pr.sf_cblocks - blk0);
                    // a stage below `pre` has its barriers armed and its weights
                    // requested already (only in the first unit, where gs = i)
                    const bool weights_sent = gs < pre;
                    // the scale blocks first, on their own barrier: their copy into
                    // TMEM then overlaps the arrival of the operand tiles
                    if (!weights_sent) mbar_arrive_expect_tx(sf_data + slot, (1 + nch_valid) * nblk * 512);
                    bulk_load(st + Cfg::A_BYTES + Cfg::B_BYTES,
                              pr.sfa + (static_cast<size_t>(w.m_tile) * pr.sf_cblocks + blk0) * 512, nblk * 512,
                              sf_data + slot, pol);
                    if (!weights_sent) {
                        load_b_scales<Cfg>(st, pr, w.n_tile, nch_valid, blk0, nblk, sf_data + slot, pol);
                        mbar_arrive_expect_tx(full + slot, Cfg::A_BYTES + Cfg::B_BYTES);
                    }
                    tma_load_2d(st, p.map_a(w.g), ks * 128, w.m_tile * 128, full + slot, pol);
                    if (!weights_sent)
                        tma_load_2d(st + Cfg::A_BYTES, p.map_b(w.g), ks * 128, w.n_tile * BN, full + slot, pol);
                    issued = gs + 1;
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        // Only MMAs are issued here (a tcgen05 instruction costs tens of cycles
        // to issue); warps 2 and 3 stage the scale factors into TMEM.
        constexpr uint32_t IDESC = idesc_block_scaled(BN, MX);
        int gs = 0, ul = 0, commits = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++ul) {
            const Unit w = decode_unit(p, u);
            const GemmProblemDev &pr = p.problem(w.g);
            const int k_steps_total = (pr.k + 63) / 64;
            if (ul > 0 && !mbar_wait(acc_empty, (ul - 1) & 1, &g_gemm_error, kErrWaitAccum, p.wait_ns)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            bool ok = true;
            for (int i = 0; i < w.nst; ++i, ++gs) {
                const int slot = gs % STAGES;
                const uint32_t ph = (gs / STAGES) & 1;
                // one wait per stage: the scale-copy threads commit sf_full only
                // after they also saw the stage's operand tiles land
                if (!mbar_wait(sf_full + slot, ph, &g_gemm_error, kErrWaitFull, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint8_t *st = smem + slot * Cfg::STAGE_BYTES;
                const uint32_t a_base = smem_u32(st);
                const uint32_t b_base = smem_u32(st + Cfg::A_BYTES);
                const uint32_t tsfa = tmem_sf + slot * Cfg::SF_COLS;
                const uint32_t tsfb = tsfa + Cfg::SF_COLS_A;
                const int ks = w.s_begin + i;
                // K step kk of the stage starts 32 bytes (2 descriptor units) further
                const uint64_t ad = sdesc_sw128(a_base);
                const uint64_t bd = sdesc_sw128(b_base);
                const int ksteps = min(4, k_steps_total - ks * 4);
                auto mma_step = [&](int kk) {
                    const int blk = MX ? kk / 2 : kk;
                    const uint32_t sfid = MX ? static_cast<uint32_t>(kk & 1) * 2u : 0u;
                    const uint32_t idesc = idesc_with_sf_ids(IDESC, sfid, sfid);
                    const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                    if constexpr (MX)
                        mma_mxf4(tmem_acc, ad + 2 * kk, bd + 2 * kk, idesc, tsfa + blk * 4, tsfb + blk * Cfg::NCH * 4, acc);
                    else
                        mma_nvf4(tmem_acc, ad + 2 * kk, bd + 2 * kk, idesc, tsfa + blk * 4, tsfb + blk * Cfg::NCH * 4, acc);
                };
                // the issuing thread is the bottleneck: full stages go unrolled
                if (ksteps == 4) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) mma_step(kk);
                } else {
                    for (int kk = 0; kk < ksteps; ++kk) mma_step(kk);
                }
                tc_commit(empty + slot);
            }
            // arrives once every MMA issued above has completed (also on abort)
            tc_commit(accf);
            ++commits;
            if (!ok) {
                *abort_flag = 1;
                break;
            }
        }
        // The epilogue waits for every commit unless it stopped early; the
        // accumulator must not be in use when TMEM is released.
        if (commits > 0) mbar_wait(accf, (commits - 1) & 1, &g_gemm_error, kErrWaitDrain);
    } else if (warp == 2 || warp == 3) {
        if (lane == 0) {
            // ----------------------------------------- scale staging, smem -> TMEM
            // Lane 0 of warps 2 and 3 share the copies of each stage (even and odd
            // K blocks): one tcgen05.cp takes tens of cycles to issue, and a
            // stage of NVFP4 scales needs twelve. A stage's TMEM scale slot is
            // rewritten only after the stage that used it has been consumed: its
            // smem slot was refilled, which needed the MMAs' "empty" commit, so
            // the scale-data wait below orders the copies.
            int gs = 0;
            bool stop = false;
            for (int u = blockIdx.x; u < units && !stop && !*abort_flag; u += gridDim.x) {
                const Unit w = decode_unit(p, u);
                const GemmProblemDev &pr = p.problem(w.g);
                const int k_steps_total = (pr.k + 63) / 64;
                for (int i = 0; i < w.nst; ++i, ++gs) {
                    const int slot = gs % STAGES;
                    if (!mbar_wait(sf_data + slot, (gs / STAGES) & 1, &g_gemm_error, kErrWaitFull, p.wait_ns)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    uint8_t *st = smem + slot * Cfg::STAGE_BYTES;
                    const uint32_t sfa_s = smem_u32(st + Cfg::A_BYTES + Cfg::B_BYTES);
                    const uint32_t sfb_s = sfa_s + Cfg::SFA_BYTES;
                    const uint32_t tsfa = tmem_sf + slot * Cfg::SF_COLS;
                    const uint32_t tsfb = tsfa + Cfg::SF_COLS_A;
                    const int ks = w.s_begin + i;
                    const int ksteps = min(4, k_steps_total - ks * 4);
                    const int nblk = MX ? (ksteps + 1) / 2 : ksteps;
                    for (int b = warp - 2; b < nblk; b += 2) {
                        tc_cp_scale_block(tsfa + b * 4, sdesc_scale(sfa_s + b * 512));
#pragma unroll
                        for (int j = 0; j < Cfg::NCH; ++j)
                            tc_cp_scale_block(tsfb + (b * Cfg::NCH + j) * 4,
                                              sdesc_scale(sfb_s + (j * Cfg::SF_BLK + b) * 512));
                    }
                    // the MMA issuer waits only for sf_full: it also stands for the
                    // stage's operand tiles
                    if (!mbar_wait(full + slot, (gs / STAGES) & 1, &g_gemm_error, kErrWaitFull, p.wait_ns)) {
                        stop = true;
                        break;
                    }
                    tc_commit(sf_full + slot);
                }
            }
            if (stop) *abort_flag = 1;
            // every scale copy this thread issued (also those of a stage given up
            // above) completes before TMEM is released
            tc_commit(cp_done + (warp - 2));
            mbar_wait(cp_done + (warp - 2), 0, &g_gemm_error, kErrWaitDrain);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                  // TMEM lane quadrant of this warp
        const int row_in_tile = q * 32 + lane;
        const uint32_t t_row = tmem_acc + (static_cast<uint32_t>(q * 32) << 16);
        uint8_t *wbuf = epi_buf + q * 4096;     // this warp's two staging buffers
        int stores = 0;                         // TMA stores this warp has issued
        int ul = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++ul) {
            const Unit w = decode_unit(p, u);
            const GemmProblemDev &pr = p.problem(w.g);
            // one thread waits and decides for all four warps, so that they
            // leave the loop together (the split-K path has named barriers)
            if (threadIdx.x == 128) {
                const bool ok = mbar_wait(accf, ul & 1, &g_gemm_error, kErrWaitAccum, p.wait_ns);
                if (!ok) *abort_flag = 1;
                epi_go[ul & 1] = ok;
            }
            epilogue_bar();
            if (!epi_go[ul & 1]) break;
            tc_fence_after();
            const bool run = (*abort_flag == 0);
            const int row = w.m_tile * 128 + row_in_tile;
            if (EPI && p.splits == 1 && pr.epi) {
                // epilogue with alpha / beta / bias: each 32-column chunk is
                // finished and stored straight from TMEM, then TMEM is released
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(t_row + c * 32, v);
                    tmem_ld_wait();
                    const int col0 = w.n_tile * BN + c * 32;
                    if (run && row < pr.m && col0 < pr.n) {
                        uint32_t part[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int ca = min(col0 + 2 * j, pr.n - 1), cb = min(col0 + 2 * j + 1, pr.n - 1);
                            part[j] = pack2<F16>(epilogue_value<F16>(pr, __uint_as_float(v[2 * j]), row, ca),
                                                 epilogue_value<F16>(pr, __uint_as_float(v[2 * j + 1]), row, cb));
                        }
                        store_packed32(pr.c, pr.ldc, row, col0, pr.n, part);
                    }
                }
                tc_fence_before();
                mbar_arrive(acc_empty);
            } else if (p.splits == 1) {
                // drain the row into registers, release TMEM, then store
                uint32_t pk[BN / 2];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(t_row + c * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        pk[c * 16 + j] = pack2<F16>(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                }
                tc_fence_before();
                mbar_arrive(acc_empty);
                if (Cfg::TMA_EPI && pr.c_tma) {
                    // 32 x 32 sub-tiles of this warp's 32 rows, written by TMA from
                    // shared memory: each lane writes its row's 64 bytes in the
                    // 64-byte-swizzled layout of the tensor map (16-byte chunk j of
                    // row r at chunk j ^ ((r / 2) % 4)); the map clips rows past M
                    // and columns past N.
                    auto stage_subtile = [&](uint8_t *buf, int c) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            *reinterpret_cast<uint4 *>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                                make_uint4(pk[c * 16 + 4 * j], pk[c * 16 + 4 * j + 1], pk[c * 16 + 4 * j + 2],
                                           pk[c * 16 + 4 * j + 3]);
                    };
                    if (P::kTable && run && lane == 0) tma_desc_acquire(p.map_c(w.g));
                    if (run && u + static_cast<int>(gridDim.x) >= units) {
                        // The CTA's last unit: the stage ring is free (every MMA
                        // that read it has completed), so all sub-tiles are staged
                        // there at once, behind one proxy fence (a fence and a
                        // store issue cost ~0.1 us per sub-tile, measured).
#pragma unroll
                        for (int c = 0; c < BN / 32; ++c) stage_subtile(smem + (q * (BN / 32) + c) * 2048, c);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            for (int c = 0; c < BN / 32; ++c) {
                                const int col0 = w.n_tile * BN + c * 32;
                                if (col0 < pr.n)
                                    tma_store_2d(p.map_c(w.g), smem + (q * (BN / 32) + c) * 2048, col0,
                                                 w.m_tile * 128 + q * 32);
                            }
                            bulk_commit();
                        }
                    } else if (run) {
                        // otherwise through the warp's two staging buffers, while
                        // the next unit's mainloop uses the ring
#pragma unroll
                        for (int c = 0; c < BN / 32; ++c) {
                            const int col0 = w.n_tile * BN + c * 32;
                            if (col0 < pr.n) {
                                uint8_t *buf = wbuf + (stores & 1) * 2048;
                                if (stores >= 2) {
                                    if (lane == 0) bulk_wait_read<1>();   // the buffer's previous store has read it
                                    __syncwarp();
                                }
                                stage_subtile(buf, c);
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    tma_store_2d(p.map_c(w.g), buf, col0, w.m_tile * 128 + q * 32);
                                    bulk_commit();
                                }
                                ++stores;
                            }
                        }
                    }
                } else if (run && row < pr.m) {
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
                        const int col0 = w.n_tile * BN + c * 32;
                        if (col0 < pr.n) {
                            uint32_t part[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) part[j] = pk[c * 16 + j];
                            store_packed32(pr.c, pr.ldc, row, col0, pr.n, part);
                        }
                    }
                }
            } else {
                // split-K: partials [split][n_tile][BN][M] fp32 (rows < M only),
                // then the last split to arrive sums them in split order
                const size_t col_stride = static_cast<size_t>(pr.m);
                float *part = p.partials + (static_cast<size_t>(w.split) * pr.n_tiles + w.n_tile) * BN * col_stride;
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(t_row + c0, v);
                    tmem_ld_wait();
                    if (run && row < pr.m) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) part[(c0 + j) * col_stride + row] = __uint_as_float(v[j]);
                    }
                }
                tc_fence_before();
                mbar_arrive(acc_empty);
                __threadfence();
                epilogue_bar();
                if (threadIdx.x == 128) {
                    // a split that gave up adds 2^20 as well: the last split then
                    // leaves C unwritten instead of summing missing partials
                    const int old = atomicAdd(p.tickets + w.tile, run ? 1 : 1 + (1 << 20));
                    const bool last = (old & 0xFFFFF) == p.splits - 1;
                    *last_flag = !last ? 0 : ((old >> 20) == 0 && run) ? 1 : 2;
                }
                epilogue_bar();
                if (*last_flag == 1) {
                    __threadfence();
                    for (int c0 = 0; c0 < BN; c0 += 32) {
                        const int col0 = w.n_tile * BN + c0;
                        if (col0 >= pr.n || row >= pr.m) break;
                        float f[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) f[j] = 0.0f;
                        for (int sp = 0; sp < p.splits; ++sp) {
                            const float *qv = p.partials + (static_cast<size_t>(sp) * pr.n_tiles + w.n_tile) * BN * col_stride;
#pragma unroll
                            for (int j = 0; j < 32; ++j) f[j] += __ldcg(qv + (c0 + j) * col_stride + row);
                        }
                        if (EPI && pr.epi) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) f[j] = epilogue_value<F16>(pr, f[j], row, min(col0 + j, pr.n - 1));
                        }
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) pk[j] = pack2<F16>(f[2 * j], f[2 * j + 1]);
                        store_packed32(pr.c, pr.ldc, row, col0, pr.n, pk);
                    }
                }
                // the last split leaves its ticket at zero, also after an abort
                if (threadIdx.x == 128 && *last_flag) p.tickets[w.tile] = 0;
                epilogue_bar();   // last_flag is reused by the next unit
            }
        }
        // the C stores by TMA have read their staging buffers before the CTA
        // leaves (their writes complete with the grid, before any dependent
        // grid's dependency wait returns)
        if (Cfg::TMA_EPI && lane == 0) bulk_wait_read<0>();
    }
    __syncwarp();

    // ----------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0) {
        // copies still in flight (only after an abort) must land before exit
        for (int i = max(0, issued - STAGES); i < issued; ++i) {
            mbar_wait(sf_data + (i % STAGES), (i / STAGES) & 1, &g_gemm_error, kErrWaitDrain);
            mbar_wait(full + (i % STAGES), (i / STAGES) & 1, &g_gemm_error, kErrWaitDrain);
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

template <int KIND, int BN, int STAGES, class P, bool F16, bool EPI = false>
cudaError_t launch_bs_gemm(const P &params, cudaStream_t stream)
{
    using Cfg = GemmCfg<KIND, BN, STAGES>;
    auto kern = bs_gemm_kernel<KIND, BN, STAGES, P, F16, EPI>;
    static KernelOnce once;
    int sms = 0;
    const cudaError_t e = prepare_kernel(kern, Cfg::SMEM_BYTES, once, &sms);
    if (e != cudaSuccess) return e;
    const int units = params.total_tiles * params.splits;
    const int grid = min(units, max(1, sms));
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    P launch_params = params;
    launch_params.wait_ns = wait_limit_ns();
    return cudaLaunchKernelEx(&cfg, kern, launch_params);
}

constexpr int kMxStages = 4;        // BN = 256
constexpr int kMxNarrowStages = 6;  // BN = 128: 34 KB stages
constexpr int kNvBN = 256, kNvStages = 4;

template <int MAXG>
void fill_problem(GemmParams<MAXG> &P, int g, const GemmProblemHost &h, int bn, int vec, int &tiles)
{
    P.tma[g] = h.tma;
    P.tmb[g] = h.tmb;
    P.tmc[g] = h.tmc;
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
    d.epi = h.epi ? 1 : 0;
    d.alpha = h.alpha;
    d.beta = h.beta;
    d.bias = static_cast<const uint16_t *>(h.bias);
    d.c_tma = h.c_tma ? 1 : 0;
    tiles += d.m_tiles * d.n_tiles;
}

}  // namespace

int gemm_block_n_nv() { return kNvBN; }

cudaError_t launch_gemm_mx(const GemmProblemHost &prob, int bn, int splits, float *partials, int *tickets,
                           cudaStream_t stream)
{
    if (bn != 128 && bn != 256) return cudaErrorInvalidValue;
    GemmParams<1> P;
    memset(&P, 0, sizeof(P));
    int tiles = 0;
    fill_problem(P, 0, prob, bn, 32, tiles);
    P.num_groups = 1;
    P.total_tiles = tiles;
    P.splits = splits;
    P.partials = partials;
    P.tickets = tickets;
    if (prob.epi) {
        if (bn == 128) return launch_bs_gemm<0, 128, kMxNarrowStages, GemmParams<1>, false, true>(P, stream);
        return launch_bs_gemm<0, 256, kMxStages, GemmParams<1>, false, true>(P, stream);
    }
    if (bn == 128) return launch_bs_gemm<0, 128, kMxNarrowStages, GemmParams<1>, false>(P, stream);
    return launch_bs_gemm<0, 256, kMxStages, GemmParams<1>, false>(P, stream);
}

// The grouped launch: problems in kernel parameters up to kMaxGroups, else in
// the device table (filled here, on the stream, before the launch).
template <int KIND, int BN, int STAGES, bool F16>
cudaError_t launch_grouped(const GemmProblemHost *probs, int num_groups, void *table, int vec, cudaStream_t stream)
{
    if (num_groups <= kMaxGroups) {
        GemmParams<kMaxGroups> P;
        memset(&P, 0, sizeof(P));
        int tiles = 0;
        for (int g = 0; g < num_groups; ++g) fill_problem(P, g, probs[g], BN, vec, tiles);
        P.num_groups = num_groups;
        P.total_tiles = tiles;
        P.splits = 1;
        return launch_bs_gemm<KIND, BN, STAGES, GemmParams<kMaxGroups>, F16>(P, stream);
    }
    if (!table || (reinterpret_cast<uintptr_t>(table) & 63u) != 0) return cudaErrorInvalidValue;
    std::vector<uint8_t> host(group_table_bytes(num_groups), 0);
    CUtensorMap *maps = reinterpret_cast<CUtensorMap *>(host.data());
    uint8_t *recs = host.data() + static_cast<size_t>(num_groups) * kTableMaps * sizeof(CUtensorMap);
    GemmParams<1> one;
    int tiles = 0;
    for (int g = 0; g < num_groups; ++g) {
        memset(&one, 0, sizeof(one));
        int t = tiles;
        fill_problem(one, 0, probs[g], BN, vec, t);
        one.prob[0].tile_start = tiles;
        tiles = t;
        maps[g * kTableMaps + 0] = probs[g].tma;
        maps[g * kTableMaps + 1] = probs[g].tmb;
        maps[g * kTableMaps + 2] = probs[g].tmc;
        memcpy(recs + static_cast<size_t>(g) * kTableProblemBytes, &one.prob[0], sizeof(GemmProblemDev));
    }
    cudaError_t e = upload_table(table, host.data(), host.size(), stream);
    if (e != cudaSuccess) return e;
    GemmParamsTable T;
    memset(&T, 0, sizeof(T));
    T.maps = static_cast<const CUtensorMap *>(table);
    T.probs = static_cast<const uint8_t *>(table) + static_cast<size_t>(num_groups) * kTableMaps * sizeof(CUtensorMap);
    T.num_groups = num_groups;
    T.total_tiles = tiles;
    T.splits = 1;
    return launch_bs_gemm<KIND, BN, STAGES, GemmParamsTable, F16>(T, stream);
}

cudaError_t launch_gemm_nv_grouped(const GemmProblemHost *probs, int num_groups, void *table, cudaStream_t stream)
{
    return launch_grouped<1, kNvBN, kNvStages, true>(probs, num_groups, table, 16, stream);
}

cudaError_t launch_gemm_mx_grouped(const GemmProblemHost *probs, int num_groups, void *table, cudaStream_t stream)
{
    return launch_grouped<0, kNvBN, kMxStages, false>(probs, num_groups, table, 32, stream);
}

namespace {

constexpr int kUploadChunk = 30720;   // table bytes per upload launch (kernel parameters)

struct UploadChunk {
    uint4 *dst;
    uint32_t n16;                      // 16-byte words to copy
    uint32_t pad_;
    uint4 data[kUploadChunk / 16];
};

__global__ void __launch_bounds__(256) table_upload_kernel(const __grid_constant__ UploadChunk c)
{
    for (uint32_t i = threadIdx.x; i < c.n16; i += blockDim.x) c.dst[i] = c.data[i];
}

}  // namespace

cudaError_t upload_table(void *dst, const void *src, size_t bytes, cudaStream_t stream)
{
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) != 0 || bytes % 16 != 0) return cudaErrorInvalidValue;
    static UploadChunk c;   // host staging of one launch's parameters (copied at launch)
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    for (size_t off = 0; off < bytes; off += kUploadChunk) {
        const size_t n = std::min(bytes - off, static_cast<size_t>(kUploadChunk));
        c.dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(dst) + off);
        c.n16 = static_cast<uint32_t>(n / 16);
        memcpy(c.data, static_cast<const uint8_t *>(src) + off, n);
        table_upload_kernel<<<1, 256, 0, stream>>>(c);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int read_and_clear_gemm_error()
{
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(int)) != cudaSuccess) return -1;
    cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(int));
    return v;
}

}  // namespace mxfp4
