// Block-scaled FP4 GEMM on CTA pairs (tcgen05 cta_group::2), for problems
// with enough 256 x 256 output tiles to fill the GPU: the MXFP4 GEMM at large
// M (kind::mxf4, bf16 C) and the grouped NVFP4 GEMM (kind::mxf4nvf4
// scale_vec::4X, fp16 C).
//
// What it computes is the same as the single-CTA kernel in gemm.cu
// (kernelbot-amd-mxfp4-mm-517169 docstring steps 3-4 and the gemm_a4w4 call;
// kernelbot-nvfp4-group-gemm-496271 nvfp4_gemm_kernel and its loop over
// problems). The difference is the MMA: one instruction of M = 256, N = 256,
// K = 64 runs on the tensor cores of both SMs of a cluster pair. Each CTA
// holds its own 128 rows of A and one half of the 256 rows of B, so an SM
// receives 32 KB of operands per 256-deep K stage instead of the 48 KB a
// single-CTA 128 x 256 tile needs for the same work, and one thread issues the
// MMAs of two SMs.
//
// Persistent: cluster pair p walks the pair tiles p, p + pairs, ...
//   warp 0 lane 0   (both CTAs) TMA producer for this CTA's A rows and B half,
//                   its A scale blocks and the scale blocks of all 256 B rows;
//                   the copies of both CTAs complete rank 0's barriers, which
//                   rank 0 arms with the bytes of both
//   warp 1          (both CTAs) allocates / frees the pair's TMEM; lane 0 of
//                   rank 0 issues the MMAs
//   warps 2, 3      lane 0 of rank 0 copies the stage's scale blocks into both
//                   CTAs' TMEM (even / odd K blocks)
//   warps 4-11      (both CTAs) epilogue: each drains 32 accumulator rows x
//                   128 columns of this CTA into registers, hands TMEM back
//                   (arrive on rank 0's barrier) and stores C while the next
//                   tile's mainloop runs
// MMA completion is signalled to both CTAs by multicast commits. Every wait
// on an mbarrier is bounded; a final cluster barrier keeps both CTAs alive
// until neither can touch the other's shared memory, then the pair frees its
// TMEM together.
#include <cstring>
#include <vector>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mxfp4 {

__device__ int g_gemm_pair_error;

namespace {

using namespace gemm_detail;

template <int KIND, int STAGES>
struct PairCfg {
    static constexpr bool MX = KIND == 0;
    static constexpr int SF_BLK = MX ? 2 : 4;           // 512-B scale blocks per 128 rows per stage
    static constexpr uint32_t A_BYTES = 128 * 128;      // this CTA's 128 rows x 256 FP4
    static constexpr uint32_t B_BYTES = 128 * 128;      // this CTA's half of the 256 B rows
    static constexpr uint32_t SFA_BYTES = SF_BLK * 512;
    static constexpr uint32_t SFB_BYTES = 2 * SF_BLK * 512;   // both 128-row chunks of the tile's B
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr uint32_t SF_COLS_A = SF_BLK * 4;
    static constexpr uint32_t SF_COLS = 3 * SF_BLK * 4;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t BAR_BYTES = 512;
    static constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
    static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
    static_assert(256 + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    // full, sf_data, empty, sf_full per stage; accf, acc_empty, two drain
    // barriers; TMEM address, flags and the producer's stage count
    static_assert((4 * STAGES + 4) * 8 + 24 <= BAR_BYTES, "barrier area");
};

constexpr int kPairThreads = 384;        // warps 0-3: producer, MMA issuer, two scale-copy warps; 4-11: epilogue
constexpr int kPairEpiWarps = 8;

__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// The problems of a launch in kernel parameters (up to MAXG of them).
template <int MAXG>
struct PairParams {
    CUtensorMap tma[MAXG];     // packed A, box {128 B, 128 rows}
    CUtensorMap tmb[MAXG];     // packed B, box {128 B, 128 rows}
    CUtensorMap tmsfa[MAXG];   // A scale blocks [blocks, 128 u32], box {128, SF_BLK}
    CUtensorMap tmsfb[MAXG];   // B scale blocks, same
    GemmProblemDev prob[MAXG];
    int num_groups;
    int total_tiles;
    uint64_t wait_ns;          // limit of the waits that guard work
    static constexpr bool kTable = false;
    static constexpr bool kColumnsFastest = MAXG == 1;   // tile order of a single problem
    __device__ __forceinline__ const CUtensorMap *map_a(int g) const { return &tma[g]; }
    __device__ __forceinline__ const CUtensorMap *map_b(int g) const { return &tmb[g]; }
    __device__ __forceinline__ const CUtensorMap *map_sfa(int g) const { return &tmsfa[g]; }
    __device__ __forceinline__ const CUtensorMap *map_sfb(int g) const { return &tmsfb[g]; }
    __device__ __forceinline__ const GemmProblemDev &problem(int g) const { return prob[g]; }
};

// The problems of a launch in a device table (any number): per group the
// maps A, B, A scales, B scales, then the problem record.
struct PairParamsTable {
    const CUtensorMap *maps;   // [num_groups][kTableMaps]
    const uint8_t *probs;      // [num_groups][kTableProblemBytes]
    int num_groups;
    int total_tiles;
    uint64_t wait_ns;
    static constexpr bool kTable = true;
    static constexpr bool kColumnsFastest = false;
    __device__ __forceinline__ const CUtensorMap *map_a(int g) const { return maps + g * kTableMaps; }
    __device__ __forceinline__ const CUtensorMap *map_b(int g) const { return maps + g * kTableMaps + 1; }
    __device__ __forceinline__ const CUtensorMap *map_sfa(int g) const { return maps + g * kTableMaps + 2; }
    __device__ __forceinline__ const CUtensorMap *map_sfb(int g) const { return maps + g * kTableMaps + 3; }
    __device__ __forceinline__ const GemmProblemDev &problem(int g) const
    {
        return *reinterpret_cast<const GemmProblemDev *>(probs + static_cast<size_t>(g) * kTableProblemBytes);
    }
};

struct PairUnit {
    int g, m_pair, n_tile;
};

// Pair tiles are numbered group by group, 256-row tiles fastest, except in a
// launch of one problem, where 256-column tiles go fastest (measured at
// 8192^3: 177.3 against 178.4 us; grouped lists ran 0.1-0.4 us slower with it).
template <class P>
__device__ __forceinline__ PairUnit decode_pair_unit(const P &p, int u)
{
    PairUnit w;
    const int g = group_of_tile(p, u);
    w.g = g;
    const GemmProblemDev &pr = p.problem(g);
    const int local = u - pr.tile_start;
    if constexpr (P::kColumnsFastest) {
        w.n_tile = local % pr.n_tiles;
        w.m_pair = local / pr.n_tiles;
    } else {
        w.m_pair = local % pr.m_tiles;
        w.n_tile = local / pr.m_tiles;
    }
    return w;
}

// Weight half of stage i (K stage i) of pair tile w for CTA `rank`: the scale
// blocks of both 128-row chunks of the tile's B (completing rank 0's scale
// barrier at sf_bar) and this CTA's 128 rows of B (rank 0's operand barrier
// at full_bar).
template <class Cfg, class P>
__device__ __forceinline__ void load_b_stage(const P &p, const PairUnit &w, const GemmProblemDev &pr, uint32_t rank,
                                             int i, uint8_t *st, uint32_t full_bar, uint32_t sf_bar, uint64_t pol)
{
    const int blk0 = i * Cfg::SF_BLK;
#pragma unroll
    for (int j = 0; j < 2; ++j)
        tma_load_2d_pair(st + Cfg::A_BYTES + Cfg::B_BYTES + Cfg::SFA_BYTES + j * Cfg::SF_BLK * 512, p.map_sfb(w.g), 0,
                         (w.n_tile * 2 + j) * pr.sf_cblocks + blk0, sf_bar, pol);
    tma_load_2d_pair(st + Cfg::A_BYTES, p.map_b(w.g), i * 128, w.n_tile * 256 + static_cast<int>(rank) * 128, full_bar,
                     pol);
}

// EPI: the variant with the alpha / beta / bias epilogue (mxfp4_gemm_a4w4_ex).
// P: PairParams<MAXG> (problems in kernel parameters) or PairParamsTable.
template <int KIND, int STAGES, class P, bool F16, bool EPI = false>
__global__ void __launch_bounds__(kPairThreads, 1) bs_gemm_pair_kernel(const __grid_constant__ P p)
{
    using Cfg = PairCfg<KIND, STAGES>;
    constexpr bool MX = Cfg::MX;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * Cfg::STAGE_BYTES);   // rank 0: both CTAs' A/B tiles landed
    uint64_t *sf_data = full + STAGES;      // rank 0: both CTAs' scale blocks landed
    uint64_t *empty = sf_data + STAGES;     // the pair's MMAs are done with the stage
    uint64_t *sf_full = empty + STAGES;     // rank 0: the stage's scales are in both TMEMs
    uint64_t *accf = sf_full + STAGES;      // the tile's accumulator is complete
    uint64_t *acc_empty = accf + 1;         // rank 0: both CTAs' epilogues drained it
    uint64_t *cp_done = acc_empty + 1;      // [2] rank 0: every scale copy of warp 2 / 3 completed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(cp_done + 2);
    volatile int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    volatile int *epi_go = abort_flag + 1;  // [2] per-tile decision of the epilogue warps
    volatile int *issued_slot = epi_go + 2; // stages this CTA's producer issued (read by rank 0 at exit)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = static_cast<int>(blockIdx.x >> 1);
    const int npairs = static_cast<int>(gridDim.x >> 1);
    const int units = p.total_tiles;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(sf_data + s, 1);
            mbar_init(empty + s, 1);
            mbar_init(sf_full + s, 2);   // one commit from each scale-copy thread
        }
        mbar_init(accf, 1);
        mbar_init(acc_empty, 2 * kPairEpiWarps);   // one arrival per epilogue warp of each CTA
        mbar_init(cp_done, 1);
        mbar_init(cp_done + 1, 1);
        *abort_flag = 0;
        fence_mbar_init();
        // a device table's maps are fetched when first used, below
        for (int g = 0; g < (P::kTable ? 0 : p.num_groups); ++g) {
            tma_prefetch_desc(p.map_a(g));
            tma_prefetch_desc(p.map_b(g));
            tma_prefetch_desc(p.map_sfa(g));
            tma_prefetch_desc(p.map_sfb(g));
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    // both CTAs' barriers exist before any arrival from the other CTA
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    // Weights (B and its scales) are read-only inputs that no kernel of this
    // library writes, so each CTA requests its half of the first pair tile's
    // first ring of weight stages before the grid-dependency wait (rank 0
    // arms those stages for all of their bytes); A and its scales follow once
    // the preceding grid has completed. Problems in a device table are read
    // only after the wait.
    int pre = 0;   // stages of the first pair tile whose weights are requested (thread 0)
    const uint64_t pol = policy_evict_last();
    if constexpr (!P::kTable) {
        if (threadIdx.x == 0 && pair < units) {
            const PairUnit w = decode_pair_unit(p, pair);
            const GemmProblemDev &pr = p.problem(w.g);
            pre = min(STAGES, (pr.k + 255) / 256);
            const uint32_t full_r0 = mapa_shared(smem_u32(full), 0);
            const uint32_t sf_r0 = mapa_shared(smem_u32(sf_data), 0);
            for (int i = 0; i < pre; ++i) {
                uint8_t *st = smem + i * Cfg::STAGE_BYTES;
                if (leader) {
                    mbar_arrive_expect_tx(sf_data + i, 2 * (Cfg::SFA_BYTES + Cfg::SFB_BYTES));
                    mbar_arrive_expect_tx(full + i, 2 * (Cfg::A_BYTES + Cfg::B_BYTES));
                }
                load_b_stage<Cfg>(p, w, pr, rank, i, st, full_r0 + i * 8, sf_r0 + i * 8, pol);
            }
        }
    }
    // every other global access waits for the preceding grid in the stream
    grid_dependency_wait();
    grid_launch_dependents();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_acc = tmem;
    const uint32_t tmem_sf = tmem + 256;
    int issued = 0;   // stages armed by the producer (warp 0 lane 0 only)

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------ TMA producer
            // Rank 0 arms its barriers with both CTAs' bytes of the stage; the
            // copies of both CTAs complete them. A rank-1 copy can land before
            // rank 0 armed the phase (the transaction count goes negative
            // meanwhile), never in an earlier phase: rank 1 refills a slot only
            // after the MMAs that needed rank 0's previous phase of it.
            // Boxes past the last row or scale block read zeros and still count
            // their full size.
            const uint32_t full_r0 = mapa_shared(smem_u32(full), 0);
            const uint32_t sf_r0 = mapa_shared(smem_u32(sf_data), 0);
            int gs = 0, g_seen = -1;
            // the first pair tile always runs: its stages below `pre` have
            // weights in flight on armed barriers, which complete only once A
            // follows
            for (int u = pair; u < units && (u == pair || !*abort_flag); u += npairs) {
                const PairUnit w = decode_pair_unit(p, u);
                const GemmProblemDev &pr = p.problem(w.g);
                if (P::kTable && w.g != g_seen) {
                    tma_desc_acquire(p.map_a(w.g));
                    tma_desc_acquire(p.map_b(w.g));
                    tma_desc_acquire(p.map_sfa(w.g));
                    tma_desc_acquire(p.map_sfb(w.g));
                    g_seen = w.g;
                }
                const int a_chunk = w.m_pair * 2 + static_cast<int>(rank);   // this CTA's 128 rows of A
                const int k_stages = (pr.k + 255) / 256;
                for (int i = 0; i < k_stages; ++i, ++gs) {
                    const int slot = gs % STAGES;
                    if (gs >= STAGES && !mbar_wait(empty + slot, ((gs / STAGES) - 1) & 1, &g_gemm_pair_error,
                                                   kErrWaitEmpty, p.wait_ns)) {
                        *abort_flag = 1;
                        break;
                    }
                    uint8_t *st = smem + slot * Cfg::STAGE_BYTES;
                    const int blk0 = i * Cfg::SF_BLK;
                    // a stage below `pre` has its barriers armed and its weights
                    // requested already (only in the first pair tile, where gs = i)
                    const bool weights_sent = gs < pre;
                    if (leader && !weights_sent) {
                        mbar_arrive_expect_tx(sf_data + slot, 2 * (Cfg::SFA_BYTES + Cfg::SFB_BYTES));
                        mbar_arrive_expect_tx(full + slot, 2 * (Cfg::A_BYTES + Cfg::B_BYTES));
                    }
                    // the scale blocks first, on their own barrier
                    tma_load_2d_pair(st + Cfg::A_BYTES + Cfg::B_BYTES, p.map_sfa(w.g), 0, a_chunk * pr.sf_cblocks + blk0,
                                     sf_r0 + slot * 8, pol);
                    if (!weights_sent) load_b_stage<Cfg>(p, w, pr, rank, i, st, full_r0 + slot * 8, sf_r0 + slot * 8, pol);
                    tma_load_2d_pair(st, p.map_a(w.g), i * 128, a_chunk * 128, full_r0 + slot * 8, pol);
                    issued = gs + 1;
                }
            }
        }
    } else if (warp == 1) {
        if (leader && lane == 0) {
            // --------------------------------------------- MMA issuer (rank 0)
            constexpr uint32_t IDESC = idesc_block_scaled(256, MX, 256);
            int gs = 0, ul = 0, commits = 0;
            for (int u = pair; u < units; u += npairs, ++ul) {
                const PairUnit w = decode_pair_unit(p, u);
                const GemmProblemDev &pr = p.problem(w.g);
                const int k_stages = (pr.k + 255) / 256;
                const int k_steps_total = (pr.k + 63) / 64;
                // the epilogues' arrivals are relaxed: they publish no data, only
                // that their TMEM loads of the accumulator have completed
                if (ul > 0 && !mbar_wait(acc_empty, (ul - 1) & 1, &g_gemm_pair_error, kErrWaitAccum, p.wait_ns)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                bool ok = true;
                for (int i = 0; i < k_stages; ++i, ++gs) {
                    const int slot = gs % STAGES;
                    const uint32_t ph = (gs / STAGES) & 1;
                    // one wait per stage: the scale-copy threads commit sf_full only
                    // after they also saw the stage's operand tiles land
                    if (!mbar_wait(sf_full + slot, ph, &g_gemm_pair_error, kErrWaitFull, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint8_t *st = smem + slot * Cfg::STAGE_BYTES;
                    const uint32_t a_base = smem_u32(st);
                    const uint32_t b_base = smem_u32(st + Cfg::A_BYTES);
                    const uint32_t tsfa = tmem_sf + slot * Cfg::SF_COLS;
                    const uint32_t tsfb = tsfa + Cfg::SF_COLS_A;
                    // K step kk of the stage starts 32 bytes (2 descriptor units) further
                    const uint64_t ad = sdesc_sw128(a_base);
                    const uint64_t bd = sdesc_sw128(b_base);
                    const int ksteps = min(4, k_steps_total - i * 4);
                    auto mma_step = [&](int kk) {
                        const int blk = MX ? kk / 2 : kk;
                        const uint32_t sfid = MX ? static_cast<uint32_t>(kk & 1) * 2u : 0u;
                        const uint32_t idesc = idesc_with_sf_ids(IDESC, sfid, sfid);
                        const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                        if constexpr (MX)
                            mma_mxf4_pair(tmem_acc, ad + 2 * kk, bd + 2 * kk, idesc, tsfa + blk * 4, tsfb + blk * 8, acc);
                        else
                            mma_nvf4_pair(tmem_acc, ad + 2 * kk, bd + 2 * kk, idesc, tsfa + blk * 4, tsfb + blk * 8, acc);
                    };
                    // the issuing thread is the bottleneck: full stages go unrolled
                    if (ksteps == 4) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) mma_step(kk);
                    } else {
                        for (int kk = 0; kk < ksteps; ++kk) mma_step(kk);
                    }
                    tc_commit_pair_mc(empty + slot, 0x3);   // both CTAs may refill the stage
                }
                // arrives in both CTAs once every MMA issued above has completed
                tc_commit_pair_mc(accf, 0x3);
                ++commits;
                if (!ok) {
                    *abort_flag = 1;
                    break;
                }
            }
            // the accumulators must not be in use when the pair frees TMEM
            if (commits > 0) mbar_wait(accf, (commits - 1) & 1, &g_gemm_pair_error, kErrWaitDrain);
        }
    } else if (warp == 2 || warp == 3) {
        if (lane == 0 && leader) {
            // ------------------------- scale staging for both CTAs (rank 0)
            // Lane 0 of warps 2 and 3 share the copies of each stage (even / odd
            // K blocks). A stage's TMEM scale slot is rewritten only after both
            // CTAs refilled the stage's smem, which needed the MMAs' "empty"
            // commit. Scale blocks past the problem (a second CTA without rows,
            // a B half past N, K blocks past K) arrive as zeros and feed only
            // accumulator rows and columns that are never stored.
            int gs = 0;
            bool stop = false;
            for (int u = pair; u < units && !stop && !*abort_flag; u += npairs) {
                const PairUnit w = decode_pair_unit(p, u);
                const GemmProblemDev &pr = p.problem(w.g);
                const int k_stages = (pr.k + 255) / 256;
                const int k_steps_total = (pr.k + 63) / 64;
                for (int i = 0; i < k_stages; ++i, ++gs) {
                    const int slot = gs % STAGES;
                    const uint32_t ph = (gs / STAGES) & 1;
                    if (!mbar_wait(sf_data + slot, ph, &g_gemm_pair_error, kErrWaitFull, p.wait_ns)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    uint8_t *st = smem + slot * Cfg::STAGE_BYTES;
                    const uint32_t sfa_s = smem_u32(st + Cfg::A_BYTES + Cfg::B_BYTES);
                    const uint32_t sfb_s = sfa_s + Cfg::SFA_BYTES;
                    const uint32_t tsfa = tmem_sf + slot * Cfg::SF_COLS;
                    const uint32_t tsfb = tsfa + Cfg::SF_COLS_A;
                    const int ksteps = min(4, k_steps_total - i * 4);
                    const int nblk = MX ? (ksteps + 1) / 2 : ksteps;
                    for (int b = warp - 2; b < nblk; b += 2) {
                        tc_cp_scale_block_pair(tsfa + b * 4, sdesc_scale(sfa_s + b * 512));
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            tc_cp_scale_block_pair(tsfb + (b * 2 + j) * 4, sdesc_scale(sfb_s + (j * Cfg::SF_BLK + b) * 512));
                    }
                    // the MMA issuer waits only for sf_full: it also stands for the
                    // stage's operand tiles
                    if (!mbar_wait(full + slot, ph, &g_gemm_pair_error, kErrWaitFull, p.wait_ns)) {
                        stop = true;
                        break;
                    }
                    tc_commit_pair(sf_full + slot);
                }
            }
            if (stop) *abort_flag = 1;
            // every scale copy this thread issued (also those of a stage given up
            // above) completes before the pair frees TMEM
            tc_commit_pair(cp_done + (warp - 2));
            mbar_wait(cp_done + (warp - 2), 0, &g_gemm_pair_error, kErrWaitDrain);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        // Eight warps: warp 4 + e reads TMEM lane quadrant e % 4 (the 32 rows
        // it may access) and columns [128 h, 128 h + 128), h = e / 4. Its two
        // pairs of 32-column loads are each in flight together, then the warp
        // hands TMEM back (a relaxed arrive on rank 0's barrier: the MMA
        // issuer only needs to know that the loads have completed) and stores.
        const int e = warp - 4;
        const int q = warp & 3;                  // TMEM lane quadrant of this warp
        const int h = e >> 2;                    // column half
        const int row_in_tile = q * 32 + lane;
        const uint32_t t_row = tmem_acc + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * 128);
        const uint32_t acc_empty_r0 = mapa_shared(smem_u32(acc_empty), 0);
        int ul = 0;
        for (int u = pair; u < units; u += npairs, ++ul) {
            const PairUnit w = decode_pair_unit(p, u);
            const GemmProblemDev &pr = p.problem(w.g);
            // one thread waits and decides for the eight warps, so that they
            // leave the loop together
            if (threadIdx.x == 128) {
                const bool ok = mbar_wait(accf, ul & 1, &g_gemm_pair_error, kErrWaitAccum, p.wait_ns);
                if (!ok) *abort_flag = 1;
                epi_go[ul & 1] = ok;
            }
            epilogue_bar();
            if (!epi_go[ul & 1]) break;
            tc_fence_after();
            const bool run = (*abort_flag == 0);
            const int row = w.m_pair * 256 + static_cast<int>(rank) * 128 + row_in_tile;
            const int col_base = w.n_tile * 256 + h * 128;
            if (EPI && pr.epi) {
                // epilogue with alpha / beta / bias: each 32-column chunk is
                // finished and stored straight from TMEM, then TMEM goes back
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    tmem_ld32(t_row + c * 32, v);
                    tmem_ld_wait();
                    const int col0 = col_base + c * 32;
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
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_r0);
                continue;
            }
            // drain this warp's 128 columns into registers (two loads in flight
            // at a time), hand TMEM back, then store
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 4; c += 2) {
                uint32_t v0[32], v1[32];
                tmem_ld32(t_row + c * 32, v0);
                tmem_ld32(t_row + (c + 1) * 32, v1);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    pk[c * 16 + j] = pack2<F16>(__uint_as_float(v0[2 * j]), __uint_as_float(v0[2 * j + 1]));
                    pk[(c + 1) * 16 + j] = pack2<F16>(__uint_as_float(v1[2 * j]), __uint_as_float(v1[2 * j + 1]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_r0);
            if (run && row < pr.m) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int col0 = col_base + c * 32;
                    if (col0 < pr.n) {
                        uint32_t part[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) part[j] = pk[c * 16 + j];
                        store_packed32(pr.c, pr.ldc, row, col0, pr.n, part);
                    }
                }
            }
        }
    }
    __syncwarp();

    // ----------------------------------------------------------- teardown
    // Copies still in flight (only after an abort) must land before either CTA
    // leaves. Rank 0's barriers count both CTAs' copies, and after an abort the
    // two producers may have issued different numbers of stages: rank 0 reads
    // rank 1's count, settles the share of each stage that only one CTA issued
    // (arms the phase with rank 1's bytes, or cancels rank 1's missing bytes),
    // then waits for every stage that can still be in flight.
    tc_fence_before();
    if (warp == 0 && lane == 0) *issued_slot = issued;
    cluster_sync();
    if (warp == 0 && lane == 0 && leader) {
        const int i0 = issued;
        const int i1 = static_cast<int>(ld_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int *>(issued_slot)), 1)));
        const int hi = max(i0, i1);
        constexpr uint32_t kSfOne = Cfg::SFA_BYTES + Cfg::SFB_BYTES;   // one CTA's bytes of a stage
        constexpr uint32_t kOpOne = Cfg::A_BYTES + Cfg::B_BYTES;
        for (int i = min(i0, i1); i < hi; ++i) {
            const int slot = i % STAGES;
            if (i >= i0) {
                mbar_arrive_expect_tx(sf_data + slot, kSfOne);
                mbar_arrive_expect_tx(full + slot, kOpOne);
            } else {
                mbar_complete_tx(sf_data + slot, kSfOne);
                mbar_complete_tx(full + slot, kOpOne);
            }
        }
        for (int i = max(0, hi - STAGES); i < hi; ++i) {
            mbar_wait(sf_data + (i % STAGES), (i / STAGES) & 1, &g_gemm_pair_error, kErrWaitDrain);
            mbar_wait(full + (i % STAGES), (i / STAGES) & 1, &g_gemm_pair_error, kErrWaitDrain);
        }
    }
    // neither CTA leaves while the other may still arrive on its barriers or
    // use its shared memory and TMEM
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, Cfg::TMEM_COLS);
    }
}

template <int KIND, int STAGES, class P, bool F16, bool EPI = false>
cudaError_t launch_pair(const P &params, cudaStream_t stream)
{
    using Cfg = PairCfg<KIND, STAGES>;
    auto kern = bs_gemm_pair_kernel<KIND, STAGES, P, F16, EPI>;
    static KernelOnce once;
    int sms = 0;
    const cudaError_t e = prepare_kernel(kern, Cfg::SMEM_BYTES, once, &sms);
    if (e != cudaSuccess) return e;
    const int pairs = min(params.total_tiles, max(1, sms / 2));
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(kPairThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    P launch_params = params;
    launch_params.wait_ns = wait_limit_ns();
    return cudaLaunchKernelEx(&cfg, kern, launch_params);
}

constexpr int kPairMxStages = 6;   // 35 KB stages
constexpr int kPairNvStages = 5;   // 38 KB stages; TMEM holds 5 stages of NVFP4 scales
static_assert(PairCfg<0, kPairMxStages>::SF_BLK == pair_sf_box_blocks(false) &&
                  PairCfg<1, kPairNvStages>::SF_BLK == pair_sf_box_blocks(true),
              "scale tensor-map boxes are one stage of scale blocks");

// Pair tiles: 256 rows of A (two CTAs) x 256 columns.
template <int MAXG>
void fill_pair_problem(PairParams<MAXG> &P, int g, const GemmProblemHost &h, int vec, int &tiles)
{
    P.tma[g] = h.tma;
    P.tmb[g] = h.tmb;
    P.tmsfa[g] = h.tmsfa;
    P.tmsfb[g] = h.tmsfb;
    GemmProblemDev &d = P.prob[g];
    d.sfa = h.sfa;
    d.sfb = h.sfb;
    d.c = h.c;
    d.ldc = h.ldc;
    d.m = h.m;
    d.n = h.n;
    d.k = h.k;
    d.m_tiles = (h.m + 255) / 256;
    d.n_tiles = (h.n + 255) / 256;
    d.tile_start = tiles;
    d.sf_cblocks = (h.k / vec + 3) / 4;
    d.epi = h.epi ? 1 : 0;
    d.alpha = h.alpha;
    d.beta = h.beta;
    d.bias = static_cast<const uint16_t *>(h.bias);
    tiles += d.m_tiles * d.n_tiles;
}

}  // namespace

int pair_tiles(int64_t m, int64_t n) { return static_cast<int>(((m + 255) / 256) * ((n + 255) / 256)); }

cudaError_t launch_gemm_mx_pair(const GemmProblemHost &prob, cudaStream_t stream)
{
    PairParams<1> P;
    memset(&P, 0, sizeof(P));
    int tiles = 0;
    fill_pair_problem(P, 0, prob, 32, tiles);
    P.num_groups = 1;
    P.total_tiles = tiles;
    if (prob.epi) return launch_pair<0, kPairMxStages, PairParams<1>, false, true>(P, stream);
    return launch_pair<0, kPairMxStages, PairParams<1>, false>(P, stream);
}

// The grouped launch: problems in kernel parameters up to kMaxGroups, else in
// the device table (filled here, on the stream, before the launch).
template <int KIND, int STAGES, bool F16>
cudaError_t launch_grouped_pair(const GemmProblemHost *probs, int num_groups, void *table, int vec,
                                cudaStream_t stream)
{
    if (num_groups <= kMaxGroups) {
        PairParams<kMaxGroups> P;
        memset(&P, 0, sizeof(P));
        int tiles = 0;
        for (int g = 0; g < num_groups; ++g) fill_pair_problem(P, g, probs[g], vec, tiles);
        P.num_groups = num_groups;
        P.total_tiles = tiles;
        return launch_pair<KIND, STAGES, PairParams<kMaxGroups>, F16>(P, stream);
    }
    if (!table || (reinterpret_cast<uintptr_t>(table) & 63u) != 0) return cudaErrorInvalidValue;
    std::vector<uint8_t> host(group_table_bytes(num_groups), 0);
    CUtensorMap *maps = reinterpret_cast<CUtensorMap *>(host.data());
    uint8_t *recs = host.data() + static_cast<size_t>(num_groups) * kTableMaps * sizeof(CUtensorMap);
    PairParams<1> one;
    int tiles = 0;
    for (int g = 0; g < num_groups; ++g) {
        memset(&one, 0, sizeof(one));
        int t = tiles;
        fill_pair_problem(one, 0, probs[g], vec, t);
        one.prob[0].tile_start = tiles;
        tiles = t;
        maps[g * kTableMaps + 0] = probs[g].tma;
        maps[g * kTableMaps + 1] = probs[g].tmb;
        maps[g * kTableMaps + 2] = probs[g].tmsfa;
        maps[g * kTableMaps + 3] = probs[g].tmsfb;
        memcpy(recs + static_cast<size_t>(g) * kTableProblemBytes, &one.prob[0], sizeof(GemmProblemDev));
    }
    cudaError_t e = upload_table(table, host.data(), host.size(), stream);
    if (e != cudaSuccess) return e;
    PairParamsTable T;
    memset(&T, 0, sizeof(T));
    T.maps = static_cast<const CUtensorMap *>(table);
    T.probs = static_cast<const uint8_t *>(table) + static_cast<size_t>(num_groups) * kTableMaps * sizeof(CUtensorMap);
    T.num_groups = num_groups;
    T.total_tiles = tiles;
    return launch_pair<KIND, STAGES, PairParamsTable, F16>(T, stream);
}

cudaError_t launch_gemm_nv_grouped_pair(const GemmProblemHost *probs, int num_groups, void *table,
                                        cudaStream_t stream)
{
    return launch_grouped_pair<1, kPairNvStages, true>(probs, num_groups, table, 16, stream);
}

cudaError_t launch_gemm_mx_grouped_pair(const GemmProblemHost *probs, int num_groups, void *table,
                                        cudaStream_t stream)
{
    return launch_grouped_pair<0, kPairMxStages, false>(probs, num_groups, table, 32, stream);
}

int read_and_clear_gemm_pair_error()
{
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_pair_error, sizeof(int)) != cudaSuccess) return -1;
    cudaMemcpyToSymbol(g_gemm_pair_error, &zero, sizeof(int));
    return v;
}

}  // namespace mxfp4
