// Fused dynamic MXFP4 quantization + block-scaled GEMM for small M
// (kernelbot-amd-mxfp4-mm-517169, "Optimization 5": the A tile is quantized on
// chip and fed straight to the matrix unit, so the quantized A never reaches
// global memory; the same page's docstring counts the round trip this saves).
//
// Design for a weight-streaming (HBM-bound) shape such as M = 16, N = 2112,
// K = 7168:
// * Swap A and B: the weight rows fill the MMA's M = 128, the few activation
//   rows (padded with zeros to MMA_N = 16/32/64) are the MMA's N. The
//   accumulator is D[n][m] = C^T, 128 TMEM lanes x MMA_N columns.
// * Grid = (ceil(N/128) weight tiles) x (S K-splits); the S CTAs of one weight
//   tile form a thread-block cluster. Each CTA streams its K-slice of 128
//   weight rows through a 4-slot TMA ring (evict-first: weights are read once);
//   the first four stages are requested before the grid-dependency wait.
// * Eight warps in four groups of 64 threads: group s owns ring slot s and
//   the CTA's K-stages s, s + 4, ... For each of its stages the group's
//   threads read the stage's bf16 A straight from global memory, two 32-element
//   blocks per thread at MMA_N = 16 (so that quantizing a stage takes one short
//   pass rather than a long serial loop in one warp), form the OCP MX scale and
//   E2M1 codes with the same arithmetic as the standalone quant kernel, and
//   write them into shared memory in the MMA's 128-byte-swizzled K-major
//   operand layout, the scales in the 512-byte blocked layout. After a named
//   barrier of the group its first thread copies both operands' scales to
//   TMEM and issues the stage's MMAs into the group's own TMEM accumulator
//   (issuing a tcgen05 instruction costs on the order of 100 cycles while an
//   N = 16 MMA is only a few cycles of tensor work, so the four groups issue in
//   parallel), then refills its ring slot with its next stage's weights.
// * Split-K reduction without global scratch: every CTA sums the four group
//   accumulators and pushes the slice of the fp32 tile that CTA r of the
//   cluster owns (weight rows r*128/S ..) into r's shared memory with remote
//   stores; after one cluster barrier each CTA sums its slice over the S
//   sources in rank order and writes C. The sum order is fixed, so results are
//   deterministic.
// Shared memory stays near 100 KB (MMA_N = 16) so two CTAs fit on an SM and
// every cluster of the grid can be resident at once.
#include <algorithm>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mxfp4 {

__device__ int g_fused_error;

namespace {

constexpr int kRing = 4;
constexpr uint32_t kWBytes = 128 * 128;   // one stage of 128 weight rows x 256 FP4
// NV selects NVFP4 (E4M3 scale per 16, kind::mxf4nvf4, fp16 C); otherwise
// MXFP4 (E8M0 per 32, kind::mxf4, bf16 C).
template <bool NV>
constexpr int kSfBlk = NV ? 4 : 2;         // 512-byte scale blocks per 128 rows per stage
// 256 threads: measured on the 16 x 2112 x 7168 call against 128 and 512
// (6.07 and 6.33 us per call against 5.78)
constexpr int kThreads = 256;
constexpr int kGroups = 4;                // warp groups; group s owns ring slot s
constexpr int kGroupThreads = kThreads / kGroups;
constexpr int kEpiParts = kThreads / 128;  // warps per TMEM lane quadrant in the epilogue
constexpr int kMaxSplits = 8;             // portable cluster size
static_assert(kGroups == kRing, "a group refills its own ring slot");

__host__ __device__ constexpr uint32_t pow2_cols_f(uint32_t n)
{
    return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 512;
}

template <int MMA_N, bool NV = false>
struct FusedCfg {
    static constexpr int SF_BLK = kSfBlk<NV>;
    static constexpr uint32_t SF_STAGE = SF_BLK * 512;     // one operand's scale bytes per stage
    // K stages (256 wide) held per CTA: each has its own quantized operand tile
    // and its own TMEM scale columns (fewer with NVFP4's larger scale blocks,
    // so that two CTAs still share an SM).
    static constexpr int MAX_ST = MMA_N <= 16 ? (NV ? 6 : 8) : 4;
    static constexpr int UPT = MMA_N * 8 / kGroupThreads;   // 32-element blocks per thread per stage
    static constexpr uint32_t ACT_TILE = MMA_N * 128;       // quantized operand bytes per stage
    static constexpr uint32_t RING_DATA = kRing * kWBytes;
    static constexpr uint32_t ACT_OFF = RING_DATA;
    static constexpr uint32_t WSF_OFF = ACT_OFF + MAX_ST * ACT_TILE;
    static constexpr uint32_t ASF_OFF = WSF_OFF + kRing * SF_STAGE;
    static constexpr uint32_t RECV_OFF = ASF_OFF + MAX_ST * SF_STAGE;
    // [source rank][m][owned rows] fp32; owned rows = ceil(128 / S) <= 128 / S + 1
    static constexpr uint32_t RECV_BYTES = MMA_N * (128 + kMaxSplits) * 4;
    static constexpr uint32_t BAR_OFF = RECV_OFF + RECV_BYTES;
    static constexpr uint32_t SMEM_BYTES = BAR_OFF + 256 + 1024;
    static constexpr uint32_t SF_COLS = 2 * SF_BLK * 4;      // per stage: weight + activation blocks
    static constexpr uint32_t ACC_COLS = kGroups * MMA_N;   // one accumulator per warp group
    static constexpr uint32_t TMEM_COLS = pow2_cols_f(ACC_COLS + MAX_ST * SF_COLS);
    static_assert(UPT >= 1 && UPT * kGroupThreads == MMA_N * 8, "quant work split");
    static_assert(ACT_TILE % 1024 == 0, "swizzled operand tiles need 1024-byte alignment");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(ACC_COLS + MAX_ST * SF_COLS <= 512, "TMEM budget");
    // full, empty per ring slot, accf; TMEM address, abort flag, every peer's abort flag
    static_assert((2 * kRing + 1) * 8 + 8 + kMaxSplits * 4 <= 256, "barrier area");
};

struct FusedArgs {
    const uint16_t *A;    // bf16 [M, K], row stride lda elements
    int64_t lda;
    const uint8_t *sfw;   // weight scales, blocked [N, K/32] (MXFP4) or [N, K/16] (NVFP4)
    uint16_t *C;          // bf16 (MXFP4) or fp16 (NVFP4) [M, N]
    int64_t ldc;
    int M, N, K;
    int splits;
    int sf_cblocks;
    uint64_t wait_ns;     // limit of the waits that guard work
};

// C element from fp32: bf16 (MXFP4) or fp16 (NVFP4), round to nearest even.
template <bool NV>
__device__ __forceinline__ uint16_t to_c(float f)
{
    if constexpr (NV)
        return __half_as_ushort(__float2half_rn(f));
    else
        return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ void group_bar(int grp)
{
    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(kGroupThreads) : "memory");
}

// Sum of the `nacc` group accumulators' columns [c0, c0 + W) of this warp's
// TMEM lane quadrant (row base t_row).
template <int W>
__device__ __forceinline__ void sum_accumulators(uint32_t t_row, int c0, int nacc, int stride, float (&f)[W])
{
#pragma unroll
    for (int j = 0; j < W; ++j) f[j] = 0.0f;
    for (int a = 0; a < nacc; ++a) {
        uint32_t v[W];
        const uint32_t addr = t_row + static_cast<uint32_t>(a * stride + c0);
        if constexpr (W == 4)
            tmem_ld4(addr, v);
        else if constexpr (W == 8)
            tmem_ld8(addr, v);
        else if constexpr (W == 16)
            tmem_ld16(addr, v);
        else
            tmem_ld32(addr, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < W; ++j) f[j] += __uint_as_float(v[j]);
    }
}

template <int MMA_N, bool NV>
__global__ void __launch_bounds__(kThreads, 2)
    fused_quant_gemm_kernel(const __grid_constant__ CUtensorMap tmw, const FusedArgs p)
{
    using Cfg = FusedCfg<MMA_N, NV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem;
    uint8_t *act = smem + Cfg::ACT_OFF;       // [stage][MMA_N rows x 128 B], 128B-swizzled
    uint8_t *ring_sf = smem + Cfg::WSF_OFF;   // [slot][SF_BLK x 512 B]
    uint8_t *act_sf = smem + Cfg::ASF_OFF;    // [stage][SF_BLK x 512 B]
    float *recv = reinterpret_cast<float *>(smem + Cfg::RECV_OFF);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::BAR_OFF);
    uint64_t *empty = full + kRing;
    uint64_t *accf = empty + kRing;              // one arrival per warp group
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accf + 1);
    volatile int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    volatile int *abort_in = abort_flag + 1;    // [kMaxSplits] the abort flag of each CTA of the cluster

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int grp = warp / (kGroupThreads / 32);
    const int gt = threadIdx.x % kGroupThreads;  // thread index within the group
    const bool leader = gt == 0;                 // issues the group's copies and tcgen05 instructions
    const int n_tile = blockIdx.x;
    const int split = blockIdx.y;
    const int k_stages = (p.K + 255) / 256;
    const int s_begin = k_stages * split / p.splits;
    const int s_end = k_stages * (split + 1) / p.splits;
    const int nst = s_end - s_begin;
    const int k_steps_total = (p.K + 63) / 64;

    const uint64_t pol_w = policy_evict_first();   // weights are read once
    auto issue_weights = [&](int i) {
        const int slot = i % kRing;
        const int ks = s_begin + i;
        const int blk0 = ks * Cfg::SF_BLK;
        const int nblk = min(Cfg::SF_BLK, p.sf_cblocks - blk0);
        mbar_arrive_expect_tx(full + slot, kWBytes + nblk * 512);
        tma_load_2d(ring + slot * kWBytes, &tmw, ks * 128, n_tile * 128, full + slot, pol_w);
        bulk_load(ring_sf + slot * Cfg::SF_STAGE, p.sfw + (static_cast<size_t>(n_tile) * p.sf_cblocks + blk0) * 512,
                  nblk * 512, full + slot, pol_w);
    };
    if (threadIdx.x == 0 && nst > 0) {
        // Warm L2 with this CTA's rows of A before the weight stream is
        // requested; the loads that use A still wait for that grid below.
        const int64_t k0 = static_cast<int64_t>(s_begin) * 256;
        const int64_t k1 = min(static_cast<int64_t>(s_end) * 256, static_cast<int64_t>(p.K));
        for (int m = 0; m < p.M; ++m)
            prefetch_l2_bulk(p.A + static_cast<int64_t>(m) * p.lda + k0, static_cast<uint32_t>((k1 - k0) * 2));
    }
    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < kRing; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(accf, kGroups);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmw);
        // Weights are read-only inputs that no kernel of this library writes,
        // so the first ring's worth of weight stages is requested before the
        // grid-dependency wait: under programmatic dependent launch the stream
        // of weights overlaps the tail of the preceding call.
        for (int i = 0; i < min(nst, kRing); ++i) issue_weights(i);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish();
    }

    // A, C and everything else in global memory is touched only after the
    // preceding grid in the stream has completed and its writes are visible.
    grid_dependency_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // --------------------- warp groups: quantize a K-stage of A, issue its MMAs
    // Group grp owns stages t = grp, grp + 4, ... and ring slot grp. Its
    // threads quantize the stage's MMA_N x 8 blocks of 32 elements (thread gt
    // takes blocks gt + 128 x), writing codes in the MMA's 128-byte-swizzled
    // K-major layout and scales in the blocked layout. Rows >= M and blocks
    // past K are zero and quantize to code 0 with scale byte 0.
    const int slot = grp;
    const uint32_t acc_tmem = tmem + static_cast<uint32_t>(grp * MMA_N);
    constexpr uint32_t IDESC = idesc_block_scaled(MMA_N, !NV);
    int last_issued = grp < min(nst, kRing) ? grp : -1;   // latest stage requested into this slot
    bool first = true;
    for (int t = grp; t < nst; t += kGroups) {
        const int ks = s_begin + t;
        if (t >= kRing && leader) {
            // the slot's previous stage has been consumed once its MMAs are done
            if (!mbar_wait(empty + slot, ((t / kRing) - 1) & 1, &g_fused_error, kErrWaitEmpty, p.wait_ns)) {
                *abort_flag = 1;
            } else {
                issue_weights(t);
                last_issued = t;
            }
        }
        uint8_t *dst = act + t * Cfg::ACT_TILE;
        uint8_t *dsf = act_sf + t * Cfg::SF_STAGE;
        constexpr int BATCH = Cfg::UPT < 2 ? Cfg::UPT : 2;   // blocks whose loads are in flight together
#pragma unroll 1
        for (int x0 = 0; x0 < Cfg::UPT; x0 += BATCH) {
            uint4 v[BATCH][4];
#pragma unroll
            for (int x = 0; x < BATCH; ++x) {
                const int u = gt + kGroupThreads * (x0 + x);
                const int m = u >> 3, j = u & 7;
                const int k0 = ks * 256 + j * 32;
                const bool ok = m < p.M && k0 < p.K;
                const uint16_t *src = p.A + static_cast<int64_t>(m) * p.lda + k0;
#pragma unroll
                for (int q = 0; q < 4; ++q) v[x][q] = ok ? ld_nc_v4(src + q * 8) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int x = 0; x < BATCH; ++x) {
                const int u = gt + kGroupThreads * (x0 + x);
                const int m = u >> 3, j = u & 7;
                uint4 codes;
                if constexpr (NV) {
                    // two 16-element groups, each with s = E4M3(fp32(amax) / 6)
                    // and codes of x / s, as the standalone NVFP4 quantizer
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t sbyte = nv_scale_byte(block_amax_bits<2>(&v[x][2 * h]));
                        const float rs = nv_recip(sbyte);
                        const uint32_t lo = nv_codes8(v[x][2 * h], rs), hi = nv_codes8(v[x][2 * h + 1], rs);
                        if (h == 0) {
                            codes.x = lo;
                            codes.y = hi;
                        } else {
                            codes.z = lo;
                            codes.w = hi;
                        }
                        const int c = 2 * j + h;   // scale column within the stage (16 per stage)
                        dsf[(c >> 2) * 512 + (m & 31) * 16 + (m >> 5) * 4 + (c & 3)] = static_cast<uint8_t>(sbyte);
                    }
                } else {
                    const uint32_t sbyte = e8m0_byte_from_amax(block_amax_bits<4>(v[x]));
                    codes.x = mx_codes8(v[x][0], sbyte);
                    codes.y = mx_codes8(v[x][1], sbyte);
                    codes.z = mx_codes8(v[x][2], sbyte);
                    codes.w = mx_codes8(v[x][3], sbyte);
                    dsf[(j >> 2) * 512 + (m & 31) * 16 + (m >> 5) * 4 + (j & 3)] = static_cast<uint8_t>(sbyte);
                }
                *reinterpret_cast<uint4 *>(dst + m * 128 + ((j ^ (m & 7)) << 4)) = codes;
            }
        }
        fence_proxy_async_smem();   // generic-proxy writes -> visible to tcgen05
        group_bar(grp);             // the stage's operand and scales are complete
        if (leader) {
            if (!mbar_wait(full + slot, (t / kRing) & 1, &g_fused_error, kErrWaitFull, p.wait_ns)) {
                *abort_flag = 1;
            } else {
                tc_fence_after();
                const uint32_t w_base = smem_u32(ring + slot * kWBytes);
                const uint32_t a_base = smem_u32(dst);
                const uint32_t wsf = smem_u32(ring_sf + slot * Cfg::SF_STAGE);
                const uint32_t asf = smem_u32(dsf);
                const uint32_t tsfw = tmem + Cfg::ACC_COLS + t * Cfg::SF_COLS;
                const uint32_t tsfa = tsfw + Cfg::SF_BLK * 4;
                const int ksteps = min(4, k_steps_total - ks * 4);
                const int nblk = NV ? ksteps : (ksteps + 1) / 2;
                for (int b = 0; b < nblk; ++b) {
                    tc_cp_scale_block(tsfw + b * 4, sdesc_scale(wsf + b * 512));
                    tc_cp_scale_block(tsfa + b * 4, sdesc_scale(asf + b * 512));
                }
                for (int kk = 0; kk < ksteps; ++kk) {
                    const uint32_t sfid = NV ? 0u : static_cast<uint32_t>(kk & 1) * 2u;
                    const int blk = NV ? kk : kk >> 1;
                    const uint32_t idesc = idesc_with_sf_ids(IDESC, sfid, sfid);
                    const uint32_t acc = (first && kk == 0) ? 0u : 1u;
                    if constexpr (NV)
                        mma_nvf4(acc_tmem, sdesc_sw128(w_base + kk * 32), sdesc_sw128(a_base + kk * 32), idesc,
                                 tsfw + blk * 4, tsfa + blk * 4, acc);
                    else
                        mma_mxf4(acc_tmem, sdesc_sw128(w_base + kk * 32), sdesc_sw128(a_base + kk * 32), idesc,
                                 tsfw + blk * 4, tsfa + blk * 4, acc);
                }
                tc_commit(empty + slot);
            }
        }
        first = false;
    }
    // The next grid in the stream may start once this grid's MMAs are issued
    // (every A load of this grid has returned): its CTAs take ~2 us to enter,
    // so their weight stream then overlaps this grid's accumulation, reduction
    // and exit instead of competing with this grid's loads of A. Measured per
    // call at 16 x 2112 x 7168: 6.65 us with the release right after the
    // dependency wait, 5.78 once the accumulators were complete, 5.74 here
    // (NVFP4: 6.43 -> 6.25).
    grid_launch_dependents();
    // one arrival per group once its MMAs are done (at once if it had none)
    if (leader) {
        if (first)
            mbar_arrive(accf);
        else
            tc_commit(accf);
    }

    // -------------------------------------------------------------- epilogue
    // Warp w reads TMEM lane quadrant w % 4 and columns [CPW (w / 4), + CPW)
    // of every group accumulator, sums them and pushes (or stores) its part.
    const int S = p.splits;
    const int nper = (128 + S - 1) / S;           // weight rows each CTA of the cluster owns
    const int nacc = min(nst, kGroups);           // accumulators that hold data
    constexpr int CPW = MMA_N / kEpiParts;        // accumulator columns per warp
    {
        // a group that gave up set the abort flag before its arrival on accf
        int acc_ok = 1;
        if (lane == 0) acc_ok = mbar_wait(accf, 0, &g_fused_error, kErrWaitAccum, p.wait_ns) && *abort_flag == 0;
        acc_ok = __shfl_sync(0xffffffffu, acc_ok, 0);
        tc_fence_after();
        const int q = warp & 3;                      // TMEM lane quadrant of this warp
        const int c0 = (warp >> 2) * CPW;
        const int n_local = q * 32 + lane;
        const int n = n_tile * 128 + n_local;
        const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
        float f[CPW];
        sum_accumulators<CPW>(t_row, c0, nacc, MMA_N, f);
        if (acc_ok) {
            if (S == 1) {
#pragma unroll
                for (int j = 0; j < CPW; ++j) {
                    const int m = c0 + j;
                    if (m < p.M && n < p.N) p.C[static_cast<int64_t>(m) * p.ldc + n] = to_c<NV>(f[j]);
                }
            } else {
                const int owner = n_local / nper;
                const uint32_t dst_base = mapa_shared(
                    smem_u32(recv) + static_cast<uint32_t>(split * MMA_N * nper + (n_local - owner * nper)) * 4,
                    static_cast<uint32_t>(owner));
#pragma unroll
                for (int j = 0; j < CPW; ++j)
                    if (c0 + j < p.M) st_shared_cluster_f32(dst_base + (c0 + j) * nper * 4, f[j]);
            }
        } else {
            *abort_flag = 1;
        }
    }

    if (S > 1) {
        // Every CTA tells every CTA of the cluster whether it gave up: an owner
        // whose slice misses a partial sum leaves C unwritten (the call then
        // reports the device error). Every CTA reaches the barrier, also after
        // an abort.
        __syncthreads();
        if (threadIdx.x < S)
            st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int *>(abort_in + split)), threadIdx.x),
                                  static_cast<uint32_t>(*abort_flag));
        cluster_sync();
        int any_abort = 0;
        for (int r = 0; r < S; ++r) any_abort |= abort_in[r];
        const int n_lo = split * nper;
        const int width = min(128, n_lo + nper) - n_lo;
        if (width > 0 && !any_abort) {
            const int cnt = width * p.M;
            for (int idx = threadIdx.x; idx < cnt; idx += kThreads) {
                const int m = idx / width;
                const int nl = idx - m * width;
                const int n = n_tile * 128 + n_lo + nl;
                if (n >= p.N) continue;
                float s = 0.0f;
                for (int r = 0; r < S; ++r) s += recv[(r * MMA_N + m) * nper + nl];
                p.C[static_cast<int64_t>(m) * p.ldc + n] = to_c<NV>(s);
            }
        }
    }

    // -------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (leader && last_issued >= 0) {
        // this slot's last copy (still in flight only after an abort) must land
        // before exit
        mbar_wait(full + slot, (last_issued / kRing) & 1, &g_fused_error, kErrWaitDrain);
    }
    if (warp == 1) {
        // every group arrives on accf once all of its MMAs and scale copies have
        // completed (at once when the epilogue already saw it)
        if (lane == 0) mbar_wait(accf, 0, &g_fused_error, kErrWaitDrain);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

template <int MMA_N, bool NV>
cudaError_t launch_fused_t(const CUtensorMap &tmw, const FusedArgs &args, int n_tiles, int splits,
                           cudaStream_t stream)
{
    using Cfg = FusedCfg<MMA_N, NV>;
    auto kern = fused_quant_gemm_kernel<MMA_N, NV>;
    static KernelOnce once;
    const cudaError_t e = prepare_kernel(kern, Cfg::SMEM_BYTES, once, nullptr);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(n_tiles, splits, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = splits;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    FusedArgs a = args;
    a.wait_ns = wait_limit_ns();
    return cudaLaunchKernelEx(&cfg, kern, tmw, a);
}

}  // namespace

bool plan_fused(int64_t M, int64_t N, int64_t K, int num_sms, FusedPlan *plan, bool nvfp4, int want_splits)
{
    if (M < 1 || M > 64 || N < 1 || K < (nvfp4 ? 16 : 32)) return false;
    const int mma_n = M <= 16 ? 16 : M <= 32 ? 32 : 64;
    const int max_st = nvfp4 ? (mma_n == 16 ? FusedCfg<16, true>::MAX_ST
                                            : mma_n == 32 ? FusedCfg<32, true>::MAX_ST : FusedCfg<64, true>::MAX_ST)
                             : (mma_n == 16 ? FusedCfg<16>::MAX_ST
                                            : mma_n == 32 ? FusedCfg<32>::MAX_ST : FusedCfg<64>::MAX_ST);
    const int64_t k_stages = (K + 255) / 256;
    const int64_t n_tiles = (N + 127) / 128;
    int64_t s = (num_sms + n_tiles / 2) / n_tiles;
    if (s > kMaxSplits) s = kMaxSplits;
    if (s < 1) s = 1;
    if (s > k_stages) s = k_stages;
    const int64_t s_min = (k_stages + max_st - 1) / max_st;
    if (want_splits > 0) s = std::min<int64_t>(std::min<int64_t>(want_splits, kMaxSplits), k_stages);
    if (s < s_min) s = s_min;
    if (s > kMaxSplits || n_tiles > 0x7fffffff) return false;
    plan->mma_n = mma_n;
    plan->splits = static_cast<int>(s);
    plan->n_tiles = static_cast<int>(n_tiles);
    return true;
}

cudaError_t launch_fused(const CUtensorMap &tmb, const void *A, int64_t lda, const uint8_t *sfb, void *C,
                         int64_t ldc, int M, int N, int K, const FusedPlan &plan, bool nvfp4, cudaStream_t stream)
{
    FusedArgs a;
    a.A = static_cast<const uint16_t *>(A);
    a.lda = lda;
    a.sfw = sfb;
    a.C = static_cast<uint16_t *>(C);
    a.ldc = ldc;
    a.M = M;
    a.N = N;
    a.K = K;
    a.splits = plan.splits;
    a.sf_cblocks = (K / (nvfp4 ? 16 : 32) + 3) / 4;
    if (nvfp4) {
        switch (plan.mma_n) {
        case 16: return launch_fused_t<16, true>(tmb, a, plan.n_tiles, plan.splits, stream);
        case 32: return launch_fused_t<32, true>(tmb, a, plan.n_tiles, plan.splits, stream);
        case 64: return launch_fused_t<64, true>(tmb, a, plan.n_tiles, plan.splits, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (plan.mma_n) {
    case 16: return launch_fused_t<16, false>(tmb, a, plan.n_tiles, plan.splits, stream);
    case 32: return launch_fused_t<32, false>(tmb, a, plan.n_tiles, plan.splits, stream);
    case 64: return launch_fused_t<64, false>(tmb, a, plan.n_tiles, plan.splits, stream);
    default: return cudaErrorInvalidValue;
    }
}

int read_and_clear_fused_error()
{
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_fused_error, sizeof(int)) != cudaSuccess) return -1;
    cudaMemcpyToSymbol(g_fused_error, &zero, sizeof(int));
    return v;
}

}  // namespace mxfp4
