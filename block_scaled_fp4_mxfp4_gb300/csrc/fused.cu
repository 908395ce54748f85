// Fused dynamic MXFP4 quantization + block-scaled GEMM for small M
// (kernelbot-amd-mxfp4-mm-517169, "Optimization 5": the A tile is quantized on
// chip and fed straight to the matrix unit, so the quantized A never reaches
// global memory; the same page's docstring counts the round trip this saves).
//
// Design for a weight-streaming (HBM-bound) shape such as M = 16, N = 2112,
// K = 7168:
// * Swap A and B: the weight rows fill the MMA's M = 128, the few activation
//   rows (padded with zeros to MMA_N = 16/32/64/128) are the MMA's N. The
//   accumulator is D[n][m] = C^T, 128 TMEM lanes x MMA_N columns.
// * Grid = (ceil(N/128) weight tiles) x (S K-splits); the S CTAs of one weight
//   tile form a thread-block cluster. Each CTA streams its K-slice of 128
//   weight rows through a 4-slot TMA ring (evict-first: weights are read once).
// * Meanwhile warps 2-5 load the CTA's K-slice of bf16 A (every row, 16-byte
//   vector loads), compute the OCP MX scale per 32-block and the E2M1 codes
//   with the same arithmetic as the standalone quant kernel, and write them
//   into shared memory directly in the MMA's 128-byte-swizzled K-major operand
//   layout, plus the scales in the 512-byte blocked layout.
// * Warp 1 lane 0 copies both operands' scales to TMEM and issues the MMAs.
// * Split-K reduction without global scratch: every CTA leaves its fp32 tile
//   in its own shared memory; after a cluster barrier each CTA sums a 1/S slice
//   of the tile over the S CTAs in rank order (distributed shared memory) and
//   writes bf16 C. The sum order is fixed, so results are deterministic.
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mxfp4 {

__device__ int g_fused_error;

namespace {

constexpr int kRing = 4;
constexpr uint32_t kWBytes = 128 * 128;   // one stage of 128 weight rows x 256 FP4
constexpr uint32_t kWSfBytes = 2 * 512;   // its two 512-byte scale blocks
constexpr int kThreads = 192;
constexpr int kMaxSplits = 16;

__host__ __device__ constexpr uint32_t pow2_cols_f(uint32_t n)
{
    return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 512;
}

template <int MMA_N>
struct FusedCfg {
    static constexpr int MAX_ST = MMA_N <= 64 ? 8 : 4;   // K stages held per CTA
    static constexpr uint32_t ACT_TILE = MMA_N * 128;     // bytes of one swizzled stage
    static constexpr uint32_t RING_DATA = kRing * kWBytes;
    static constexpr uint32_t RING_SF = kRing * kWSfBytes;
    static constexpr uint32_t ACT_DATA = MAX_ST * ACT_TILE;
    static constexpr uint32_t ACT_SF = MAX_ST * 1024;
    static constexpr uint32_t BAR_OFF = RING_DATA + RING_SF + ACT_DATA + ACT_SF;
    static constexpr uint32_t SMEM_BYTES = BAR_OFF + 256 + 1024;
    static constexpr uint32_t SF_COLS = 16;                // 8 weight + 8 activation per slot
    static constexpr uint32_t TMEM_COLS = pow2_cols_f(MMA_N + kRing * SF_COLS);
    static_assert(ACT_TILE % 1024 == 0, "swizzled operand tiles need 1024-byte alignment");
    static_assert(RING_DATA >= MMA_N * 128 * 4, "reduction tile reuses the weight ring");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct FusedArgs {
    const uint16_t *A;
    int64_t lda;
    const uint8_t *sfw;   // weight scales, blocked [N, K/32]
    __nv_bfloat16 *C;
    int64_t ldc;
    int M, N, K;
    int splits;
    int sf_cblocks;
};

template <int MMA_N>
__global__ void __launch_bounds__(kThreads, 1)
    fused_quant_gemm_kernel(const __grid_constant__ CUtensorMap tmw, const FusedArgs p)
{
    using Cfg = FusedCfg<MMA_N>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem;
    uint8_t *ring_sf = smem + Cfg::RING_DATA;
    uint8_t *act = ring_sf + Cfg::RING_SF;
    uint8_t *act_sf = act + Cfg::ACT_DATA;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::BAR_OFF);
    uint64_t *empty = full + kRing;
    uint64_t *accf = empty + kRing;
    uint64_t *act_ready = accf + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(act_ready + 1);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_tile = blockIdx.x;
    const int split = blockIdx.y;
    const int k_stages = (p.K + 255) / 256;
    const int s_begin = k_stages * split / p.splits;
    const int s_end = k_stages * (split + 1) / p.splits;
    const int nst = s_end - s_begin;
    const int k_steps_total = (p.K + 63) / 64;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < kRing; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(accf, 1);
        mbar_init(act_ready, 128);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmw);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int issued = 0;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------ weight TMA producer
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < nst; ++i) {
                const int slot = i % kRing;
                if (i >= kRing &&
                    !mbar_wait(empty + slot, ((i / kRing) - 1) & 1, &g_fused_error, kErrWaitEmpty)) {
                    *abort_flag = 1;
                    break;
                }
                const int ks = s_begin + i;
                const int blk0 = ks * 2;
                const int nblk = min(2, p.sf_cblocks - blk0);
                mbar_arrive_expect_tx(full + slot, kWBytes + nblk * 512);
                tma_load_2d(ring + slot * kWBytes, &tmw, ks * 128, n_tile * 128, full + slot, pol);
                bulk_load(ring_sf + slot * kWSfBytes,
                          p.sfw + (static_cast<size_t>(n_tile) * p.sf_cblocks + blk0) * 512, nblk * 512,
                          full + slot, pol);
                issued = i + 1;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuer
            constexpr uint32_t IDESC = idesc_block_scaled(MMA_N, true);
            bool ok = mbar_wait(act_ready, 0, &g_fused_error, kErrWaitOperand);
            if (!ok) *abort_flag = 1;
            tc_fence_after();
            for (int i = 0; ok && i < nst; ++i) {
                const int slot = i % kRing;
                if (!mbar_wait(full + slot, (i / kRing) & 1, &g_fused_error, kErrWaitFull)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t w_base = smem_u32(ring + slot * kWBytes);
                const uint32_t a_base = smem_u32(act + i * Cfg::ACT_TILE);
                const uint32_t wsf = smem_u32(ring_sf + slot * kWSfBytes);
                const uint32_t asf = smem_u32(act_sf + i * 1024);
                const uint32_t tsfw = tmem + MMA_N + slot * Cfg::SF_COLS;
                const uint32_t tsfa = tsfw + 8;
                const int ks = s_begin + i;
                const int ksteps = min(4, k_steps_total - ks * 4);
                const int nblk = (ksteps + 1) / 2;
                for (int b = 0; b < nblk; ++b) {
                    tc_cp_scale_block(tsfw + b * 4, sdesc_scale(wsf + b * 512));
                    tc_cp_scale_block(tsfa + b * 4, sdesc_scale(asf + b * 512));
                }
                for (int kk = 0; kk < ksteps; ++kk) {
                    const uint32_t sfid = static_cast<uint32_t>(kk & 1) * 2u;
                    const int blk = kk >> 1;
                    mma_mxf4(tmem, sdesc_sw128(w_base + kk * 32), sdesc_sw128(a_base + kk * 32),
                             idesc_with_sf_ids(IDESC, sfid, sfid), tsfw + blk * 4, tsfa + blk * 4,
                             (i > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(empty + slot);
            }
            tc_commit(accf);
        }
    } else {
        // ------------------------------- on-chip quantization of A (warps 2-5)
        const int tq = threadIdx.x - 64;
        const int sub = tq & 3;
        const int per_row = nst * 8;                 // 32-blocks per row in this K-slice
        const int units = MMA_N * per_row;
        for (int u0 = 0; u0 < units; u0 += 32) {
            const int u = u0 + (tq >> 2);
            const bool active = u < units;
            const int m = active ? u / per_row : 0;
            const int lb = active ? u - m * per_row : 0;
            const int kblk = s_begin * 8 + lb;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (active && m < p.M && kblk * 32 < p.K)
                v = ld_nc_v4(p.A + static_cast<int64_t>(m) * p.lda + static_cast<int64_t>(kblk) * 32 + sub * 8);
            uint32_t amax = max_abs_bits8(v);
            amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const uint32_t sbyte = e8m0_byte_from_amax(amax);
            const uint32_t codes = mx_codes8(v, sbyte);
            if (active) {
                const int t = lb >> 3, j = lb & 7;
                *reinterpret_cast<uint32_t *>(act + t * Cfg::ACT_TILE + m * 128 + ((j ^ (m & 7)) << 4) + sub * 4) =
                    codes;
                if (sub == 0)
                    act_sf[t * 1024 + (j >> 2) * 512 + (m & 31) * 16 + (m >> 5) * 4 + (j & 3)] =
                        static_cast<uint8_t>(sbyte);
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(act_ready);
    }
    __syncwarp();

    // -------------------------------------------------------------- epilogue
    float *red = reinterpret_cast<float *>(ring);   // [MMA_N][128] fp32 after the mainloop
    if (warp >= 2) {
        const bool acc_ok = mbar_wait(accf, 0, &g_fused_error, kErrWaitAccum);
        tc_fence_after();
        const int q = warp & 3;                      // TMEM lane quadrant of this warp
        const int n_local = q * 32 + lane;
        const int n = n_tile * 128 + n_local;
        const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
        for (int c0 = 0; c0 < MMA_N; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(t_row + c0, v);
            tmem_ld_wait();
            if (!acc_ok) continue;
            if (p.splits == 1) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int m = c0 + j;
                    if (m < p.M && n < p.N)
                        p.C[static_cast<int64_t>(m) * p.ldc + n] = __float2bfloat16_rn(__uint_as_float(v[j]));
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) red[(c0 + j) * 128 + n_local] = __uint_as_float(v[j]);
            }
        }
        if (!acc_ok) *abort_flag = 1;
    }

    if (p.splits > 1) {
        // every CTA of the cluster reaches both barriers, also after an abort
        cluster_sync();
        const int rank = static_cast<int>(cluster_ctarank());
        const int nper = (128 + p.splits - 1) / p.splits;
        const int n_lo = rank * nper;
        const int n_hi = min(128, n_lo + nper);
        const int width = n_hi - n_lo;
        const uint32_t red_base = smem_u32(red);
        if (width > 0) {
            const int cnt = width * p.M;
            for (int idx = threadIdx.x; idx < cnt; idx += kThreads) {
                const int m = idx / width;
                const int nl = n_lo + (idx - m * width);
                const int n = n_tile * 128 + nl;
                if (n >= p.N) continue;
                const uint32_t addr = red_base + static_cast<uint32_t>((m * 128 + nl) * 4);
                float s = 0.0f;
                for (int r = 0; r < p.splits; ++r) s += ld_shared_cluster_f32(mapa_shared(addr, r));
                p.C[static_cast<int64_t>(m) * p.ldc + n] = __float2bfloat16_rn(s);
            }
        }
        cluster_sync();
    }

    // -------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0) {
        for (int i = max(0, issued - kRing); i < issued; ++i)
            mbar_wait(full + (i % kRing), (i / kRing) & 1, &g_fused_error, kErrWaitDrain);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

template <int MMA_N>
cudaError_t launch_fused_t(const CUtensorMap &tmw, const FusedArgs &args, int n_tiles, int splits,
                           cudaStream_t stream)
{
    using Cfg = FusedCfg<MMA_N>;
    auto kern = fused_quant_gemm_kernel<MMA_N>;
    static uint64_t configured = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!(configured & (1ull << (dev & 63)))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        configured |= 1ull << (dev & 63);
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(n_tiles, splits, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = splits;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmw, args);
}

}  // namespace

bool plan_fused(int64_t M, int64_t N, int64_t K, int num_sms, FusedPlan *plan)
{
    if (M < 1 || M > 64 || N < 1 || K < 32) return false;
    const int mma_n = M <= 16 ? 16 : M <= 32 ? 32 : 64;
    const int max_st = FusedCfg<16>::MAX_ST;
    const int64_t k_stages = (K + 255) / 256;
    const int64_t n_tiles = (N + 127) / 128;
    int64_t s = (num_sms + n_tiles / 2) / n_tiles;
    if (s > 8) s = 8;
    if (s < 1) s = 1;
    if (s > k_stages) s = k_stages;
    const int64_t s_min = (k_stages + max_st - 1) / max_st;
    if (s < s_min) s = s_min;
    if (s > kMaxSplits || n_tiles > 0x7fffffff) return false;
    plan->mma_n = mma_n;
    plan->splits = static_cast<int>(s);
    plan->n_tiles = static_cast<int>(n_tiles);
    return true;
}

cudaError_t launch_fused_mx(const CUtensorMap &tmb, const void *A, int64_t lda, const uint8_t *sfb,
                            void *C, int64_t ldc, int M, int N, int K, const FusedPlan &plan,
                            cudaStream_t stream)
{
    FusedArgs a;
    a.A = static_cast<const uint16_t *>(A);
    a.lda = lda;
    a.sfw = sfb;
    a.C = static_cast<__nv_bfloat16 *>(C);
    a.ldc = ldc;
    a.M = M;
    a.N = N;
    a.K = K;
    a.splits = plan.splits;
    a.sf_cblocks = (K / 32 + 3) / 4;
    switch (plan.mma_n) {
    case 16: return launch_fused_t<16>(tmb, a, plan.n_tiles, plan.splits, stream);
    case 32: return launch_fused_t<32>(tmb, a, plan.n_tiles, plan.splits, stream);
    case 64: return launch_fused_t<64>(tmb, a, plan.n_tiles, plan.splits, stream);
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
