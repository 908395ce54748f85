// Host-side interface between the C-ABI layer (api.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace mxfp4 {

// Problems a grouped launch carries in its kernel parameters; longer lists
// go through a table in the caller's workspace.
constexpr int kMaxGroups = 16;

// Device problem table: per group kTableMaps tensor maps (A, B, then C for the
// single-CTA kernel or A scales, B scales for the CTA-pair kernel) and one
// problem record of kTableProblemBytes.
constexpr int kTableMaps = 4;
constexpr size_t kTableProblemBytes = 128;
constexpr size_t group_table_bytes(int num_groups)
{
    return static_cast<size_t>(num_groups) * (kTableMaps * sizeof(CUtensorMap) + kTableProblemBytes);
}

// Default limit of every bounded wait in the kernels (2 s of %globaltimer).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Limit of the waits that guard work in kernels launched from now on
// (mxfp4_set_wait_limit_ns); the waits on a kernel's exit path keep the
// default. Process-wide, read at every launch.
uint64_t wait_limit_ns();
void set_wait_limit_ns(uint64_t ns);

// Per-device, set-once facts of one kernel instantiation: its dynamic
// shared-memory limit is raised once per device and the device's SM count is
// read once. Safe when launches come from several host threads (at worst two
// threads both set the same attribute).
struct KernelOnce {
    std::atomic<uint64_t> done{0};
    std::atomic<int> sms[64];
};

template <typename Kern>
cudaError_t prepare_kernel(Kern kern, uint32_t smem_bytes, KernelOnce &once, int *sms)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << dev;
    if (!(once.done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes));
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        once.sms[dev].store(n, std::memory_order_relaxed);
        once.done.fetch_or(bit, std::memory_order_release);
    }
    if (sms) *sms = once.sms[dev].load(std::memory_order_relaxed);
    return cudaSuccess;
}

// ---------------------------------------------------------------- quant.cu
// Every quantization launch uses programmatic dependent launch and reads A
// only after the preceding grid has completed. feeds_gemm: the next launch
// is this library's GEMM on the quantized activations, which may start once
// every CTA has passed that wait (it reads only weights before its own
// wait); otherwise the next grid starts when this one has exited, and the
// codes and scales are made visible device-wide before each CTA exits.
cudaError_t launch_quant_mx(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq,
                            int64_t ldq, void *sf, int num_sms, cudaStream_t stream, bool feeds_gemm = false);
cudaError_t launch_quant_nv(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq,
                            int64_t ldq, void *sf, int num_sms, cudaStream_t stream);
// One matrix of a grouped NVFP4 quantization (bf16 A [M, K] -> packed codes
// [M, K/2] with row stride ldq bytes + blocked E4M3 scales).
struct QuantGroupHost {
    const void *A;
    int64_t M, K, lda;
    void *Aq;
    int64_t ldq;
    void *sf;
};
// All `count` (1..kMaxGroups) matrices in one launch.
cudaError_t launch_quant_nv_grouped(const QuantGroupHost *groups, int count, int num_sms, cudaStream_t stream,
                                    bool feeds_gemm = false);

// --------------------------------------------------------- rmsnorm_quant.cu
// Fused RMSNorm (bf16 weight [K], eps) + MXFP4 quantization of bf16 X [M, K].
cudaError_t launch_rmsnorm_mx_quant(const void *X, int64_t M, int64_t K, int64_t ldx, const void *w, float eps,
                                    void *Aq, int64_t ldq, void *sf, float *rstd, double *sumsq, int num_sms,
                                    cudaStream_t stream);

// ----------------------------------------------------------------- gemm.cu
// One GEMM problem as the tile scheduler sees it.
struct GemmProblemHost {
    CUtensorMap tma;          // packed A [m, k/2] u8, box {128 B, 128 rows}, 128B swizzle
    CUtensorMap tmb;          // packed B [n, k/2] u8, box {128 B, bn rows}, 128B swizzle
    const uint8_t *sfa;       // blocked scales of A
    const uint8_t *sfb;       // blocked scales of B
    void *c;                  // bf16 (MXFP4) or fp16 (NVFP4) [m, n]
    int64_t ldc;              // elements
    int m, n, k;
    // optional epilogue C = alpha * acc + beta * C + bias[n] (epi false: C = acc)
    bool epi;
    float alpha, beta;
    const void *bias;         // [n] in C's type, or null
    // CTA-pair kernels only: the scale buffers as [blocks, 128 u32] with a box of
    // one stage's K-blocks (2 for MXFP4, 4 for NVFP4)
    CUtensorMap tmsfa;
    CUtensorMap tmsfb;
    // single-CTA kernel: C as a 16-bit [m, n] tensor, box {32, 32}, 64-byte
    // swizzle, for tiles stored by TMA (c_tma; else C is stored directly)
    CUtensorMap tmc;
    bool c_tma;
};

// Tile width along N of the grouped NVFP4 GEMM (box rows of tmb).
int gemm_block_n_nv();

// MXFP4 (kind::mxf4, bf16 C) with tiles of 128 x bn, bn = 128 or 256 (the box
// rows of prob.tmb). splits > 1 needs `partials` (splits * n_tiles * bn * M
// floats) and zeroed `tickets` (one int per tile).
cudaError_t launch_gemm_mx(const GemmProblemHost &prob, int bn, int splits, float *partials,
                           int *tickets, cudaStream_t stream);
// Grouped NVFP4 (kind::mxf4nvf4, fp16 C), one launch over all groups. More
// than kMaxGroups problems need `table`: group_table_bytes(num_groups) bytes
// of device memory (64-byte aligned), filled on `stream` before the launch.
cudaError_t launch_gemm_nv_grouped(const GemmProblemHost *probs, int num_groups, void *table,
                                   cudaStream_t stream);
// Grouped MXFP4 (kind::mxf4, bf16 C), one launch over all groups; `table` as above.
cudaError_t launch_gemm_mx_grouped(const GemmProblemHost *probs, int num_groups, void *table,
                                   cudaStream_t stream);
int read_and_clear_gemm_error();

// ------------------------------------------------------------ gemm_pair.cu
// The same GEMMs on CTA pairs (tcgen05 cta_group::2, 256 x 256 tiles, no
// split-K) for problems with enough tiles to fill the GPU. prob.tmb boxes are
// 128 rows (each CTA loads half of a tile's B).
int pair_tiles(int64_t m, int64_t n);   // 256 x 256 tiles of an m x n output
// scale blocks per tmsfa / tmsfb box (one stage): 2 for MXFP4, 4 for NVFP4
constexpr int pair_sf_box_blocks(bool nvfp4) { return nvfp4 ? 4 : 2; }
cudaError_t launch_gemm_mx_pair(const GemmProblemHost &prob, cudaStream_t stream);
cudaError_t launch_gemm_nv_grouped_pair(const GemmProblemHost *probs, int num_groups, void *table,
                                        cudaStream_t stream);
cudaError_t launch_gemm_mx_grouped_pair(const GemmProblemHost *probs, int num_groups, void *table,
                                        cudaStream_t stream);

// Copies `bytes` (a multiple of 16) from host memory into the device table
// `dst` (16-byte aligned) on `stream` with kernels that carry the bytes in
// their parameters: stream-ordered, capturable in a CUDA graph, and the host
// buffer may be reused as soon as this returns.
cudaError_t upload_table(void *dst, const void *src, size_t bytes, cudaStream_t stream);
int read_and_clear_gemm_pair_error();

// ---------------------------------------------------------------- fused.cu
struct FusedPlan {
    int mma_n;       // activation rows padded to the MMA N
    int splits;      // K splits = cluster size
    int n_tiles;     // ceil(N / 128)
};
// Whether the fused small-M kernel can run (M, K) and with which plan.
// nvfp4: E4M3 scales per 16 and fp16 C (else MXFP4: E8M0 per 32, bf16 C).
// want_splits > 0 asks for that many K-splits (clamped to what the kernel
// can run); 0 takes the shape-derived rule.
bool plan_fused(int64_t M, int64_t N, int64_t K, int num_sms, FusedPlan *plan, bool nvfp4 = false,
                int want_splits = 0);

// One entry of the measured split-K table (csrc/split_table.inc): the
// K-splits that were fastest for a shape. which: 0 = two-kernel GEMM path
// (bucket = 128-row tiles of M), 1 = fused MXFP4, 2 = fused NVFP4 (bucket =
// MMA width 16 / 32 / 64 of the padded activation rows).
struct SplitEntry {
    int which, bucket;
    int64_t n, k;
    int splits;
};
// tmb: packed weights [N, K/2], box {128 B, 128 rows}, 128B swizzle.
cudaError_t launch_fused(const CUtensorMap &tmb, const void *A, int64_t lda, const uint8_t *sfb,
                         void *C, int64_t ldc, int M, int N, int K, const FusedPlan &plan, bool nvfp4,
                         cudaStream_t stream);
int read_and_clear_fused_error();

}  // namespace mxfp4
