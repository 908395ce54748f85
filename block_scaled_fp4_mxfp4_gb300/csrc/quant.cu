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
// Work unit: one warp x one 1024-element chunk of one row. The warp loads the
// chunk with 16-byte vectors, 512 contiguous bytes per instruction (the access
// that streams at full HBM bandwidth), and passes it through a 2 KB shared
// buffer so that each lane then holds 32 consecutive elements: one MXFP4
// block or two NVFP4 blocks. A lane takes its blocks' largest magnitudes with
// packed bf16 max operations, encodes its 16 bytes of codes and stores them
// with one vector store (the warp writes 512 contiguous bytes); the scale
// bytes of four consecutive blocks meet in one lane by two (MXFP4) or one
// (NVFP4) shuffles and go out as one 32-bit word of the blocked layout. Rows
// past M up to the next multiple of 128 and K-blocks past K inside a written
// word get the pad byte (0x7F for E8M0 = 1.0, 0x00 for E4M3). One launch may
// quantize up to kMaxGroups matrices (the grouped path); a single matrix is a
// table of one. Launches use programmatic dependent launch: A is read after
// the wait for the preceding grid (a small A is prefetched into L2 before
// it), and inside a quant -> GEMM call the GEMM is released right after that
// wait so that it streams its weights while A is quantized.
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mxfp4 {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kQuantWarps = kQuantThreads / 32;
constexpr int kChunk = 1024;            // elements per work unit (one warp)
// A of at most this many bytes is prefetched into L2 before the dependency
// wait (a larger one would only double the requests of the loads that follow)
constexpr int64_t kQuantPrefetchMaxBytes = 16ll << 20;
// resident blocks per SM (16 KB of shared memory each): MXFP4 fits in 40
// registers, NVFP4's reciprocal and scale conversion want a few more
template <int VEC>
constexpr int kQuantBlocksPerSm = VEC == 32 ? 6 : 5;

// The matrices of one launch: the work units of matrix g are the global
// units [first[g], first[g + 1]), row-major over (row padded to 128, chunk).
struct QuantGroupsDev {
    const uint16_t *A[kMaxGroups];
    uint8_t *Aq[kMaxGroups];
    uint8_t *sf[kMaxGroups];
    int64_t lda[kMaxGroups], ldq[kMaxGroups];
    int64_t first[kMaxGroups + 1];
    int M[kMaxGroups], K[kMaxGroups], nchunk[kMaxGroups];
    int vec_store[kMaxGroups];   // code rows 16-byte aligned: one vector store per lane
    int count;
    int feeds_gemm;              // let the next grid start right after the dependency wait
    int prefetch;                // A is small: pull it into L2 before the dependency wait
};

// Position of 16-byte slot s of a warp's chunk buffer: the slot's bank group
// (s mod 8) is XORed with (s / 8) mod 8, so that both the loading pattern
// (slot 32 j + lane) and the reading pattern (slot 4 lane + j) touch eight
// distinct bank groups in every quarter-warp.
__device__ __forceinline__ int swz(int s) { return s ^ ((s >> 3) & 7); }

template <int VEC>
__global__ void __launch_bounds__(kQuantThreads, kQuantBlocksPerSm<VEC>) quant_kernel(const __grid_constant__ QuantGroupsDev q)
{
    constexpr int BPL = 32 / VEC;                 // blocks per lane (1 or 2)
    constexpr uint32_t PAD = VEC == 32 ? 0x7Fu : 0x00u;
    __shared__ uint4 chunk_buf[kQuantWarps][kChunk / 8];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t units = q.first[q.count];
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kQuantWarps;
    if (q.prefetch && lane == 0) {
        // A small A is requested into L2 while the preceding grid still runs
        // (this grid starts early under programmatic dependent launch): the
        // loads after the wait then hit L2. L2 is the point of coherence, so
        // a later write of the preceding grid still reaches those loads.
        int g = 0;
        for (int64_t u = static_cast<int64_t>(blockIdx.x) * kQuantWarps + warp; u < units; u += nwarps) {
            while (u >= q.first[g + 1]) ++g;
            const int64_t local = u - q.first[g];
            const int nch = q.nchunk[g];
            const int64_t r = local / nch;
            const int k0 = static_cast<int>(local - r * nch) * kChunk;
            if (r < q.M[g])
                prefetch_l2_bulk(q.A[g] + r * q.lda[g] + k0, static_cast<uint32_t>(min(kChunk, q.K[g] - k0) * 2));
        }
    }
    // Launched with programmatic dependent launch: A is read only after the
    // preceding grid has completed. The GEMM of a quant -> GEMM call may
    // start right after that and request its weights; it reads what this
    // grid writes only after its own dependency wait.
    grid_dependency_wait();
    if (q.feeds_gemm) grid_launch_dependents();
    uint4 *buf = chunk_buf[warp];
    int g = 0;
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * kQuantWarps + warp; u < units; u += nwarps) {
        while (u >= q.first[g + 1]) ++g;         // units only grow along the loop
        const int64_t local = u - q.first[g];
        const int nch = q.nchunk[g];
        const int64_t r = local / nch;
        const int k0 = static_cast<int>(local - r * nch) * kChunk;
        const int K = q.K[g];
        const int C = K / VEC;                   // scale columns (K-blocks)
        const int cblocks = (C + 3) / 4;         // scale words per row
        const int kl = k0 + 32 * lane;           // first element of this lane's span
        uint32_t sb[BPL];
#pragma unroll
        for (int t = 0; t < BPL; ++t) sb[t] = PAD;
        if (r < q.M[g]) {
            const uint16_t *src = q.A[g] + r * q.lda[g] + k0;
            uint4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = 256 * j + 8 * lane;
                v[j] = (k0 + e < K) ? ld_nc_v4(src + e) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) buf[swz(32 * j + lane)] = v[j];
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = buf[swz(4 * lane + j)];
            __syncwarp();                        // the buffer is free for the next unit
            if (kl < K) {
                uint32_t w[4];
#pragma unroll
                for (int t = 0; t < BPL; ++t) {
                    constexpr int NV = VEC / 8;  // 16-byte vectors per block
                    const uint32_t amax = block_amax_bits<NV>(v + t * NV);
                    if constexpr (VEC == 32) {
                        sb[t] = e8m0_byte_from_amax(amax);
#pragma unroll
                        for (int i = 0; i < NV; ++i) w[t * NV + i] = mx_codes8(v[t * NV + i], sb[t]);
                    } else {
                        sb[t] = nv_scale_byte(amax);
                        const float rs = nv_recip(sb[t]);
#pragma unroll
                        for (int i = 0; i < NV; ++i) w[t * NV + i] = nv_codes8(v[t * NV + i], rs);
                    }
                }
                uint8_t *dst = q.Aq[g] + r * q.ldq[g] + kl / 2;
                if (q.vec_store[g]) {
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) reinterpret_cast<uint32_t *>(dst)[i] = w[i];
                }
            }
        }
        // four consecutive K-blocks' scale bytes meet in one lane as one word
        uint32_t word;
        if constexpr (VEC == 32) {
            word = sb[0];
            word |= __shfl_down_sync(0xffffffffu, word, 1) << 8;
            word |= __shfl_down_sync(0xffffffffu, word, 2) << 16;
        } else {
            word = sb[0] | (sb[1] << 8);
            word |= __shfl_down_sync(0xffffffffu, word, 1) << 16;
        }
        constexpr int LPW = 4 / BPL;             // lanes per scale word
        const int wi = (k0 / VEC + lane * BPL) / 4;
        if ((lane % LPW) == 0 && wi < cblocks) {
            // the word's place: 128-row chunk, K-word, row within a 32-row group, group
            *reinterpret_cast<uint32_t *>(q.sf[g] + ((r >> 7) * cblocks + wi) * 512 + (r & 31) * 16 +
                                          ((r >> 5) & 3) * 4) = word;
        }
    }
    // A grid that starts when this one has exited (the implicit trigger) may
    // read weights quantized here before its dependency wait: the codes and
    // scales are performed device-wide before the CTA leaves. (The GEMM that
    // a quant -> GEMM call releases early reads them only after its wait.)
    if (!q.feeds_gemm) __threadfence();
}

template <int VEC>
cudaError_t launch_quant(const QuantGroupHost *groups, int count, int num_sms, cudaStream_t stream, bool feeds_gemm)
{
    if (count < 1 || count > kMaxGroups) return cudaErrorInvalidValue;
    QuantGroupsDev q;
    memset(&q, 0, sizeof(q));
    q.count = count;
    q.feeds_gemm = feeds_gemm ? 1 : 0;
    int64_t a_bytes = 0;
    q.first[0] = 0;
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
        q.nchunk[g] = static_cast<int>((h.K + kChunk - 1) / kChunk);
        q.vec_store[g] = ((reinterpret_cast<uintptr_t>(h.Aq) & 15u) == 0 && (h.ldq & 15) == 0) ? 1 : 0;
        q.first[g + 1] = q.first[g] + (h.M + 127) / 128 * 128 * q.nchunk[g];
        a_bytes += h.M * h.K * 2;
    }
    q.prefetch = a_bytes <= kQuantPrefetchMaxBytes ? 1 : 0;
    for (int g = count + 1; g <= kMaxGroups; ++g) q.first[g] = q.first[count];
    const int64_t units = q.first[count];
    int64_t blocks = (units + kQuantWarps - 1) / kQuantWarps;
    const int64_t cap = static_cast<int64_t>(num_sms) * kQuantBlocksPerSm<VEC>;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(kQuantThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quant_kernel<VEC>, q);
}

}  // namespace

cudaError_t launch_quant_nv_grouped(const QuantGroupHost *groups, int count, int num_sms, cudaStream_t stream,
                                    bool feeds_gemm)
{
    return launch_quant<16>(groups, count, num_sms, stream, feeds_gemm);
}

cudaError_t launch_quant_mx(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq,
                            int64_t ldq, void *sf, int num_sms, cudaStream_t stream, bool feeds_gemm)
{
    const QuantGroupHost one{A, M, K, lda, Aq, ldq, sf};
    return launch_quant<32>(&one, 1, num_sms, stream, feeds_gemm);
}

cudaError_t launch_quant_nv(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq,
                            int64_t ldq, void *sf, int num_sms, cudaStream_t stream)
{
    const QuantGroupHost one{A, M, K, lda, Aq, ldq, sf};
    return launch_quant<16>(&one, 1, num_sms, stream, false);
}

}  // namespace mxfp4
