// Fused RMSNorm + MXFP4 quantization: bf16 X [M, K] and a bf16 weight w [K]
// -> packed E2M1 codes [M, K/2] and E8M0 scales (blocked layout, pad 0x7F) of
//   y_k = fp32(fp32(x_k * r) * w_k),   r = fp32(1 / sqrt(ss / K + eps)),
//   ss = sum_k x_k^2 (exact, rounded once to fp64; r from it in fp64),
// each 32-value block of y quantized by the OCP MX rule as mxfp4_quantize
// does. kernelbot-amd-mxfp4-mm-683203 names this fused activation step (the
// fused RMSNorm + MXFP4 quantization its "hot path" cites) without its
// arithmetic; the rule above is this library's reading of it.
//
// One CTA per row (grid-stride over the rows padded to 128). The sum of
// squares is formed exactly in 128-bit integers: a bf16 x is m * 2^(E - 134)
// with an 8-bit m, so x^2 = m^2 * 2^(2E - 268); every square is shifted to a
// common exponent set by the row's largest E (80 bits of headroom: exact
// whenever all nonzero magnitudes of the row lie within 2^40 of the largest,
// and no overflow for K < 2^31) and added with carries. Integer addition does
// not depend on the order, so the 256 threads and the cross-warp reduction
// give the same sum as any other order; it is rounded once to fp64 (round to
// nearest even), which is the correctly rounded exact sum the reading asks for. The row is then
// read a third time (from L2) to form y, quantize it and store codes and
// scale words exactly as the quantization kernel does.
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mxfp4 {
namespace {

constexpr int kRmsThreads = 256;
constexpr int kRmsWarps = kRmsThreads / 32;
constexpr int kRmsHeadroom = 80;   // fractional bits of the fixed-point sum

struct U128 {
    unsigned long long lo, hi;
};

__device__ __forceinline__ void add128(U128 &a, unsigned long long lo, unsigned long long hi)
{
    const unsigned long long s = a.lo + lo;
    a.hi += hi + (s < lo ? 1ull : 0ull);
    a.lo = s;
}

// Biased exponent (1 for zero and subnormals) and 8-bit significand of a bf16.
__device__ __forceinline__ void bf16_parts(uint32_t h, int &e, uint32_t &m)
{
    const uint32_t E = (h >> 7) & 0xFFu;
    m = E ? ((h & 0x7Fu) | 0x80u) : (h & 0x7Fu);
    e = E ? static_cast<int>(E) : 1;
}

// m^2 * 2^s as a 128-bit integer (s <= kRmsHeadroom; s < 0 drops the bits
// below 2^0).
__device__ __forceinline__ void square_term(uint32_t m, int s, unsigned long long &lo, unsigned long long &hi)
{
    const unsigned long long v = static_cast<unsigned long long>(m * m);   // < 2^16
    lo = 0;
    hi = 0;
    if (s >= 64) {
        hi = v << (s - 64);
    } else if (s >= 0) {
        lo = v << s;
        if (s > 48) hi = v >> (64 - s);
    } else if (s > -16) {
        lo = v >> (-s);
    }
}

// (hi * 2^64 + lo) * 2^e2 rounded to the nearest double (ties to even).
__device__ __forceinline__ double u128_to_double(U128 a, int e2)
{
    if (a.hi == 0 && a.lo == 0) return 0.0;
    unsigned long long top = a.lo;
    int shift = 0;
    if (a.hi != 0) {
        const int lz = __clzll(static_cast<long long>(a.hi));
        shift = 64 - lz;
        top = lz ? ((a.hi << lz) | (a.lo >> (64 - lz))) : a.hi;
        const unsigned long long dropped = lz ? (a.lo << lz) : a.lo;
        if (dropped != 0) top |= 1ull;      // sticky bit, 11 places below the rounding point
    }
    const double d = __ull2double_rn(top);  // the one rounding
    const int n = shift + e2;               // in [-346, 224]: an exact power-of-two scaling
    return d * __longlong_as_double(static_cast<long long>(1023 + n) << 52);
}

__global__ void __launch_bounds__(kRmsThreads) rmsnorm_mx_quant_kernel(const uint16_t *__restrict__ X, int M, int K,
                                                                       int64_t ldx, const uint16_t *__restrict__ w,
                                                                       float eps, uint8_t *__restrict__ Aq,
                                                                       int64_t ldq, uint8_t *__restrict__ sf)
{
    __shared__ int s_emax[kRmsWarps];       // per-warp largest magnitude (bf16 bits)
    __shared__ unsigned long long s_lo[kRmsWarps], s_hi[kRmsWarps];
    __shared__ float s_r;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nvec = K / 8;                 // 16-byte vectors per row
    const int C = K / 32;                   // scale columns
    const int cblocks = (C + 3) / 4;
    const int nseg = (K + 255) / 256;
    const int64_t rows = (static_cast<int64_t>(M) + 127) / 128 * 128;

    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const bool row_ok = r < M;
        const uint16_t *xrow = X + r * ldx;
        float rs = 0.0f;
        if (row_ok) {
            // pass 1: the largest magnitude of the row (bf16 magnitudes order as integers)
            uint32_t mm = 0;
            for (int i = tid; i < nvec; i += kRmsThreads) mm = max(mm, max_abs_bits8(ld_nc_v4(xrow + i * 8)));
            mm = __reduce_max_sync(0xffffffffu, mm);
            if (lane == 0) s_emax[warp] = static_cast<int>(mm);
            __syncthreads();
            mm = 0;
#pragma unroll
            for (int i = 0; i < kRmsWarps; ++i) mm = max(mm, static_cast<uint32_t>(s_emax[i]));
            // its exponent (1 for subnormals, 0 for an all-zero row)
            const int emax = mm ? max(static_cast<int>(mm >> 7), 1) : 0;
            // pass 2: exact sum of squares at the common exponent. A square whose
            // shift is at least 48 (|x| within 2^16 of the largest) goes to a
            // 64-bit per-vector sum (< 8 * 2^48), added to the 128-bit
            // accumulator once per vector; smaller ones take the general path.
            const int base = kRmsHeadroom - 2 * emax;
            U128 acc{0ull, 0ull};
            for (int i = tid; i < nvec; i += kRmsThreads) {
                const uint4 v = ld_nc_v4(xrow + i * 8);
                const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
                unsigned long long fast = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    int e;
                    uint32_t m;
                    bf16_parts((wv[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu, e, m);
                    const int sh = 2 * e + base;
                    if (sh >= 48) {
                        fast += static_cast<unsigned long long>(m * m) << (sh - 48);
                    } else if (m != 0) {
                        unsigned long long lo, hi;
                        square_term(m, sh, lo, hi);
                        add128(acc, lo, hi);
                    }
                }
                add128(acc, fast << 48, fast >> 16);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const unsigned long long lo = __shfl_xor_sync(0xffffffffu, acc.lo, o);
                const unsigned long long hi = __shfl_xor_sync(0xffffffffu, acc.hi, o);
                add128(acc, lo, hi);
            }
            if (lane == 0) {
                s_lo[warp] = acc.lo;
                s_hi[warp] = acc.hi;
            }
            __syncthreads();
            if (tid == 0) {
                U128 t{0ull, 0ull};
                for (int i = 0; i < kRmsWarps; ++i) add128(t, s_lo[i], s_hi[i]);
                // sum = t * 2^(2 emax - 268 - headroom)
                const double ss = u128_to_double(t, 2 * emax - 268 - kRmsHeadroom);
                const double ms = ss / static_cast<double>(K) + static_cast<double>(eps);
                const double r64 = ms > 0.0 ? 1.0 / sqrt(ms) : 0.0;
                s_r = __double2float_rn(r64);
            }
            __syncthreads();
            rs = s_r;
        }
        // pass 3: y, its MXFP4 codes and scale words (one warp per 256-element segment)
        uint8_t *qrow = Aq + r * ldq;
        uint8_t *sfrow = sf + (static_cast<size_t>(r >> 7) * cblocks) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
        for (int seg = warp; seg < nseg; seg += kRmsWarps) {
            const int blk = seg * 8 + lane / 4;         // scale column of this lane
            const int k = blk * 32 + (lane % 4) * 8;    // first element of this lane
            const bool ok = row_ok && blk < C;
            float y[8];
            uint32_t amax = 0;
            if (ok) {
                const uint4 xv = ld_nc_v4(xrow + k);
                const uint4 wv = ld_nc_v4(w + k);
                const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    y[2 * j] = __fmul_rn(__fmul_rn(__uint_as_float(xa[j] << 16), rs), __uint_as_float(wa[j] << 16));
                    y[2 * j + 1] = __fmul_rn(__fmul_rn(__uint_as_float(xa[j] & 0xFFFF0000u), rs),
                                             __uint_as_float(wa[j] & 0xFFFF0000u));
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) amax = max(amax, __float_as_uint(y[j]) & 0x7FFFFFFFu);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) y[j] = 0.0f;
            }
            amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            // OCP MX: e = floor(log2 amax) - 2, clamped below at -127 (byte 0)
            const uint32_t E = amax >> 23;
            const uint32_t sbyte = E >= 2 ? E - 2 : 0;
            const float mult = __uint_as_float((254u - sbyte) << 23);   // 2^-e, exact
            const uint32_t codes = e2m1x8_rn_sat(y[0] * mult, y[1] * mult, y[2] * mult, y[3] * mult,
                                                 y[4] * mult, y[5] * mult, y[6] * mult, y[7] * mult);
            if (ok) *reinterpret_cast<uint32_t *>(qrow + k / 2) = codes;
            const uint32_t mine = ok ? sbyte : 0x7Fu;
            const int base = lane & ~15;
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) word |= __shfl_sync(0xffffffffu, mine, base + j * 4) << (8 * j);
            const int widx = seg * 2 + lane / 16;
            if ((lane & 15) == 0 && widx < cblocks)
                *reinterpret_cast<uint32_t *>(sfrow + static_cast<size_t>(widx) * 512) = word;
        }
        __syncthreads();   // the shared slots are reused by the next row
    }
}

}  // namespace

cudaError_t launch_rmsnorm_mx_quant(const void *X, int64_t M, int64_t K, int64_t ldx, const void *w, float eps,
                                    void *Aq, int64_t ldq, void *sf, int num_sms, cudaStream_t stream)
{
    if (M < 1 || K < 1 || M > 0x7fffffff || K > 0x7fffffff) return cudaErrorInvalidValue;
    const int64_t rows = (M + 127) / 128 * 128;
    int64_t blocks = rows;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    rmsnorm_mx_quant_kernel<<<static_cast<unsigned>(blocks), kRmsThreads, 0, stream>>>(
        static_cast<const uint16_t *>(X), static_cast<int>(M), static_cast<int>(K), ldx,
        static_cast<const uint16_t *>(w), eps, static_cast<uint8_t *>(Aq), ldq, static_cast<uint8_t *>(sf));
    return cudaGetLastError();
}

}  // namespace mxfp4
