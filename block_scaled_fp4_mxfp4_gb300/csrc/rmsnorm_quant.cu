// Fused RMSNorm + MXFP4 quantization: bf16 X [M, K] and a bf16 weight w [K]
// -> packed E2M1 codes [M, K/2] and E8M0 scales (blocked layout, pad 0x7F) of
//   y_k = fp32(fp32(x_k * r) * w_k),   r = fp32(1 / sqrt(ss / K + eps)),
//   ss = sum_k x_k^2 (exact, rounded once to fp64; r from it in fp64),
// each 32-value block of y quantized by the OCP MX rule as mxfp4_quantize
// does. kernelbot-amd-mxfp4-mm-683203 names this fused activation step (the
// fused RMSNorm + MXFP4 quantization its "hot path" cites) without its
// arithmetic; the rule above is this library's reading of it.
//
// One CTA per row at a time (several CTAs per SM, grid-stride over the rows
// padded to 128). Thread t of a CTA of T threads holds the 16-byte vectors
// t, t + T, ..., t + (VPT - 1) T of the row in registers, so the row is read
// from memory once and the three passes (largest magnitude, sum of squares,
// quantization) run on registers; four consecutive lanes hold one 32-value
// block, so block maxima take two shuffles and the code stores of a warp are
// 128 contiguous bytes. (Rows longer than VPT * T vectors are taken in chunks
// of that size, reloaded in each pass.)
//
// The sum of squares is exact for every finite input. A bf16 x is m * 2^(E-134)
// with an 8-bit m (E the exponent field, 1 for subnormals), so x^2 is
// m^2 * 2^(2E - 268). Relative to the row's largest exponent field Emax:
//  * E >= Emax - 16 (the common case): u = m * 2^(E - Emax + 16) < 2^24 is an
//    integer and u^2 is accumulated exactly with one wide multiply-add into a
//    64-bit sum (at most 128 terms between flushes, < 2^55);
//  * Emax - 56 <= E < Emax - 16: m^2 shifted to a 128-bit fixed point with 80
//    fractional bits below 2 (Emax) (the 64-bit sums are added into it too;
//    < K * 2^96, no overflow for K < 2^31);
//  * smaller E: m^2 goes to a 576-bit integer in shared memory whose bit 0 is
//    2^-266 (the smallest square), kept as 18 64-bit counters of 32-bit limbs
//    that take shared atomic adds. Rows never reach this path unless their
//    magnitudes span more than 2^40; the 128-bit sum is then added into the
//    limbs and carries are propagated before the rounding.
// Integer addition does not depend on the order, so the threads and the
// cross-warp reduction give the same exact sum as any other order; it is
// rounded once to fp64 (round to nearest even: 64 leading bits plus a sticky
// bit for everything below them), which is the correctly rounded exact sum the
// reading asks for.
#include <atomic>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mxfp4 {
namespace {

constexpr int kRmsMaxThreads = 512;
constexpr int kRmsHeadroom = 80;   // fractional bits of the 128-bit fixed-point sum
constexpr int kRmsFastSpan = 16;   // exponent fields within this of the largest take the 64-bit sum
constexpr int kRmsLimbs = 18;      // 32-bit limbs of the exact integer (576 bits >= 522 + 31 + carries)

struct U128 {
    unsigned long long lo, hi;
};

__device__ __forceinline__ void add128(U128 &a, unsigned long long lo, unsigned long long hi)
{
    const unsigned long long s = a.lo + lo;
    a.hi += hi + (s < lo ? 1ull : 0ull);
    a.lo = s;
}

// a << s for s < 32, and 0 for every larger s taken as unsigned (a negative
// s included): the shift saturates instead of wrapping.
__device__ __forceinline__ uint32_t shl_sat(uint32_t a, int s)
{
    uint32_t d;
    asm("shl.b32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(s));
    return d;
}

// acc + a * b with a 64-bit product (one wide multiply-add).
__device__ __forceinline__ unsigned long long mad_wide(uint32_t a, uint32_t b, unsigned long long acc)
{
    unsigned long long d;
    asm("mad.wide.u32 %0, %1, %2, %3;" : "=l"(d) : "r"(a), "r"(b), "l"(acc));
    return d;
}

// m^2 * 2^s as a 128-bit integer, 0 <= s <= kRmsHeadroom.
__device__ __forceinline__ void square_term(uint32_t m, int s, unsigned long long &lo, unsigned long long &hi)
{
    const unsigned long long v = static_cast<unsigned long long>(m * m);   // < 2^16
    lo = 0;
    hi = 0;
    if (s >= 64) {
        hi = v << (s - 64);
    } else {
        lo = v << s;
        if (s > 48) hi = v >> (64 - s);
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

// The exact sum held as limbs (32-bit values in limb[0 .. kRmsLimbs), bit 0 =
// 2^-266) after `win` (a 128-bit sum whose bit 0 is bit q of the limbs) has
// been added and carries propagated, rounded to the nearest double. One
// thread; limb counters are < 2^63, so no addition here overflows.
__device__ double limbs_to_double(unsigned long long *limb, U128 win, int q)
{
    const uint32_t w[4] = {static_cast<uint32_t>(win.lo), static_cast<uint32_t>(win.lo >> 32),
                           static_cast<uint32_t>(win.hi), static_cast<uint32_t>(win.hi >> 32)};
    const int l0 = q >> 5, b = q & 31;
    unsigned long long prev = 0;
    for (int i = 0; i < 5; ++i) {
        const unsigned long long cur = i < 4 ? static_cast<unsigned long long>(w[i]) << b : 0ull;
        limb[l0 + i] += (cur & 0xFFFFFFFFull) + (prev >> 32);
        prev = cur;
    }
    unsigned long long carry = 0;
    for (int i = 0; i < kRmsLimbs; ++i) {
        const unsigned long long x = limb[i] + carry;
        limb[i] = x & 0xFFFFFFFFull;
        carry = x >> 32;
    }
    int top = kRmsLimbs - 1;
    while (top > 0 && limb[top] == 0) --top;
    if (limb[top] == 0) return 0.0;
    const unsigned long long hi = limb[top], mid = top >= 1 ? limb[top - 1] : 0ull,
                             low = top >= 2 ? limb[top - 2] : 0ull;
    const int lz = __clz(static_cast<int>(hi));
    const unsigned long long wv = (hi << 32) | mid;
    unsigned long long bits = (wv << lz) | (lz ? (low >> (32 - lz)) : 0ull);
    bool sticky = ((low << lz) & 0xFFFFFFFFull) != 0;
    for (int i = 0; i + 2 < top; ++i) sticky |= limb[i] != 0;
    if (sticky) bits |= 1ull;               // below the rounding point of the 64 leading bits
    const double d = __ull2double_rn(bits);
    const int n = 32 * top - lz - 298;      // bits * 2^n is the value (n in [-329, 246])
    return d * __longlong_as_double(static_cast<long long>(1023 + n) << 52);
}

// The 16-byte vectors a thread holds: chunk c, slot j is vector (c VPT + j) T + tid.
template <int VPT>
__device__ __forceinline__ void load_chunk(uint4 (&v)[VPT], const uint16_t *xrow, int c, int T, int tid, int nvec)
{
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int idx = (c * VPT + j) * T + tid;
        v[j] = idx < nvec ? ld_nc_v4(xrow + static_cast<int64_t>(idx) * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// The squares of the elements with E < e_lo (every element when e_lo > 255)
// among chunk c of this thread's vectors, reloaded from memory (this path is
// rare): the 128-bit sum of those inside its window, the others added into the
// limbs. Returns the sum and whether any square went to the limbs.
struct GeneralSum {
    U128 acc;
    bool dropped;
};

__device__ __noinline__ GeneralSum general_squares(const uint16_t *xrow, int c, int vpt, int T, int tid, int nvec,
                                                   int e_lo, int emax, unsigned long long *limb)
{
    const int base = kRmsHeadroom - 2 * emax;
    GeneralSum g{{0ull, 0ull}, false};
    for (int j = 0; j < vpt; ++j) {
        const int idx = (c * vpt + j) * T + tid;
        if (idx >= nvec) break;
        const uint4 v = ld_nc_v4(xrow + static_cast<int64_t>(idx) * 8);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t h = (wv[t >> 1] >> ((t & 1) * 16)) & 0xFFFFu;
            const uint32_t E = (h >> 7) & 0xFFu;
            if ((h & 0x7FFFu) == 0 || static_cast<int>(E) >= e_lo) continue;
            const uint32_t m = E ? ((h & 0x7Fu) | 0x80u) : (h & 0x7Fu);
            const int e = E ? static_cast<int>(E) : 1;
            const int sh = 2 * e + base;
            if (sh >= 0) {
                unsigned long long lo, hi;
                square_term(m, sh, lo, hi);
                add128(g.acc, lo, hi);
            } else {
                const int p = 2 * e - 2;   // bit of m^2 in the limbs
                const unsigned long long x = static_cast<unsigned long long>(m * m) << (p & 31);
                atomicAdd(limb + (p >> 5), x & 0xFFFFFFFFull);
                if (x >> 32) atomicAdd(limb + (p >> 5) + 1, x >> 32);
                g.dropped = true;
            }
        }
    }
    return g;
}

// Launch bounds per vectors-per-thread: up to 16 vectors use at most 256
// threads (rms_shape), so the register cap is set by the CTAs wanted per SM.
template <int VPT>
struct RmsBounds {
    static constexpr int threads = VPT == 16 ? kRmsMaxThreads : 256;
    static constexpr int blocks = VPT <= 4 ? 4 : (VPT == 8 ? 3 : 1);
};

template <int VPT>
__global__ void __launch_bounds__(RmsBounds<VPT>::threads, RmsBounds<VPT>::blocks)
    rmsnorm_mx_quant_kernel(const uint16_t *__restrict__ X, int M, int K, int64_t ldx, const uint16_t *__restrict__ w,
                            float eps, uint8_t *__restrict__ Aq, int64_t ldq, uint8_t *__restrict__ sf,
                            float *__restrict__ rstd, double *__restrict__ sumsq)
{
    __shared__ uint32_t s_max[kRmsMaxThreads / 32];
    __shared__ unsigned long long s_lo[kRmsMaxThreads / 32], s_hi[kRmsMaxThreads / 32];
    __shared__ unsigned long long s_limb[kRmsLimbs];
    __shared__ float s_r;
    const int T = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = T >> 5;
    const int nvec = K / 8;                 // 16-byte vectors per row
    const int cblocks = (K / 32 + 3) / 4;   // scale words per row
    const int nchunk = (nvec + VPT * T - 1) / (VPT * T);
    const int64_t rows = (static_cast<int64_t>(M) + 127) / 128 * 128;
    uint4 v[VPT];

    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        uint8_t *sfrow = sf + (static_cast<size_t>(r >> 7) * cblocks) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
        if (r >= M) {   // a padding row of the blocked layout: its scale words only
            for (int i = tid; i < cblocks; i += T)
                *reinterpret_cast<uint32_t *>(sfrow + static_cast<size_t>(i) * 512) = 0x7F7F7F7Fu;
            continue;
        }
        const uint16_t *xrow = X + r * ldx;
        if (nchunk == 1) load_chunk<VPT>(v, xrow, 0, T, tid, nvec);

        // pass 1: the largest magnitude (bf16 magnitudes order as integers)
        uint32_t mx2 = 0;
        for (int c = 0; c < nchunk; ++c) {
            if (nchunk > 1) load_chunk<VPT>(v, xrow, c, T, tid, nvec);
#pragma unroll
            for (int j = 0; j < VPT; ++j) mx2 = umax16x2(mx2, max_abs_pair8(v[j]));
        }
        uint32_t mm = __reduce_max_sync(0xffffffffu, max(mx2 & 0xFFFFu, mx2 >> 16));
        if (lane == 0) s_max[warp] = mm;
        if (tid < kRmsLimbs) s_limb[tid] = 0;
        __syncthreads();
        mm = 0;
        for (int i = 0; i < nwarps; ++i) mm = max(mm, s_max[i]);
        // its exponent field (1 for subnormals, 0 for an all-zero row)
        const int emax = mm ? max(static_cast<int>(mm >> 7), 1) : 0;

        // pass 2: the exact sum of squares
        U128 acc{0ull, 0ull};
        bool dropped = false;
        if (emax > kRmsFastSpan) {
            const int e_lo = emax - kRmsFastSpan;
            const uint32_t thr = static_cast<uint32_t>(e_lo) << 7;   // magnitudes below take the slow paths
            for (int c = 0; c < nchunk; ++c) {
                if (nchunk > 1) load_chunk<VPT>(v, xrow, c, T, tid, nvec);
                unsigned long long fast = 0;
                uint32_t low2 = 0xFFFFFFFFu;   // per half: smallest nonzero magnitude - 1 (zero -> 0xFFFF)
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t x = wv[i];
                        const uint32_t a = x & 0x7FFF7FFFu;
                        low2 = umin16x2(low2, (a + 0x7FFF7FFFu) ^ 0x80008000u);
                        const uint32_t u0 = shl_sat((x & 0x7Fu) | 0x80u, static_cast<int>((x >> 7) & 0xFFu) - e_lo);
                        const uint32_t u1 = shl_sat(((x >> 16) & 0x7Fu) | 0x80u,
                                                    static_cast<int>((x >> 23) & 0xFFu) - e_lo);
                        fast = mad_wide(u0, u0, fast);
                        fast = mad_wide(u1, u1, fast);
                    }
                }
                // u^2 = m^2 2^(2E - 2 Emax + 32): 2^48 units of the 128-bit sum
                add128(acc, fast << 48, fast >> 16);
                if (min(low2 & 0xFFFFu, low2 >> 16) < thr - 1) {
                    const GeneralSum g = general_squares(xrow, c, VPT, T, tid, nvec, e_lo, emax, s_limb);
                    add128(acc, g.acc.lo, g.acc.hi);
                    dropped |= g.dropped;
                }
            }
        } else if (emax > 0) {
            // the whole row lies below 2^-110: every square takes the 128-bit path
            for (int c = 0; c < nchunk; ++c) {
                const GeneralSum g = general_squares(xrow, c, VPT, T, tid, nvec, 1 << 30, emax, s_limb);
                add128(acc, g.acc.lo, g.acc.hi);
                dropped |= g.dropped;
            }
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
        const int any_dropped = __syncthreads_or(dropped);
        if (tid == 0) {
            U128 t{0ull, 0ull};
            for (int i = 0; i < nwarps; ++i) add128(t, s_lo[i], s_hi[i]);
            // sum = t * 2^(2 Emax - 268 - headroom) (+ the limbs when any square fell below)
            const double ss = any_dropped ? limbs_to_double(s_limb, t, 2 * emax - 268 - kRmsHeadroom + 266)
                                          : u128_to_double(t, 2 * emax - 268 - kRmsHeadroom);
            const double ms = ss / static_cast<double>(K) + static_cast<double>(eps);
            const double r64 = ms > 0.0 ? 1.0 / sqrt(ms) : 0.0;
            const float r32 = __double2float_rn(r64);
            s_r = r32;
            if (rstd) rstd[r] = r32;
            if (sumsq) sumsq[r] = ss;
        }
        __syncthreads();
        const float rs = s_r;

        // pass 3: y, its MXFP4 codes and scale words
        uint8_t *qrow = Aq + r * ldq;
        for (int c = 0; c < nchunk; ++c) {
            if (nchunk > 1) load_chunk<VPT>(v, xrow, c, T, tid, nvec);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int idx = (c * VPT + j) * T + tid;   // this lane's vector; 4 lanes per block
                const bool ok = idx < nvec;
                float y[8];
                float amax = 0.0f;
                if (ok) {
                    const uint4 wv = __ldg(reinterpret_cast<const uint4 *>(w) + idx);
                    const uint32_t xa[4] = {v[j].x, v[j].y, v[j].z, v[j].w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        y[2 * i] = __fmul_rn(__fmul_rn(__uint_as_float(xa[i] << 16), rs), __uint_as_float(wa[i] << 16));
                        y[2 * i + 1] = __fmul_rn(__fmul_rn(__uint_as_float(xa[i] & 0xFFFF0000u), rs),
                                                 __uint_as_float(wa[i] & 0xFFFF0000u));
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(y[i]));
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[i] = 0.0f;
                }
                uint32_t ab = __float_as_uint(amax);
                ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, 1));
                ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, 2));
                // OCP MX: e = floor(log2 amax) - 2, clamped below at -127 (byte 0)
                const uint32_t E = ab >> 23;
                const uint32_t sbyte = E >= 2 ? E - 2 : 0;
                const float mult = __uint_as_float((254u - sbyte) << 23);   // 2^-e, exact
                const uint32_t codes = e2m1x8_rn_sat(y[0] * mult, y[1] * mult, y[2] * mult, y[3] * mult,
                                                     y[4] * mult, y[5] * mult, y[6] * mult, y[7] * mult);
                if (ok) *reinterpret_cast<uint32_t *>(qrow + static_cast<int64_t>(idx) * 4) = codes;
                const uint32_t mine = ok ? sbyte : 0x7Fu;
                const int b16 = lane & 16;
                uint32_t word = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) word |= __shfl_sync(0xffffffffu, mine, b16 + i * 4) << (8 * i);
                const int widx = idx >> 4;   // lanes 0 and 16 hold a multiple of 16
                if ((lane & 15) == 0 && widx < cblocks)
                    *reinterpret_cast<uint32_t *>(sfrow + static_cast<size_t>(widx) * 512) = word;
            }
        }
        // No barrier is needed before the next row: its writes of s_max, s_limb,
        // s_lo/s_hi and s_r each follow a barrier that every read of this row's
        // values precedes.
    }
}

// Vectors per thread and threads per CTA for rows of nvec vectors: about 128
// threads holding up to 16 vectors each; rows longer than 16 * 512 vectors
// are taken in chunks of that size.
void rms_shape(int nvec, int &vpt, int &threads)
{
    vpt = 1;
    while (vpt < 16 && vpt * 2 * 128 <= nvec) vpt *= 2;
    const int t = (nvec + vpt - 1) / vpt;
    threads = min(kRmsMaxThreads, max(32, (t + 31) / 32 * 32));
}

template <int VPT>
cudaError_t launch_vpt(const void *X, int M, int K, int64_t ldx, const void *w, float eps, void *Aq, int64_t ldq,
                       void *sf, float *rstd, double *sumsq, int threads, int num_sms, cudaStream_t stream)
{
    static std::atomic<int> occ_cache[kRmsMaxThreads / 32 + 1];
    std::atomic<int> &slot = occ_cache[threads / 32];
    int occ = slot.load(std::memory_order_relaxed);
    if (occ == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, rmsnorm_mx_quant_kernel<VPT>, threads, 0);
        if (e != cudaSuccess) return e;
        occ = max(occ, 1);
        slot.store(occ, std::memory_order_relaxed);
    }
    const int64_t rows = (static_cast<int64_t>(M) + 127) / 128 * 128;
    const int64_t blocks = min(rows, static_cast<int64_t>(num_sms) * occ);
    rmsnorm_mx_quant_kernel<VPT><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<const uint16_t *>(X), M, K, ldx, static_cast<const uint16_t *>(w), eps,
        static_cast<uint8_t *>(Aq), ldq, static_cast<uint8_t *>(sf), rstd, sumsq);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm_mx_quant(const void *X, int64_t M, int64_t K, int64_t ldx, const void *w, float eps,
                                    void *Aq, int64_t ldq, void *sf, float *rstd, double *sumsq, int num_sms,
                                    cudaStream_t stream)
{
    if (M < 1 || K < 1 || M > 0x7fffffff || K > 0x7fffffff) return cudaErrorInvalidValue;
    int vpt = 1, threads = 32;
    rms_shape(static_cast<int>(K / 8), vpt, threads);
    const int m = static_cast<int>(M), k = static_cast<int>(K);
    switch (vpt) {
    case 1: return launch_vpt<1>(X, m, k, ldx, w, eps, Aq, ldq, sf, rstd, sumsq, threads, num_sms, stream);
    case 2: return launch_vpt<2>(X, m, k, ldx, w, eps, Aq, ldq, sf, rstd, sumsq, threads, num_sms, stream);
    case 4: return launch_vpt<4>(X, m, k, ldx, w, eps, Aq, ldq, sf, rstd, sumsq, threads, num_sms, stream);
    case 8: return launch_vpt<8>(X, m, k, ldx, w, eps, Aq, ldq, sf, rstd, sumsq, threads, num_sms, stream);
    default: return launch_vpt<16>(X, m, k, ldx, w, eps, Aq, ldq, sf, rstd, sumsq, threads, num_sms, stream);
    }
}

}  // namespace mxfp4
