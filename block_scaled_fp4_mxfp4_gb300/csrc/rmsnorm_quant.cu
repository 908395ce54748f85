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
// Sum of squares, exact for every finite input. A bf16 x is m * 2^(E - 134)
// with an 8-bit m (E the exponent field, taken as 1 for subnormals), so x^2
// is m^2 * 2^(2E - 268). Relative to the row's largest exponent field Emax:
//  * E >= Emax - 14 (nearly every element): x * 2^(148 - Emax) is an integer u
//    with |u| < 2^22, formed by one fused multiply-add with 1.5 * 2^23 (its
//    bits minus those of the constant), and u^2 is accumulated exactly by a
//    wide multiply-add into a 64-bit sum (at most 128 terms between flushes)
//    that is added into a 128-bit fixed point with 80 fractional bits below
//    2 (Emax) (< K * 2^96: no overflow for K < 2^31);
//  * elements below that window are rare; a thread whose smallest magnitude
//    lies below it finds the vectors that hold them and, one vector at a time,
//    takes the fast path's rounded square back out and adds the exact one:
//    for E >= Emax - 28 through a second such window (x * 2^(162 - Emax)),
//    for E >= Emax - 40 as m^2 shifted into the 128-bit sum, and below that
//    into a 576-bit integer in shared memory whose bit 0 is 2^-266 (the
//    smallest square), kept as 18 64-bit counters of 32-bit limbs that take
//    shared atomic adds; the 128-bit sum is then added into the limbs and
//    carries are propagated.
// Integer addition does not depend on the order, so the threads and the
// cross-warp reduction give the same exact sum S as any other order.
//
// r. ss = RN64(S) (64 leading bits of S and a sticky bit, rounded once), and
// r = RN32(RN64(1 / RN64(sqrt(RN64(RN64(ss / K) + eps))))), the fp64 sequence
// of the reading. Dependent fp64 operations take tens of cycles each on this
// GPU, so the sequence runs only when its result is not already decided: a
// float-float evaluation z of 1 / sqrt(S / K + eps) (error analysis at
// rstd_fast) lies within 2^-39 z of the fp64 sequence's value, and when no
// fp32 rounding midpoint lies within 2^-38 z of z, RN32 of the fp64 value is
// RN32(z). Otherwise (about one row in 2^14; always for K >= 2^24 or a result
// outside the normal fp32 range) the fp64 sequence runs.
#include <atomic>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mxfp4 {
namespace {

constexpr int kRmsMaxThreads = 512;
constexpr int kRmsHeadroom = 80;       // fractional bits of the 128-bit fixed-point sum
constexpr int kRmsFastSpan = 14;       // exponent fields within this of the largest take the 64-bit sum
constexpr int kRmsFastMinEmax = 21;    // 2^(148 - Emax) is a normal fp32 power of two
constexpr int kRmsLimbs = 18;          // 32-bit limbs of the exact integer (576 bits >= 522 + 31 + carries)
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr int kMagicBits = 0x4B400000;
constexpr int kRmsWStageMax = 32768;   // largest weight staged as fp32 (bytes): K <= 8192

struct U128 {
    unsigned long long lo, hi;
};

__device__ __forceinline__ void add128(U128 &a, unsigned long long lo, unsigned long long hi)
{
    const unsigned long long s = a.lo + lo;
    a.hi += hi + (s < lo ? 1ull : 0ull);
    a.lo = s;
}

__device__ __forceinline__ void sub128(U128 &a, unsigned long long lo, unsigned long long hi)
{
    const unsigned long long s = a.lo - lo;
    a.hi -= hi + (a.lo < lo ? 1ull : 0ull);
    a.lo = s;
}

// acc + a * b with a signed 64-bit product (one wide multiply-add).
__device__ __forceinline__ long long mad_wide_s(int a, int b, long long acc)
{
    long long d;
    asm("mad.wide.s32 %0, %1, %2, %3;" : "=l"(d) : "r"(a), "r"(b), "l"(acc));
    return d;
}

// Two products of fp32 pairs in one instruction (each rounded to nearest even).
__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

// The fast path's integer for one fp32 element x (scale = 2^(148 - Emax)):
// exact when x lies in its window, the rounded value otherwise.
__device__ __forceinline__ int fast_u(float x, float scale)
{
    return __float_as_int(__fmaf_rn(x, scale, kMagic)) - kMagicBits;
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

// A nonnegative value as (top + below) * 2^n: top holds its 64 leading bits
// (bit 63 set unless the value is 0) and `sticky` whether `below` (< 1) is
// nonzero.
struct Lead64 {
    unsigned long long top;
    int n;
    bool sticky;
};

// (hi * 2^64 + lo) * 2^e2.
__device__ __forceinline__ Lead64 lead_of_u128(U128 a, int e2)
{
    Lead64 r{0ull, 0, false};
    if (a.hi != 0) {
        const int lz = __clzll(static_cast<long long>(a.hi));
        r.top = lz ? ((a.hi << lz) | (a.lo >> (64 - lz))) : a.hi;
        r.sticky = (lz ? (a.lo << lz) : a.lo) != 0;
        r.n = 64 - lz + e2;
    } else if (a.lo != 0) {
        const int lz = __clzll(static_cast<long long>(a.lo));
        r.top = a.lo << lz;
        r.n = e2 - lz;
    }
    return r;
}

// The exact sum held as limbs (32-bit values in limb[0 .. kRmsLimbs), bit 0 =
// 2^-266) after `win` (a 128-bit sum whose bit 0 is bit q of the limbs) has
// been added and carries propagated. One thread; the limb counters stay
// below 2^63, so no addition here overflows.
__device__ Lead64 lead_of_limbs(unsigned long long *limb, U128 win, int q)
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
    Lead64 r{0ull, 0, false};
    int top = kRmsLimbs - 1;
    while (top > 0 && limb[top] == 0) --top;
    if (limb[top] == 0) return r;
    const unsigned long long hi = limb[top], mid = top >= 1 ? limb[top - 1] : 0ull,
                             low = top >= 2 ? limb[top - 2] : 0ull;
    const int lz = __clz(static_cast<int>(hi));
    r.top = (((hi << 32) | mid) << lz) | (lz ? (low >> (32 - lz)) : 0ull);
    bool sticky = ((low << lz) & 0xFFFFFFFFull) != 0;
    for (int i = 0; i + 2 < top; ++i) sticky |= limb[i] != 0;
    r.sticky = sticky;
    r.n = 32 * top - lz - 298;   // n in [-329, 246]
    return r;
}

// RN64 of the value: the sticky bit lies below the rounding point of the 64
// leading bits, so one conversion rounds correctly.
__device__ __forceinline__ double lead_to_double(const Lead64 &v)
{
    if (v.top == 0) return 0.0;
    const double d = __ull2double_rn(v.top | (v.sticky ? 1ull : 0ull));
    return d * __longlong_as_double(static_cast<long long>(1023 + v.n) << 52);   // exact scaling
}

// x * 2^e in two power-of-two steps (exact for normal results; a result
// below the normal range takes an absolute error under 2^-149).
__device__ __forceinline__ float scale2(float x, int e)
{
    const int e1 = max(-126, min(127, e));
    const int e2 = max(-126, min(127, e - e1));
    return __fmul_rn(__fmul_rn(x, __int_as_float((127 + e1) << 23)), __int_as_float((127 + e2) << 23));
}

// floor(log2 x) of a positive finite fp32 (subnormals included).
__device__ __forceinline__ int ilog2f(float x)
{
    const int b = __float_as_int(x);
    const int E = (b >> 23) & 0xFF;
    return E ? E - 127 : -118 - __clz(b);
}

// r = RN32(RN64(1 / RN64(sqrt(RN64(RN64(ss / K) + eps))))) for S = (top +
// below) * 2^n, ss = RN64(S), decided without fp64; false when it cannot be.
// Every operation below is an explicit rounded fp32 intrinsic, so none is
// contracted.
//
// Quantities are scaled by 2^-k2 (k2 even) so that A' = (S/K + eps) 2^-k2 lies
// in [1/2, 8); r = RN32(2^(-k2/2) rho), rho the fp64 sequence's value for A'
// (the scaling commutes with every rounding while results are normal, which
// is checked at the end). Relative error of the estimate z of A'^(-1/2):
//  * S from its 48 leading bits (s_hi + s_lo): 2^-47; ss against S: 2^-53;
//  * S'/K as q_hi + q_lo, q_hi = RN(s_hi RN(1/K)), remainder by fma (K < 2^24
//    is exact in fp32), q_lo = RN(RN(rem + s_lo) RN(1/K)): below 2^-44.4;
//  * + eps' by an exact two-sum, the low parts added with one rounding: 2^-46;
//    so A' is known to 2^-43.9, which moves A'^(-1/2) by 2^-44.9;
//  * y0 = rsqrt.approx(a_hi); h = A' y0^2 - 1 with y0^2 and a_hi p_hi split
//    exactly by fma and t_hi - 1 exact (t_hi in [1/2, 2]); |h| <= 2^-18 is
//    required (else false), so h's own rounding is below 2^-42 and its low
//    terms' below 2^-45.9;
//  * z = y0 (1 - c), c = h (1/2 - 3h/8), the series of (1 + h)^(-1/2) (its
//    truncation 5/16 |h|^3 < 2^-55): c's error below 2^-42.9 (half of h's,
//    plus its own rounding), y0 c rounded: 2^-42;
// in all below 2^-40.4; the fp64 sequence's four roundings move its value by
// at most 2.5 * 2^-53 from the exact A^(-1/2). So the fp64 value lies within
// 2^-39 z of z, and RN32 of it is RN32(z) whenever no fp32 rounding midpoint
// lies within 2^-38 z of z.
__device__ bool rstd_fast(const Lead64 &S, int K, float eps, float &r)
{
    if (K >= (1 << 24)) return false;
    const bool s0 = S.top == 0, e0 = !(eps > 0.0f);
    if (s0 && e0) {   // ss / K + eps == 0: r = 0
        r = 0.0f;
        return true;
    }
    const int kb = 31 - __clz(K);   // 2^kb <= K < 2^(kb+1)
    // S/K in [2^(ls-1), 2^(ls+1)), eps in [2^le, 2^(le+1))
    const int ls = s0 ? -100000 : S.n + 63 - kb;
    const int le = e0 ? -100000 : ilog2f(eps);
    const int k2 = max(ls, le) & ~1;
    const float Kf = static_cast<float>(K);
    const float invK = __frcp_rn(Kf);
    const float s_hi = scale2(static_cast<float>(static_cast<uint32_t>(S.top >> 40)), S.n + 40 - k2);
    const float s_lo = scale2(static_cast<float>(static_cast<uint32_t>((S.top >> 16) & 0xFFFFFFu)), S.n + 16 - k2);
    const float q_hi = __fmul_rn(s_hi, invK);
    const float rem = __fadd_rn(__fmaf_rn(-q_hi, Kf, s_hi), s_lo);
    const float q_lo = __fmul_rn(rem, invK);
    const float ep = scale2(eps, -k2);
    // two-sum of q_hi and eps', then the low parts
    const float a0 = __fadd_rn(q_hi, ep);
    const float bv = __fsub_rn(a0, q_hi);
    const float t = __fadd_rn(__fsub_rn(q_hi, __fsub_rn(a0, bv)), __fsub_rn(ep, bv));
    const float a_lo0 = __fadd_rn(t, q_lo);
    const float a_hi = __fadd_rn(a0, a_lo0);   // fast two-sum: |a0| >= |a_lo0|
    const float a_lo = __fsub_rn(a_lo0, __fsub_rn(a_hi, a0));
    const float y0 = rsqrtf(a_hi);
    const float p_hi = __fmul_rn(y0, y0);
    const float p_lo = __fmaf_rn(y0, y0, -p_hi);
    const float t_hi = __fmul_rn(a_hi, p_hi);
    const float t_lo = __fmaf_rn(a_hi, p_hi, -t_hi);
    const float small = __fmaf_rn(a_hi, p_lo, __fmaf_rn(a_lo, p_hi, t_lo));
    const float h = __fadd_rn(__fsub_rn(t_hi, 1.0f), small);
    if (!(fabsf(h) <= 0x1p-18f)) return false;
    const float c = __fmul_rn(h, __fmaf_rn(-0.375f, h, 0.5f));
    const float lo = -__fmul_rn(y0, c);
    const float cz = __fadd_rn(y0, lo);                  // RN32(z), z = y0 + lo
    const float e = __fadd_rn(__fsub_rn(y0, cz), lo);    // z - cz, exact (|y0| >= |lo|)
    const float ulp_below = __fsub_rn(cz, __int_as_float(__float_as_int(cz) - 1));
    if (!(__fadd_rn(2.0f * fabsf(e), cz * 0x1p-38f) < ulp_below)) return false;
    const int ez = ((__float_as_int(cz) >> 23) & 0xFF) - (k2 >> 1);
    if (ez < 1 || ez > 254) return false;                // r would not be a normal fp32
    r = __int_as_float(__float_as_int(cz) - ((k2 >> 1) << 23));
    return true;
}

// The fp64 sequence itself.
__device__ float rstd_fp64(double ss, int K, float eps)
{
    const double ms = ss / static_cast<double>(K) + static_cast<double>(eps);
    const double r64 = ms > 0.0 ? 1.0 / sqrt(ms) : 0.0;
    return __double2float_rn(r64);
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

// The exact squares of the nonzero elements of magnitude (bf16 bits) below
// `below` among chunk c of this thread's vectors, reloaded from memory (this
// path is rare): those within the 128-bit sum's window added to it, the
// others into the limbs (shared atomics).
struct GeneralSum {
    U128 add;
    bool dropped;
};

__device__ __noinline__ GeneralSum exact_squares(const uint16_t *xrow, int c, int vpt, int T, int tid, int nvec,
                                                 uint32_t below, int emax, unsigned long long *limb)
{
    GeneralSum g{{0ull, 0ull}, false};
    for (int j = 0; j < vpt; ++j) {
        const int idx = (c * vpt + j) * T + tid;
        if (idx >= nvec) break;
        const uint4 v = ld_nc_v4(xrow + static_cast<int64_t>(idx) * 8);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t h = (wv[t >> 1] >> ((t & 1) * 16)) & 0xFFFFu;
            if ((h & 0x7FFFu) == 0 || (h & 0x7FFFu) >= below) continue;
            const uint32_t E = (h >> 7) & 0xFFu;
            const uint32_t m = E ? ((h & 0x7Fu) | 0x80u) : (h & 0x7Fu);
            const int e = E ? static_cast<int>(E) : 1;
            const int sh = 2 * e + kRmsHeadroom - 2 * emax;
            if (sh >= 0) {
                unsigned long long lo, hi;
                square_term(m, sh, lo, hi);
                add128(g.add, lo, hi);
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

// Per half-word lane: the smallest nonzero magnitude minus one of two packed
// bf16 values (a zero maps to 0xFFFF), folded into m.
__device__ __forceinline__ uint32_t min_nonzero2(uint32_t m, uint32_t w)
{
    return umin16x2(m, ((w & 0x7FFF7FFFu) + 0x7FFF7FFFu) ^ 0x80008000u);
}

// Lane-wise bf16 minimum of |a| and |b| (the sign bit of each result lane is
// not meaningful). Finite inputs only.
__device__ __forceinline__ uint32_t absmin_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("min.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Elements of one vector below the fast window (nonzero magnitude bits below
// thr), branch-free: their fast-path integers squared into `back` (to be taken
// out again), the squares of those at or above thr2 in the second window into
// `f2`, and whether any lies below thr2.
__device__ __forceinline__ void slow_vector(const uint4 &v, uint32_t thr, uint32_t thr2, float scale, float scale2,
                                            long long &back, long long &f2, bool &deep)
{
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t h = (t & 1) ? (wv[t >> 1] >> 16) : (wv[t >> 1] & 0xFFFFu);
        const uint32_t a = h & 0x7FFFu;
        const bool oow = a - 1u < thr - 1u;   // 0 < a < thr
        const float xf = __uint_as_float(h << 16);
        const int u = oow ? fast_u(xf, scale) : 0;
        const bool in2 = a >= thr2;
        const int u2 = (oow && in2) ? fast_u(xf, scale2) : 0;
        back = mad_wide_s(u, u, back);
        f2 = mad_wide_s(u2, u2, f2);
        deep |= oow && !in2;
    }
}

// Largest CTA and register budget per vectors-per-thread: up to 6 vectors per
// thread at 64 registers, 7 or 8 at 80, up to 14 at 96, 16 at 128 (CTAs of up
// to 256 threads, 512 with 16 vectors).
template <int VPT>
struct RmsBounds {
    static constexpr int threads = VPT == 16 ? kRmsMaxThreads : 256;
    static constexpr int regs = VPT <= 6 ? 64 : (VPT <= 8 ? 80 : (VPT < 16 ? 96 : 128));
};

template <int VPT>
__global__ void __launch_bounds__(RmsBounds<VPT>::threads) __maxnreg__(RmsBounds<VPT>::regs)
    rmsnorm_mx_quant_kernel(const uint16_t *__restrict__ X, int M, int K, int64_t ldx, const uint16_t *__restrict__ w,
                            float eps, uint8_t *__restrict__ Aq, int64_t ldq, uint8_t *__restrict__ sf,
                            float *__restrict__ rstd, double *__restrict__ sumsq, int wstage)
{
    // with `wstage`: the weight as fp32, vector i's first four values at
    // s_w[i] and its last four at s_w[nvec + i] (conflict-free 16-byte reads)
    extern __shared__ float4 s_w[];
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

    if (wstage) {   // read by pass 3 only after the first row's barriers
        for (int i = tid; i < nvec; i += T) {
            const uint4 wv = __ldg(reinterpret_cast<const uint4 *>(w) + i);
            s_w[i] = make_float4(__uint_as_float(wv.x << 16), __uint_as_float(wv.x & 0xFFFF0000u),
                                 __uint_as_float(wv.y << 16), __uint_as_float(wv.y & 0xFFFF0000u));
            s_w[nvec + i] = make_float4(__uint_as_float(wv.z << 16), __uint_as_float(wv.z & 0xFFFF0000u),
                                        __uint_as_float(wv.w << 16), __uint_as_float(wv.w & 0xFFFF0000u));
        }
    }

    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        uint8_t *sfrow = sf + (static_cast<size_t>(r >> 7) * cblocks) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
        if (r >= M) {   // a padding row of the blocked layout: its scale words only
            for (int i = tid; i < cblocks; i += T)
                *reinterpret_cast<uint32_t *>(sfrow + static_cast<size_t>(i) * 512) = 0x7F7F7F7Fu;
            continue;
        }
        const uint16_t *xrow = X + r * ldx;
        if (nchunk == 1) load_chunk<VPT>(v, xrow, 0, T, tid, nvec);

        // pass 1: the largest and the smallest magnitude (a zero counts: it
        // only sends the thread to the exact check below); two chains of each
        uint32_t mxa = 0, mxb = 0, mna = 0x7FFF7FFFu, mnb = 0x7FFF7FFFu;
        for (int c = 0; c < nchunk; ++c) {
            if (nchunk > 1) load_chunk<VPT>(v, xrow, c, T, tid, nvec);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                mxa = absmax_bf16x2(mxa, v[j].x);
                mna = absmin_bf16x2(mna, v[j].x);
                mxb = absmax_bf16x2(mxb, v[j].y);
                mnb = absmin_bf16x2(mnb, v[j].y);
                mxa = absmax_bf16x2(mxa, v[j].z);
                mna = absmin_bf16x2(mna, v[j].z);
                mxb = absmax_bf16x2(mxb, v[j].w);
                mnb = absmin_bf16x2(mnb, v[j].w);
            }
        }
        const uint32_t mx2 = absmax_bf16x2(mxa, mxb), mn2 = absmin_bf16x2(mna, mnb);
        uint32_t mm = __reduce_max_sync(0xffffffffu, max(mx2 & 0x7FFFu, (mx2 >> 16) & 0x7FFFu));
        if (lane == 0) s_max[warp] = mm;
        if (tid < kRmsLimbs) s_limb[tid] = 0;
        __syncthreads();
        mm = 0;
        for (int i = 0; i < nwarps; ++i) mm = max(mm, s_max[i]);
        // its exponent field (1 for subnormals, 0 for an all-zero row)
        const int emax = mm ? max(static_cast<int>(mm >> 7), 1) : 0;

        // pass 2: the exact sum of squares (128-bit units of 2^(2 Emax - 348))
        U128 acc{0ull, 0ull};
        bool dropped = false;
        if (emax >= kRmsFastMinEmax) {
            const int e_lo = emax - kRmsFastSpan;
            const uint32_t thr = static_cast<uint32_t>(e_lo) << 7;   // magnitudes below leave the window
            const float scale = __int_as_float((148 - emax + 127) << 23);
            const bool slow = min(mn2 & 0x7FFFu, (mn2 >> 16) & 0x7FFFu) < thr;
            for (int c = 0; c < nchunk; ++c) {
                if (nchunk > 1) load_chunk<VPT>(v, xrow, c, T, tid, nvec);
                long long fa = 0, fb = 0;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int u0 = fast_u(__uint_as_float(wv[i] << 16), scale);
                        const int u1 = fast_u(__uint_as_float(wv[i] & 0xFFFF0000u), scale);
                        fa += static_cast<long long>(u0) * u0;
                        fb += static_cast<long long>(u1) * u1;
                    }
                }
                // u^2 = x^2 2^(296 - 2 Emax): 2^-52 units of the 128-bit sum
                const unsigned long long f = static_cast<unsigned long long>(fa + fb);
                add128(acc, f << 52, f >> 12);
                if (slow) {
                    // Elements below the window, found vector by vector: the fast
                    // path's rounded square comes back out; those within 14 more
                    // binades take a second window (x * 2^(162 - Emax) is an
                    // integer below 2^22 there, its square in 2^-24 units), the
                    // rest their exact square.
                    const bool second = emax >= 35;
                    const uint32_t thr2 = second ? thr - (kRmsFastSpan << 7) : thr;
                    const float scale2 = second ? __int_as_float((162 - emax + 127) << 23) : 0.0f;
                    long long f2 = 0, back = 0;
                    bool deep = false;
                    uint32_t flagged = 0;   // vectors holding such elements
#pragma unroll
                    for (int j = 0; j < VPT; ++j) {
                        const uint32_t vm = min_nonzero2(min_nonzero2(min_nonzero2(min_nonzero2(
                                                0xFFFFFFFFu, v[j].x), v[j].y), v[j].z), v[j].w);
                        flagged |= (min(vm & 0xFFFFu, vm >> 16) < thr - 1 ? 1u : 0u) << j;
                    }
                    while (flagged) {   // one copy of the element code, fed by selects
                        const int jf = __ffs(flagged) - 1;
                        flagged &= flagged - 1;
                        uint4 t = v[0];
#pragma unroll
                        for (int j = 1; j < VPT; ++j)
                            if (j == jf) t = v[j];
                        slow_vector(t, thr, thr2, scale, scale2, back, f2, deep);
                    }
                    const unsigned long long f2u = static_cast<unsigned long long>(f2);
                    const unsigned long long bu = static_cast<unsigned long long>(back);
                    add128(acc, f2u << 24, f2u >> 40);
                    sub128(acc, bu << 52, bu >> 12);
                    if (deep) {   // 28 binades or more below the largest
                        const GeneralSum g = exact_squares(xrow, c, VPT, T, tid, nvec, thr2, emax, s_limb);
                        add128(acc, g.add.lo, g.add.hi);
                        dropped |= g.dropped;
                    }
                }
            }
        } else if (emax > 0) {
            // the whole row lies below 2^-106: every square takes the 128-bit path
            for (int c = 0; c < nchunk; ++c) {
                const GeneralSum g = exact_squares(xrow, c, VPT, T, tid, nvec, 0x8000u, emax, s_limb);
                add128(acc, g.add.lo, g.add.hi);
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
            // S = t * 2^(2 Emax - 348), plus the limbs when any square fell below
            const Lead64 S = any_dropped ? lead_of_limbs(s_limb, t, 2 * emax - 82)
                                         : lead_of_u128(t, 2 * emax - 268 - kRmsHeadroom);
            float r32;
            if (!rstd_fast(S, K, eps, r32)) r32 = rstd_fp64(lead_to_double(S), K, eps);
            s_r = r32;
            if (rstd) rstd[r] = r32;
            if (sumsq) sumsq[r] = lead_to_double(S);
        }
        __syncthreads();
        const float rs = s_r;

        // pass 3: y, its MXFP4 codes and scale words
        uint8_t *qrow = Aq + r * ldq;
        const float2 rs2 = make_float2(rs, rs);
        for (int c = 0; c < nchunk; ++c) {
            if (nchunk > 1) load_chunk<VPT>(v, xrow, c, T, tid, nvec);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int idx = (c * VPT + j) * T + tid;   // this lane's vector; 4 lanes per block
                const bool ok = idx < nvec;                // else x is zero (load_chunk): y = 0, nothing stored
                const int wi = min(idx, nvec - 1);
                float wf[8];
                if (wstage) {
                    const float4 wa = s_w[wi], wb = s_w[nvec + wi];
                    wf[0] = wa.x; wf[1] = wa.y; wf[2] = wa.z; wf[3] = wa.w;
                    wf[4] = wb.x; wf[5] = wb.y; wf[6] = wb.z; wf[7] = wb.w;
                } else {
                    const uint4 wv = __ldg(reinterpret_cast<const uint4 *>(w) + wi);
                    const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        wf[2 * i] = __uint_as_float(wa[i] << 16);
                        wf[2 * i + 1] = __uint_as_float(wa[i] & 0xFFFF0000u);
                    }
                }
                const uint32_t xa[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                float2 y[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 xf = make_float2(__uint_as_float(xa[i] << 16), __uint_as_float(xa[i] & 0xFFFF0000u));
                    y[i] = mul2(mul2(xf, rs2), make_float2(wf[2 * i], wf[2 * i + 1]));
                }
                float amax = fmaxf(fmaxf(fabsf(y[0].x), fabsf(y[0].y)), fmaxf(fabsf(y[1].x), fabsf(y[1].y)));
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(y[2].x), fabsf(y[2].y)), fmaxf(fabsf(y[3].x), fabsf(y[3].y))));
                uint32_t ab = __float_as_uint(amax);
                ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, 1));
                ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, 2));
                // OCP MX: e = floor(log2 amax) - 2, clamped below at -127 (byte 0)
                const uint32_t E = ab >> 23;
                const uint32_t sbyte = E >= 2 ? E - 2 : 0;
                const float mult = __uint_as_float((254u - sbyte) << 23);   // 2^-e, exact
                const float2 m2 = make_float2(mult, mult);
#pragma unroll
                for (int i = 0; i < 4; ++i) y[i] = mul2(y[i], m2);
                const uint32_t codes =
                    e2m1x8_rn_sat(y[0].x, y[0].y, y[1].x, y[1].y, y[2].x, y[2].y, y[3].x, y[3].y);
                if (ok) *reinterpret_cast<uint32_t *>(qrow + static_cast<int64_t>(idx) * 4) = codes;
                // scale word of lanes 0-15 / 16-31: the bytes of lanes +0, +4, +8, +12
                // (blocks 0-3 of the word), gathered in two exchanges
                uint32_t pw = ok ? sbyte : 0x7Fu;
                const uint32_t o1 = __shfl_xor_sync(0xffffffffu, pw, 4);
                pw = (lane & 4) ? (o1 | (pw << 8)) : (pw | (o1 << 8));
                const uint32_t o2 = __shfl_xor_sync(0xffffffffu, pw, 8);
                const uint32_t word = (lane & 8) ? (o2 | (pw << 16)) : (pw | (o2 << 16));
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

// Vectors per thread (one of the compiled counts) and threads per CTA for rows
// of nvec vectors. With rows to spare (more than two per SM) CTAs of up to 128
// threads (up to 16 vectors each) keep more rows in flight per SM; with few
// rows, CTAs of up to 256 threads shorten each row's dependent chain. Rows
// longer than 16 vectors per thread widen the CTA up to 512 threads, then
// are taken in chunks.
constexpr int kVptChoices[] = {1, 2, 3, 4, 5, 6, 7, 8, 10, 12, 14, 16};

void rms_shape(int nvec, bool few_rows, int &vpt, int &threads)
{
    const int cta = few_rows ? 256 : 128;
    if (nvec <= 16 * cta) {
        const int need = (nvec + cta - 1) / cta;
        vpt = 16;
        for (int c : kVptChoices) {
            if (c >= need) {
                vpt = c;
                break;
            }
        }
        const int t = (nvec + vpt - 1) / vpt;
        threads = max(32, (t + 31) / 32 * 32);
    } else {
        vpt = 16;
        const int t = (nvec + 15) / 16;
        threads = min(kRmsMaxThreads, (t + 31) / 32 * 32);
    }
}

template <int VPT>
cudaError_t launch_vpt(const void *X, int M, int K, int64_t ldx, const void *w, float eps, void *Aq, int64_t ldq,
                       void *sf, float *rstd, double *sumsq, int threads, int num_sms, cudaStream_t stream)
{
    static std::atomic<int> occ_cache[kRmsMaxThreads / 32 + 1];
    std::atomic<int> &slot = occ_cache[threads / 32];
    int occ = slot.load(std::memory_order_relaxed);
    if (occ == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, rmsnorm_mx_quant_kernel<VPT>, threads,
                                                                      kRmsWStageMax);
        if (e != cudaSuccess) return e;
        occ = max(occ, 1);
        slot.store(occ, std::memory_order_relaxed);
    }
    const int64_t rows = (static_cast<int64_t>(M) + 127) / 128 * 128;
    const int64_t blocks = min(rows, static_cast<int64_t>(num_sms) * occ);
    // the weight is staged as fp32 in shared memory when it fits
    const int nvec = K / 8;
    const int wstage = nvec * 32 <= kRmsWStageMax ? 1 : 0;
    const size_t smem = wstage ? static_cast<size_t>(nvec) * 32 : 0;
    rmsnorm_mx_quant_kernel<VPT><<<static_cast<unsigned>(blocks), threads, smem, stream>>>(
        static_cast<const uint16_t *>(X), M, K, ldx, static_cast<const uint16_t *>(w), eps,
        static_cast<uint8_t *>(Aq), ldq, static_cast<uint8_t *>(sf), rstd, sumsq, wstage);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm_mx_quant(const void *X, int64_t M, int64_t K, int64_t ldx, const void *w, float eps,
                                    void *Aq, int64_t ldq, void *sf, float *rstd, double *sumsq, int num_sms,
                                    cudaStream_t stream)
{
    if (M < 1 || K < 1 || M > 0x7fffffff || K > 0x7fffffff) return cudaErrorInvalidValue;
    int vpt = 1, threads = 32;
    rms_shape(static_cast<int>(K / 8), M <= 2 * static_cast<int64_t>(num_sms), vpt, threads);
    const int m = static_cast<int>(M), k = static_cast<int>(K);
#define MXFP4_RMS_CASE(V) \
    case V: return launch_vpt<V>(X, m, k, ldx, w, eps, Aq, ldq, sf, rstd, sumsq, threads, num_sms, stream);
    switch (vpt) {
        MXFP4_RMS_CASE(1)
        MXFP4_RMS_CASE(2)
        MXFP4_RMS_CASE(3)
        MXFP4_RMS_CASE(4)
        MXFP4_RMS_CASE(5)
        MXFP4_RMS_CASE(6)
        MXFP4_RMS_CASE(7)
        MXFP4_RMS_CASE(8)
        MXFP4_RMS_CASE(10)
        MXFP4_RMS_CASE(12)
        MXFP4_RMS_CASE(14)
    default: return launch_vpt<16>(X, m, k, ldx, w, eps, Aq, ldq, sf, rstd, sumsq, threads, num_sms, stream);
    }
#undef MXFP4_RMS_CASE
}

}  // namespace mxfp4
