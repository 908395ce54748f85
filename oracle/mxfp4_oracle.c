/*
 * CPU oracle for block-scaled FP4 quantization and GEMM (MXFP4 and NVFP4).
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this file's library. The product
 * path (the CUDA library) never calls into it and shares no code with it.
 *
 * Plain, slow, single-threaded loops in double precision. Every function
 * names the passage of the source pages it restates:
 *   [MM-517169]  kernelbot-amd-mxfp4-mm-517169 (fused quant + GEMM submission)
 *   [MM-683203]  kernelbot-amd-mxfp4-mm-683203 (quant + shuffle + hsaco GEMM)
 *   [NV-496271]  kernelbot-nvfp4-group-gemm-496271 (NVFP4 grouped GEMM)
 * The rounding rule is the OCP MX rule (shared exponent = floor(log2 amax) - 2,
 * E2M1 round-half-to-even saturating at +-6, amax = 0 -> scale 2^-127). The
 * pages' own scale rules differ from it; they are kept here only as
 * `orc_mx_block_variant` so a test can show that they differ.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- codecs -- */

/* E2M1 magnitudes in code order 0..7: [MM-517169] module docstring ("FP4 E2M1
 * representable magnitudes") and the level comment above _quant_to_fp4. */
static const double kE2M1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Decode one 4-bit E2M1 code. Bit 3 is the sign ([MM-517169] _fused_quant_gemm_kernel,
 * comment "0b0xxx = positive, 0b1xxx = negative"); code 0x8 is -0. */
double orc_e2m1_decode(int code)
{
    double m = kE2M1Mag[code & 7];
    return (code & 8) ? -m : m;
}

/* Encode a real value to E2M1: round to the nearest level, a tie goes to the
 * level with the even code index (round-half-to-even on the 1-bit mantissa),
 * magnitudes >= 6 saturate to 6, and the IEEE sign is kept even when the
 * magnitude rounds to 0 (so -0 and tiny negatives give 0x8). */
int orc_e2m1_encode(double v)
{
    int sign = signbit(v) ? 8 : 0;
    double a = fabs(v);
    int idx;
    if (a >= 6.0) {
        idx = 7;
    } else {
        int i = 0;
        while (i < 7 && kE2M1Mag[i + 1] <= a) i++;
        /* kE2M1Mag[i] <= a < kE2M1Mag[i+1] */
        double mid = 0.5 * (kE2M1Mag[i] + kE2M1Mag[i + 1]); /* exact */
        if (a < mid)
            idx = i;
        else if (a > mid)
            idx = i + 1;
        else
            idx = (i % 2 == 0) ? i : i + 1;
    }
    return sign | idx;
}

/* E8M0 byte b encodes 2^(b-127); 127 is 1.0 ([MM-683203] key trick 2). 0xFF is
 * NaN and is never produced here. */
double orc_e8m0_decode(int b)
{
    if (b == 0xFF) return NAN;
    return ldexp(1.0, b - 127);
}

/* FP8 E4M3 (the "fn" variant: bias 7, subnormals, no infinities, S.1111.111 =
 * NaN) used as the NVFP4 per-16 scale ([NV-496271] VEC_SIZE constant and the
 * float8_e4m3fn scale tensors of _prepare_scale_for_tma). */
double orc_e4m3_decode(int b)
{
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round a non-negative finite value to E4M3, nearest-even, saturating at the
 * largest finite magnitude 448 (byte 0x7E). Used to form NVFP4 scales. */
int orc_e4m3_encode_satfinite(double f)
{
    if (!(f > 0.0)) return 0;
    if (f >= 448.0) return 0x7E;
    int e = ilogb(f);
    if (e < -6) {
        /* subnormal range: multiples of 2^-9 */
        double k = nearbyint(ldexp(f, 9));
        return (int)k; /* k == 8 is byte 0x08 == 2^-6, the smallest normal */
    }
    double k = nearbyint(ldexp(f, 3 - e)); /* in [8, 16] */
    if (k >= 16.0) {
        k = 8.0;
        e += 1;
    }
    int b = ((e + 7) << 3) | ((int)k - 8);
    if (b > 0x7E) b = 0x7E;
    return b;
}

/* bf16 bit pattern -> double (exact). */
double orc_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static float bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------ scale layout ----- */

/* Byte offset of element (r, c) of a logical [R, C] scale matrix stored in the
 * 128x4 blocked layout. [NV-496271] _prepare_scale_for_tma docstring: the
 * reordered tensor is indexed [i%32, (i%128)/32, i/128, j%4, j/4] and is then
 * permuted to the contiguous order [i/128, j/4, i%32, (i%128)/32, j%4], i.e.
 * 512-byte blocks of 128 rows x 4 columns. */
int64_t orc_sf_offset(int64_t r, int64_t c, int64_t C)
{
    int64_t cblocks = (C + 3) / 4;
    return ((r / 128) * cblocks + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

/* Size in bytes of a blocked scale buffer for a logical [R, C] matrix. */
int64_t orc_sf_bytes(int64_t R, int64_t C)
{
    return ((R + 127) / 128) * ((C + 3) / 4) * 512;
}

/* Pack a linear row-major [R, C] scale matrix into the blocked layout; cells
 * that no (r, c) maps to are set to `pad` ([MM-683203] key trick 2: padding
 * holds 127 so a padded cell acts as scale 1.0). */
void orc_sf_pack(const uint8_t *lin, int64_t R, int64_t C, uint8_t pad, uint8_t *blk)
{
    memset(blk, pad, (size_t)orc_sf_bytes(R, C));
    for (int64_t r = 0; r < R; r++)
        for (int64_t c = 0; c < C; c++) blk[orc_sf_offset(r, c, C)] = lin[r * C + c];
}

void orc_sf_unpack(const uint8_t *blk, int64_t R, int64_t C, uint8_t *lin)
{
    for (int64_t r = 0; r < R; r++)
        for (int64_t c = 0; c < C; c++) lin[r * C + c] = blk[orc_sf_offset(r, c, C)];
}

/* ---------------------------------------------------- MXFP4 quantize ----- */

/* OCP MX shared exponent of one block: floor(log2 amax) - 2, clamped to
 * [-127, 127]; amax = 0 gives -127 (scale 2^-127). ilogb is exact on the
 * double image of any bf16, subnormals included. */
int orc_mx_shared_exponent(double amax)
{
    if (amax == 0.0) return -127;
    int e = ilogb(amax) - 2;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* Quantize one row-block of 32 values (given as doubles that are exactly bf16
 * values) under the OCP rule: scale byte into *sb, codes into code[32].
 * [MM-517169] module docstring steps "abs-max per 32, E8M0 scale, pack to
 * fp4x2"; [MM-683203] _quant_shuffled (the same per-32 quant op). */
void orc_mx_quantize_block(const double *x, int *sb, int *code)
{
    double amax = 0.0;
    for (int i = 0; i < 32; i++)
        if (fabs(x[i]) > amax) amax = fabs(x[i]);
    int e = orc_mx_shared_exponent(amax);
    *sb = e + 127;
    for (int i = 0; i < 32; i++) code[i] = orc_e2m1_encode(ldexp(x[i], -e)); /* exact scaling */
}

/* The pages' differing scale rules, for comparison only.
 *   variant 1: [MM-517169] _e8m0_scale, scale = 2^floor(log2(amax/6 + 1e-30)),
 *              elements by _quant_to_fp4 (clamp to [0,6], strict-< thresholds).
 *   variant 2: [MM-517169] module docstring, scale = 2^round(log2(amax/6)),
 *              same element rule.
 * Writes the scale's base-2 exponent to *e_out and the codes (sign bit 3). */
void orc_mx_block_variant(const double *x, int variant, int *e_out, int *code)
{
    double amax = 0.0;
    for (int i = 0; i < 32; i++)
        if (fabs(x[i]) > amax) amax = fabs(x[i]);
    int e;
    if (variant == 1)
        e = (int)floor(log2(amax / 6.0 + 1e-30));
    else
        e = (amax > 0.0) ? (int)nearbyint(log2(amax / 6.0)) : -127;
    *e_out = e;
    static const double th[7] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0};
    for (int i = 0; i < 32; i++) {
        double s = fabs(x[i]) / ldexp(1.0, e);
        if (s > 6.0) s = 6.0;
        int q = 7;
        for (int t = 0; t < 7; t++)
            if (s < th[t]) {
                q = t;
                break;
            }
        code[i] = (signbit(x[i]) ? 8 : 0) | q;
    }
}

/* Quantize a bf16 matrix A [M, K] (row stride lda elements) to MXFP4:
 *   q  : [M, K/2] bytes, row stride ldq bytes, low nibble = even k
 *        ([MM-517169] docstring "low nibble = first, high nibble = second");
 *   sf : blocked [M, K/32] E8M0 scale buffer, pad cells 0x7F.
 * Returns 0, or -1 if K is not a multiple of 32. */
int orc_mx_quantize(const uint16_t *A, int64_t M, int64_t K, int64_t lda, uint8_t *q, int64_t ldq,
                    uint8_t *sf)
{
    if (K % 32 != 0) return -1;
    int64_t C = K / 32;
    memset(sf, 0x7F, (size_t)orc_sf_bytes(M, C));
    double x[32];
    int code[32], sb;
    for (int64_t r = 0; r < M; r++) {
        for (int64_t b = 0; b < C; b++) {
            for (int i = 0; i < 32; i++) x[i] = orc_bf16_to_double(A[r * lda + b * 32 + i]);
            orc_mx_quantize_block(x, &sb, code);
            sf[orc_sf_offset(r, b, C)] = (uint8_t)sb;
            for (int j = 0; j < 16; j++)
                q[r * ldq + b * 16 + j] = (uint8_t)((code[2 * j] & 15) | ((code[2 * j + 1] & 15) << 4));
        }
    }
    return 0;
}

/* ---------------------------------------------------- NVFP4 quantize ----- */

/* Quantize a bf16 matrix to NVFP4 (E2M1 codes, one E4M3 scale per 16 along K,
 * blocked layout, pad 0). The pages consume NVFP4 operands that an external
 * generator produced ([NV-496271] custom_kernel inputs) and do not state its
 * rule; the reading used here, in fp32 as a GPU computes it:
 *   s = E4M3_satfinite_RNE(fp32(amax) / 6),  q_i = E2M1_RNE_sat(fp32(x_i) / s),
 * and s == 0 gives all-zero magnitudes (signs kept). Returns 0, or -1 if K % 16. */
int orc_nv_quantize(const uint16_t *A, int64_t M, int64_t K, int64_t lda, uint8_t *q, int64_t ldq,
                    uint8_t *sf)
{
    if (K % 16 != 0) return -1;
    int64_t C = K / 16;
    memset(sf, 0x00, (size_t)orc_sf_bytes(M, C));
    for (int64_t r = 0; r < M; r++) {
        for (int64_t b = 0; b < C; b++) {
            float xs[16];
            float amax = 0.0f;
            for (int i = 0; i < 16; i++) {
                xs[i] = bf16_to_float(A[r * lda + b * 16 + i]);
                if (fabsf(xs[i]) > amax) amax = fabsf(xs[i]);
            }
            volatile float ratio = amax / 6.0f; /* fp32, round-to-nearest-even */
            int sb = orc_e4m3_encode_satfinite((double)ratio);
            float s = (float)orc_e4m3_decode(sb);
            sf[orc_sf_offset(r, b, C)] = (uint8_t)sb;
            int code[16];
            for (int i = 0; i < 16; i++) {
                if (s == 0.0f) {
                    code[i] = signbit(xs[i]) ? 8 : 0;
                } else {
                    volatile float v = xs[i] / s; /* fp32 division */
                    code[i] = orc_e2m1_encode((double)v);
                }
            }
            for (int j = 0; j < 8; j++)
                q[r * ldq + b * 8 + j] = (uint8_t)((code[2 * j] & 15) | ((code[2 * j + 1] & 15) << 4));
        }
    }
    return 0;
}

/* ---------------------------------------------------------- dequant ------ */

/* Dequantize an FP4 matrix [R, K] (packed bytes, row stride ld) with blocked
 * scales of vector length vec (32: E8M0, 16: E4M3) into doubles [R, K]. */
void orc_dequant(const uint8_t *q, int64_t ld, const uint8_t *sf, int64_t R, int64_t K, int vec,
                 double *out)
{
    int64_t C = K / vec;
    for (int64_t r = 0; r < R; r++)
        for (int64_t k = 0; k < K; k++) {
            uint8_t byte = q[r * ld + k / 2];
            int code = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
            uint8_t sb = sf[orc_sf_offset(r, k / vec, C)];
            double s = (vec == 32) ? orc_e8m0_decode(sb) : orc_e4m3_decode(sb);
            out[r * K + k] = orc_e2m1_decode(code) * s;
        }
}

/* ------------------------------------------------------------ GEMM ------ */

/* One output element of the block-scaled FP4 GEMM by its definition:
 *   C[m,n] = sum_k (qa[m,k] * sa[m,k/vec]) * (qb[n,k] * sb[n,k/vec])
 * accumulated in double, and S[m,n] = sum_k |a_k b_k| for the tolerance.
 * [MM-517169] docstring steps 3-4 (dot against B, fp32 accumulate, bf16 C);
 * [NV-496271] nvfp4_gemm_kernel (dot_scaled of e2m1 with per-16 scales). */
static void gemm_elem(const uint8_t *qa, int64_t ldqa, const uint8_t *sfa, const uint8_t *qb,
                      int64_t ldqb, const uint8_t *sfb, int64_t K, int vec, int64_t m, int64_t n,
                      double *c, double *s)
{
    int64_t C = K / vec;
    double acc = 0.0, aabs = 0.0;
    for (int64_t k = 0; k < K; k++) {
        uint8_t ba = qa[m * ldqa + k / 2], bb = qb[n * ldqb + k / 2];
        int ca = (k % 2 == 0) ? (ba & 15) : (ba >> 4);
        int cb = (k % 2 == 0) ? (bb & 15) : (bb >> 4);
        uint8_t ea = sfa[orc_sf_offset(m, k / vec, C)];
        uint8_t eb = sfb[orc_sf_offset(n, k / vec, C)];
        double sa = (vec == 32) ? orc_e8m0_decode(ea) : orc_e4m3_decode(ea);
        double sbv = (vec == 32) ? orc_e8m0_decode(eb) : orc_e4m3_decode(eb);
        double p = (orc_e2m1_decode(ca) * sa) * (orc_e2m1_decode(cb) * sbv);
        acc += p;
        aabs += fabs(p);
    }
    *c = acc;
    *s = aabs;
}

/* Full reference GEMM: C_ref [M, N] and S [M, N] (row-major doubles). */
void orc_gemm_full(const uint8_t *qa, int64_t ldqa, const uint8_t *sfa, const uint8_t *qb,
                   int64_t ldqb, const uint8_t *sfb, int64_t M, int64_t N, int64_t K, int vec,
                   double *cref, double *sabs)
{
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++)
            gemm_elem(qa, ldqa, sfa, qb, ldqb, sfb, K, vec, m, n, &cref[m * N + n], &sabs[m * N + n]);
}

/* Sampled reference GEMM: the same definition at npairs (rows[i], cols[i]). */
void orc_gemm_sampled(const uint8_t *qa, int64_t ldqa, const uint8_t *sfa, const uint8_t *qb,
                      int64_t ldqb, const uint8_t *sfb, int64_t K, int vec, const int64_t *rows,
                      const int64_t *cols, int64_t npairs, double *cref, double *sabs)
{
    for (int64_t i = 0; i < npairs; i++)
        gemm_elem(qa, ldqa, sfa, qb, ldqb, sfb, K, vec, rows[i], cols[i], &cref[i], &sabs[i]);
}

/* Tolerance check of the contract: |C_gpu - C_ref| <= 2^-8 * S + 1e-3 per
 * element. Returns the number of failing elements; *worst gets the largest
 * ratio |diff| / bound seen. */
int64_t orc_check_tolerance(const double *cgpu, const double *cref, const double *sabs, int64_t n,
                            double *worst)
{
    int64_t bad = 0;
    double w = 0.0;
    for (int64_t i = 0; i < n; i++) {
        double bound = ldexp(sabs[i], -8) + 1e-3;
        double d = fabs(cgpu[i] - cref[i]);
        if (!(d <= bound)) bad++;
        double r = d / bound;
        if (r > w || r != r) w = r;
    }
    *worst = w;
    return bad;
}
