/*
 * Oracle: number formats (E2M1, E4M3, BF16, E8M0 exponents) and the token
 * scale.  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Each encoder is written as "enumerate the representable values and take the
 * nearest", the textbook definition of round-to-nearest, rather than with bit
 * tricks, so that it can be checked by eye.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "oracle.h"

/* E2M1 magnitudes, indexed by the 3-bit magnitude field (exponent bias 1, one
 * mantissa bit).  TE PR #3753 "Add NVFP4 EP dispatch and combine backward",
 * PR description: tokens travel as "E2M1 codes".  Reading R1: code =
 * (sign << 3) | magnitude index. */
static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double or_e2m1_value(int code)
{
    double m = kE2M1[code & 7];
    return (code & 8) ? -m : m;
}

/* Round to the nearest E2M1 magnitude; an exact tie goes to the even index
 * (the one whose mantissa bit is 0), values above 6 saturate to 6, and the
 * sign of the input (also of a zero result) is kept (reading R2, R5). */
int or_e2m1_rne(double v)
{
    int sign = signbit(v) ? 8 : 0;
    double a = fabs(v);
    if (a >= 6.0) /* saturate; also keeps huge |v| out of the distance test */
        return sign | 7;
    int best = 0;
    double best_d = fabs(a - kE2M1[0]);
    for (int i = 1; i < 8; ++i) {
        double d = fabs(a - kE2M1[i]);
        if (d < best_d || (d == best_d && (i % 2) == 0)) {
            best = i;
            best_d = d;
        }
    }
    return sign | best;
}

/* Stochastic rounding to E2M1 with a 16-bit random number r16 (reading R13):
 * with lo <= |v| < hi the neighbouring grid values and f = (|v|-lo)/(hi-lo),
 * round up to hi iff r16 + 65536 f >= 65536 (an exact comparison: 65536 f is
 * exact in double), i.e. with probability floor(65536 f)/65536 over the
 * 65536 values of r16.  Grid values never move; |v| >= 6 gives 6.  Sign
 * kept. */
int or_e2m1_sr(double v, unsigned r16)
{
    int sign = signbit(v) ? 8 : 0;
    double a = fabs(v);
    if (a >= 6.0)
        return sign | 7;
    int i = 0;
    while (i < 7 && kE2M1[i + 1] <= a)
        ++i;
    double lo = kE2M1[i], hi = kE2M1[i + 1];
    double f = (a - lo) / (hi - lo);
    int up = ((double)(r16 & 0xffffu) + f * 65536.0) >= 65536.0;
    return sign | (up ? i + 1 : i);
}

/* E4M3 ("fn" variant): bias 7, 3 mantissa bits, subnormals, no infinity, code
 * 0x7f / 0xff is NaN, largest finite value 448.  TE PR #3753, PR description:
 * "E4M3 block scales"; TE PR #3270 "EP dispatch with unfused MXFP8
 * quantization", review thread: E4M3 only. */
double or_e4m3_value(int code)
{
    int mag = code & 0x7f;
    if (mag == 0x7f)
        return NAN;
    int e = mag >> 3, m = mag & 7;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return (code & 0x80) ? -v : v;
}

/* Nearest E4M3 value, ties to the even code, |v| > 448 saturates to 448
 * ("satfinite").  The positive finite codes 0..126 are in increasing value
 * order, so a binary search finds the bracketing pair. */
int or_e4m3_rne_sat(double v)
{
    int sign = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    if (a >= 448.0)
        return sign | 126;
    int lo = 0, hi = 126; /* value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (or_e4m3_value(mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double dlo = a - or_e4m3_value(lo), dhi = or_e4m3_value(hi) - a;
    int pick;
    if (dlo < dhi)
        pick = lo;
    else if (dhi < dlo)
        pick = hi;
    else
        pick = (lo % 2 == 0) ? lo : hi;
    return sign | pick;
}

double or_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a finite value to the nearest BF16, ties to even.  The value is first
 * converted to float (exact for the values the oracle produces: they have at
 * most 24 significant bits and are at least 2^-149), then the low 16 bits of
 * the binary32 pattern are rounded away with ties to even. */
uint16_t or_bf16_rne(double v)
{
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* Token scale exponent (reading R3): the smallest integer k >= -126 with
 * amax <= 2688 * 2^k, where 2688 = 6 * 448 is the largest value a block can
 * hold (E2M1 max times E4M3 max).  TE PR #3753, PR description: each token
 * carries one FP32 scale, restricted to powers of two. */
int or_token_scale_exp(double amax)
{
    int k = -126;
    while (amax > 2688.0 * ldexp(1.0, k))
        ++k;
    return k;
}

/* MXFP8 block exponent (reading R14): the smallest integer e in [-127, 127]
 * with bmax <= 448 * 2^e, so that no element saturates.  TE PR #3270, sequence
 * diagram: the data is quantised to E4M3 with E8M0 block scales. */
int or_mx_scale_exp(double bmax)
{
    int e = -127;
    while (e < 127 && bmax > 448.0 * ldexp(1.0, e))
        ++e;
    return e;
}

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 * as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplications, the key
 * advanced by the Weyl constants between rounds. */
void or_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)M0 * c0;
        uint64_t p1 = (uint64_t)M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += W0;
        k1 += W1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 16 bits of x in reverse order (bit 0 <-> bit 15). */
static unsigned reverse16(unsigned x)
{
    unsigned r = 0;
    for (int b = 0; b < 16; ++b)
        if (x & (1u << b))
            r |= 1u << (15 - b);
    return r;
}

/* The 16-bit random number of element idx in a given stream (reading R13).
 * One Philox call covers 16 consecutive elements: counter = (lo32(n),
 * hi32(n), stream, 0) with n = idx / 16, key = (lo32(seed), hi32(seed)).
 * Element idx uses output word q = (idx / 4) mod 4; with b0..b3 the bytes of
 * that word (b0 the least significant), A = b2 * 256 + b0 and
 * B = b3 * 256 + b1, the four elements of the word take, for j = idx mod 4:
 * j = 0: A, j = 1: A bit-reversed, j = 2: B, j = 3: B bit-reversed. */
unsigned or_sr_u16(uint64_t seed, uint32_t stream, uint64_t idx)
{
    uint64_t n = idx / 16;
    uint32_t ctr[4] = {(uint32_t)n, (uint32_t)(n >> 32), stream, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    or_philox4x32_10(ctr, key, out);
    uint32_t w = out[(idx / 4) % 4];
    unsigned b0 = w & 0xffu, b1 = (w >> 8) & 0xffu, b2 = (w >> 16) & 0xffu, b3 = w >> 24;
    unsigned A = (b2 << 8) | b0, B = (b3 << 8) | b1;
    switch (idx % 4) {
    case 0: return A;
    case 1: return reverse16(A);
    case 2: return B;
    default: return reverse16(B);
    }
}

/* 16-point random Hadamard transform (reading R9): u_i = sigma_i * d_i / 4,
 * exact in FP32 for decoded NVFP4 values, then the in-place Walsh-Hadamard
 * butterflies for len = 1, 2, 4, 8, each sum and difference rounded to FP32.
 * sigma_i = -1 where bit i of sign_mask is set.  y = 1/4 * H16 * diag(sigma)
 * * d, with H16 the Sylvester Hadamard matrix, H[i][l] = (-1)^popcount(i & l).
 * The 1/4 = 1/sqrt(16) normalisation is the one under which "post-RHT amax
 * <= 4x rowwise amax" holds (TE PR #3755 "Optionally derive FC1 dy NVFP4
 * amaxes from the dGLU epilogue", PR description). */
void or_rht16_f32(const float d[16], uint16_t sign_mask, float y[16])
{
    float u[16];
    for (int i = 0; i < 16; ++i) {
        float s = ((sign_mask >> i) & 1u) ? -0.25f : 0.25f;
        u[i] = s * d[i];
    }
    for (int len = 1; len < 16; len *= 2) {
        for (int a = 0; a < 16; ++a) {
            if (a & len)
                continue;
            float p = u[a], q = u[a + len];
            u[a] = p + q;
            u[a + len] = p - q;
        }
    }
    for (int i = 0; i < 16; ++i)
        y[i] = u[i];
}

/* Batch forms of the scalar encoders, for exhaustive checks. */
void or_e2m1_rne_batch(const double *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint8_t)or_e2m1_rne(v[i]);
}

void or_e2m1_sr_batch(const double *v, const uint16_t *r16, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint8_t)or_e2m1_sr(v[i], r16[i]);
}

void or_e4m3_rne_sat_batch(const double *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint8_t)or_e4m3_rne_sat(v[i]);
}

void or_sr_u16s(uint64_t seed, uint32_t stream, uint64_t idx0, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint16_t)or_sr_u16(seed, stream, idx0 + (uint64_t)i);
}
