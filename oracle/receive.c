/*
 * Oracle: direct receive, packed rows -> grouped rowwise + columnwise-RHT
 * NVFP4 operands with per-expert amax metadata.  TEST INFRASTRUCTURE ONLY
 * (see oracle.h).
 *
 * TE PR #3753 "Add NVFP4 EP dispatch and combine backward", PR description:
 * the expert GEMM's grouped NVFP4 operands are made directly from the received
 * rows, reading them once; the rowwise operand keeps the codes the sender
 * wrote, and the RHT-transformed columnwise values are requantised with a
 * per-expert scale that comes from a bound, so neither a BF16 round trip nor an amax pass is needed.
 * TE PR #3755 "Optionally derive FC1 dy NVFP4 amaxes from the dGLU
 * epilogue", PR description: after the RHT no columnwise value exceeds four
 * times the rowwise amax.
 * TE PR #3324 "Enable NVFP4 row-scaled (per-token) backward for
 * GroupedLinear", description: row-scaled (per-token) NVFP4 operands.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "oracle.h"

static float get_f32(const uint8_t *p) { float v; memcpy(&v, p, 4); return v; }

/* Per-expert metadata (readings R11, R17):
 *   amax_row = max over the expert's rows of the trailer's A_t
 *   amax_col = fl32(4 * amax_row)                      (the 4x bound)
 *   S_enc    = min(fl32(2688 / amax_col), FLT_MAX) if amax_col > 0, else 1 */
void or_expert_amax(const uint8_t *rows, int64_t H, const int32_t *offsets,
                    int E, float *amax_row, float *amax_col, float *scale_enc)
{
    size_t S = or_row_bytes(H);
    for (int e = 0; e < E; ++e) {
        float a = 0.0f;
        for (int32_t r = offsets[e]; r < offsets[e + 1]; ++r) {
            float at = get_f32(rows + (size_t)r * S + S - 12);
            if (at > a)
                a = at;
        }
        float ac = 4.0f * a;
        float se = 1.0f;
        if (ac > 0.0f) {
            se = 2688.0f / ac;
            if (se > FLT_MAX)
                se = FLT_MAX;
        }
        amax_row[e] = a;
        amax_col[e] = ac;
        scale_enc[e] = se;
    }
}

/* Decoded value of element h of a packed row: sign * G[m] * s_b * S_t, exact
 * (at most 6 significant bits, magnitude >= 2^-136) and therefore exact in
 * float as well (reading R10). */
static float decode(const uint8_t *row, int64_t H, size_t S, int64_t h)
{
    int code = (row[h / 2] >> ((h % 2) * 4)) & 0xf;
    double sb = or_e4m3_value(row[H / 2 + h / 16]);
    double St = (double)get_f32(row + S - 16);
    return (float)(or_e2m1_value(code) * sb * St);
}

void or_nvfp4_direct_receive(const uint8_t *rows, int64_t R_cap, int64_t H,
                             const int32_t *offsets, int E,
                             const uint8_t *expert_mask,
                             uint8_t *rw_codes, uint8_t *rw_scales,
                             float *rw_row_scale, uint8_t *cw_codes,
                             uint8_t *cw_scales, float *amax_row,
                             float *amax_col, float *scale_enc,
                             int rounding, uint64_t seed,
                             uint16_t sign_mask, int64_t *report)
{
    size_t S = or_row_bytes(H);
    (void)R_cap;
    for (int i = 0; i < 4; ++i)
        report[i] = 0;
    or_expert_amax(rows, H, offsets, E, amax_row, amax_col, scale_enc);

    for (int e = 0; e < E; ++e) {
        if (expert_mask && !expert_mask[e])
            continue;
        int64_t off = offsets[e];
        int64_t n = offsets[e + 1] - offsets[e];

        /* rowwise operand (reading R8): the sender's codes and block scales,
         * the token scale as the per-row FP32 scale */
        for (int64_t r = off; r < off + n; ++r) {
            const uint8_t *row = rows + (size_t)r * S;
            memcpy(rw_codes + (size_t)r * (H / 2), row, (size_t)(H / 2));
            memcpy(rw_scales + (size_t)r * (H / 16), row + H / 2, (size_t)(H / 16));
            rw_row_scale[r] = get_f32(row + S - 16);
        }

        /* columnwise operand (readings R9-R13): per hidden column h and per
         * block of 16 consecutive rows of this expert, RHT along the rows,
         * then an E4M3 block scale from the bound-derived per-expert scale
         * and E2M1 codes.  Layout: expert e's codes are [H][n/2] bytes at
         * byte off*H/2, its scales [H][n/16] at byte off*H/16. */
        float se = scale_enc[e];
        float ce = se / 6.0f;
        float bound = 4.0f * amax_row[e];
        uint8_t *cc = cw_codes + (size_t)off * (size_t)(H / 2);
        uint8_t *cs = cw_scales + (size_t)off * (size_t)(H / 16);
        for (int64_t h = 0; h < H; ++h) {
            for (int64_t j = 0; j < n / 16; ++j) {
                float d[16], y[16];
                float dmax = 0.0f;
                for (int i = 0; i < 16; ++i) {
                    d[i] = decode(rows + (size_t)(off + 16 * j + i) * S, H, S, h);
                    dmax = fmaxf(dmax, fabsf(d[i]));
                }
                or_rht16_f32(d, sign_mask, y);
                float bmax = 0.0f;
                for (int i = 0; i < 16; ++i) {
                    float ay = fabsf(y[i]);
                    bmax = fmaxf(bmax, ay);
                    if (ay > bound)
                        report[1] += 1;
                    if (ay > 4.0f * dmax)
                        report[3] += 1;
                }
                float sprod = bmax * ce;
                int s = or_e4m3_rne_sat((double)sprod);
                if ((double)sprod > 448.0)
                    report[0] += 1;
                float sval = (float)or_e4m3_value(s);
                float r = (sval == 0.0f) ? 0.0f : se / sval;
                cs[h * (n / 16) + j] = (uint8_t)s;
                for (int i = 0; i < 16; ++i) {
                    float v = fabsf(y[i]) * r;
                    if (v > 6.0f)
                        report[2] += 1;
                    double sv = signbit(y[i]) ? -(double)v : (double)v;
                    int64_t pos = 16 * j + i; /* row within the expert */
                    int code;
                    if (rounding == 1)
                        code = or_e2m1_sr(sv, or_sr_u16(seed, 1u,
                                   (uint64_t)off * (uint64_t)H + (uint64_t)h * (uint64_t)n + (uint64_t)pos));
                    else
                        code = or_e2m1_rne(sv);
                    size_t byte = (size_t)h * (size_t)(n / 2) + (size_t)(pos / 2);
                    if (pos % 2 == 0)
                        cc[byte] = (uint8_t)((cc[byte] & 0xf0) | code);
                    else
                        cc[byte] = (uint8_t)((cc[byte] & 0x0f) | (code << 4));
                }
            }
        }
    }
}

/* Scale-factor layout of a block-scaled GEMM operand (reading R23).  TE PR
 * #3753 "Add NVFP4 EP dispatch and combine backward", commit "... under NVFP4
 * autocast": the combine backward returns the gradient as a "swizzled NVFP4
 * GroupedTensor" that holds only GEMM operands; the pages do not spell the
 * layout out.  The one taken is the tiled layout that Blackwell block-scaled
 * matrix multiplies read: the scale matrix SF[M][Kb] (M a multiple of 128, Kb
 * a multiple of 4) is cut into tiles of 128 rows x 4 scale columns, stored
 * one after another with the tiles along Kb contiguous (tile (mt, kt) at
 * (mt * Kb/4 + kt) * 512); inside a tile, element (m, kb) is at
 *   (m mod 32) * 16 + ((m mod 128) / 32) * 4 + (kb mod 4).
 * lin is row-major [M][Kb]; out receives the M*Kb bytes in tiled order. */
void or_scale_swizzle(const uint8_t *lin, int64_t M, int64_t Kb, uint8_t *out)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < Kb; ++kb) {
            int64_t tile = (m / 128) * (Kb / 4) + kb / 4;
            int64_t in_tile = (m % 32) * 16 + ((m % 128) / 32) * 4 + kb % 4;
            out[tile * 512 + in_tile] = lin[m * Kb + kb];
        }
    }
}

/* Columnwise RHT operand of a BF16 input with a supplied per-expert amax
 * (reading R24).  TE PR #3755 "Optionally derive FC1 dy NVFP4 amaxes from the
 * dGLU epilogue", PR description: the exact amax known to the dGLU epilogue,
 * rounded to BF16, is the rowwise amax; four times it bounds the columnwise
 * values after the RHT, so no separate amax pass over the grouped tensor is
 * made.
 *   x        BF16 [R_cap][H], rows in expert order (expert e: rows
 *            [offsets[e], offsets[e+1]), a multiple of 16 rows)
 *   amax_in  [E] the supplied amax of each expert
 * Per expert: amax_row = BF16_RNE(amax_in), amax_col = fl32(4 amax_row),
 * S_enc as for the direct receive (R11).  Per hidden column and block of 16
 * consecutive rows: d = the BF16 values (exact in float), the same RHT,
 * block scale and codes as the direct receive's columnwise operand (R9, R11,
 * R12); stochastic rounding draws from Philox stream 2 with element index
 * off*H + h*n + row-in-expert (R13). */
void or_nvfp4_colwise_rht_bf16(const uint16_t *x, int64_t R_cap, int64_t H,
                               const int32_t *offsets, int E,
                               const float *amax_in, uint8_t *cw_codes,
                               uint8_t *cw_scales, float *amax_row,
                               float *amax_col, float *scale_enc,
                               int rounding, uint64_t seed,
                               uint16_t sign_mask, int64_t *report)
{
    (void)R_cap;
    for (int i = 0; i < 4; ++i)
        report[i] = 0;
    for (int e = 0; e < E; ++e) {
        uint16_t ab = or_bf16_rne((double)amax_in[e]);
        uint32_t bits = (uint32_t)ab << 16;
        float a;
        memcpy(&a, &bits, 4);
        float ac = 4.0f * a;
        float se = 1.0f;
        if (ac > 0.0f) {
            se = 2688.0f / ac;
            if (se > FLT_MAX)
                se = FLT_MAX;
        }
        amax_row[e] = a;
        amax_col[e] = ac;
        scale_enc[e] = se;

        int64_t off = offsets[e];
        int64_t n = offsets[e + 1] - offsets[e];
        float ce = se / 6.0f;
        uint8_t *cc = cw_codes + (size_t)off * (size_t)(H / 2);
        uint8_t *cs = cw_scales + (size_t)off * (size_t)(H / 16);
        for (int64_t h = 0; h < H; ++h) {
            for (int64_t j = 0; j < n / 16; ++j) {
                float d[16], y[16];
                float dmax = 0.0f;
                for (int i = 0; i < 16; ++i) {
                    uint32_t b = (uint32_t)x[(size_t)(off + 16 * j + i) * (size_t)H + (size_t)h] << 16;
                    memcpy(&d[i], &b, 4);
                    dmax = fmaxf(dmax, fabsf(d[i]));
                }
                or_rht16_f32(d, sign_mask, y);
                float bmax = 0.0f;
                for (int i = 0; i < 16; ++i) {
                    float ay = fabsf(y[i]);
                    bmax = fmaxf(bmax, ay);
                    if (ay > ac)
                        report[1] += 1;
                    if (ay > 4.0f * dmax)
                        report[3] += 1;
                }
                float sprod = bmax * ce;
                int s = or_e4m3_rne_sat((double)sprod);
                if ((double)sprod > 448.0)
                    report[0] += 1;
                float sval = (float)or_e4m3_value(s);
                float r = (sval == 0.0f) ? 0.0f : se / sval;
                cs[h * (n / 16) + j] = (uint8_t)s;
                for (int i = 0; i < 16; ++i) {
                    float v = fabsf(y[i]) * r;
                    if (v > 6.0f)
                        report[2] += 1;
                    double sv = signbit(y[i]) ? -(double)v : (double)v;
                    int64_t pos = 16 * j + i; /* row within the expert */
                    int code;
                    if (rounding == 1)
                        code = or_e2m1_sr(sv, or_sr_u16(seed, 2u,
                                   (uint64_t)off * (uint64_t)H + (uint64_t)h * (uint64_t)n + (uint64_t)pos));
                    else
                        code = or_e2m1_rne(sv);
                    size_t byte = (size_t)h * (size_t)(n / 2) + (size_t)(pos / 2);
                    if (pos % 2 == 0)
                        cc[byte] = (uint8_t)((cc[byte] & 0xf0) | code);
                    else
                        cc[byte] = (uint8_t)((cc[byte] & 0x0f) | (code << 4));
                }
            }
        }
    }
}
