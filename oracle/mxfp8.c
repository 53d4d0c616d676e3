/*
 * Oracle: MXFP8 pack with the routing gather.  TEST INFRASTRUCTURE ONLY (see
 * oracle.h).
 *
 * TE PR #3270 "EP dispatch with unfused MXFP8 quantization": bfloat16 tokens
 * are quantised to MXFP8 (E4M3 data with E8M0 block scales, sequence diagram;
 * only E4M3, review thread), and the received data and its block scales sit
 * in one buffer the caller provides, data first, scales after (Changes).
 *
 * Reading R14: 32-element blocks; the block exponent e is the smallest integer
 * in [-127, 127] with max|x| <= 448 * 2^e (no element saturates), stored as
 * the E8M0 byte e + 127; each element is E4M3_RNE(x / 2^e).  Buffer layout:
 * data [R_cap][H] bytes, then scales [R_cap][H/32] bytes.  Padding rows are
 * the packing of an all-zero token (data 0, scale byte 0).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "oracle.h"

static void mx_token(const uint16_t *x, int64_t H, uint8_t *data, uint8_t *scales)
{
    for (int64_t b = 0; b < H / 32; ++b) {
        double bmax = 0.0;
        for (int i = 0; i < 32; ++i)
            bmax = fmax(bmax, fabs(or_bf16_value(x[b * 32 + i])));
        int e = or_mx_scale_exp(bmax);
        scales[b] = (uint8_t)(e + 127);
        for (int i = 0; i < 32; ++i) {
            double v = or_bf16_value(x[b * 32 + i]) / ldexp(1.0, e);
            data[b * 32 + i] = (uint8_t)or_e4m3_rne_sat(v);
        }
    }
}

void or_mxfp8_pack(const uint16_t *tokens, int64_t T, int64_t H,
                   const int32_t *dest, int k, const int32_t *offsets,
                   const int32_t *counts, int E, uint8_t *buf, int64_t R_cap)
{
    uint8_t *data = buf;
    uint8_t *scales = buf + (size_t)R_cap * (size_t)H;
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int32_t d = dest[t * k + j];
            if (d < 0)
                continue;
            mx_token(tokens + t * H, H, data + (size_t)d * H, scales + (size_t)d * (H / 32));
        }
    }
    for (int e = 0; e < E; ++e) {
        for (int32_t r = offsets[e] + counts[e]; r < offsets[e + 1]; ++r) {
            memset(data + (size_t)r * H, 0, (size_t)H);
            memset(scales + (size_t)r * (H / 32), 0, (size_t)(H / 32));
        }
    }
}

/* Columnwise (wgrad) MXFP8 operand of an expert-grouped BF16 tensor (reading
 * R25).  TE PR #3270 "EP dispatch with unfused MXFP8 quantization",
 * Description: the combine backward returns the expert-output gradient as a
 * per-expert MXFP8 GroupedTensor; the expert GEMM's weight gradient reduces
 * over the tokens, so its operand takes its 32-element blocks along the token
 * axis.  Per expert e (rows [offsets[e], offsets[e+1]), a multiple of 32), per
 * hidden column h and per block of 32 consecutive rows: the R14 exponent and
 * E4M3 elements.  Buffer: data, expert e as [H][n_e] bytes at byte
 * offsets[e]*H (the rows of column h along the bytes); then, from byte
 * R_cap*H, scales, expert e as [H][n_e/32] bytes at offsets[e]*H/32. */
void or_mxfp8_colwise(const uint16_t *x, int64_t R_cap, int64_t H,
                      const int32_t *offsets, int E, uint8_t *buf)
{
    uint8_t *data = buf;
    uint8_t *scales = buf + (size_t)R_cap * (size_t)H;
    for (int e = 0; e < E; ++e) {
        int64_t off = offsets[e], n = offsets[e + 1] - offsets[e];
        for (int64_t h = 0; h < H; ++h) {
            for (int64_t b = 0; b < n / 32; ++b) {
                double bmax = 0.0;
                for (int i = 0; i < 32; ++i)
                    bmax = fmax(bmax, fabs(or_bf16_value(x[(off + 32 * b + i) * H + h])));
                int ex = or_mx_scale_exp(bmax);
                scales[(size_t)off * (size_t)(H / 32) + (size_t)h * (size_t)(n / 32) + (size_t)b] =
                    (uint8_t)(ex + 127);
                for (int i = 0; i < 32; ++i) {
                    double v = or_bf16_value(x[(off + 32 * b + i) * H + h]) / ldexp(1.0, ex);
                    data[(size_t)off * (size_t)H + (size_t)h * (size_t)n + (size_t)(32 * b + i)] =
                        (uint8_t)or_e4m3_rne_sat(v);
                }
            }
        }
    }
}
