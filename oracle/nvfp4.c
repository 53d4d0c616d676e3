/*
 * Oracle: NVFP4 row pack and unpack.  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * TE PR #3753 "Add NVFP4 EP dispatch and combine backward", PR description
 * and the review thread on the EP header comment: a token is quantised once,
 * on the sending side, into a single row of E2M1 codes with an E4M3 scale per
 * 16 elements and an FP32 token scale that is a power of two; without direct
 * receive the received rows are turned back into BF16.
 *
 * Row layout (reading R6), S = roundup16(9H/16 + 16) bytes:
 *   [0, H/2)        E2M1 codes, element 2i in the low nibble of byte i
 *   [H/2, 9H/16)    E4M3 block scales, one per 16 elements, in block order
 *   [9H/16, S-16)   zero
 *   [S-16, S)       trailer: f32 token scale S_t, f32 token amax A_t,
 *                   u32 source token id (0xFFFFFFFF on a padding row), u32 0
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "oracle.h"

size_t or_row_bytes(int64_t H)
{
    size_t raw = (size_t)(9 * H / 16 + 16);
    return (raw + 15) / 16 * 16;
}

static void put_f32(uint8_t *p, float v) { memcpy(p, &v, 4); }
static void put_u32(uint8_t *p, uint32_t v) { memcpy(p, &v, 4); }
static float get_f32(const uint8_t *p) { float v; memcpy(&v, p, 4); return v; }

/* Quantise one BF16 token into one packed row.
 *  A_t = max |x| (exact; TE PR #3755, test commit: the test checks that each
 *        rowwise amax is the BF16 input's own), S_t = 2^k_t (reading R3).
 *  s_b = E4M3_RNE_sat(B_b / (6 S_t)) with B_b the block's max |x| (R4).
 *  code = E2M1(x / (s_b S_t)), RNE or stochastic (R5, R13); s_b = 0 gives
 *        magnitude 0 with the sign kept (R2).
 * Stochastic rounding draws element (t_index * H + h) of stream 0. */
void or_nvfp4_pack_token(const uint16_t *x, int64_t H, uint32_t token_id,
                         int rounding, uint64_t seed, uint64_t t_index,
                         uint8_t *row)
{
    size_t S = or_row_bytes(H);
    memset(row, 0, S);
    double amax = 0.0;
    for (int64_t h = 0; h < H; ++h)
        amax = fmax(amax, fabs(or_bf16_value(x[h])));
    int kt = or_token_scale_exp(amax);
    double St = ldexp(1.0, kt);
    for (int64_t b = 0; b < H / 16; ++b) {
        double bmax = 0.0;
        for (int i = 0; i < 16; ++i)
            bmax = fmax(bmax, fabs(or_bf16_value(x[b * 16 + i])));
        int sb = or_e4m3_rne_sat(bmax / (6.0 * St));
        double s = or_e4m3_value(sb) * St;
        row[H / 2 + b] = (uint8_t)sb;
        for (int i = 0; i < 16; ++i) {
            int64_t h = b * 16 + i;
            double xv = or_bf16_value(x[h]);
            int code;
            if (s == 0.0) {
                code = signbit(xv) ? 8 : 0;
            } else {
                double v = xv / s;
                if (rounding == 1)
                    code = or_e2m1_sr(v, or_sr_u16(seed, 0u, t_index * (uint64_t)H + (uint64_t)h));
                else
                    code = or_e2m1_rne(v);
            }
            row[h / 2] |= (uint8_t)((h % 2) ? (code << 4) : code);
        }
    }
    put_f32(row + S - 16, (float)St);
    put_f32(row + S - 12, (float)amax);
    put_u32(row + S - 8, token_id);
    put_u32(row + S - 4, 0u);
}

/* A padding row is the packing of an all-zero token with id 0xFFFFFFFF
 * (reading R7). */
static void pad_row(int64_t H, uint8_t *row)
{
    size_t S = or_row_bytes(H);
    memset(row, 0, S);
    put_f32(row + S - 16, (float)ldexp(1.0, -126));
    put_f32(row + S - 12, 0.0f);
    put_u32(row + S - 8, 0xFFFFFFFFu);
}

void or_nvfp4_pack(const uint16_t *tokens, int64_t T, int64_t H,
                   const int32_t *dest, int k, const int32_t *offsets,
                   const int32_t *counts, int E, uint8_t *rows,
                   int64_t R_cap, int rounding, uint64_t seed)
{
    size_t S = or_row_bytes(H);
    (void)R_cap;
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int32_t d = dest[t * k + j];
            if (d < 0)
                continue;
            /* the sender packs once; every destination gets the same bytes */
            or_nvfp4_pack_token(tokens + t * H, H, (uint32_t)t, rounding, seed,
                                (uint64_t)t, rows + (size_t)d * S);
        }
    }
    for (int e = 0; e < E; ++e)
        for (int32_t r = offsets[e] + counts[e]; r < offsets[e + 1]; ++r)
            pad_row(H, rows + (size_t)r * S);
}

/* Decode rows [0, R) to BF16 (reading R15): sign * G[m] * s_b * S_t, exact in
 * double, then rounded to BF16 (exact unless below BF16's normal range). */
void or_nvfp4_unpack(const uint8_t *rows, int64_t R_cap, int64_t H,
                     const int32_t *offsets, int E, uint16_t *out)
{
    size_t S = or_row_bytes(H);
    int64_t R = offsets[E];
    (void)R_cap;
    for (int64_t r = 0; r < R; ++r) {
        const uint8_t *row = rows + (size_t)r * S;
        double St = (double)get_f32(row + S - 16);
        for (int64_t h = 0; h < H; ++h) {
            int code = (row[h / 2] >> ((h % 2) * 4)) & 0xf;
            double sb = or_e4m3_value(row[H / 2 + h / 16]);
            double v = or_e2m1_value(code) * sb * St;
            out[r * H + h] = or_bf16_rne(v);
        }
    }
}
