/*
 * Plain CPU oracle for the NVFP4 expert-parallel pack / direct-receive path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the two are checked against each other, never built from one
 * another.
 *
 * Every function is the slow, obviously-correct restatement of one step of the
 * method described by four TransformerEngine pull-request pages:
 *   [EP-NVFP4]   TE PR #3753 "[Common][PyTorch] Add NVFP4 EP dispatch and
 *                combine backward"
 *   [EP-MXFP8]   TE PR #3270 "[Common][PyTorch] EP dispatch with unfused MXFP8
 *                quantization"
 *   [ROW-SCALED] TE PR #3324 "[PyTorch] Enable NVFP4 row-scaled (per-token)
 *                backward for GroupedLinear"
 *   [DGLU-AMAX]  TE PR #3755 "[PyTorch] Optionally derive FC1 dy NVFP4 amaxes
 *                from the dGLU epilogue"
 * Where the pages leave a step open, the reading taken is stated beside the
 * function (the readings are numbered R1..R22 and listed in the design notes).
 *
 * Precision: exact-real steps are done in double (every product and quotient
 * used is either exact in double or provably on the same side of every
 * rounding boundary); the columnwise re-quantisation is specified in FP32
 * (single IEEE binary32 operations, round to nearest even, no fused
 * multiply-add) and is done here in float with floating-point contraction
 * disabled at compile time.
 *
 * Parity status: every function below is pinned by a CPU test against an
 * independent formulation (brute force, closed form, library routine or
 * published test vector).  No function here is "parity unpinned".
 */
#ifndef NVFP4_ORACLE_H
#define NVFP4_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats ------------------------------------------------------ */
double   or_e2m1_value(int code);                  /* 4-bit code -> value           */
int      or_e2m1_rne(double v);                    /* nearest, ties to even index   */
int      or_e2m1_sr(double v, unsigned r16);       /* stochastic, 16 random bits    */
double   or_e4m3_value(int code);                  /* 8-bit code -> value (NaN: 0x7f/0xff) */
int      or_e4m3_rne_sat(double v);                /* nearest, ties even, saturating */
double   or_bf16_value(uint16_t bits);
uint16_t or_bf16_rne(double v);                    /* exact for |v| >= 2^-149 with <= 24 bits */
int      or_token_scale_exp(double amax);          /* k_t of the power-of-two token scale */
int      or_mx_scale_exp(double bmax);             /* E8M0 exponent of an MXFP8 block */
void     or_e2m1_rne_batch(const double *v, int64_t n, uint8_t *out);
void     or_e2m1_sr_batch(const double *v, const uint16_t *r16, int64_t n, uint8_t *out);
void     or_e4m3_rne_sat_batch(const double *v, int64_t n, uint8_t *out);

/* ---- counter-based random numbers ---------------------------------------- */
void     or_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
unsigned or_sr_u16(uint64_t seed, uint32_t stream, uint64_t idx);
void     or_sr_u16s(uint64_t seed, uint32_t stream, uint64_t idx0, int64_t n, uint16_t *out);

/* ---- 16-point random Hadamard transform along tokens ------------------- */
void     or_rht16_f32(const float d[16], uint16_t sign_mask, float y[16]);

/* ---- the hot path ---------------------------------------------------------- */
size_t   or_row_bytes(int64_t H);
uint32_t or_route_plan(const int32_t *topk, int64_t T, int k, int E, int A,
                       int32_t *offsets, int32_t *counts, int32_t *dest);
void     or_nvfp4_pack_token(const uint16_t *x, int64_t H, uint32_t token_id,
                             int rounding, uint64_t seed, uint64_t t_index,
                             uint8_t *row);
void     or_nvfp4_pack(const uint16_t *tokens, int64_t T, int64_t H,
                       const int32_t *dest, int k, const int32_t *offsets,
                       const int32_t *counts, int E, uint8_t *rows,
                       int64_t R_cap, int rounding, uint64_t seed);
void     or_nvfp4_unpack(const uint8_t *rows, int64_t R_cap, int64_t H,
                         const int32_t *offsets, int E, uint16_t *out);
void     or_expert_amax(const uint8_t *rows, int64_t H, const int32_t *offsets,
                        int E, float *amax_row, float *amax_col,
                        float *scale_enc);
/* report[0] = blocks whose E4M3 scale saturated at 448
 * report[1] = post-RHT values above 4 x rowwise amax of their expert
 * report[2] = elements whose value before E2M1 rounding exceeded 6
 * report[3] = post-RHT values above 4 x max |decoded input| of their block
 *             (an exact invariant: must always be 0)                        */
void     or_nvfp4_direct_receive(const uint8_t *rows, int64_t R_cap, int64_t H,
                                 const int32_t *offsets, int E,
                                 const uint8_t *expert_mask,
                                 uint8_t *rw_codes, uint8_t *rw_scales,
                                 float *rw_row_scale, uint8_t *cw_codes,
                                 uint8_t *cw_scales, float *amax_row,
                                 float *amax_col, float *scale_enc,
                                 int rounding, uint64_t seed,
                                 uint16_t sign_mask, int64_t *report);
/* BF16-input columnwise RHT operand with a supplied per-expert amax (R24);
 * report as for or_nvfp4_direct_receive (report[1]: values above 4 x the
 * rounded supplied amax). */
void     or_nvfp4_colwise_rht_bf16(const uint16_t *x, int64_t R_cap, int64_t H,
                                   const int32_t *offsets, int E,
                                   const float *amax_in, uint8_t *cw_codes,
                                   uint8_t *cw_scales, float *amax_row,
                                   float *amax_col, float *scale_enc,
                                   int rounding, uint64_t seed,
                                   uint16_t sign_mask, int64_t *report);
/* Columnwise MXFP8 operand of an expert-grouped BF16 tensor (R25). */
void     or_mxfp8_colwise(const uint16_t *x, int64_t R_cap, int64_t H,
                          const int32_t *offsets, int E, uint8_t *buf);
/* Tiled scale-factor layout (R23): M % 128 == 0, Kb % 4 == 0. */
void     or_scale_swizzle(const uint8_t *lin, int64_t M, int64_t Kb, uint8_t *out);
void     or_mxfp8_pack(const uint16_t *tokens, int64_t T, int64_t H,
                       const int32_t *dest, int k, const int32_t *offsets,
                       const int32_t *counts, int E, uint8_t *buf,
                       int64_t R_cap);

#ifdef __cplusplus
}
#endif
#endif
