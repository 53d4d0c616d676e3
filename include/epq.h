/*
 * epq.h -- C ABI of libepq.so: NVFP4 / MXFP8 expert-parallel token
 * quantisation on one GB300 (sm_103a).
 *
 * The method is the one described by four TransformerEngine pull-request
 * pages, cited below by title and section:
 *   TE PR #3753 "[Common][PyTorch] Add NVFP4 EP dispatch and combine backward"
 *   TE PR #3270 "[Common][PyTorch] EP dispatch with unfused MXFP8 quantization"
 *   TE PR #3324 "[PyTorch] Enable NVFP4 row-scaled (per-token) backward for
 *               GroupedLinear"
 *   TE PR #3755 "[PyTorch] Optionally derive FC1 dy NVFP4 amaxes from the dGLU
 *               epilogue"
 * The cross-GPU expert-parallel transport of those pages is replaced, on one
 * GPU, by a local routing plan that places every (token, expert) pair in an
 * expert-contiguous, alignment-padded row order.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers named "device" are CUDA device memory owned by the caller; the
 *   library never allocates, frees or synchronises, and never keeps a pointer
 *   after the call returns.  Every call only enqueues work on `stream` (a
 *   cudaStream_t passed as void*; NULL = the legacy default stream), so these
 *   calls can be captured in a CUDA graph (ep_route_plan_noalloc aside: this
 *   header makes no statement about capturing it).
 * - Device guard: the call makes the device that owns the first input pointer
 *   current for its duration (and restores the previous device); every other
 *   pointer must live on that same device, else EP_ERR_DEVICE (TE PR #3753,
 *   commit "guard the NVFP4 EP bindings with the input tensor's device").
 * - Errors found on the host (null pointer, bad size, bad argument, too small
 *   a buffer, pointer on the wrong device) return a negative ep_status before
 *   anything is enqueued.  A failed launch returns EP_ERR_CUDA.  Errors that
 *   only the data can reveal (a bad routing id, a wait that gave up) are ORed
 *   into the caller's device word *dev_status as EP_DEV_ERR_* bits and the
 *   offending item is skipped; kernels never trap.  The caller reads
 *   dev_status after its own synchronisation.
 * - Outputs are bit-deterministic for a given input, routing, seed and sign
 *   mask.  Rows in [R, R_cap) of every row-indexed output are left untouched,
 *   R = expert_offsets[E].
 * - Shapes: T tokens, H hidden (H % 32 == 0), k routing slots per token
 *   (1 <= k <= 32), E experts (1 <= E <= 1024), A per-expert alignment
 *   (A > 0, A % 128 == 0), R_cap rows of capacity (< 2^31).
 */
#ifndef EPQ_H
#define EPQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EP_OK = 0,
    EP_ERR_NULL = -1,      /* a required pointer is NULL                    */
    EP_ERR_SHAPE = -2,     /* T, H, k, E out of range or H % 32 != 0        */
    EP_ERR_ALIGN = -3,     /* A not a positive multiple of 128, or a
                              pointer not 16-byte aligned                   */
    EP_ERR_CAPACITY = -4,  /* R_cap or a workspace too small                */
    EP_ERR_ARG = -5,       /* bad rounding mode or other argument           */
    EP_ERR_DEVICE = -6,    /* pointer not device memory of the input device */
    EP_ERR_CUDA = -7       /* a CUDA call failed                            */
} ep_status;

enum { EP_ROUND_RNE = 0, EP_ROUND_SR = 1 };

/* Bits ORed into *dev_status by the kernels. */
enum {
    EP_DEV_ERR_BAD_EXPERT = 1u,  /* routing id outside [-1, E): slot dropped  */
    EP_DEV_ERR_DUP_EXPERT = 2u,  /* id repeated within a token: later dropped */
    EP_DEV_ERR_TIMEOUT = 4u,     /* a bounded wait gave up; outputs invalid   */
    EP_DEV_ERR_CAPACITY = 8u     /* expert_offsets[E] > R_cap: rows skipped   */
};

/* Bytes of one packed NVFP4 row: roundup16(9H/16 + 16). */
size_t ep_nvfp4_row_bytes(int64_t H);

/* Upper bound on R = sum_e ceil(c_e / A) * A over any routing: T*k + E*(A-1). */
int64_t ep_rows_capacity(int64_t T, int k, int E, int A);

/* Device workspace needed by ep_route_plan: 16 + ceil(T/512) * E * 4 bytes.
 * Its first 16 bytes hold a grid-barrier count and generation: they must be
 * zero before the workspace is first used, and every call that completes
 * leaves them usable for the next call (a zero-filled buffer can be reused
 * indefinitely by calls on one stream; calls that may overlap need separate
 * workspaces). */
size_t ep_route_workspace_bytes(int64_t T, int k, int E);

/*
 * ep_route_plan -- expert-contiguous placement of every (token, slot).
 * TE PR #3270, description and sequence diagram: dispatch returns the received
 * rows "expert-major" as a per-expert grouped tensor; review thread: each
 * expert slot is aligned to a multiple of 128 rows for the grouped packed
 * scales; TE PR #3753, commit "layer_args": the backward takes (top_k,
 * alignment, topk_idx_dtype).
 *   topk_idx        device int32 [T, k], row-major; -1 = dropped slot.  An id
 *                   >= E or < -1 sets EP_DEV_ERR_BAD_EXPERT and is dropped; an
 *                   id repeated within a token sets EP_DEV_ERR_DUP_EXPERT and
 *                   the later slot is dropped.
 *   expert_offsets  device int32 [E+1] out: expert e owns rows
 *                   [offsets[e], offsets[e+1]); offsets[E] = R.
 *   expert_counts   device int32 [E] out: c_e, tokens routed to e.  The
 *                   n_e - c_e trailing rows of expert e are padding rows.
 *   dest            device int32 [T*k] out: row of (t, j), or -1 if dropped.
 *                   Within an expert, rows follow ascending token order.
 *   workspace       device, ws_bytes >= ep_route_workspace_bytes(T, k, E),
 *                   zero-filled before its first use (see above).
 *   R_cap           capacity the rows buffers will have; must be at least
 *                   ep_rows_capacity(T, k, E, A) (EP_ERR_CAPACITY otherwise).
 * One cooperative launch (all CTAs resident, one grid barrier whose wait is
 * bounded: EP_DEV_ERR_TIMEOUT if it gives up); T = 0 is allowed (all offsets
 * and counts 0).
 */
ep_status ep_route_plan(const int32_t *topk_idx, int64_t T, int k, int E, int A,
                        int64_t R_cap, int32_t *expert_offsets,
                        int32_t *expert_counts, int32_t *dest, void *workspace,
                        size_t ws_bytes, uint32_t *dev_status, void *stream);

/* Size of the scratch array inside the library that ep_route_plan_noalloc
 * uses in place of a caller's workspace. */
#define EP_ROUTE_STATIC_SCRATCH_BYTES 262144

/*
 * ep_route_plan_noalloc -- ep_route_plan without a workspace argument.
 * The pages have no counterpart: this is a library convenience.  It is for
 * callers that cannot allocate device memory for a workspace: a runtime or
 * plugin host that owns the whole GPU's memory in its own pool and passes an
 * extension only its inputs and outputs, or a latency-critical loop where a
 * cudaMalloc would synchronise the device.
 *   Arguments, outputs and device status: as ep_route_plan.  Results are
 *   identical to ep_route_plan's for the same inputs.
 *   Limit: ep_route_workspace_bytes(T, k, E) must not exceed
 *   EP_ROUTE_STATIC_SCRATCH_BYTES (256 KiB: e.g. T <= 130560 tokens at
 *   E = 256); larger problems return EP_ERR_CAPACITY and launch nothing.
 *   Memory: allocates nothing, on any call.  The scratch is a fixed device
 *   array of EP_ROUTE_STATIC_SCRATCH_BYTES that every GPU which loads the
 *   library holds until the process exits.  The first call on a device looks
 *   up that device's scratch address (cudaGetSymbolAddress), and so does the
 *   first call after the device's context was replaced (e.g. by
 *   cudaDeviceReset); make those calls before any stream capture: one made
 *   while `stream` is capturing returns EP_ERR_ARG and enqueues nothing.
 *   Each call clears the scratch's barrier words on `stream` before its
 *   kernel.
 *   Concurrency: all calls on a device share one scratch array, so calls
 *   whose work may overlap on the GPU (different streams, or several host
 *   threads) race and give wrong plans; order them on one stream, or use
 *   ep_route_plan with a workspace per stream.
 */
ep_status ep_route_plan_noalloc(const int32_t *topk_idx, int64_t T, int k,
                                int E, int A, int64_t R_cap,
                                int32_t *expert_offsets,
                                int32_t *expert_counts, int32_t *dest,
                                uint32_t *dev_status, void *stream);

/*
 * ep_nvfp4_pack -- quantise each BF16 token once into a packed NVFP4 row and
 * write that row to each of its destinations; fill padding rows.
 * TE PR #3753, PR description and the review thread on the EP header comment:
 * each token is quantised a single time on the sending side, into a row of
 * E2M1 codes with E4M3 scales per 16 elements and an FP32 token scale that is
 * a power of two; the combine backward takes the recipe's stochastic rounding.
 *   tokens_bf16     device bf16 [T, H] row-major, finite values.
 *   dest, expert_offsets, expert_counts: as produced by ep_route_plan.
 *   rows            device u8 [R_cap, S], S = ep_nvfp4_row_bytes(H), 16-byte
 *                   aligned.  Row layout: [0, H/2) E2M1 codes (element 2i in
 *                   the low nibble of byte i); [H/2, 9H/16) E4M3 block scales,
 *                   one per 16 elements; zeros up to S-16; trailer at S-16 =
 *                   {f32 token scale S_t = 2^k, f32 token amax A_t,
 *                   u32 source token id, u32 0}.  A padding row is the packing
 *                   of an all-zero token with id 0xFFFFFFFF.
 *   expert_amax     device f32 [E] or NULL.  When given, the token amax A_t of
 *                   every row written is max-reduced into expert_amax[e] of
 *                   the row's expert e (on the bit patterns: all values are
 *                   >= 0), so that afterwards it holds the largest A_t over
 *                   the rows of each expert (padding rows have A_t = 0): the
 *                   per-expert amax ep_nvfp4_direct_receive can take instead
 *                   of reducing the row trailers itself.  The caller fills it
 *                   first (zeros, or the partial maxima of earlier packs into
 *                   the same rows).  4-byte aligned.  With it, the next kernel
 *                   on `stream` may start (programmatic dependent launch) only
 *                   as the pack's CTAs finish their work, not when they
 *                   start.
 *   rounding        EP_ROUND_RNE or EP_ROUND_SR (element codes only; scales
 *                   are always round-to-nearest-even).  SR gives element
 *                   idx = t*H + h a 16-bit number R from Philox4x32-10 keyed
 *                   by `seed`, counter (idx/16, idx/2^36, stream 0, 0): word
 *                   (idx/4)%4 of the output, bytes b0..b3, A = b2:b0,
 *                   B = b3:b1; idx%4 = 0, 1, 2, 3 takes A, A bit-reversed,
 *                   B, B bit-reversed; the code rounds up iff
 *                   R + 65536 f >= 65536 (f: position between the two
 *                   neighbouring E2M1 values).
 * Numerics: A_t = max|x|; k = smallest integer >= -126 with A_t <= 2688*2^k;
 * s_b = E4M3_RNE(max|x_block| / (6*S_t)); code = E2M1(x / (s_b*S_t)), nearest
 * with ties to even, saturating at 6, sign kept (also for zero).
 */
ep_status ep_nvfp4_pack(const void *tokens_bf16, int64_t T, int64_t H,
                        const int32_t *dest, int k,
                        const int32_t *expert_offsets,
                        const int32_t *expert_counts, int E, uint8_t *rows,
                        int64_t R_cap, float *expert_amax, int rounding,
                        uint64_t seed, uint32_t *dev_status, void *stream);

/*
 * ep_nvfp4_dispatch -- ep_route_plan followed by ep_nvfp4_pack, in one call.
 * TE PR #3753, PR description: the NVFP4 dispatch routes each token and sends
 * it as one packed NVFP4 row; here the routing plan and the pack run back to
 * back on `stream`.
 *   Arguments: those of ep_route_plan (topk_idx, T, k, E, A, R_cap,
 *   expert_offsets, expert_counts, dest, workspace, ws_bytes) and of
 *   ep_nvfp4_pack (tokens_bf16, H, rows, expert_amax, rounding, seed); every
 *   check of both calls is made before anything is enqueued.  expert_amax
 *   (f32 [E] or NULL) is set to zero by the routing kernel before the pack
 *   max-reduces into it, so after the call it holds each expert's amax.  Outputs, device status and
 *   errors: exactly those of the two calls made in that order.
 *   Timing: the routing kernel starts only after all earlier work on `stream`
 *   has finished, so the pack kernel reads and encodes its first tokens while
 *   the routing kernel still runs and waits for it only before reading `dest`
 *   (the separate ep_nvfp4_pack reads no token before that wait).
 */
ep_status ep_nvfp4_dispatch(const int32_t *topk_idx, const void *tokens_bf16,
                            int64_t T, int64_t H, int k, int E, int A,
                            int64_t R_cap, int32_t *expert_offsets,
                            int32_t *expert_counts, int32_t *dest,
                            void *workspace, size_t ws_bytes, uint8_t *rows,
                            float *expert_amax, int rounding, uint64_t seed,
                            uint32_t *dev_status, void *stream);

/*
 * ep_nvfp4_unpack -- decode packed rows to BF16 (the path used when direct
 * receive is off).  TE PR #3753, PR description: without direct receive the
 * received rows are turned back into BF16; commit "grad direct-receive
 * opt-out": the opt-out returns that BF16 decode.
 *   rows            device u8 [R_cap, S] (ep_nvfp4_pack layout).
 *   out_bf16        device bf16 [R_cap, H]; rows [0, R) written with
 *                   BF16(sign * E2M1 value * s_b * S_t) (exact in BF16 except
 *                   below its normal range, where it is rounded to nearest).
 */
ep_status ep_nvfp4_unpack(const uint8_t *rows, int64_t R_cap, int64_t H,
                          const int32_t *expert_offsets, int E, void *out_bf16,
                          uint32_t *dev_status, void *stream);

/* Outputs of ep_nvfp4_direct_receive (all device memory). */
typedef struct {
    uint8_t *rw_codes;      /* u8 [R_cap, H/2]  rowwise codes (sender's)      */
    uint8_t *rw_scales;     /* u8 [R_cap, H/16] rowwise E4M3 block scales     */
    float *rw_row_scale;    /* f32 [R_cap]      per-row FP32 scale S_t        */
    uint8_t *cw_codes;      /* u8 [R_cap*H/2]  columnwise RHT codes; expert e:
                               [H][n_e/2] bytes at byte offsets[e]*H/2, the
                               rows (tokens) of column h along the bytes     */
    uint8_t *cw_scales;     /* u8 [R_cap*H/16] columnwise E4M3 scales; expert
                               e: [H][n_e/16] at byte offsets[e]*H/16        */
    float *amax_row;        /* f32 [E] rowwise amax of each expert            */
    float *amax_col;        /* f32 [E] columnwise amax bound = 4 * amax_row   */
    float *cw_scale_enc;    /* f32 [E] columnwise encode scale S_enc          */
} ep_nvfp4_grouped;

/*
 * ep_nvfp4_direct_receive -- build the expert GEMM's grouped NVFP4 operands
 * straight from the packed rows, in one pass over them.
 * TE PR #3753, PR description: the rowwise operand keeps the codes the sender
 * produced, and the columnwise RHT operand is requantised with a per-expert
 * scale derived from a bound, which avoids both a trip through BF16 and a pass
 * that measures the amax; TE PR #3755, PR description: after the RHT no
 * columnwise value exceeds four times the rowwise amax; TE PR #3324,
 * description: NVFP4 operands with one FP32 scale per row (per token).
 *   rows            device u8 [R_cap, S]; R_cap * H above 2^36 (element
 *                   positions of 36 bits or more) -> EP_ERR_CAPACITY.
 *   expert_amax     device f32 [E] or NULL: each expert's amax, the largest
 *                   token amax A_t over its rows, already reduced (as
 *                   ep_nvfp4_pack / ep_nvfp4_dispatch leave it); the outputs
 *                   are then identical and no trailer pass is made (below one
 *                   128-row tile of capacity the trailers are read anyway, to
 *                   the same result).  NULL: the call reduces the trailers
 *                   itself.  4-byte aligned (EP_ERR_ALIGN otherwise).
 *   out             host pointer to the output descriptor.  The rowwise group
 *                   (rw_codes, rw_scales, rw_row_scale) may be all NULL to skip
 *                   it; everything else is required.
 *   rounding, seed  columnwise element rounding; SR counter = (p/16, 0,
 *                   stream 1, 0) with p = offsets[e]*H + h*n_e + row-in-expert.
 *   rht_sign_mask   bit i set = sign -1 on the i-th row of every 16-row block.
 * Per expert: amax_row = max of the rows' token amaxes; amax_col = 4*amax_row;
 * S_enc = min(2688/amax_col, FLT_MAX) (1 if amax_col = 0).  Per hidden column
 * and 16-row block: y = (1/4) H16 diag(sigma) d over the decoded values d;
 * s = E4M3_RNE_sat(max|y| * (S_enc/6)); code = E2M1(|y| * (S_enc/s)) with the
 * sign of y (FP32, single-rounded operations, in this order).
 * Kernels on `stream`: without expert_amax, the per-expert metadata from the
 * row trailers (4 bytes per row), then the tile transform, which reads S_enc
 * back; with it, the tile transform alone (it writes the metadata too).
 */
ep_status ep_nvfp4_direct_receive(const uint8_t *rows, int64_t R_cap,
                                  int64_t H, const int32_t *expert_offsets,
                                  int E, const float *expert_amax,
                                  const ep_nvfp4_grouped *out,
                                  int rounding, uint64_t seed,
                                  uint16_t rht_sign_mask, uint32_t *dev_status,
                                  void *stream);

/*
 * ep_nvfp4_direct_receive_swizzled -- ep_nvfp4_direct_receive with both scale
 * tensors in the tiled layout that block-scaled GEMMs read.
 * TE PR #3753, commit "... under NVFP4 autocast": the combine backward hands
 * FC2's gradient over as a grouped NVFP4 tensor whose scales are already in
 * the GEMM's swizzled order and which carries GEMM operands only.  The pages
 * do not spell the layout out; the one used is the
 * Blackwell block-scaled operand layout: a scale matrix SF[M][Kb] is cut into
 * 512-byte tiles of 128 rows x 4 scale columns, tile (mt, kt) at byte
 * (mt*Kb/4 + kt)*512, and element (m, kb) of a tile at
 * (m mod 32)*16 + ((m mod 128)/32)*4 + (kb mod 4).
 *   Arguments, codes, row scales, metadata and errors: as
 *   ep_nvfp4_direct_receive, plus H % 128 != 0 -> EP_ERR_SHAPE.
 *   rw_scales: the [R, H/16] matrix of rows [0, R) in that layout (expert
 *   slots are whole 128-row tiles); bytes past R*H/16 are left untouched.
 *   cw_scales: expert e's [H, n_e/16] matrix in that layout, at byte
 *   offsets[e]*H/16 (the same place and size as the linear form).
 */
ep_status ep_nvfp4_direct_receive_swizzled(const uint8_t *rows, int64_t R_cap,
                                           int64_t H,
                                           const int32_t *expert_offsets,
                                           int E, const float *expert_amax,
                                           const ep_nvfp4_grouped *out,
                                           int rounding, uint64_t seed,
                                           uint16_t rht_sign_mask,
                                           uint32_t *dev_status,
                                           void *stream);

/*
 * ep_nvfp4_colwise_rht_bf16 -- the columnwise RHT operand of an expert-grouped
 * BF16 tensor, with the per-expert amax supplied by its producer.
 * TE PR #3755 "Optionally derive FC1 dy NVFP4 amaxes from the dGLU epilogue",
 * PR description: the dGLU epilogue's exact amax, rounded to BF16, serves as
 * the rowwise amax; four times it bounds the columnwise amax after the RHT, so
 * the grouped tensor needs no amax pass of its own.
 *   x_bf16          device bf16 [R_cap, H], rows in expert order: expert e
 *                   owns rows [expert_offsets[e], expert_offsets[e+1]), a
 *                   whole number of 128-row tiles (as ep_route_plan gives);
 *                   a slot that is not raises EP_DEV_ERR_BAD_EXPERT and its
 *                   rows are skipped.  Finite values.
 *   amax_in         device f32 [E]: the supplied amax of each expert.
 *   cw_codes, cw_scales, amax_row, amax_col, cw_scale_enc: as the columnwise
 *                   part of ep_nvfp4_grouped (layout R12: expert e's codes
 *                   [H][n_e/2] at byte offsets[e]*H/2, scales [H][n_e/16] at
 *                   byte offsets[e]*H/16).
 * Per expert: amax_row = BF16_RNE(amax_in), amax_col = 4*amax_row, S_enc =
 * min(2688/amax_col, FLT_MAX) (1 if 0).  Per hidden column and block of 16
 * rows: the same transform, block scale and codes as the direct receive's
 * columnwise operand with the BF16 values as input; SR draws from Philox
 * stream 2 (counter as for the direct receive).  The data is read once.
 */
ep_status ep_nvfp4_colwise_rht_bf16(const void *x_bf16, int64_t R_cap,
                                    int64_t H, const int32_t *expert_offsets,
                                    int E, const float *amax_in,
                                    uint8_t *cw_codes, uint8_t *cw_scales,
                                    float *amax_row, float *amax_col,
                                    float *cw_scale_enc, int rounding,
                                    uint64_t seed, uint16_t rht_sign_mask,
                                    uint32_t *dev_status, void *stream);

/*
 * ep_mxfp8_pack -- MXFP8 variant of the pack with the same routing gather.
 * TE PR #3270, description: bfloat16 tokens are quantised to MXFP8 and
 * dispatched; sequence diagram: the quantisation step yields E4M3 data with
 * E8M0 block scales; Changes: the received data and its block scales live in
 * one buffer the caller provides, the data region first and the scales
 * after it.
 *   buf             device u8: data [R_cap, H] then scales [R_cap, H/32].
 * Per 32-element block: e = smallest integer in [-127, 127] with
 * max|x| <= 448*2^e, scale byte e + 127, element E4M3_RNE(x / 2^e).
 * Padding rows are all zero (data and scale bytes).
 */
ep_status ep_mxfp8_pack(const void *tokens_bf16, int64_t T, int64_t H,
                        const int32_t *dest, int k,
                        const int32_t *expert_offsets,
                        const int32_t *expert_counts, int E, uint8_t *buf,
                        int64_t R_cap, uint32_t *dev_status, void *stream);

/*
 * ep_mxfp8_colwise -- the columnwise (weight-gradient) MXFP8 operand of an
 * expert-grouped BF16 tensor: 32-element blocks along the token axis.
 * TE PR #3270, Description: the combine backward returns the expert-output
 * gradient as a per-expert MXFP8 GroupedTensor; Changes: data and block
 * scales in one caller-supplied buffer, data first.
 *   x_bf16          device bf16 [R_cap, H], rows in expert order (expert e:
 *                   rows [expert_offsets[e], expert_offsets[e+1]), whole
 *                   128-row tiles, else EP_DEV_ERR_BAD_EXPERT and the expert
 *                   is skipped).  Finite values.
 *   buf             device u8: data, expert e as [H][n_e] bytes at byte
 *                   expert_offsets[e]*H (column h's rows along the bytes);
 *                   then, from byte R_cap*H, scales, expert e as [H][n_e/32]
 *                   at expert_offsets[e]*H/32.  Bytes of rows past R are left
 *                   untouched.
 * Per column and 32-row block: e = smallest integer in [-127, 127] with
 * max|x| <= 448*2^e, scale byte e + 127, element E4M3_RNE(x / 2^e) (as
 * ep_mxfp8_pack along the other axis).
 */
ep_status ep_mxfp8_colwise(const void *x_bf16, int64_t R_cap, int64_t H,
                           const int32_t *expert_offsets, int E, uint8_t *buf,
                           uint32_t *dev_status, void *stream);

/* Human-readable name of a status code. */
const char *ep_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* EPQ_H */
