/*
 * Oracle: routing plan (the one-GPU stand-in for the expert-parallel
 * transport).  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * TE PR #3270 "EP dispatch with unfused MXFP8 quantization": the dispatch
 * returns "expert-major" received rows as a per-expert grouped tensor
 * (description, sequence diagram), the routing is prepared once and cached
 * (review thread on ep_prepare), and each expert slot is aligned to a multiple
 * of 128 rows (review thread: "each expert slot is 128-aligned").
 * TE PR #3753 "Add NVFP4 EP dispatch and combine backward": the combine
 * backward takes (top_k, alignment, topk_idx_dtype) (commit "layer_args").
 *
 * Reading R7: ids are int32 in [0, E), or -1 for a dropped slot.  An id out
 * of range, or an id repeated within one token, sets a status bit and that
 * slot is dropped (the first occurrence of a repeated id is kept).  Rows of an
 * expert hold its tokens in ascending token order; expert e occupies
 * n_e = ceil(c_e / A) * A rows starting at offsets[e].
 */
#include <stdint.h>
#include <stdlib.h>

#include "oracle.h"

#define OR_BAD_EXPERT 1u
#define OR_DUP_EXPERT 2u

uint32_t or_route_plan(const int32_t *topk, int64_t T, int k, int E, int A,
                       int32_t *offsets, int32_t *counts, int32_t *dest)
{
    uint32_t status = 0;
    /* 1. validate every slot; dest[] temporarily holds the expert id or -1 */
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int32_t e = topk[t * k + j];
            int32_t keep = e;
            if (e == -1) {
                keep = -1;
            } else if (e < 0 || e >= E) {
                status |= OR_BAD_EXPERT;
                keep = -1;
            } else {
                for (int jj = 0; jj < j; ++jj) {
                    if (topk[t * k + jj] == e) {
                        status |= OR_DUP_EXPERT;
                        keep = -1;
                    }
                }
            }
            dest[t * k + j] = keep;
        }
    }
    /* 2. per-expert counts and aligned offsets */
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t i = 0; i < T * (int64_t)k; ++i)
        if (dest[i] >= 0)
            counts[dest[i]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        int32_t n = (counts[e] + A - 1) / A * A;
        offsets[e + 1] = offsets[e] + n;
    }
    /* 3. destinations: walk tokens in ascending order, filling each expert */
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int32_t e = dest[t * k + j];
            if (e < 0)
                continue;
            dest[t * k + j] = offsets[e] + fill[e];
            fill[e] += 1;
        }
    }
    free(fill);
    return status;
}
