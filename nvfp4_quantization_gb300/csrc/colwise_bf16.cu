// Columnwise RHT operand of a BF16 input with a supplied per-expert amax.
//
// TE PR #3755 "Optionally derive FC1 dy NVFP4 amaxes from the dGLU epilogue",
// PR description: the producer (the dGLU epilogue) already knows the exact
// amax; its BF16 rounding is used as the rowwise amax, four times that bounds
// every columnwise value after the RHT, and no separate amax pass over the
// grouped tensor is made.  The input is the
// expert-grouped BF16 gradient; the per-expert encode scale comes from the
// supplied amax, so the data is read once.
//
// Work unit of a warp: 64 rows x 64 columns of one expert (expert slots are
// multiples of 128 rows), 8 KB of BF16 that the warp's own two-stage TMA ring
// brings into shared memory; the warp requests the unit after next as soon as
// its 64 words per lane are in registers, so two units per warp (192 KB per
// SM) are in flight while it computes.  Lane l takes the column pair l of the
// unit: its 64 rows (four 16-row blocks) x 2 columns, runs the 16-point
// transform on FP32 pairs, derives the E4M3 block scales from S_enc and writes
// each column's 32 code bytes (one sector) and 4 scale bytes in one store
// each.  The same arithmetic, in the same order, as the direct receive's
// columnwise operand, with the BF16 values as the decoded input.
#include <float.h>

#include "epq_device.cuh"
#include "epq_internal.h"

namespace epq {

constexpr int kCbMaxExperts = 1024;

constexpr int kCbWarps = 12;         // RHT operand: warps of a CTA, one CTA per SM
constexpr int kCbStages = 2;         // TMA stages per warp
constexpr int kCbUnitRows = 64;
constexpr int kCbUnitWords = 32;     // 64 BF16 columns = 128 bytes per row
constexpr uint32_t kCbUnitBytes = kCbUnitRows * kCbUnitWords * 4;

struct CbRcp {
    float v[128];   // RN(1 / s) for every E4M3 code s (0 for s = 0), computed on the host
};

struct __align__(128) CbSmem {
    uint32_t stage[kCbWarps][kCbStages][kCbUnitRows * kCbUnitWords];
    uint64_t full[kCbWarps][kCbStages];
    float rcp[128];
    // followed by the expert offsets [E + 1] (int) and S_enc [E] (float)
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return u2f(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return u2f(w & 0xffff0000u); }

// x rounded to BF16 (nearest, ties to even), as FP32.
__device__ __forceinline__ float round_bf16(float x)
{
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(x));
    return u2f((uint32_t)h << 16);
}

// Last e with offs[e] <= row.
__device__ __forceinline__ int cb_expert_of_row(const int *offs, int E, int row)
{
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offs[mid] <= row)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// One 16-row block of the column pair held in w[0..15] (low halves: column
// h0, high halves: h0 + 1): the scaled transform, the two block scales (byte
// 0: column h0) and the two columns' 8 code bytes.  pos: Philox position of
// the block's first element in column h0 (SR only); n: the expert's rows.
template <bool kSR>
__device__ __forceinline__ void cb_block(const uint32_t *w, uint32_t sign_mask, float se, const float *rcp_s,
                                         const PhiloxKey &key, uint64_t pos, int n, uint32_t &s2, uint2 &c0,
                                         uint2 &c1)
{
    // u = sigma d / 4 (exact) and the first butterfly stage: one rounding
    // each, fl(u_a + u_b) and fl(u_a - u_b), as FMAs of exact products
    float2 u[16];
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float sa = ((sign_mask >> i) & 1u) ? -0.25f : 0.25f;
        const float sb = ((sign_mask >> (i + 1)) & 1u) ? -0.25f : 0.25f;
        const float2 da = mul2(make_float2(bf16_lo(w[i]), bf16_hi(w[i])), make_float2(sa, sa));
        const float2 db = make_float2(bf16_lo(w[i + 1]), bf16_hi(w[i + 1]));
        u[i] = __ffma2_rn(db, make_float2(sb, sb), da);
        u[i + 1] = __ffma2_rn(db, make_float2(-sb, -sb), da);
    }
#pragma unroll
    for (int len = 2; len < 16; len <<= 1) {
#pragma unroll
        for (int a = 0; a < 16; ++a) {
            if (a & len)
                continue;
            const float2 p = u[a], q = u[a + len];
            u[a] = add2(p, q);
            u[a + len] = sub2(p, q);
        }
    }
    const float p0 = max3_abs(fabsf(u[0].x), u[1].x, u[2].x), q0 = max3_abs(fabsf(u[0].y), u[1].y, u[2].y);
    const float p1 = max3_abs(fabsf(u[3].x), u[4].x, u[5].x), q1 = max3_abs(fabsf(u[3].y), u[4].y, u[5].y);
    const float p2 = max3_abs(fabsf(u[6].x), u[7].x, u[8].x), q2 = max3_abs(fabsf(u[6].y), u[7].y, u[8].y);
    const float p3 = max3_abs(fabsf(u[9].x), u[10].x, u[11].x), q3 = max3_abs(fabsf(u[9].y), u[10].y, u[11].y);
    const float p4 = max3_abs(fabsf(u[12].x), u[13].x, u[14].x), q4 = max3_abs(fabsf(u[12].y), u[13].y, u[14].y);
    const float b0 = fmaxf(fmaxf(p0, p1), max3_abs(fmaxf(p2, p3), p4, u[15].x));
    const float b1 = fmaxf(fmaxf(q0, q1), max3_abs(fmaxf(q2, q3), q4, u[15].y));
    const float ce = __fdiv_rn(se, 6.0f);
    s2 = cvt_e4m3x2(b0 * ce, b1 * ce);
    float2 r2;
    const float2 sv = f16x2_to_f32x2(cvt_f16x2_from_e4m3x2(s2 & 0xffffu));
    if (se >= 0x1p-100f && se <= 0x1p100f) {
        // r = fl32(S_enc / s) by one Markstein step from RN(1/s); s = 0 gives 0
        const float2 y2 = make_float2(rcp_s[s2 & 0xffu], rcp_s[(s2 >> 8) & 0xffu]);
        const float2 se2 = make_float2(se, se);
        const float2 qq = mul2(se2, y2);
        const float2 ee = __ffma2_rn(make_float2(-sv.x, -sv.y), qq, se2);
        r2 = __ffma2_rn(ee, y2, qq);
    } else {
        r2 = make_float2(sv.x == 0.0f ? 0.0f : __fdiv_rn(se, sv.x), sv.y == 0.0f ? 0.0f : __fdiv_rn(se, sv.y));
    }
#pragma unroll
    for (int i = 0; i < 16; ++i)
        u[i] = mul2(u[i], r2);
    if (kSR) {
        // rows 4q .. 4q + 3 of the block take word q of its column's Philox output (stream 2)
        const Philox4 ra = sr_bytes16_36(key, 2u, pos);
        const Philox4 rb = sr_bytes16_36(key, 2u, pos + (uint64_t)n);
        c0 = make_uint2(cvt_e2m1x8_sr(u[0].x, u[1].x, u[2].x, u[3].x, u[4].x, u[5].x, u[6].x, u[7].x, ra.x, ra.y),
                        cvt_e2m1x8_sr(u[8].x, u[9].x, u[10].x, u[11].x, u[12].x, u[13].x, u[14].x, u[15].x, ra.z,
                                      ra.w));
        c1 = make_uint2(cvt_e2m1x8_sr(u[0].y, u[1].y, u[2].y, u[3].y, u[4].y, u[5].y, u[6].y, u[7].y, rb.x, rb.y),
                        cvt_e2m1x8_sr(u[8].y, u[9].y, u[10].y, u[11].y, u[12].y, u[13].y, u[14].y, u[15].y, rb.z,
                                      rb.w));
    } else {
        c0 = make_uint2(cvt_e2m1x8(u[0].x, u[1].x, u[2].x, u[3].x, u[4].x, u[5].x, u[6].x, u[7].x),
                        cvt_e2m1x8(u[8].x, u[9].x, u[10].x, u[11].x, u[12].x, u[13].x, u[14].x, u[15].x));
        c1 = make_uint2(cvt_e2m1x8(u[0].y, u[1].y, u[2].y, u[3].y, u[4].y, u[5].y, u[6].y, u[7].y),
                        cvt_e2m1x8(u[8].y, u[9].y, u[10].y, u[11].y, u[12].y, u[13].y, u[14].y, u[15].y));
    }
}

__device__ __forceinline__ void st_global_32B(uint8_t *p, uint2 a, uint2 b, uint2 c, uint2 d, bool v8)
{
    if (v8) {
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x), "r"(a.y),
                     "r"(b.x), "r"(b.y), "r"(c.x), "r"(c.y), "r"(d.x), "r"(d.y)
                     : "memory");
    } else {
        reinterpret_cast<uint4 *>(p)[0] = make_uint4(a.x, a.y, b.x, b.y);
        reinterpret_cast<uint4 *>(p)[1] = make_uint4(c.x, c.y, d.x, d.y);
    }
}

template <bool kSR>
__global__ void __launch_bounds__(kCbWarps * 32, 1)
colwise_rht_bf16_kernel(const __grid_constant__ CUtensorMap tm_x, int H, int R_cap,
                        const int32_t *__restrict__ offsets, int E, const float *__restrict__ amax_in,
                        uint8_t *__restrict__ cw_codes, uint8_t *__restrict__ cw_scales, float *__restrict__ amax_row,
                        float *__restrict__ amax_col, float *__restrict__ scale_enc,
                        const __grid_constant__ PhiloxKey key, uint32_t sign_mask, uint32_t *__restrict__ status,
                        const __grid_constant__ CbRcp rcp, int codes_v8)
{
    extern __shared__ uint8_t cb_smem_raw[];
    CbSmem &sm = *reinterpret_cast<CbSmem *>((reinterpret_cast<uintptr_t>(cb_smem_raw) + 127) & ~(uintptr_t)127);
    int *offs = reinterpret_cast<int *>(&sm + 1);        // [E + 1]
    float *se_s = reinterpret_cast<float *>(offs + E + 1);  // [E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (lane == 0) {
        for (int s = 0; s < kCbStages; ++s)
            mbar_init(&sm.full[warp][s], 1);
        fence_mbar_init();
        if (warp == 0)
            tma_prefetch_desc(&tm_x);
    }
    pdl_launch_dependents();
    pdl_wait();
    for (int i = tid; i <= E; i += blockDim.x)
        offs[i] = __ldg(offsets + i);
    for (int i = tid; i < 128; i += blockDim.x)
        sm.rcp[i] = rcp.v[i];
    // per expert: amax_row = BF16_RNE(supplied amax), amax_col = 4 amax_row,
    // S_enc = min(2688 / amax_col, FLT_MAX) (1 when amax_col = 0)
    for (int e = tid; e < E; e += blockDim.x) {
        const float a = round_bf16(__ldg(amax_in + e));
        float ac;
        const float se = colwise_encode_scale(a, ac);
        se_s[e] = se;
        if (blockIdx.x == 0) {
            amax_row[e] = a;
            amax_col[e] = ac;
            scale_enc[e] = se;
        }
    }
    __syncthreads();
    int R = offs[E];
    if (R > R_cap) {
        if (blockIdx.x == 0 && tid == 0)
            raise_status(status, kDevErrCapacity);
        R = R_cap;
    }
    const int ngrp = (H + 63) / 64;   // 64-column groups of a row
    const int64_t n_units = (int64_t)(R / kCbUnitRows) * ngrp;
    const int64_t stride = (int64_t)gridDim.x * kCbWarps;
    const int64_t u0 = (int64_t)blockIdx.x * kCbWarps + warp;
    uint32_t *const stg = sm.stage[warp][0];
    uint64_t *const full = sm.full[warp];
    auto issue = [&](int64_t u, int s) {
        const int rb = (int)(u / ngrp), cg = (int)(u % ngrp);
        mbar_arrive_expect_tx(&full[s], kCbUnitBytes);
        tma_load_2d(stg + s * (kCbUnitRows * kCbUnitWords), &tm_x, 128 * cg, kCbUnitRows * rb, &full[s]);
    };
    int issued = 0;
    if (lane == 0) {
        for (int s = 0; s < kCbStages; ++s) {
            if (u0 + s * stride >= n_units)
                break;
            issue(u0 + s * stride, s);
            ++issued;
        }
    }
    issued = __shfl_sync(0xffffffffu, issued, 0);

    int it = 0;
    for (int64_t wu = u0; wu < n_units; wu += stride, ++it) {
        const int s = it % kCbStages;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (uint32_t)(it / kCbStages) & 1u))) {
            if (lane == 0)
                raise_status(status, kDevErrTimeout);
            break;
        }
        uint32_t w[kCbUnitRows];
        const uint32_t *src = stg + s * (kCbUnitRows * kCbUnitWords) + lane;
#pragma unroll
        for (int r = 0; r < kCbUnitRows; ++r)
            w[r] = src[r * kCbUnitWords];
        // every lane's reads of the stage are done before it is refilled
        __syncwarp();
        if (wu + kCbStages * stride < n_units) {
            if (lane == 0)
                issue(wu + kCbStages * stride, s);
            ++issued;
        }
        const int rb = (int)(wu / ngrp), cg = (int)(wu % ngrp);
        const int row0 = kCbUnitRows * rb;
        const int e = cb_expert_of_row(offs, E, row0);
        const int off = offs[e], n = offs[e + 1] - off, rl = row0 - off;
        if ((off & 127) != 0 || (n & 127) != 0) {
            // an expert slot that is not whole 128-row tiles: skipped
            if (lane == 0)
                raise_status(status, kDevErrBadExpert);
            continue;
        }
        const int h0 = 64 * cg + 2 * lane;   // columns h0 and h0 + 1
        if (h0 >= H)
            continue;
        const float se = se_s[e];
        const uint64_t pos = (uint64_t)off * (uint64_t)H + (uint64_t)h0 * (uint64_t)n + (uint64_t)rl;
        uint32_t s2[4];
        uint2 c0[4], c1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            cb_block<kSR>(w + 16 * j, sign_mask, se, sm.rcp, key, pos + 16 * j, n, s2[j], c0[j], c1[j]);
        uint8_t *d0 = cw_codes + (int64_t)off * (H / 2) + (int64_t)h0 * (n / 2) + rl / 2;
        st_global_32B(d0, c0[0], c0[1], c0[2], c0[3], codes_v8 != 0);
        st_global_32B(d0 + n / 2, c1[0], c1[1], c1[2], c1[3], codes_v8 != 0);
        uint8_t *cs = cw_scales + (int64_t)off * (H / 16) + (int64_t)h0 * (n / 16) + rl / 16;
        *reinterpret_cast<uint32_t *>(cs) = pack4(s2[0] & 0xffu, s2[1] & 0xffu, s2[2] & 0xffu, s2[3] & 0xffu);
        *reinterpret_cast<uint32_t *>(cs + n / 16) =
            pack4((s2[0] >> 8) & 0xffu, (s2[1] >> 8) & 0xffu, (s2[2] >> 8) & 0xffu, (s2[3] >> 8) & 0xffu);
    }
    // never leave with a load of this warp's ring still in flight (after a
    // wait that gave up)
    if (lane == 0)
        for (int i = it; i < issued; ++i)
            (void)mbar_wait_bounded(&full[i % kCbStages], (uint32_t)(i / kCbStages) & 1u);
}

// ---------------------------------------------------------------- MXFP8 columnwise
// The weight-gradient operand of the MXFP8 recipe (TE PR #3270 "EP dispatch
// with unfused MXFP8 quantization", Description: the combine backward returns
// the expert-output gradient as a per-expert MXFP8 GroupedTensor): blocks of
// 32 consecutive rows of one expert per hidden column, the E8M0 exponent e the
// smallest in [-127, 127] with max|x| <= 448 * 2^e, elements E4M3_RNE(x / 2^e).
// Work unit of a warp: 128 rows x 64 columns of one expert (16 KB of BF16),
// streamed through the warp's own two-stage TMA ring; lane l takes the column
// pair l and the unit's four 32-row blocks in turn, reading each block's 32
// words from the stage: the two columns' block maxima on the BF16 bit
// patterns, 32 data bytes per column (one sector) per block, so each column's
// 128-byte line of the unit comes from one lane, and after the four blocks the
// column's 4 scale bytes in one store.
constexpr int kMxWarps = 6;          // warps of a CTA, one CTA per SM
constexpr int kMxUnitRows = 128;
constexpr uint32_t kMxUnitBytes = kMxUnitRows * kCbUnitWords * 4;

struct __align__(128) MxSmem {
    uint32_t stage[kMxWarps][kCbStages][kMxUnitRows * kCbUnitWords];
    uint64_t full[kMxWarps][kCbStages];
    // followed by the expert offsets [E + 1] (int)
};

template <bool kV8>
__global__ void __launch_bounds__(kMxWarps * 32, 1)
mxfp8_colwise_kernel(const __grid_constant__ CUtensorMap tm_x, int H, int R_cap, const int32_t *__restrict__ offsets,
                     int E, uint8_t *__restrict__ buf, uint32_t *__restrict__ status)
{
    extern __shared__ uint8_t mx_smem_raw[];
    MxSmem &sm = *reinterpret_cast<MxSmem *>((reinterpret_cast<uintptr_t>(mx_smem_raw) + 127) & ~(uintptr_t)127);
    int *offs = reinterpret_cast<int *>(&sm + 1);   // [E + 1]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (lane == 0) {
        for (int s = 0; s < kCbStages; ++s)
            mbar_init(&sm.full[warp][s], 1);
        fence_mbar_init();
        if (warp == 0)
            tma_prefetch_desc(&tm_x);
    }
    pdl_launch_dependents();
    pdl_wait();
    for (int i = tid; i <= E; i += blockDim.x)
        offs[i] = __ldg(offsets + i);
    __syncthreads();
    int R = offs[E];
    if (R > R_cap) {
        if (blockIdx.x == 0 && tid == 0)
            raise_status(status, kDevErrCapacity);
        R = R_cap;
    }
    uint8_t *data = buf;
    uint8_t *scales = buf + (int64_t)R_cap * H;
    const int ngrp = (H + 63) / 64;
    const int64_t n_units = (int64_t)(R / kMxUnitRows) * ngrp;
    const int64_t stride = (int64_t)gridDim.x * kMxWarps;
    const int64_t u0 = (int64_t)blockIdx.x * kMxWarps + warp;
    uint32_t *const stg = sm.stage[warp][0];
    uint64_t *const full = sm.full[warp];
    auto issue = [&](int64_t u, int s) {
        const int rb = (int)(u / ngrp), cg = (int)(u % ngrp);
        mbar_arrive_expect_tx(&full[s], kMxUnitBytes);
        tma_load_2d(stg + s * (kMxUnitRows * kCbUnitWords), &tm_x, 128 * cg, kMxUnitRows * rb, &full[s]);
    };
    int issued = 0;
    if (lane == 0) {
        for (int s = 0; s < kCbStages; ++s) {
            if (u0 + s * stride >= n_units)
                break;
            issue(u0 + s * stride, s);
            ++issued;
        }
    }
    issued = __shfl_sync(0xffffffffu, issued, 0);

    int it = 0;
    for (int64_t wu = u0; wu < n_units; wu += stride, ++it) {
        const int s = it % kCbStages;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (uint32_t)(it / kCbStages) & 1u))) {
            if (lane == 0)
                raise_status(status, kDevErrTimeout);
            break;
        }
        const int rb = (int)(wu / ngrp), cg = (int)(wu % ngrp);
        const int row0 = kMxUnitRows * rb;
        const int e = cb_expert_of_row(offs, E, row0);
        const int off = offs[e], n = offs[e + 1] - off, rl = row0 - off;
        const bool bad = (off & 127) != 0 || (n & 127) != 0;
        if (bad && lane == 0)
            raise_status(status, kDevErrBadExpert);   // an expert slot that is not whole 128-row tiles: skipped
        const int h0 = 64 * cg + 2 * lane;            // columns h0 and h0 + 1
        if (!bad && h0 < H) {
            const uint32_t *src = stg + s * (kMxUnitRows * kCbUnitWords) + lane;
            uint8_t *dp = data + (int64_t)off * H + (int64_t)h0 * n + rl;
            uint32_t sw0 = 0u, sw1 = 0u;
#pragma unroll 1
            for (int b = 0; b < 4; ++b) {
                uint32_t wv[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    wv[i] = src[(32 * b + i) * kCbUnitWords];
                // block maxima of both columns on the bit patterns (finite BF16:
                // for non-negative values integer order is value order)
                uint32_t m = wv[0];
#pragma unroll
                for (int i = 1; i < 32; ++i)
                    asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(wv[i]));
                m &= 0x7fff7fffu;
                float f[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint32_t bm = q ? (m >> 16) : (m & 0xffffu);
                    // smallest e in [-127, 127] with B <= 448 * 2^e; 448 = 1.75 * 2^8,
                    // i.e. BF16 exponent field 135 with mantissa field 96
                    const int ef = (int)((bm >> 7) & 0xffu), mt = (int)(bm & 0x7fu);
                    int ex = (ef == 0) ? -127 : ef - 135 + (mt > 96 ? 1 : 0);
                    ex = max(-127, min(127, ex));
                    f[q] = (ex <= 126) ? exp2i(-ex) : u2f(0x00400000u);   // 2^-e
                    if (q)
                        sw1 |= (uint32_t)(ex + 127) << (8 * b);
                    else
                        sw0 |= (uint32_t)(ex + 127) << (8 * b);
                }
                uint32_t d0[8], d1[8];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float2 a0 = mul2(make_float2(bf16_lo(wv[i]), bf16_lo(wv[i + 1])), make_float2(f[0], f[0]));
                    const float2 a1 = mul2(make_float2(bf16_lo(wv[i + 2]), bf16_lo(wv[i + 3])), make_float2(f[0], f[0]));
                    const float2 c0 = mul2(make_float2(bf16_hi(wv[i]), bf16_hi(wv[i + 1])), make_float2(f[1], f[1]));
                    const float2 c1 = mul2(make_float2(bf16_hi(wv[i + 2]), bf16_hi(wv[i + 3])), make_float2(f[1], f[1]));
                    d0[i / 4] = cvt_e4m3x2(a0.x, a0.y) | (cvt_e4m3x2(a1.x, a1.y) << 16);
                    d1[i / 4] = cvt_e4m3x2(c0.x, c0.y) | (cvt_e4m3x2(c1.x, c1.y) << 16);
                }
                st_global_32B(dp + 32 * b, make_uint2(d0[0], d0[1]), make_uint2(d0[2], d0[3]),
                              make_uint2(d0[4], d0[5]), make_uint2(d0[6], d0[7]), kV8);
                st_global_32B(dp + n + 32 * b, make_uint2(d1[0], d1[1]), make_uint2(d1[2], d1[3]),
                              make_uint2(d1[4], d1[5]), make_uint2(d1[6], d1[7]), kV8);
            }
            uint8_t *sp = scales + (int64_t)off * (H / 32) + (int64_t)h0 * (n / 32) + rl / 32;
            *reinterpret_cast<uint32_t *>(sp) = sw0;
            *reinterpret_cast<uint32_t *>(sp + n / 32) = sw1;
        }
        // every lane's reads of the stage are done: load it with the unit after next
        __syncwarp();
        if (wu + kCbStages * stride < n_units) {
            if (lane == 0)
                issue(wu + kCbStages * stride, s);
            ++issued;
        }
    }
    // never leave with a load of this warp's ring in flight (after a wait that gave up)
    if (lane == 0)
        for (int i = it; i < issued; ++i)
            (void)mbar_wait_bounded(&full[i % kCbStages], (uint32_t)(i / kCbStages) & 1u);
}

cudaError_t launch_mxfp8_colwise(const LaunchCtx &c, const uint16_t *x, int R_cap, int H, const int32_t *offsets,
                                 int E, uint8_t *buf, uint32_t *status)
{
    CUtensorMap tm_x;
    if (!make_map(&tm_x, x, 2 * (uint64_t)H, (uint64_t)(R_cap > 0 ? R_cap : 1), 2 * (uint64_t)H,
                  kCbUnitWords * 4, kMxUnitRows))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(MxSmem) + 128 + (size_t)(E + 1) * 4;
    const bool v8 = (reinterpret_cast<uintptr_t>(buf) & 31u) == 0;
    static std::atomic<uint32_t> done[2][2] = {};
    auto kern = v8 ? mxfp8_colwise_kernel<true> : mxfp8_colwise_kernel<false>;
    cudaError_t err = ensure_smem_limit(kern, c.device, (int)(sizeof(MxSmem) + 128 + (kCbMaxExperts + 1) * 4),
                                        done[v8 ? 1 : 0]);
    if (err != cudaSuccess)
        return err;
    const int64_t units = (int64_t)(R_cap / kMxUnitRows) * ((H + 63) / 64);
    int64_t grid = (units + kMxWarps - 1) / kMxWarps;
    if (grid > c.num_sms)
        grid = c.num_sms;   // one resident CTA per SM
    if (grid < 1)
        grid = 1;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kMxWarps * 32), smem, c.stream, tm_x, H, R_cap, offsets, E,
                      buf, status);
}

static CbRcp make_cb_rcp()
{
    CbRcp t;
    for (int code = 0; code < 128; ++code) {
        const int ex = code >> 3, mt = code & 7;
        const float v = ex == 0 ? (float)mt * (1.0f / 512.0f) : (1.0f + (float)mt / 8.0f) * ldexpf(1.0f, ex - 7);
        t.v[code] = (v == 0.0f || code == 127) ? 0.0f : 1.0f / v;   // IEEE single division: RN(1/v)
    }
    return t;
}

cudaError_t launch_colwise_rht_bf16(const LaunchCtx &c, const uint16_t *x, int R_cap, int H, const int32_t *offsets,
                                    int E, const float *amax_in, uint8_t *cw_codes, uint8_t *cw_scales,
                                    float *amax_row, float *amax_col, float *scale_enc, int rounding, uint64_t seed,
                                    uint32_t sign_mask, uint32_t *status)
{
    static const CbRcp rcp = make_cb_rcp();
    // the input as a byte tensor [R_cap][2H]; a box is one unit, 64 rows x 128
    // bytes (a last column group past H reads zeros and is not stored)
    CUtensorMap tm_x;
    if (!make_map(&tm_x, x, 2 * (uint64_t)H, (uint64_t)(R_cap > 0 ? R_cap : 1), 2 * (uint64_t)H,
                  kCbUnitWords * 4, kCbUnitRows))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(CbSmem) + 128 + (size_t)(2 * E + 1) * 4;
    static std::atomic<uint32_t> done[2][2] = {};
    auto kern = rounding == 1 ? colwise_rht_bf16_kernel<true> : colwise_rht_bf16_kernel<false>;
    cudaError_t err = ensure_smem_limit(kern, c.device, (int)(sizeof(CbSmem) + 128 + (2 * kCbMaxExperts + 1) * 4),
                                        done[rounding == 1 ? 1 : 0]);
    if (err != cudaSuccess)
        return err;
    const int64_t units = (int64_t)(R_cap / kCbUnitRows) * ((H + 63) / 64);
    int64_t grid = (units + kCbWarps - 1) / kCbWarps;
    if (grid > c.num_sms)
        grid = c.num_sms;   // one resident CTA per SM
    if (grid < 1)
        grid = 1;
    const int v8 = (reinterpret_cast<uintptr_t>(cw_codes) & 31u) == 0;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kCbWarps * 32), smem, c.stream, tm_x, H, R_cap, offsets, E,
                      amax_in, cw_codes, cw_scales, amax_row, amax_col, scale_enc, philox_key(seed), sign_mask,
                      status, rcp, v8);
}

} // namespace epq
