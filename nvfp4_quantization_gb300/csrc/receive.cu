// Direct receive: packed NVFP4 rows -> the expert GEMM's grouped rowwise and
// columnwise-RHT NVFP4 operands, in one pass over the rows.
//
// TE PR #3753 "Add NVFP4 EP dispatch and combine backward", PR description:
// the receiver builds the NVFP4 GroupedTensor straight from the rows in one
// pass; the rowwise operand reuses the sender's codes; the columnwise RHT
// operand is quantised with a bound-derived per-expert scale (no BF16 round
// trip, no amax pass over the data).  TE PR #3755 "Optionally derive FC1 dy
// NVFP4 amaxes from the dGLU epilogue", PR description: the post-RHT
// columnwise amax is bounded by 4x the rowwise amax.
//
// Kernel 1 (expert_amax): one CTA per expert reduces the 4-byte token amaxes
// in the row trailers (the rows' data is not read) into amax_row, the 4x
// bound amax_col and the encode scale S_enc.
//
// Kernel 2 (direct_receive): persistent CTAs walk tiles of 128 rows x 256
// hidden columns (a tile never straddles two experts: expert slots are
// multiples of 128 rows), row-tile-major so that concurrently running CTAs
// share row trailers and complete each other's output sectors in L2.  One
// producer thread streams tiles into a 4-stage shared-memory ring with 2-D
// TMA loads (codes box 128 B x 128 rows, scales 16 B x 128, trailers
// 16 B x 128).  The rowwise operand leaves straight from the ring with a TMA
// store (codes) and 16-byte stores (scales, token scale).  Each of 128
// consumer threads owns two adjacent hidden columns (one code byte per row):
// it decodes 16 rows at a time exactly into FP32 pairs using a per-tile
// table of (E4M3 block scale x token scale x sigma / 4), runs the 16-point
// Walsh-Hadamard butterflies on packed FP32 pairs, derives the E4M3 block
// scale from the expert's S_enc, re-encodes to E2M1 (RNE or Philox-driven
// stochastic rounding) and keeps the 64 code bytes and 8 scale bytes of each
// column in registers until the tile is done, then writes them as whole
// 16-byte chunks of the [H][n_e] columnwise layout.
#include <cudaTypedefs.h>
#include <float.h>
#include <string.h>

#include "epq_device.cuh"
#include "epq_internal.h"

namespace epq {

constexpr int kTileRows = 128;
constexpr int kTileCols = 256;
constexpr int kCodeBytes = kTileCols / 2;    // 128
constexpr int kScaleBytes = kTileCols / 16;  // 16
constexpr int kStages = 4;
constexpr int kConsumers = 128;              // 4 warps, 2 columns per thread
constexpr int kThreads = kConsumers + 32;    // + 1 producer warp
constexpr uint32_t kStageTx = kTileRows * (kCodeBytes + kScaleBytes + 16);
constexpr int kTabStride = kTileRows + 4;    // pad: 4 column blocks per warp hit distinct banks

struct __align__(128) DrSmem {
    uint8_t codes[kStages][kTileRows][kCodeBytes];
    uint8_t scales[kStages][kTileRows][kScaleBytes];
    uint32_t trailer[kStages][kTileRows][4];
    float table[2][kScaleBytes][kTabStride];  // [buf][column block][row]
    float rtab[2][128];                       // [buf][E4M3 code] -> S_enc / s
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int abort_flag;
    int consumed;
};

// --------------------------------------------------------------- kernel 1
__global__ void __launch_bounds__(256)
expert_amax_kernel(const uint8_t *__restrict__ rows, int R_cap, int64_t S,
                   const int32_t *__restrict__ offsets, int E, float *__restrict__ amax_row,
                   float *__restrict__ amax_col, float *__restrict__ scale_enc,
                   uint32_t *__restrict__ status)
{
    __shared__ uint32_t wm[8];
    pdl_launch_dependents();
    pdl_wait();
    const int e = blockIdx.x;
    int lo = offsets[e], hi = offsets[e + 1];
    if (hi > R_cap) {
        if (threadIdx.x == 0)
            raise_status(status, kDevErrCapacity);
        hi = R_cap;
    }
    uint32_t m = 0; // token amaxes are non-negative: compare their bit patterns
    for (int r = lo + threadIdx.x; r < hi; r += blockDim.x)
        m = max(m, __ldg(reinterpret_cast<const uint32_t *>(rows + (int64_t)r * S + S - 12)));
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0)
        wm[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < 8; ++i)
            m = max(m, wm[i]);
        const float a = u2f(m);
        const float ac = 4.0f * a;
        float se = 1.0f;
        if (ac > 0.0f)
            se = fminf(__fdiv_rn(2688.0f, ac), FLT_MAX);
        amax_row[e] = a;
        amax_col[e] = ac;
        scale_enc[e] = se;
    }
}

// --------------------------------------------------------------- kernel 2
struct DrArgs {
    const int32_t *offsets;
    int E;
    int H;
    int R_cap;
    int n_strips;
    uint8_t *rw_scales;
    float *rw_row_scale;
    uint8_t *cw_codes;
    uint8_t *cw_scales;
    const float *scale_enc;
    uint64_t seed;
    uint32_t sign_mask;
    uint32_t *status;
    int do_rowwise;
};

__device__ __forceinline__ int expert_of_row(const int32_t *offsets, int E, int row)
{
    int lo = 0, hi = E - 1; // last e with offsets[e] <= row
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(offsets + mid) <= row)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void st16g(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

template <bool kSR>
__device__ __forceinline__ void consumer_loop(DrSmem &sm, const CUtensorMap *tm_rw, const DrArgs &p,
                                              int n_units)
{
    const int c = threadIdx.x; // 0..127
    const int H = p.H;
    int it = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++it) {
        const int s = it % kStages;
        const uint32_t ph = (uint32_t)(it / kStages) & 1u;
        const int buf = it & 1;
        bool failed = false;
        if (!mbar_wait_bounded(&sm.full[s], ph)) {
            failed = true;
            sm.abort_flag = 1;
            raise_status(p.status, kDevErrTimeout);
        }
        const int rt = u / p.n_strips, st = u - rt * p.n_strips;
        const int row0 = rt * kTileRows;
        const int e = expert_of_row(p.offsets, p.E, row0);
        const int off_e = __ldg(p.offsets + e);
        const int n_e = __ldg(p.offsets + e + 1) - off_e;
        const int rl = row0 - off_e;

        // rowwise operand: codes by TMA store, scales and token scale by threads
        if (p.do_rowwise && !failed) {
            if (c == 0) {
                tma_store_2d(tm_rw, st * kCodeBytes, row0, &sm.codes[s][0][0]);
                tma_store_commit();
            }
            const int nb = min(kScaleBytes, H / 16 - st * kScaleBytes);
            uint8_t *dst = p.rw_scales + (int64_t)(row0 + c) * (H / 16) + st * kScaleBytes;
            const uint8_t *src = &sm.scales[s][c][0];
            if (nb == kScaleBytes && ((H / 16) % 16) == 0) {
                st16g(dst, *reinterpret_cast<const uint4 *>(src));
            } else {
                for (int b = 0; b < nb; b += 2)
                    *reinterpret_cast<uint16_t *>(dst + b) = *reinterpret_cast<const uint16_t *>(src + b);
            }
            if (st == 0)
                p.rw_row_scale[row0 + c] = u2f(sm.trailer[s][c][0]);
        }

        // per-tile tables: decode scale of (row c, column block cb) with the
        // RHT sign and the 1/4 folded in (exact), and S_enc / s per E4M3 code
        {
            float rs = u2f(sm.trailer[s][c][0]) * 0.25f;
            if ((p.sign_mask >> (c & 15)) & 1u)
                rs = -rs;
            const uint32_t *sc4 = reinterpret_cast<const uint32_t *>(&sm.scales[s][c][0]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t w = sc4[q];
                const float2 a = f16x2_to_f32x2(cvt_f16x2_from_e4m3x2(w & 0xffffu));
                const float2 b = f16x2_to_f32x2(cvt_f16x2_from_e4m3x2(w >> 16));
                sm.table[buf][4 * q + 0][c] = a.x * rs;
                sm.table[buf][4 * q + 1][c] = a.y * rs;
                sm.table[buf][4 * q + 2][c] = b.x * rs;
                sm.table[buf][4 * q + 3][c] = b.y * rs;
            }
            const float se = __ldg(p.scale_enc + e);
            const float sv = e4m3_to_f32((uint32_t)c);
            sm.rtab[buf][c] = (sv == 0.0f) ? 0.0f : __fdiv_rn(se, sv);
        }
        // one decision for all consumers: stop if any wait gave up
        if (named_bar_or(1, kConsumers, failed || sm.abort_flag != 0))
            break;

        const float se = __ldg(p.scale_enc + e);
        const float ce = __fdiv_rn(se, 6.0f);
        const int h0 = st * kTileCols + 2 * c;
        if (h0 < H) {
            const int cb = c >> 3;
            uint32_t cw0[16], cw1[16];
            uint32_t sc0[2] = {0u, 0u}, sc1[2] = {0u, 0u};
#pragma unroll
            for (int blk = 0; blk < 8; ++blk) {
                const float4 *tp = reinterpret_cast<const float4 *>(&sm.table[buf][cb][blk * 16]);
                float scv[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 t4 = tp[q];
                    scv[4 * q + 0] = t4.x; scv[4 * q + 1] = t4.y;
                    scv[4 * q + 2] = t4.z; scv[4 * q + 3] = t4.w;
                }
                float2 u[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint32_t byte = sm.codes[s][blk * 16 + i][c];
                    const float2 qv = f16x2_to_f32x2(cvt_f16x2_from_e2m1x2(byte));
                    u[i] = mul2(qv, make_float2(scv[i], scv[i]));
                }
                // 16-point Walsh-Hadamard butterflies, len = 1, 2, 4, 8
#pragma unroll
                for (int len = 1; len < 16; len <<= 1) {
#pragma unroll
                    for (int a = 0; a < 16; ++a) {
                        if (a & len)
                            continue;
                        const float2 x = u[a], y = u[a + len];
                        u[a] = add2(x, y);
                        u[a + len] = sub2(x, y);
                    }
                }
                float b0 = 0.0f, b1 = 0.0f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    b0 = fmaxf(b0, fabsf(u[i].x));
                    b1 = fmaxf(b1, fabsf(u[i].y));
                }
                const uint32_t s2 = cvt_e4m3x2(b0 * ce, b1 * ce);
                const uint32_t s0 = s2 & 0xffu, s1 = (s2 >> 8) & 0xffu;
                const float2 r2 = make_float2(sm.rtab[buf][s0], sm.rtab[buf][s1]);
                sc0[blk >> 2] |= s0 << (8 * (blk & 3));
                sc1[blk >> 2] |= s1 << (8 * (blk & 3));
                float2 v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[i] = mul2(u[i], r2);
                if (kSR) {
                    const uint64_t pos = (uint64_t)off_e * (uint64_t)H + (uint64_t)h0 * (uint64_t)n_e +
                                         (uint64_t)(rl + blk * 16);
                    const Philox4 ra = sr_bytes16(p.seed, 1u, pos);
                    const Philox4 rb = sr_bytes16(p.seed, 1u, pos + (uint64_t)n_e);
                    const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w};
                    const uint32_t wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        v[i].x = sr_e2m1_value(v[i].x, (wa[i >> 2] >> (8 * (i & 3))) & 0xffu);
                        v[i].y = sr_e2m1_value(v[i].y, (wb[i >> 2] >> (8 * (i & 3))) & 0xffu);
                    }
                }
                uint32_t a0 = 0u, a1 = 0u, b0w = 0u, b1w = 0u;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    a0 |= cvt_e2m1x2(v[2 * m].x, v[2 * m + 1].x) << (8 * m);
                    a1 |= cvt_e2m1x2(v[8 + 2 * m].x, v[8 + 2 * m + 1].x) << (8 * m);
                    b0w |= cvt_e2m1x2(v[2 * m].y, v[2 * m + 1].y) << (8 * m);
                    b1w |= cvt_e2m1x2(v[8 + 2 * m].y, v[8 + 2 * m + 1].y) << (8 * m);
                }
                cw0[2 * blk] = a0;
                cw0[2 * blk + 1] = a1;
                cw1[2 * blk] = b0w;
                cw1[2 * blk + 1] = b1w;
            }
            // columns h0 and h0+1: 64 code bytes and 8 scale bytes each
            uint8_t *cc = p.cw_codes + (int64_t)off_e * (H / 2) + (int64_t)(rl / 2);
            uint8_t *cs = p.cw_scales + (int64_t)off_e * (H / 16) + (int64_t)(rl / 16);
            uint8_t *d0 = cc + (int64_t)h0 * (n_e / 2);
            uint8_t *d1 = d0 + (n_e / 2);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                st16g(d0 + 16 * q, make_uint4(cw0[4 * q], cw0[4 * q + 1], cw0[4 * q + 2], cw0[4 * q + 3]));
                st16g(d1 + 16 * q, make_uint4(cw1[4 * q], cw1[4 * q + 1], cw1[4 * q + 2], cw1[4 * q + 3]));
            }
            *reinterpret_cast<uint2 *>(cs + (int64_t)h0 * (n_e / 16)) = make_uint2(sc0[0], sc0[1]);
            *reinterpret_cast<uint2 *>(cs + (int64_t)(h0 + 1) * (n_e / 16)) = make_uint2(sc1[0], sc1[1]);
        }

        // release the stage (after the rowwise TMA store has read it)
        if (c == 0 && p.do_rowwise)
            tma_store_wait_read0();
        __syncwarp();
        if ((c & 31) == 0)
            mbar_arrive(&sm.empty[s]);
    }
    if (c == 0) {
        sm.consumed = it;
        if (p.do_rowwise)
            tma_store_wait0();
    }
}

__global__ void __launch_bounds__(kThreads, 2)
direct_receive_kernel(const __grid_constant__ CUtensorMap tm_codes,
                      const __grid_constant__ CUtensorMap tm_scales,
                      const __grid_constant__ CUtensorMap tm_trailer,
                      const __grid_constant__ CUtensorMap tm_rw, DrArgs p, int sr)
{
    extern __shared__ uint8_t smem_raw[];
    DrSmem &sm = *reinterpret_cast<DrSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kConsumers / 32);
        }
        sm.abort_flag = 0;
        sm.consumed = 0;
        fence_mbar_init();
    }
    if (warp == kConsumers / 32 && lane == 0) {
        tma_prefetch_desc(&tm_codes);
        tma_prefetch_desc(&tm_scales);
        tma_prefetch_desc(&tm_trailer);
    }
    __syncthreads();
    pdl_launch_dependents();
    pdl_wait();

    int R = __ldg(p.offsets + p.E);
    if (R > p.R_cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            raise_status(p.status, kDevErrCapacity);
        R = p.R_cap;
    }
    const int n_units = (R / kTileRows) * p.n_strips;

    int issued = 0;
    if (warp == kConsumers / 32) {
        if (lane == 0) {
            for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++issued) {
                const int s = issued % kStages;
                const uint32_t ph = (uint32_t)(issued / kStages) & 1u;
                if (!mbar_wait_bounded(&sm.empty[s], ph ^ 1u)) {
                    sm.abort_flag = 1;
                    raise_status(p.status, kDevErrTimeout);
                    break;
                }
                if (sm.abort_flag)
                    break;
                const int rt = u / p.n_strips, st = u - rt * p.n_strips;
                mbar_arrive_expect_tx(&sm.full[s], kStageTx);
                tma_load_2d(&sm.codes[s][0][0], &tm_codes, st * kCodeBytes, rt * kTileRows, &sm.full[s]);
                tma_load_2d(&sm.scales[s][0][0], &tm_scales, st * kScaleBytes, rt * kTileRows, &sm.full[s]);
                tma_load_2d(&sm.trailer[s][0][0], &tm_trailer, 0, rt * kTileRows, &sm.full[s]);
            }
        }
    } else if (sr) {
        consumer_loop<true>(sm, &tm_rw, p, n_units);
    } else {
        consumer_loop<false>(sm, &tm_rw, p, n_units);
    }
    __syncthreads();
    // never leave with a tile load still in flight (only after an abort)
    if (warp == kConsumers / 32 && lane == 0) {
        for (int i = sm.consumed; i < issued; ++i)
            (void)mbar_wait_bounded(&sm.full[i % kStages], (uint32_t)(i / kStages) & 1u);
    }
}

// --------------------------------------------------------------- host
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2-D byte tensor [outer][inner] with a row pitch of `pitch` bytes.
static bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t pitch,
                     uint32_t box_inner, uint32_t box_outer)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_direct_receive(const LaunchCtx &c, const uint8_t *rows, int R_cap, int H,
                                  const int32_t *offsets, int E, const GroupedOut &out,
                                  int rounding, uint64_t seed, uint32_t sign_mask,
                                  uint32_t *status)
{
    const int64_t S = row_bytes(H);
    cudaError_t err = launch_pdl(expert_amax_kernel, dim3(E), dim3(256), 0, c.stream, rows, R_cap, S,
                                 offsets, E, out.amax_row, out.amax_col, out.scale_enc, status);
    if (err != cudaSuccess || R_cap < kTileRows)
        return err;

    CUtensorMap tm_codes, tm_scales, tm_trailer, tm_rw;
    memset(&tm_rw, 0, sizeof(tm_rw));
    const uint64_t rc = (uint64_t)R_cap;
    if (!make_map(&tm_codes, rows, (uint64_t)H / 2, rc, (uint64_t)S, kCodeBytes, kTileRows) ||
        !make_map(&tm_scales, rows + H / 2, (uint64_t)H / 16, rc, (uint64_t)S, kScaleBytes, kTileRows) ||
        !make_map(&tm_trailer, rows + S - 16, 16, rc, (uint64_t)S, 16, kTileRows))
        return cudaErrorInvalidValue;
    const int do_rw = out.rw_codes != nullptr;
    if (do_rw && !make_map(&tm_rw, out.rw_codes, (uint64_t)H / 2, rc, (uint64_t)H / 2, kCodeBytes, kTileRows))
        return cudaErrorInvalidValue;

    DrArgs a;
    a.offsets = offsets;
    a.E = E;
    a.H = H;
    a.R_cap = R_cap;
    a.n_strips = (H + kTileCols - 1) / kTileCols;
    a.rw_scales = out.rw_scales;
    a.rw_row_scale = out.rw_row_scale;
    a.cw_codes = out.cw_codes;
    a.cw_scales = out.cw_scales;
    a.scale_enc = out.scale_enc;
    a.seed = seed;
    a.sign_mask = sign_mask;
    a.status = status;
    a.do_rowwise = do_rw;

    const size_t smem = sizeof(DrSmem) + 1024;
    static int done[2] = {0, 0};
    err = ensure_smem_limit(direct_receive_kernel, c.device, (int)smem, done);
    if (err != cudaSuccess)
        return err;
    const int64_t max_units = (int64_t)(R_cap / kTileRows) * a.n_strips;
    int64_t grid = 2 * (int64_t)c.num_sms;
    if (grid > max_units)
        grid = max_units;
    if (grid < 1)
        grid = 1;
    return launch_pdl(direct_receive_kernel, dim3((unsigned)grid), dim3(kThreads), smem, c.stream, tm_codes,
                      tm_scales, tm_trailer, tm_rw, a, rounding == 1 ? 1 : 0);
}

} // namespace epq
