// Direct receive: packed NVFP4 rows -> the expert GEMM's grouped rowwise and
// columnwise-RHT NVFP4 operands, in one pass over the rows' data.
//
// TE PR #3753 "Add NVFP4 EP dispatch and combine backward", PR description:
// the grouped NVFP4 operands are made directly from the received rows, reading
// them once: rowwise, the codes the sender wrote are kept; columnwise, after
// the RHT, values are requantised with a per-expert scale taken from a bound
// rather than measured (nothing goes back through BF16).  TE PR #3755
// "Optionally derive FC1 dy NVFP4 amaxes from the dGLU epilogue", PR
// description: four times the rowwise amax bounds the columnwise amax after
// the RHT.
//
// Work unit: a tile of 128 rows x 256 hidden columns (a tile never straddles
// two experts: expert slots are multiples of 128 rows).  Persistent CTAs take
// the tiles in row-major order, round robin, so the whole grid sweeps the
// rows once, front to back.
//
// Given the per-expert amax the pack reduced as it wrote the rows, one launch:
// the tile kernel waits on the pack, issues its first tile loads, and derives
// every expert's S_enc from the amax itself (CTA 0 writes the metadata).  From
// the rows alone, two launches: expert_amax_kernel reduces each expert's
// 4-byte token amaxes from the row trailers (the rows' data is not read) into
// the expert's metadata and encode scale S_enc, and the tile kernel, launched
// behind it with programmatic dependent launch, starts its first tile loads
// while the amax kernel runs and reads S_enc once per CTA after waiting for it.
//
// Stages: a shared-memory ring of tiles (2 stages and 3 CTAs per SM for RNE,
// 3 stages and 2 CTAs per SM for SR) loaded by 2-D TMA (codes 128 B
// x 128 rows, scales 16 B x 128, row trailers 16 B x 128).  There is no
// producer warp: thread 0 issues the first tile's loads as the CTA starts
// (the other stages' once it has arrived), and the last warp to finish with a stage (an acquire-release counter) writes the metadata of the
// tile kStages ahead (expert, its offsets, S_enc) and issues its loads.
//
// Warps (8): the rowwise operand leaves straight from the ring (TMA
// stores of the codes and, when H % 256 == 0, of the scales; the token scale
// by threads).  For the columnwise operand each thread owns two adjacent
// hidden columns (one code byte per row) and 64 of the 128 rows: it decodes
// 16 rows at a time exactly into FP32 pairs with a per-tile table of (E4M3
// block scale x token scale x sigma / 4), runs the 16-point Walsh-Hadamard
// butterflies on packed FP32 pairs, derives the E4M3 block scale from S_enc,
// re-encodes to E2M1 (RNE or Philox-driven stochastic rounding) and writes
// each column's 32 code bytes as one sector of the [H][n_e] columnwise
// layout; the warp holding rows 64..127 hands its scale bytes to the warp
// holding rows 0..63 so each column's 8 scale bytes leave in one store.
#include <cudaTypedefs.h>
#include <float.h>
#include <math.h>
#include <string.h>

#include "epq_device.cuh"
#include "epq_internal.h"

namespace epq {

constexpr int kTileRows = 128;
constexpr int kTileCols = 256;
constexpr int kCodeBytes = kTileCols / 2;    // 128
constexpr int kScaleBytes = kTileCols / 16;  // 16
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers;         // no producer warp: the last warp to free a stage refills it
constexpr uint32_t kStageTx = kTileRows * (kCodeBytes + kScaleBytes + 16);
constexpr int kMaxExperts = 1024;

struct StageMeta {
    int e, off, n;
    float se, ce;        // S_enc and fl32(S_enc / 6)
};

template <int NS>   // ring stages
struct __align__(128) DrSmem {
    static constexpr int kNS = NS;
    uint8_t codes[NS][kTileRows][kCodeBytes];
    uint8_t scales[NS][kTileRows][kScaleBytes];
    uint32_t trailer[NS][kTileRows][4];
    union {   // rows padded to 80 bytes: the 16 column blocks' rows start on different banks
        uint2 t16[kConsumerWarps][16][10];       // per warp: [column block][row pair] (w2, w2 with -w_b)
        float t32[kConsumerWarps][16][20];       // per warp: [column block][row] FP32 decode scale
    } tab;
    uint8_t outc[2][kConsumerWarps][2048];       // [tile parity][warp = row block]: 256 columns x 8 code bytes
    uint8_t outs[2][kConsumerWarps][256];        // [tile parity][warp]: a scale byte per column
    float rcp[128];                             // [E4M3 code s] -> RN(1 / s), 0 for s = 0
    StageMeta meta[NS];
    uint64_t full[NS];
    uint64_t stg_full[2];                       // outc / outs [parity] written by all 8 warps
    uint64_t stg_empty[2];                      // outc / outs [parity] read (stored) by all 8 warps
    uint32_t rel[NS];                      // warps done with the stage's current tile
    int abort_flag;
    int consumed;                               // fewest tiles any warp finished
    int issued;                                 // tiles whose loads were issued
    // followed, in the launch's dynamic shared memory, by expert_offsets
    // (E + 1 ints, copied once) and the S_enc of every expert (E floats)
};

template <class Sm>
__device__ __forceinline__ int *smem_offs(Sm &sm) { return reinterpret_cast<int *>(&sm + 1); }
template <class Sm>
__device__ __forceinline__ float *smem_se(Sm &sm, int E) { return reinterpret_cast<float *>(smem_offs(sm) + E + 1); }

// Three ring stages and two CTAs per SM in both modes: a thread holds its 16
// code words, its 8 decode-scale pairs and the 16 butterfly pairs, which
// needs more than the 80 registers three CTAs per SM would leave.
template <bool kSR>
struct DrCfg {
    static constexpr int kStages = 3;
    static constexpr int kCtasPerSm = 2;
    using Smem = DrSmem<kStages>;
};
// each CTA gets at most (228 KB - 1 KB reserved per CTA) / CTAs per SM
// (with the per-expert arrays of up to 256 experts)
static_assert(sizeof(DrCfg<true>::Smem) + 1024 + 8 * 256 + 4 <= 113 * 1024, "direct receive must fit two CTAs per SM");

struct DrArgs {
    const uint8_t *rows;
    int64_t S;
    const int32_t *offsets;
    int E;
    int H;
    int R_cap;
    int n_strips;
    uint8_t *rw_scales;
    float *rw_row_scale;
    uint8_t *cw_codes;
    uint8_t *cw_scales;
    float *scale_enc;
    PhiloxKey key;     // round keys of the SR seed
    uint32_t sign_mask;
    uint32_t *status;
    int do_rowwise;
    int cw_v8;         // cw_codes is 32-byte aligned: 32-byte stores
    float rcp[128];    // RN(1 / s) for every E4M3 code s (0 for s = 0), computed on the host
    int rws_tma;       // rowwise scales leave by TMA store (H % 256 == 0)
    // per-expert amax reduced by the pack (else S_enc comes from the amax
    // kernel through scale_enc); last, so the fields above keep their offsets
    // (moving them made the SR kernel spill)
    const float *amax_in;
    float *amax_row, *amax_col;
    int grid_q, grid_r;   // the grid's CTA count divided by n_strips: quotient, remainder
};

// Tiles of a CTA: u = blockIdx.x + k * gridDim.x, k = 0, 1, ... over the tiles
// numbered row-major (u = row_tile * n_strips + strip).  At any moment the grid
// works on one contiguous band of row tiles, all strips of each: complete
// rowwise rows and, because expert slots are contiguous row ranges, whole
// columnwise column runs are written within a short window, so the output
// reaches DRAM in whole pages instead of scattered lines.

// Last e with offs[e] <= row (offs in shared memory).
__device__ __forceinline__ int expert_of_row(const int *offs, int E, int row)
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

// Issue the TMA loads of a tile into stage s, expecting their bytes on the
// stage's barrier (one thread).
template <class Sm>
__device__ __forceinline__ void issue_tile(Sm &sm, const CUtensorMap *tmc, const CUtensorMap *tms,
                                           const CUtensorMap *tmt, int s, int rt, int st)
{
    const int row0 = rt * kTileRows;
    mbar_expect_tx(&sm.full[s], kStageTx);
    tma_load_2d(&sm.codes[s][0][0], tmc, st * kCodeBytes, row0, &sm.full[s]);
    tma_load_2d(&sm.scales[s][0][0], tms, st * kScaleBytes, row0, &sm.full[s]);
    tma_load_2d(&sm.trailer[s][0][0], tmt, 0, row0, &sm.full[s]);
}

// The CTA's tiles u = blockIdx.x + it * gridDim.x in turn, as row tile
// u / n_strips and strip u % n_strips, stepped without a division per tile.
struct TileWalk {
    int u, rt, st;
    __device__ __forceinline__ explicit TileWalk(const DrArgs &p)
        : u((int)blockIdx.x), rt((int)blockIdx.x / p.n_strips), st((int)blockIdx.x % p.n_strips)
    {
    }
    __device__ __forceinline__ void next(const DrArgs &p)
    {
        u += (int)gridDim.x;
        rt += p.grid_q;
        st += p.grid_r;
        if (st >= p.n_strips) {
            st -= p.n_strips;
            ++rt;
        }
    }
};

// The tile this CTA takes it-th; false past the CTA's share.
__device__ __forceinline__ bool tile_of(const DrArgs &p, int n_units, int it, int &rt, int &st)
{
    const int u = (int)blockIdx.x + it * (int)gridDim.x;
    if (u >= n_units)
        return false;
    rt = u / p.n_strips;
    st = u % p.n_strips;
    return true;
}

// The stage's tile metadata: expert, its slot, S_enc and S_enc / 6.
template <class Sm>
__device__ __forceinline__ void stage_meta(Sm &sm, const DrArgs &p, int s, int rt)
{
    const int *offs = smem_offs(sm);
    const int e = expert_of_row(offs, p.E, rt * kTileRows);
    const int off = offs[e];
    const float se = smem_se(sm, p.E)[e];
    sm.meta[s] = StageMeta{e, off, offs[e + 1] - off, se, __fdiv_rn(se, 6.0f)};
}

// Per-expert metadata (one CTA per expert, grid-stride): the rowwise amax is
// the largest 4-byte token amax in the expert's row trailers (the rows' data
// is not read), the columnwise amax its 4x bound, S_enc = 2688 / amax_col.
// The tile kernel that follows reads S_enc back.
constexpr int kAmaxThreads = 512;

__global__ void __launch_bounds__(kAmaxThreads)
expert_amax_kernel(const uint8_t *__restrict__ rows, int64_t S, const int32_t *__restrict__ offsets, int E,
                   int R_cap, float *__restrict__ amax_row, float *__restrict__ amax_col,
                   float *__restrict__ scale_enc)
{
    __shared__ uint32_t red[kAmaxThreads / 32];
    pdl_wait();
    // the tile kernel may start now: the rows it reads are complete
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    const uint8_t *amax_at = rows + S - 12;   // A_t inside each row's trailer
    for (int e = blockIdx.x; e < E; e += gridDim.x) {
        const int off = __ldg(offsets + e);
        const int end = min(__ldg(offsets + e + 1), R_cap);
        uint32_t m = 0; // non-negative floats compare as their bit patterns
        for (int r = off + tid; r < end; r += 8 * kAmaxThreads) {
            uint32_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int rr = r + j * kAmaxThreads;
                v[j] = rr < end ? __ldg(reinterpret_cast<const uint32_t *>(amax_at + (int64_t)rr * S)) : 0u;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                m = max(m, v[j]);
        }
        m = __reduce_max_sync(0xffffffffu, m);
        if ((tid & 31) == 0)
            red[tid >> 5] = m;
        __syncthreads();
        if (tid == 0) {
            uint32_t x = 0u;
            for (int w = 0; w < kAmaxThreads / 32; ++w)
                x = max(x, red[w]);
            const float a = u2f(x);
            float ac;
            const float se = colwise_encode_scale(a, ac);
            amax_row[e] = a;
            amax_col[e] = ac;
            scale_enc[e] = se;
        }
        __syncthreads();
    }
}

__device__ __forceinline__ void st16g(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// 32-byte store (one full sector); p must be 32-byte aligned.
__device__ __forceinline__ void st32g(void *p, uint4 a, uint4 b)
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x), "r"(a.y),
                 "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
}

// Byte P of a word of code bytes -> f16x2 of its two E2M1 codes (exact; the
// low nibble to the low half).
template <int P>
__device__ __forceinline__ uint32_t e2m1_byte_f16x2(uint32_t w)
{
    uint32_t r;
    if (P == 0)
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
            : "=r"(r) : "r"(w));
    else if (P == 1)
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b1;\n\t}"
            : "=r"(r) : "r"(w));
    else if (P == 2)
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b2;\n\t}"
            : "=r"(r) : "r"(w));
    else
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b3;\n\t}"
            : "=r"(r) : "r"(w));
    return r;
}

// Byte offset, in a warp's code staging area (256 columns x 8 bytes: its
// 16-row block of every column of the strip), of columns 8l + 2p and
// 8l + 2p + 1: lane l's 64 bytes with their 16-byte chunks rotated by l mod 4,
// so that the 32 lanes' 16-byte stores of one column pair fall on distinct
// banks.
__device__ __forceinline__ int stage_off(int l, int p) { return 64 * l + 16 * (p ^ (l & 3)); }

// The thread's 16-row block of 8 columns, one column pair (code byte P of
// the 16 code words) at a time: decode, the RHT, block scales, E2M1 codes
// (RNE, or SR with the Philox words of the pair's two columns).  The pair's
// 16 code bytes and 2 scale bytes go to the warp's staging areas.
//   kF16: t16 holds the 8 row pairs' (w2, -w2 high) decode-scale words as
//   f16 pairs, values scaled by 2^-K (se, ce scaled by 2^K); else t32 holds
//   the 16 rows' FP32 decode scales and r = S_enc / s is an IEEE division.
template <bool kSR, bool kF16, int P>
__device__ __forceinline__ void rht_pair(const uint32_t (&cw)[16], const uint2 (&t16)[8], const float (&t32)[16],
                                         const float *rcp, float se, float ce, const Philox4 &ra, const Philox4 &rb,
                                         uint8_t *outc, uint8_t *outs, int lane)
{
    float2 u[16];
    if (kF16) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w2 = t16[i].x, nw2 = t16[i].y;
            const uint32_t qa = e2m1_byte_f16x2<P>(cw[2 * i]);
            const uint32_t qb = e2m1_byte_f16x2<P>(cw[2 * i + 1]);
            // d_a = q_a w_a exactly (f16 x f16 in FP32), then the len-1
            // butterfly d_a +- q_b w_b with one rounding each
            const float dax = fma_f16h<0, 0>(qa, w2, -0.0f), day = fma_f16h<1, 0>(qa, w2, -0.0f);
            u[2 * i] = make_float2(fma_f16h<0, 1>(qb, w2, dax), fma_f16h<1, 1>(qb, w2, day));
            u[2 * i + 1] = make_float2(fma_f16h<0, 1>(qb, nw2, dax), fma_f16h<1, 1>(qb, nw2, day));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float wa = t32[2 * i], wb = t32[2 * i + 1];
            const float2 qa = f16x2_to_f32x2(e2m1_byte_f16x2<P>(cw[2 * i]));
            const float2 qb = f16x2_to_f32x2(e2m1_byte_f16x2<P>(cw[2 * i + 1]));
            const float2 da = mul2(qa, make_float2(wa, wa));
            u[2 * i] = __ffma2_rn(qb, make_float2(wb, wb), da);
            u[2 * i + 1] = __ffma2_rn(qb, make_float2(-wb, -wb), da);
        }
    }
    // remaining Walsh-Hadamard butterflies, len = 2, 4, 8
#pragma unroll
    for (int len = 2; len < 16; len <<= 1) {
#pragma unroll
        for (int a = 0; a < 16; ++a) {
            if (a & len)
                continue;
            const float2 x = u[a], y = u[a + len];
            u[a] = add2(x, y);
            u[a + len] = sub2(x, y);
        }
    }
    // block maxima as a tree of 3-input maxima
    const float p0 = max3_abs(fabsf(u[0].x), u[1].x, u[2].x), q0 = max3_abs(fabsf(u[0].y), u[1].y, u[2].y);
    const float p1 = max3_abs(fabsf(u[3].x), u[4].x, u[5].x), q1 = max3_abs(fabsf(u[3].y), u[4].y, u[5].y);
    const float p2 = max3_abs(fabsf(u[6].x), u[7].x, u[8].x), q2 = max3_abs(fabsf(u[6].y), u[7].y, u[8].y);
    const float p3 = max3_abs(fabsf(u[9].x), u[10].x, u[11].x), q3 = max3_abs(fabsf(u[9].y), u[10].y, u[11].y);
    const float p4 = max3_abs(fabsf(u[12].x), u[13].x, u[14].x), q4 = max3_abs(fabsf(u[12].y), u[13].y, u[14].y);
    const float b0 = max3_abs(max3_abs(p0, p1, p2), p3, max3_abs(p4, u[15].x, 0.0f));
    const float b1 = max3_abs(max3_abs(q0, q1, q2), q3, max3_abs(q4, u[15].y, 0.0f));
    const float2 bc = mul2(make_float2(b0, b1), make_float2(ce, ce));
    const uint32_t s2 = cvt_e4m3x2(bc.x, bc.y);
    float2 r2;
    if (kF16) {
        // r = fl32(S_enc / s) by one Markstein step from y = RN(1/s): q = RN(S_enc y),
        // e = S_enc - s q (exact), r = RN(q + e y) is the correctly rounded
        // quotient (S_enc within 2^(+-100)); s = 0 gives y = 0 and r = 0
        const float2 y2 = make_float2(rcp[s2 & 0xffu], rcp[(s2 >> 8) & 0xffu]);
        const float2 sv = f16x2_to_f32x2(cvt_f16x2_from_e4m3x2(s2));
        const float2 se2 = make_float2(se, se);
        const float2 q = mul2(se2, y2);
        const float2 e = __ffma2_rn(make_float2(-sv.x, -sv.y), q, se2);
        r2 = __ffma2_rn(e, y2, q);
    } else {
        const float2 sv = f16x2_to_f32x2(cvt_f16x2_from_e4m3x2(s2));
        r2 = make_float2(sv.x == 0.0f ? 0.0f : __fdiv_rn(se, sv.x), sv.y == 0.0f ? 0.0f : __fdiv_rn(se, sv.y));
    }
#pragma unroll
    for (int i = 0; i < 16; ++i)
        u[i] = mul2(u[i], r2);
    uint4 cc;
    if (kSR) {
        // rows 4q .. 4q + 3 of the block take word q of its column's Philox output
        cc = make_uint4(cvt_e2m1x8_sr(u[0].x, u[1].x, u[2].x, u[3].x, u[4].x, u[5].x, u[6].x, u[7].x, ra.x, ra.y),
                        cvt_e2m1x8_sr(u[8].x, u[9].x, u[10].x, u[11].x, u[12].x, u[13].x, u[14].x, u[15].x, ra.z,
                                      ra.w),
                        cvt_e2m1x8_sr(u[0].y, u[1].y, u[2].y, u[3].y, u[4].y, u[5].y, u[6].y, u[7].y, rb.x, rb.y),
                        cvt_e2m1x8_sr(u[8].y, u[9].y, u[10].y, u[11].y, u[12].y, u[13].y, u[14].y, u[15].y, rb.z,
                                      rb.w));
    } else {
        cc = make_uint4(cvt_e2m1x8(u[0].x, u[1].x, u[2].x, u[3].x, u[4].x, u[5].x, u[6].x, u[7].x),
                        cvt_e2m1x8(u[8].x, u[9].x, u[10].x, u[11].x, u[12].x, u[13].x, u[14].x, u[15].x),
                        cvt_e2m1x8(u[0].y, u[1].y, u[2].y, u[3].y, u[4].y, u[5].y, u[6].y, u[7].y),
                        cvt_e2m1x8(u[8].y, u[9].y, u[10].y, u[11].y, u[12].y, u[13].y, u[14].y, u[15].y));
    }
    *reinterpret_cast<uint4 *>(outc + stage_off(lane, P)) = cc;
    *reinterpret_cast<uint16_t *>(outs + 8 * lane + 2 * P) = (uint16_t)s2;
}

// The Philox outputs of columns h and h + 1 of one 16-row block: counters
// n and n + nstep (n = (off_e H + h n_e + row) / 16, nstep = n_e / 16).  The
// call's element positions are below R_cap * H <= 2^36 (the boundary refuses
// larger buffers), so every counter of the call fits the first word (32-bit
// arithmetic is exact) and the counter's second word, n / 2^32, is 0.
__device__ __forceinline__ void pair_random(const PhiloxKey &K, uint32_t n, uint32_t nstep, Philox4 &ra, Philox4 &rb)
{
    ra = philox4x32_10(n, 0u, 1u, 0u, K);
    rb = philox4x32_10(n + nstep, 0u, 1u, 0u, K);
}

// The thread's four column pairs (8 columns x 16 rows).  With stochastic
// rounding the Philox outputs of the next pair are computed alongside the
// current pair's arithmetic (independent work for the scheduler).
template <bool kSR, bool kF16>
__device__ __forceinline__ void rht_thread(const uint32_t (&cw)[16], const uint2 (&t16)[8], const float (&t32)[16],
                                           const float *rcp, float se, float ce, const PhiloxKey &K, uint32_t nbase,
                                           uint32_t nstep, uint8_t *outc, uint8_t *outs, int lane)
{
    Philox4 ra, rb, na, nb;
    if (kSR)
        pair_random(K, nbase, nstep, ra, rb);
    if (kSR)
        pair_random(K, nbase + 2 * nstep, nstep, na, nb);
    rht_pair<kSR, kF16, 0>(cw, t16, t32, rcp, se, ce, ra, rb, outc, outs, lane);
    if (kSR) {
        ra = na;
        rb = nb;
        pair_random(K, nbase + 4 * nstep, nstep, na, nb);
    }
    rht_pair<kSR, kF16, 1>(cw, t16, t32, rcp, se, ce, ra, rb, outc, outs, lane);
    if (kSR) {
        ra = na;
        rb = nb;
        pair_random(K, nbase + 6 * nstep, nstep, na, nb);
    }
    rht_pair<kSR, kF16, 2>(cw, t16, t32, rcp, se, ce, ra, rb, outc, outs, lane);
    rht_pair<kSR, kF16, 3>(cw, t16, t32, rcp, se, ce, na, nb, outc, outs, lane);
}

// The FP32-table path (a row block whose token exponents spread too far for
// the f16 decode scales): rare, kept out of line.
template <bool kSR>
__device__ __noinline__ void rht_thread_f32(const uint32_t (&cw)[16], const float (&t32)[16], const float *rcp,
                                            float se, float ce, const PhiloxKey &K, uint32_t nbase, uint32_t nstep,
                                            uint8_t *outc, uint8_t *outs, int lane)
{
    const uint2 t16[8] = {};
    rht_thread<kSR, false>(cw, t16, t32, rcp, se, ce, K, nbase, nstep, outc, outs, lane);
}

// The store phase of one staged tile (expert slot at row `off`, n rows;
// rows rl .. rl + 127 of the expert; strip st): thread c takes column
// h = 256 st + c, its 64 code bytes (two full sectors of the [H][n_e / 2]
// layout) and its 8 scale bytes.
template <bool kSwz, class Sm>
__device__ __forceinline__ void store_tile(const Sm &sm, const DrArgs &p, int par, int off, int n, int rl, int st)
{
    const int c = threadIdx.x, H = p.H;
    const int h = st * kTileCols + c;
    if (h >= H)
        return;
    const int l = c >> 3, pp = (c >> 1) & 3, half = c & 1;
    const int off8 = stage_off(l, pp) + 8 * half;
    uint32_t v[16];
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
        const uint2 x = *reinterpret_cast<const uint2 *>(&sm.outc[par][w][off8]);
        v[2 * w] = x.x;
        v[2 * w + 1] = x.y;
    }
    uint8_t *d = p.cw_codes + (int64_t)off * (H / 2) + (int64_t)h * (n / 2) + rl / 2;
    if (p.cw_v8) {
        st32g(d, make_uint4(v[0], v[1], v[2], v[3]), make_uint4(v[4], v[5], v[6], v[7]));
        st32g(d + 32, make_uint4(v[8], v[9], v[10], v[11]), make_uint4(v[12], v[13], v[14], v[15]));
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            st16g(d + 16 * q, make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
    }
    // scale byte of row block w is byte (c & 3) of word c >> 2 of warp w's area
    uint32_t sw[8];
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w)
        sw[w] = reinterpret_cast<const uint32_t *>(sm.outs[par][w])[c >> 2];
    const uint32_t sel = (uint32_t)(c & 3) * 0x11u | 0x0040u;   // byte c & 3 of two words
    const uint32_t lo = __byte_perm(__byte_perm(sw[0], sw[1], sel) & 0xffffu, __byte_perm(sw[2], sw[3], sel), 0x5410);
    const uint32_t hi = __byte_perm(__byte_perm(sw[4], sw[5], sel) & 0xffffu, __byte_perm(sw[6], sw[7], sel), 0x5410);
    if (kSwz) {
        // tiled layout: the 4 scale bytes of a column's 64 rows are one word
        // of the expert's tile (column / 128, row-in-expert / 64)
        uint8_t *tt = p.cw_scales + (int64_t)off * (H / 16) + ((int64_t)(h >> 7) * (n / 64) + rl / 64) * 512 +
                      ((h & 127) >> 5) * 4 + (h & 31) * 16;
        *reinterpret_cast<uint32_t *>(tt) = lo;
        *reinterpret_cast<uint32_t *>(tt + 512) = hi;
    } else {
        uint8_t *cs = p.cw_scales + (int64_t)off * (H / 16) + (int64_t)h * (n / 16) + rl / 16;
        *reinterpret_cast<uint2 *>(cs) = make_uint2(lo, hi);
    }
}

// A bounded wait on phase `k & 1` of a staging barrier; false (with the
// abort flag and the timeout status set) if it gave up or another warp has.
template <class Sm>
__device__ __forceinline__ bool stage_wait(Sm &sm, uint64_t *bar, int k, const DrArgs &p)
{
    if (mbar_wait_bounded(bar, (uint32_t)k & 1u) && !sm.abort_flag)
        return true;
    if ((threadIdx.x & 31) == 0) {
        sm.abort_flag = 1;
        raise_status(p.status, kDevErrTimeout);
    }
    return false;
}

// Warp w computes row block w (rows 16w .. 16w + 15) of the tile, lane l the
// columns 8l .. 8l + 7 of the strip (the code bytes 4l .. 4l + 3 of each row:
// a warp's loads cover whole 128-byte rows).  A column's 128 rows thus come
// from all 8 warps: each warp stages its 8 code bytes and one scale byte per
// column (two staging buffers, used by alternate tiles), and thread c stores
// column c's 64 code bytes (two full sectors) and 8 scale bytes once all 8
// warps have staged the tile.  That store phase of a tile runs after the
// warp's compute of the next one, so the warps reach it at different times:
// the stores do not leave in one burst, and a warp waits only for the
// slowest warp of the tile before.  Per buffer, stg_full counts the 8 warps'
// stagings and stg_empty their store phases (a buffer is written again two
// tiles later, after every warp has stored from it).
template <bool kSR, bool kSwz, class Sm>
__device__ __forceinline__ int consumer_loop(Sm &sm, const CUtensorMap *tm_rw, const CUtensorMap *tm_rws,
                                             const CUtensorMap *tmc, const CUtensorMap *tms,
                                             const CUtensorMap *tmt, const DrArgs &p, int n_units)
{
    const int c = threadIdx.x;          // 0 .. kConsumers-1
    const int warp = c >> 5, lane = c & 31;
    const int H = p.H;
    int done = 0;
    bool ok = true;
    int prev_off = 0, prev_n = 0, prev_rl = 0, prev_st = 0;   // the tile before, staged, not yet stored
    int it = 0;
    for (TileWalk tw(p); tw.u < n_units; tw.next(p), ++it) {
        const int rt = tw.rt, st = tw.st;
        const int s = it % Sm::kNS;
        const uint32_t ph = (uint32_t)(it / Sm::kNS) & 1u;
        if (!mbar_wait_bounded(&sm.full[s], ph) || sm.abort_flag) {
            if (lane == 0) {
                sm.abort_flag = 1;
                raise_status(p.status, kDevErrTimeout);
            }
            ok = false;
            break;
        }
        const StageMeta m = sm.meta[s];
        const int row0 = rt * kTileRows;
        const int rl = row0 - m.off;
        const int par = it & 1;
        uint8_t *outc = sm.outc[par][warp];
        uint8_t *outs = sm.outs[par][warp];

        // rowwise operand: codes by TMA store, scales and token scale by threads
        if (p.do_rowwise && c < kTileRows) {
            if (c == 0) {
                tma_store_2d(tm_rw, st * kCodeBytes, row0, &sm.codes[s][0][0]);
                if (p.rws_tma)
                    tma_store_2d(tm_rws, st * kScaleBytes, row0, &sm.scales[s][0][0]);
                tma_store_commit();
            }
            if (!p.rws_tma && !kSwz) {
                const int nb = min(kScaleBytes, H / 16 - st * kScaleBytes);
                uint8_t *dst = p.rw_scales + (int64_t)(row0 + c) * (H / 16) + st * kScaleBytes;
                const uint8_t *src = &sm.scales[s][c][0];
                for (int b = 0; b < nb; b += 2)
                    *reinterpret_cast<uint16_t *>(dst + b) = *reinterpret_cast<const uint16_t *>(src + b);
            }
            if (st == 0)
                p.rw_row_scale[row0 + c] = u2f(sm.trailer[s][c][0]);
        }
        if (p.do_rowwise && kSwz) {
            // tiled layout: the strip's scale columns 16 st .. 16 st + 15 of
            // rows row0 .. row0 + 127 are the 512-byte tiles (rt, 4 st + g),
            // g = 0..3, one contiguous run; word (g, i, q) of the run (i =
            // row mod 32, q = row / 32) holds the 4 scale bytes of group g of
            // row 32 q + i
            const int ng = min(4, (H / 16 - st * kScaleBytes) / 4);
            uint8_t *run = p.rw_scales + ((int64_t)rt * (H / 64) + 4 * st) * 512;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int w = c + kThreads * j, gg = w >> 7, i = (w >> 2) & 31, q = w & 3;
                if (gg < ng)
                    *reinterpret_cast<uint32_t *>(run + 4 * w) =
                        *reinterpret_cast<const uint32_t *>(&sm.scales[s][32 * q + i][4 * gg]);
            }
        }

        // Decode-scale table of the warp's 16 rows and the strip's 16 column
        // blocks: lane l builds row pair l & 7 (rows 16w + 2(l & 7), + 1) of
        // the column blocks 4(l >> 3) .. + 3.  When the token exponents k of
        // the rows with a nonzero scale lie within 13 of their maximum K,
        // every s_b 2^(k - K - 2) is an exact f16 (no lower bit below 2^-24,
        // at most 112): the table then holds, per column block and row pair,
        // (w_a, w_b) and (w_a, -w_b) as f16 pairs (the RHT sign and the 1/4
        // folded in), and the block arithmetic runs on the values scaled by
        // 2^-K, with S_enc and S_enc / 6 scaled by 2^K (powers of two: every
        // rounding is the same as unscaled).
        const int rp = lane & 7, bq = lane >> 3;
        const int ra0 = 16 * warp + 2 * rp, ra1 = ra0 + 1;
        const uint32_t st0 = sm.trailer[s][ra0][0], st1 = sm.trailer[s][ra1][0];
        const uint32_t w40 = *reinterpret_cast<const uint32_t *>(&sm.scales[s][ra0][4 * bq]);
        const uint32_t w41 = *reinterpret_cast<const uint32_t *>(&sm.scales[s][ra1][4 * bq]);
        const int k0 = (int)(st0 >> 23) - 127, k1 = (int)(st1 >> 23) - 127;
        int kmax = max(w40 ? k0 : -1000, w41 ? k1 : -1000);
        int kmin = min(w40 ? k0 : 1000, w41 ? k1 : 1000);
        kmax = __reduce_max_sync(0xffffffffu, kmax);
        kmin = __reduce_min_sync(0xffffffffu, kmin);
        const int K = kmax >= kmin ? kmax : 0;
        const float se16 = m.se * exp2i(K), ce16 = m.ce * exp2i(K);
        const bool f16 = kmin >= K - 13 && se16 >= 0x1p-100f && se16 <= 0x1p100f;
        const bool neg0 = (p.sign_mask >> (2 * rp)) & 1u, neg1 = (p.sign_mask >> (2 * rp + 1)) & 1u;
        if (f16) {
            float f0 = w40 ? exp2i(k0 - K - 2) : 0.0f, f1 = w41 ? exp2i(k1 - K - 2) : 0.0f;
            if (neg0)
                f0 = -f0;
            if (neg1)
                f1 = -f1;
            const uint32_t fp = cvt_f16x2(f0, f1);
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                // (s_b of row a, s_b of row b) -> f16 pair, times (f_a, f_b): exact
                const uint32_t sb = __byte_perm(w40, w41, (uint32_t)(b | ((b + 4) << 4)));
                const uint32_t w2 = hmul2_rn(cvt_f16x2_from_e4m3x2(sb), fp);
                sm.tab.t16[warp][4 * bq + b][rp] = make_uint2(w2, w2 ^ 0x80000000u);
            }
        } else {
            float rs0 = u2f(st0) * 0.25f, rs1 = u2f(st1) * 0.25f;
            if (neg0)
                rs0 = -rs0;
            if (neg1)
                rs1 = -rs1;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                sm.tab.t32[warp][4 * bq + b][2 * rp] = e4m3_to_f32((w40 >> (8 * b)) & 0xffu) * rs0;
                sm.tab.t32[warp][4 * bq + b][2 * rp + 1] = e4m3_to_f32((w41 >> (8 * b)) & 0xffu) * rs1;
            }
        }
        __syncwarp();

        // this tile's staging buffer was last read by the store phase of the
        // tile two before
        if (it >= 2 && !stage_wait(sm, &sm.stg_empty[par], (it - 2) >> 1, p)) {
            ok = false;
            break;
        }
        // columns h0 .. h0 + 7 (all inside H, which is a multiple of 32)
        const int h0 = st * kTileCols + 8 * lane;
        if (h0 < H) {
            uint32_t cw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                cw[i] = *reinterpret_cast<const uint32_t *>(&sm.codes[s][16 * warp + i][4 * lane]);
            // Philox counter of column h0, this row block: (off_e H + h0 n_e + row) / 16,
            // with off_e, n_e and the row multiples of 16 and the whole below 2^32
            const uint32_t nstep = (uint32_t)(m.n >> 4);
            const uint32_t nbase = kSR ? (uint32_t)(m.off >> 4) * (uint32_t)H + (uint32_t)h0 * nstep +
                                             (uint32_t)((rl + 16 * warp) >> 4)
                                       : 0u;
            float t32[16];
            if (f16) {
                uint2 t16[8];
                const uint4 *tp = reinterpret_cast<const uint4 *>(&sm.tab.t16[warp][lane >> 1][0]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 v = tp[j];
                    t16[2 * j] = make_uint2(v.x, v.y);
                    t16[2 * j + 1] = make_uint2(v.z, v.w);
                }
                rht_thread<kSR, true>(cw, t16, t32, sm.rcp, se16, ce16, p.key, nbase, nstep, outc, outs, lane);
            } else {
                const float4 *tp = reinterpret_cast<const float4 *>(&sm.tab.t32[warp][lane >> 1][0]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 v = tp[j];
                    t32[4 * j] = v.x;
                    t32[4 * j + 1] = v.y;
                    t32[4 * j + 2] = v.z;
                    t32[4 * j + 3] = v.w;
                }
                rht_thread_f32<kSR>(cw, t32, sm.rcp, m.se, m.ce, p.key, nbase, nstep, outc, outs, lane);
            }
        }

        // release the stage (the rowwise TMA store having read it); the
        // last warp to release it refills it with the tile kStages ahead
        if (c == 0 && p.do_rowwise)
            tma_store_wait_read0();
        __syncwarp();
        if (lane == 0) {
            uint32_t before;
            asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                         : "=r"(before)
                         : "r"((uint32_t)__cvta_generic_to_shared(&sm.rel[s]))
                         : "memory");
            if (before == kConsumerWarps - 1) {
                sm.rel[s] = 0u;
                int rt2, st2;
                if (tile_of(p, n_units, it + Sm::kNS, rt2, st2)) {
                    stage_meta(sm, p, s, rt2);
                    // bytes expected before the arrival, so the phase waits for them;
                    // the arrival releases the metadata
                    issue_tile(sm, tmc, tms, tmt, s, rt2, st2);
                    mbar_arrive(&sm.full[s]);
                    atomicAdd(&sm.issued, 1);
                }
            }
            // this warp's staging of the tile is written
            mbar_arrive(&sm.stg_full[par]);
        }
        // the tile before: once all 8 warps staged it, store it and free its buffer
        if (it >= 1) {
            if (!stage_wait(sm, &sm.stg_full[par ^ 1], (it - 1) >> 1, p)) {
                ok = false;
                break;
            }
            store_tile<kSwz>(sm, p, par ^ 1, prev_off, prev_n, prev_rl, prev_st);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.stg_empty[par ^ 1]);
        }
        prev_off = m.off;
        prev_n = m.n;
        prev_rl = rl;
        prev_st = st;
        done = it + 1;
    }
    // the last tile
    if (ok && done >= 1 && stage_wait(sm, &sm.stg_full[(done - 1) & 1], (done - 1) >> 1, p))
        store_tile<kSwz>(sm, p, (done - 1) & 1, prev_off, prev_n, prev_rl, prev_st);
    if (c == 0 && p.do_rowwise)
        tma_store_wait0();
    return done;
}

// kSwz: both scale tensors in the tiled layout of block-scaled GEMM operands.
template <bool kSR, bool kSwz>
__global__ void __launch_bounds__(kThreads, DrCfg<kSR>::kCtasPerSm)
direct_receive_kernel(const __grid_constant__ CUtensorMap tm_codes,
                      const __grid_constant__ CUtensorMap tm_scales,
                      const __grid_constant__ CUtensorMap tm_trailer,
                      const __grid_constant__ CUtensorMap tm_rw, const __grid_constant__ CUtensorMap tm_rws,
                      const __grid_constant__ DrArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    using Sm = typename DrCfg<kSR>::Smem;
    Sm &sm = *reinterpret_cast<Sm *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < Sm::kNS; ++i) {
            mbar_init(&sm.full[i], 1);
            sm.rel[i] = 0u;
        }
        mbar_init(&sm.stg_full[0], kConsumerWarps);
        mbar_init(&sm.stg_full[1], kConsumerWarps);
        mbar_init(&sm.stg_empty[0], kConsumerWarps);
        mbar_init(&sm.stg_empty[1], kConsumerWarps);
        sm.abort_flag = 0;
        sm.consumed = 0x7fffffff;
        fence_mbar_init();
        tma_prefetch_desc(&tm_codes);
        tma_prefetch_desc(&tm_scales);
        tma_prefetch_desc(&tm_trailer);
    }
    // The rows and the offsets were complete before this grid could start
    // (expert_amax_kernel lets it launch only after its own wait on the pack
    // has returned), so the first tile's loads go out before the wait on the
    // amax kernel (only S_enc comes from it), and even before the expert
    // offsets are read: tile 0 of this CTA is loaded if it lies inside the
    // row capacity, and dropped unused if it lies past the rows in use.
    // With the amax supplied (p.amax_in) the grid before this one is the pack
    // itself, and no row may be read before the wait on it.
    // The other stages' tiles are issued by lane 0 of warps 1 .. kStages - 1,
    // one each, as soon as their rows may be read: the issue of a tile's
    // three boxes holds its thread for a while, and done by thread 0 after
    // tile 0 had arrived it kept warp 0 (and with it the whole tile) from
    // starting.  Their bytes are expected on the stages' barriers at the
    // issue; thread 0 writes the metadata and arrives (releasing both) after
    // the barrier that follows S_enc.
    const int rt0 = (int)blockIdx.x / p.n_strips, st0 = (int)blockIdx.x % p.n_strips;
    const int pre = rt0 < p.R_cap / kTileRows ? 1 : 0;
    if (threadIdx.x == 0 && pre && !p.amax_in)
        issue_tile(sm, &tm_codes, &tm_scales, &tm_trailer, 0, rt0, st0);
    __syncthreads();
    pdl_launch_dependents();

    for (int i = threadIdx.x; i <= p.E; i += blockDim.x)
        smem_offs(sm)[i] = __ldg(p.offsets + i);
    for (int i = threadIdx.x; i < 128; i += blockDim.x)
        sm.rcp[i] = p.rcp[i];
    __syncthreads();
    int R = smem_offs(sm)[p.E];
    if (R > p.R_cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            raise_status(p.status, kDevErrCapacity);
        R = p.R_cap;
    }
    const int n_units = (R / kTileRows) * p.n_strips;
    const bool use0 = (int)blockIdx.x < n_units;   // tile 0 holds rows in use
    const int wn = (int)threadIdx.x >> 5;            // the stage whose tile this thread issues
    int rtn = 0, stn = 0;
    const bool issuer = (threadIdx.x & 31) == 0 && wn >= 1 && wn < Sm::kNS && tile_of(p, n_units, wn, rtn, stn);
    if (issuer && !p.amax_in)
        issue_tile(sm, &tm_codes, &tm_scales, &tm_trailer, wn, rtn, stn);

    pdl_wait();
    if (threadIdx.x == 0 && pre && p.amax_in)
        issue_tile(sm, &tm_codes, &tm_scales, &tm_trailer, 0, rt0, st0);
    if (issuer && p.amax_in)
        issue_tile(sm, &tm_codes, &tm_scales, &tm_trailer, wn, rtn, stn);
    if (p.amax_in) {
        // S_enc of every expert from the supplied amax; CTA 0 writes the metadata
        for (int i = threadIdx.x; i < p.E; i += blockDim.x) {
            const float a = p.amax_in[i];
            float ac;
            const float se = colwise_encode_scale(a, ac);
            smem_se(sm, p.E)[i] = se;
            if (blockIdx.x == 0) {
                p.amax_row[i] = a;
                p.amax_col[i] = ac;
                p.scale_enc[i] = se;
            }
        }
    } else {
        for (int i = threadIdx.x; i < p.E; i += blockDim.x)
            smem_se(sm, p.E)[i] = p.scale_enc[i];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // metadata of the first stages' tiles; each arrival releases its
        // stage (a dropped tile 0's arrival only lets its bytes be waited
        // for before the exit)
        int issued = pre;
        if (pre) {
            if (use0)
                stage_meta(sm, p, 0, rt0);
            mbar_arrive(&sm.full[0]);
            for (int n = 1; n < Sm::kNS; ++n) {
                int rt, st;
                if (!tile_of(p, n_units, n, rt, st))
                    break;
                stage_meta(sm, p, n, rt);
                mbar_arrive(&sm.full[n]);
                issued = n + 1;
            }
        }
        sm.issued = issued;
    }

    const int done = consumer_loop<kSR, kSwz>(sm, &tm_rw, &tm_rws, &tm_codes, &tm_scales, &tm_trailer, p, n_units);
    if (lane == 0)
        atomicMin(&sm.consumed, done);
    __syncthreads();
    // never leave with a tile load still in flight (after an abort, when
    // warps may have stopped at different tiles, or for a dropped tile 0)
    if (threadIdx.x == 0) {
        for (int i = sm.consumed; i < sm.issued; ++i)
            (void)mbar_wait_bounded(&sm.full[i % Sm::kNS], (uint32_t)(i / Sm::kNS) & 1u);
    }
}

// --------------------------------------------------------------- host
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2-D byte tensor [outer][inner] with a row pitch of `pitch` bytes.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t pitch,
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
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_direct_receive(const LaunchCtx &c, const uint8_t *rows, int R_cap, int H,
                                  const int32_t *offsets, int E, const GroupedOut &out,
                                  int rounding, uint64_t seed, uint32_t sign_mask,
                                  uint32_t *status, bool swz, const float *amax_in)
{
    const int64_t S = row_bytes(H);
    // fewer than 128 rows of capacity: no tile can exist, and the amax kernel
    // alone writes the metadata (from the trailers: the same values)
    if (R_cap < kTileRows)
        amax_in = nullptr;
    cudaError_t err = cudaSuccess;
    if (!amax_in)
        err = launch_pdl(expert_amax_kernel, dim3((unsigned)E), dim3(kAmaxThreads), 0, c.stream, rows, S, offsets, E,
                         R_cap, out.amax_row, out.amax_col, out.scale_enc);
    if (err != cudaSuccess || R_cap < kTileRows)
        return err;

    CUtensorMap tm_codes, tm_scales, tm_trailer, tm_rw, tm_rws;
    memset(&tm_rw, 0, sizeof(tm_rw));
    memset(&tm_rws, 0, sizeof(tm_rws));
    const uint64_t rc = (uint64_t)R_cap;
    if (!make_map(&tm_codes, rows, (uint64_t)H / 2, rc, (uint64_t)S, kCodeBytes, kTileRows) ||
        !make_map(&tm_scales, rows + H / 2, (uint64_t)H / 16, rc, (uint64_t)S, kScaleBytes, kTileRows) ||
        !make_map(&tm_trailer, rows + S - 16, 16, rc, (uint64_t)S, 16, kTileRows))
        return cudaErrorInvalidValue;
    const int do_rw = out.rw_codes != nullptr;
    if (do_rw && !make_map(&tm_rw, out.rw_codes, (uint64_t)H / 2, rc, (uint64_t)H / 2, kCodeBytes, kTileRows))
        return cudaErrorInvalidValue;
    // rowwise scales by TMA when every strip is a whole 16-byte box and the
    // row pitch H/16 is a multiple of 16 bytes
    const int rws_tma = do_rw && !swz && H % kTileCols == 0 &&
                        make_map(&tm_rws, out.rw_scales, (uint64_t)H / 16, rc, (uint64_t)H / 16, kScaleBytes, kTileRows);

    DrArgs a;
    a.rows = rows;
    a.S = S;
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
    a.amax_in = amax_in;
    a.amax_row = out.amax_row;
    a.amax_col = out.amax_col;
    a.key = philox_key(seed);
    a.sign_mask = sign_mask;
    a.status = status;
    a.do_rowwise = do_rw;
    a.cw_v8 = (reinterpret_cast<uintptr_t>(out.cw_codes) & 31u) == 0;
    a.rws_tma = rws_tma;
    for (int code = 0; code < 128; ++code) {
        const int ex = code >> 3, mt = code & 7;
        const float v = ex == 0 ? (float)mt * (1.0f / 512.0f) : (1.0f + (float)mt / 8.0f) * ldexpf(1.0f, ex - 7);
        a.rcp[code] = (v == 0.0f || code == 127) ? 0.0f : 1.0f / v;   // IEEE single division: RN(1/v)
    }

    const bool sr = rounding == 1;
    const size_t smem_fixed = (sr ? sizeof(DrCfg<true>::Smem) : sizeof(DrCfg<false>::Smem)) + 1024;
    const size_t smem = smem_fixed + (size_t)(2 * E + 1) * 4;
    static std::atomic<uint32_t> done[4][2] = {};
    auto kern = sr ? (swz ? direct_receive_kernel<true, true> : direct_receive_kernel<true, false>)
                   : (swz ? direct_receive_kernel<false, true> : direct_receive_kernel<false, false>);
    // the limit is set once per device, for the largest expert count
    err = ensure_smem_limit(kern, c.device, (int)(smem_fixed + (2 * kMaxExperts + 1) * 4),
                            done[(sr ? 2 : 0) + (swz ? 1 : 0)]);
    if (err != cudaSuccess)
        return err;
    const int64_t max_units = (int64_t)(R_cap / kTileRows) * a.n_strips;
    int64_t grid = (int64_t)(sr ? DrCfg<true>::kCtasPerSm : DrCfg<false>::kCtasPerSm) * c.num_sms;
    if (grid > max_units)
        grid = max_units;
    if (grid < 1)
        grid = 1;
    a.grid_q = (int)grid / a.n_strips;
    a.grid_r = (int)grid % a.n_strips;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, c.stream, tm_codes, tm_scales, tm_trailer,
                      tm_rw, tm_rws, a);
}

} // namespace epq
