// Sender-side pack kernels with the routing gather fused in.
//
// NVFP4 (TE PR #3753 "Add NVFP4 EP dispatch and combine backward", PR
// description: a token is quantised once and sent as a single row holding
// E2M1 codes, an E4M3 scale for every 16 elements and an FP32 token scale that
// is a power of two; in the combine backward the codes are stochastically
// rounded) and MXFP8 (TE PR #3270 "EP dispatch with unfused MXFP8
// quantization": E4M3 data with E8M0 scales per 32 elements, data and scales
// in one buffer).
//
// One CTA per token.  A thread owns CPT chunks of 32 consecutive elements
// (64 bytes of BF16, read with four 16-byte streaming loads issued before any
// use), so a token is read from HBM exactly once; the block maxima and the
// token amax are computed on the BF16 bit patterns (for finite non-negative
// BF16, integer order is value order), the token is encoded once in
// registers and stored to each of its k destination rows with coalesced
// 16-byte stores.  Extra CTAs after the token CTAs write the padding rows.
#include <math.h>

#include "epq_device.cuh"
#include "epq_internal.h"

namespace epq {

constexpr int kMaxThreads = 256;

__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void st16(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Max of |x| over the 16 BF16 values held in w[0..7], as a BF16 bit pattern.
// max.xorsign.abs keeps max(|a|, |b|) per half (its sign is discarded).
__device__ __forceinline__ uint32_t absmax16_bits(const uint32_t *w)
{
    uint32_t m = w[0];
#pragma unroll
    for (int i = 1; i < 8; ++i)
        asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(w[i]));
    m &= 0x7fff7fffu;
    return max(m & 0xffffu, m >> 16);
}

// CTA-wide max of a non-negative value; sm has room for one word per warp.
__device__ __forceinline__ uint32_t cta_max(uint32_t v, uint32_t *sm)
{
    v = __reduce_max_sync(0xffffffffu, v);
    const int warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    if ((threadIdx.x & 31) == 0)
        sm[warp] = v;
    __syncthreads();
    uint32_t m = 0;
    for (int i = 0; i < nw; ++i)
        m = max(m, sm[i]);
    return m;
}

// Token scale exponent from the token amax (a BF16 bit pattern): the smallest
// k >= -126 with A <= 2688 * 2^k.  2688 = 1.3125 * 2^11, i.e. BF16 exponent
// field 138 with mantissa field 40.
__device__ __forceinline__ int token_scale_exp(uint32_t a_bits)
{
    const int ef = (a_bits >> 7) & 0xff, mt = a_bits & 0x7f;
    if (ef == 0)
        return -126;
    return max(-126, ef - 138 + (mt > 40 ? 1 : 0));
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return u2f(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return u2f(w & 0xffff0000u); }

// Correctly rounded quotient of (x0, x1) by 6: the correctly rounded
// reciprocal y6 = RN(1/6) and one Markstein correction step
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. R&D 34(1), 1990): q0 = x y6,
// r = x - 6 q0 (exact), q = q0 + r y6.
__device__ __forceinline__ float2 div6_rn(float2 x)
{
    const float y6 = 1.0f / 6.0f;
    const float2 q0 = mul2(x, make_float2(y6, y6));
    const float2 r = __ffma2_rn(q0, make_float2(-6.0f, -6.0f), x);
    return __ffma2_rn(r, make_float2(y6, y6), q0);
}

// Block of 16 elements (w[0..7]) -> 8 bytes of E2M1 codes of x / s.
//  fast: yn = -RN(1/s); the negated correctly rounded quotient comes from one
//        Markstein step, v' = -(x/s): q0' = x yn, r = x + q0' s (exact),
//        v' = q0' + r yn.  Encoding -v and flipping the sign bit of every
//        code afterwards (one XOR per 8 codes) gives the codes of x / s with
//        the sign of x kept also for zeros (x = -0 yields v' = +0).
//  slow: IEEE division by -s (tokens whose scale is outside 2^[-100, 100]).
template <bool kSR>
__device__ __forceinline__ uint2 encode_block16(const uint32_t *w, float s, float yn, bool fast,
                                                const uint32_t *rnd)
{
    float v[16];
    const float2 yn2 = make_float2(yn, yn), s2 = make_float2(s, s);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 x = make_float2(bf16lo(w[i]), bf16hi(w[i]));
        float2 q;
        if (fast) {
            const float2 q0 = mul2(x, yn2);
            const float2 r = __ffma2_rn(q0, s2, x);
            q = __ffma2_rn(r, yn2, q0);
        } else if (s == 0.0f) {
            q = mul2(x, make_float2(-0.0f, -0.0f));
        } else {
            q = make_float2(__fdiv_rn(x.x, -s), __fdiv_rn(x.y, -s));
        }
        v[2 * i] = q.x;
        v[2 * i + 1] = q.y;
    }
    if (kSR) // elements 4q .. 4q + 3 take the random word rnd[q]
        return make_uint2(cvt_e2m1x8_sr(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7], rnd[0], rnd[1]) ^ 0x88888888u,
                          cvt_e2m1x8_sr(v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15], rnd[2], rnd[3]) ^
                              0x88888888u);
    return make_uint2(cvt_e2m1x8(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]) ^ 0x88888888u,
                      cvt_e2m1x8(v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]) ^ 0x88888888u);
}

// Padding rows: for every expert e, rows [offsets[e] + counts[e], offsets[e+1]).
// One warp per row, rows spread over all padding CTAs.  kind 0 = NVFP4 row
// (zeros + trailer {2^-126, 0, 0xFFFFFFFF, 0}), kind 1 = MXFP8 row (zeros).
__device__ void fill_padding(int kind, int pad_cta, int pad_ctas, const int32_t *offsets,
                             const int32_t *counts, int E, int R_cap, uint8_t *base, int64_t S,
                             int H, uint32_t *status)
{
    __shared__ int pexcl[1025];
    __shared__ int wtmp[32];
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        pexcl[e] = (offsets[e + 1] - offsets[e]) - counts[e];
    __syncthreads();
    // exclusive prefix (serial per warp-slice is plenty for E <= 1024)
    {
        const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
        const int per = (E + nt - 1) / nt, b = min(tid * per, E), en = min(b + per, E);
        int sum = 0;
        for (int i = b; i < en; ++i)
            sum += pexcl[i];
        int x = sum;
        for (int o = 1; o < 32; o <<= 1) {
            const int yv = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += yv;
        }
        if (lane == 31)
            wtmp[warp] = x;
        __syncthreads();
        if (warp == 0) {
            const int nw = (nt + 31) / 32;
            int v = (lane < nw) ? wtmp[lane] : 0;
            for (int o = 1; o < 32; o <<= 1) {
                const int yv = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o)
                    v += yv;
            }
            wtmp[lane] = v;
        }
        __syncthreads();
        int run = (warp ? wtmp[warp - 1] : 0) + x - sum;
        for (int i = b; i < en; ++i) {
            const int v = pexcl[i];
            pexcl[i] = run;
            run += v;
        }
        if (tid == 0)
            pexcl[E] = wtmp[31];
        __syncthreads();
    }
    const int total = pexcl[E];
    const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int g = pad_cta * nw + (threadIdx.x >> 5); g < total; g += pad_ctas * nw) {
        int lo = 0, hi = E - 1; // last e with pexcl[e] <= g
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pexcl[mid] <= g)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int e = lo;
        const int r = offsets[e] + counts[e] + (g - pexcl[e]);
        if (r < 0 || r >= R_cap) {
            if (lane == 0)
                raise_status(status, kDevErrCapacity);
            continue;
        }
        if (kind == 0) {
            uint8_t *row = base + (int64_t)r * S;
            for (int64_t o = (int64_t)lane * 16; o < S - 16; o += 32 * 16)
                st16(row + o, make_uint4(0u, 0u, 0u, 0u));
            if (lane == 0)
                st16(row + S - 16, make_uint4(0x00800000u /* 2^-126 */, 0u, 0xffffffffu, 0u));
        } else {
            uint8_t *row = base + (int64_t)r * H;
            for (int o = lane * 16; o < H; o += 32 * 16)
                st16(row + o, make_uint4(0u, 0u, 0u, 0u));
            uint8_t *sc = base + (int64_t)R_cap * H + (int64_t)r * (H / 32);
            for (int o = lane; o < H / 32; o += 32)
                sc[o] = 0;
        }
    }
}

// RN(1/v) for every E4M3 code 0..127 (0 for v = 0; entry 127 unused),
// computed on the host with IEEE single-precision division.
struct RcpTable {
    float v[128];
};

template <int CPT>
__device__ __forceinline__ void load_token(uint32_t (&w)[CPT][16], const uint8_t *src, int nq)
{
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int q = threadIdx.x + c * blockDim.x;
        if (q < nq) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint4 v = ld_stream16(src + (int64_t)q * 64 + p * 16);
                w[c][4 * p + 0] = v.x; w[c][4 * p + 1] = v.y;
                w[c][4 * p + 2] = v.z; w[c][4 * p + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                w[c][i] = 0u;
        }
    }
}

// Persistent: token CTAs walk tokens blockIdx.x, + n_tok_ctas, ...; the next
// token's BF16 data is requested before the current one is encoded, so its
// loads are in flight during the encode and the stores.  CTAs from n_tok_ctas on write the padding rows.
template <int CPT, bool kSR>
__global__ void __launch_bounds__(kMaxThreads)
nvfp4_pack_kernel(const uint16_t *__restrict__ tokens, int T, int H, const int32_t *__restrict__ dest,
                  int k, const int32_t *__restrict__ offsets, const int32_t *__restrict__ counts, int E,
                  uint8_t *__restrict__ rows, int64_t S, int R_cap, const __grid_constant__ PhiloxKey key,
                  uint32_t *__restrict__ status, int n_tok_ctas, int pad_ctas,
                  const __grid_constant__ RcpTable rcp, const int32_t *__restrict__ topk,
                  float *__restrict__ expert_amax)
{
    __shared__ uint32_t wmax[2][kMaxThreads / 32];
    __shared__ float srcp[128];
    if (!expert_amax)   // as in the warp kernel: a reader of the amax is let in as CTAs finish
        pdl_launch_dependents();
    pdl_wait();
    if ((int)blockIdx.x >= n_tok_ctas) {
        fill_padding(0, blockIdx.x - n_tok_ctas, pad_ctas, offsets, counts, E, R_cap, rows, S, H, status);
        if (expert_amax)
            pdl_launch_dependents();
        return;
    }
    for (int i = threadIdx.x; i < 128; i += blockDim.x)
        srcp[i] = rcp.v[i];
    const int nq = H / 32;
    const uint8_t *base = reinterpret_cast<const uint8_t *>(tokens);

    int t = blockIdx.x;
    uint32_t w[CPT][16];
    if (t < T)
        load_token<CPT>(w, base + (int64_t)t * H * 2, nq);
    for (int iter = 0; t < T; t += n_tok_ctas, ++iter) {
        // the next token's loads go out before this token is encoded
        const int tn = t + n_tok_ctas;
        uint32_t wn[CPT][16];
        if (tn < T)
            load_token<CPT>(wn, base + (int64_t)tn * H * 2, nq);
        uint32_t bmax[CPT][2];
        uint32_t amax = 0;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            bmax[c][0] = absmax16_bits(&w[c][0]);
            bmax[c][1] = absmax16_bits(&w[c][8]);
            amax = max(amax, max(bmax[c][0], bmax[c][1]));
        }
        // CTA amax (the barrier also publishes srcp on the first token)
        const uint32_t a_bits = cta_max(amax, wmax[iter & 1]);
        const int kt = token_scale_exp(a_bits);
        const float St = exp2i(kt);
        const bool fast = (kt >= -100 && kt <= 100);
        const float inv_st = fast ? exp2i(-kt) : 0.0f;

        uint4 codes[CPT];
        uint32_t sb2s[CPT];
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            const float2 bf = make_float2(u2f(bmax[c][0] << 16), u2f(bmax[c][1] << 16));
            float2 qs;
            if (fast) {
                qs = div6_rn(mul2(bf, make_float2(inv_st, inv_st)));  // B / (6 S_t), correctly rounded
            } else {
                const float six_st = 6.0f * St;
                qs = make_float2(__fdiv_rn(bf.x, six_st), __fdiv_rn(bf.y, six_st));
            }
            const uint32_t sb2 = cvt_e4m3x2(qs.x, qs.y);
            sb2s[c] = sb2;
            const float2 sbf = f16x2_to_f32x2(cvt_f16x2_from_e4m3x2(sb2));
            const float s0 = sbf.x * St, s1 = sbf.y * St;
            // -RN(1/(s_b S_t)) = -RN(1/s_b) 2^-k, exact for |k| <= 100
            const float yn0 = fast ? -srcp[sb2 & 0xffu] * inv_st : 0.0f;
            const float yn1 = fast ? -srcp[(sb2 >> 8) & 0xffu] * inv_st : 0.0f;
            const int q = threadIdx.x + c * blockDim.x;
            uint2 c0, c1;
            if (kSR) {
                const uint64_t idx0 = (uint64_t)t * (uint64_t)H + (uint64_t)q * 32u;
                const Philox4 r0 = sr_bytes16(key, 0u, idx0);
                const Philox4 r1 = sr_bytes16(key, 0u, idx0 + 16u);
                const uint32_t rr0[4] = {r0.x, r0.y, r0.z, r0.w};
                const uint32_t rr1[4] = {r1.x, r1.y, r1.z, r1.w};
                c0 = encode_block16<true>(&w[c][0], s0, yn0, fast, rr0);
                c1 = encode_block16<true>(&w[c][8], s1, yn1, fast, rr1);
            } else {
                c0 = encode_block16<false>(&w[c][0], s0, yn0, fast, nullptr);
                c1 = encode_block16<false>(&w[c][8], s1, yn1, fast, nullptr);
            }
            codes[c] = make_uint4(c0.x, c0.y, c1.x, c1.y);
        }

        for (int j = 0; j < k; ++j) {
            const int d = __ldg(dest + (int64_t)t * k + j);
            if (d < 0)
                continue;
            if (d >= R_cap) {
                if (threadIdx.x == 0)
                    raise_status(status, kDevErrCapacity);
                continue;
            }
            uint8_t *row = rows + (int64_t)d * S;
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                const int q = threadIdx.x + c * blockDim.x;
                if (q < nq) {
                    st16(row + (int64_t)q * 16, codes[c]);
                    *reinterpret_cast<uint16_t *>(row + H / 2 + q * 2) = (uint16_t)sb2s[c];
                }
            }
            if (threadIdx.x == 0) {
                st16(row + S - 16, make_uint4(f2u(St), a_bits << 16, (uint32_t)t, 0u));
            } else if (threadIdx.x == 1) {
                for (int64_t o = 9 * (int64_t)H / 16; o < S - 16; o += 2)
                    *reinterpret_cast<uint16_t *>(row + o) = 0;
            }
        }
        // thread j: slot j's expert takes A_t into its max
        if (expert_amax && (int)threadIdx.x < k) {
            const int d = __ldg(dest + (int64_t)t * k + threadIdx.x);
            if (d >= 0 && d < R_cap) {
                const int e = topk ? __ldg(topk + (int64_t)t * k + threadIdx.x) : expert_of_dest(offsets, E, d);
                if (e >= 0 && e < E)
                    red_max_nonneg(expert_amax + e, u2f(a_bits << 16));
            }
        }
        if (tn < T) {
#pragma unroll
            for (int c = 0; c < CPT; ++c)
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[c][i] = wn[c][i];
        }
    }
    if (expert_amax)
        pdl_launch_dependents();
}

// Encode NB blocks held by one lane (block b = lane + 32 b of the token).
template <int NB, bool kFast, bool kSR>
__device__ __forceinline__ void encode_lane_blocks(const uint32_t (&w)[NB][8], const uint32_t (&bm)[NB], float St,
                                                   float inv_st, const float *srcp, const PhiloxKey &key, uint64_t t,
                                                   int H, int lane, uint2 (&code)[NB], uint32_t (&sbyte)[NB])
{
#pragma unroll
    for (int b = 0; b < NB; b += 2) {
        const int b1 = (b + 1 < NB) ? b + 1 : b;
        const float2 bf = make_float2(u2f(bm[b] << 16), u2f(bm[b1] << 16));
        float2 qs;
        if (kFast) {
            qs = div6_rn(mul2(bf, make_float2(inv_st, inv_st)));  // B / (6 S_t), correctly rounded
        } else {
            const float six_st = 6.0f * St;
            qs = make_float2(__fdiv_rn(bf.x, six_st), __fdiv_rn(bf.y, six_st));
        }
        const uint32_t sb2 = cvt_e4m3x2(qs.x, qs.y);
        const float2 sbf = f16x2_to_f32x2(cvt_f16x2_from_e4m3x2(sb2));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int bb = b + h;
            if (bb < NB) {
                const uint32_t sc = (sb2 >> (8 * h)) & 0xffu;
                const float s = (h ? sbf.y : sbf.x) * St;
                const float yn = kFast ? -srcp[sc] * inv_st : 0.0f;
                sbyte[bb] = sc;
                if (kSR) {
                    const uint64_t idx0 = t * (uint64_t)H + (uint64_t)(lane + 32 * bb) * 16u;
                    const Philox4 r = sr_bytes16(key, 0u, idx0);
                    const uint32_t rr[4] = {r.x, r.y, r.z, r.w};
                    code[bb] = encode_block16<true>(w[bb], s, yn, kFast, rr);
                } else {
                    code[bb] = encode_block16<false>(w[bb], s, yn, kFast, nullptr);
                }
            }
        }
    }
}

// Warp-per-token pack (H % 512 == 0, H <= 8192).  Lane l owns the 16-element
// blocks l, l + 32, ... of a token (32 contiguous bytes each).  Each warp
// streams its tokens through kBuf shared-memory buffers with 1-D bulk copies
// (TMA) issued kBuf tokens ahead, copies a token into registers, refills the
// buffer, reduces the token amax with a warp reduction, encodes its blocks
// and stores them to every destination row.  CTAs past the token CTAs write
// the padding rows.
//
// `early` (set only when the routing kernel just before this one on the
// stream was launched without programmatic dependency, so every earlier
// kernel, and with it whatever wrote the tokens, finished before it began):
// the tokens are complete when this grid starts, so each warp copies and
// encodes its first token while the routing kernel still runs, and waits for
// it only before reading the destinations.  Otherwise nothing is read before
// the wait but an L2 prefetch of the first two tokens (it returns no data).
constexpr int kPackWarps = 4;
// One buffer per warp: the next token's copy is issued as soon as the current
// one is in registers, so it overlaps the encode and the stores; a second
// buffer bought nothing but shared memory (it capped residency at one CTA per
// SM at H = 7168, three at H = 4096).
constexpr int kBuf = 1;

template <int NB, bool kSR>
__global__ void __launch_bounds__(32 * kPackWarps)
nvfp4_pack_warp_kernel(const uint16_t *__restrict__ tokens, int T, int H, const int32_t *__restrict__ dest,
                       int k, const int32_t *__restrict__ offsets, const int32_t *__restrict__ counts, int E,
                       uint8_t *__restrict__ rows, int64_t S, int R_cap, const __grid_constant__ PhiloxKey key,
                       uint32_t *__restrict__ status, int n_tok_ctas, int pad_ctas,
                       const __grid_constant__ RcpTable rcp, int early, const int32_t *__restrict__ topk,
                       float *__restrict__ expert_amax)
{
    extern __shared__ __align__(128) uint8_t pbuf[];   // [kPackWarps][kBuf][2H]
    __shared__ float srcp[128];
    __shared__ uint64_t bar[kPackWarps][kBuf];
    // With the per-expert amax reduced here, the next kernel (a direct receive
    // that reads it) is let in only as this grid's CTAs finish their work (each
    // triggers at its end): started earlier, its CTAs would sit on the SMs this
    // grid's CTAs still need; it reads nothing before its wait on this grid.
    if (!expert_amax)
        pdl_launch_dependents();
    if ((int)blockIdx.x >= n_tok_ctas) {
        pdl_wait();
        fill_padding(0, blockIdx.x - n_tok_ctas, pad_ctas, offsets, counts, E, R_cap, rows, S, H, status);
        if (expert_amax)
            pdl_launch_dependents();
        return;
    }
    // Before the wait for the routing plan: pull this warp's first tokens
    // into L2.  Under `early` the first token's bulk copy starts at once and
    // the next token's copy is issued as soon as the first has arrived, so
    // nothing is prefetched (an early prefetch would only compete with the
    // first copies).
    if (!early && (threadIdx.x & 31) == 0) {
        const int tw = blockIdx.x * kPackWarps + (threadIdx.x >> 5);
        for (int q = 0; q < kBuf + 1; ++q) {
            const int t = tw + q * n_tok_ctas * kPackWarps;
            if (t < T)
                bulk_prefetch_l2(reinterpret_cast<const uint8_t *>(tokens) + (int64_t)t * 2 * H, 2u * (uint32_t)H);
        }
    }
    if (!early)
        pdl_wait();
    for (int i = threadIdx.x; i < 128; i += blockDim.x)
        srcp[i] = rcp.v[i];
    if (threadIdx.x == 0) {
        for (int i = 0; i < kPackWarps * kBuf; ++i)
            mbar_init(&bar[0][0] + i, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = n_tok_ctas * kPackWarps;
    const uint32_t tok_bytes = 2u * (uint32_t)H;
    uint8_t *mybuf = pbuf + (size_t)warp * kBuf * tok_bytes;
    const uint8_t *gtok = reinterpret_cast<const uint8_t *>(tokens);
    const int t0 = blockIdx.x * kPackWarps + warp;
    if (lane == 0) {
#pragma unroll
        for (int b = 0; b < kBuf; ++b) {
            const int t = t0 + b * nw;
            if (t < T) {
                mbar_arrive_expect_tx(&bar[warp][b], tok_bytes);
                bulk_load(mybuf + b * tok_bytes, gtok + (int64_t)t * tok_bytes, tok_bytes, &bar[warp][b]);
            }
        }
    }
    int i = 0;
    const int n_mine = t0 < T ? (T - 1 - t0) / nw + 1 : 0;   // tokens of this warp
    for (int t = t0; t < T; t += nw, ++i) {
        const int b = i % kBuf;
        if (!mbar_wait_bounded(&bar[warp][b], (uint32_t)(i / kBuf) & 1u)) {
            if (lane == 0) {
                raise_status(status, kDevErrTimeout);
                // leave no bulk copy in flight: wait (bounded) for the ones issued
                const int issued = min(n_mine, i + kBuf);
                for (int j = i; j < issued; ++j)
                    (void)mbar_wait_bounded(&bar[warp][j % kBuf], (uint32_t)(j / kBuf) & 1u);
            }
            break;
        }
        const uint8_t *src = mybuf + b * tok_bytes;
        uint32_t w[NB][8];
#pragma unroll
        for (int q = 0; q < NB; ++q) {
            const uint4 v0 = *reinterpret_cast<const uint4 *>(src + (lane + 32 * q) * 32);
            const uint4 v1 = *reinterpret_cast<const uint4 *>(src + (lane + 32 * q) * 32 + 16);
            w[q][0] = v0.x; w[q][1] = v0.y; w[q][2] = v0.z; w[q][3] = v0.w;
            w[q][4] = v1.x; w[q][5] = v1.y; w[q][6] = v1.z; w[q][7] = v1.w;
        }
        // (the first token's destinations, under `early`, only after the wait)
        int dl = (lane < k && (i > 0 || !early)) ? __ldg(dest + (int64_t)t * k + lane) : -1;
        uint32_t bm[NB];
        uint32_t amax = 0;
#pragma unroll
        for (int q = 0; q < NB; ++q) {
            bm[q] = absmax16_bits(w[q]);
            amax = max(amax, bm[q]);
        }
        const uint32_t a_bits = __reduce_max_sync(0xffffffffu, amax);
        // every lane's reads of this buffer are done (they fed the reduction):
        // refill it with the token kBuf iterations ahead
        if (lane == 0) {
            const int tn = t + kBuf * nw;
            if (tn < T) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bar[warp][b], tok_bytes);
                bulk_load(mybuf + b * tok_bytes, gtok + (int64_t)tn * tok_bytes, tok_bytes, &bar[warp][b]);
            }
        }
        const int kt = token_scale_exp(a_bits);
        const float St = exp2i(kt);
        uint2 code[NB];
        uint32_t sbyte[NB];
        if (kt >= -100 && kt <= 100)
            encode_lane_blocks<NB, true, kSR>(w, bm, St, exp2i(-kt), srcp, key, (uint64_t)t, H, lane, code, sbyte);
        else
            encode_lane_blocks<NB, false, kSR>(w, bm, St, 0.0f, srcp, key, (uint64_t)t, H, lane, code, sbyte);
        if (i == 0 && early) {
            pdl_wait();
            if (lane < k)
                dl = __ldg(dest + (int64_t)t * k + lane);
        }
        for (int j = 0; j < k; ++j) {
            const int d = __shfl_sync(0xffffffffu, dl, j);
            if (d < 0)
                continue;
            if (d >= R_cap) {
                if (lane == 0)
                    raise_status(status, kDevErrCapacity);
                continue;
            }
            uint8_t *row = rows + (int64_t)d * S;
#pragma unroll
            for (int q = 0; q < NB; ++q) {
                const int u = lane + 32 * q;
                *reinterpret_cast<uint2 *>(row + (int64_t)u * 8) = code[q];
                row[H / 2 + u] = (uint8_t)sbyte[q];
            }
            if (lane == 0)
                st16(row + S - 16, make_uint4(f2u(St), a_bits << 16, (uint32_t)t, 0u));
            else if (lane == 1)
                for (int64_t o = 9 * (int64_t)H / 16; o < S - 16; o += 2)
                    *reinterpret_cast<uint16_t *>(row + o) = 0;
        }
        // the expert of each written row takes the token amax A_t into its max
        // (lane j: slot j; the routing plan zeroed the array, or the caller did)
        if (expert_amax && lane < k && dl >= 0 && dl < R_cap) {
            const int e = topk ? __ldg(topk + (int64_t)t * k + lane) : expert_of_dest(offsets, E, dl);
            if (e >= 0 && e < E)
                red_max_nonneg(expert_amax + e, u2f(a_bits << 16));
        }
    }
    if (expert_amax)
        pdl_launch_dependents();
}

// One MXFP8 block of 32 values (16 words of BF16 pairs) -> its 32 E4M3 bytes
// (o, in element order) and its E8M0 scale byte: e = the smallest integer in
// [-127, 127] with max|x| <= 448 * 2^e, elements E4M3_RNE(x / 2^e).
__device__ __forceinline__ void mxfp8_encode32(const uint32_t (&w)[16], uint32_t (&o)[8], uint32_t &sbyte)
{
    const uint32_t b = max(absmax16_bits(&w[0]), absmax16_bits(&w[8]));
    // smallest e in [-127, 127] with B <= 448 * 2^e; 448 = 1.75 * 2^8, i.e.
    // BF16 exponent field 135 with mantissa field 96
    const int ef = (b >> 7) & 0xff, mt = b & 0x7f;
    int e = (ef == 0) ? -127 : ef - 135 + (mt > 96 ? 1 : 0);
    e = max(-127, min(127, e));
    const float f = (e <= 126) ? exp2i(-e) : u2f(0x00400000u); // 2^-e
    const float2 f2 = make_float2(f, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 a = mul2(make_float2(bf16lo(w[2 * i]), bf16hi(w[2 * i])), f2);
        const float2 bb = mul2(make_float2(bf16lo(w[2 * i + 1]), bf16hi(w[2 * i + 1])), f2);
        o[i] = cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(bb.x, bb.y) << 16);
    }
    sbyte = (uint32_t)(e + 127);
}

// Block q's 32 bytes and scale byte to every destination row of its token.
// The scale bytes of four neighbouring blocks (lanes 4i .. 4i + 3 of a warp)
// leave as one word when a row's scales are a whole number of words; the four
// lanes of a group are then all present (the block size is a multiple of 32
// and q < nq holds for all four or none), and only they take part in the
// exchange.
__device__ __forceinline__ void mxfp8_store_block(const uint32_t (&o)[8], uint32_t sbyte, int q, int nq, int H,
                                                  const int *sdest, int k, uint8_t *buf, uint8_t *scales, int R_cap,
                                                  uint32_t *status)
{
    const bool wordwise = (nq & 3) == 0;
    uint32_t sw = sbyte << (8 * (q & 3));
    if (wordwise) {
        const uint32_t grp = 0xfu << (threadIdx.x & 28u);
        sw |= __shfl_xor_sync(grp, sw, 1);
        sw |= __shfl_xor_sync(grp, sw, 2);
    }
    for (int j = 0; j < k; ++j) {
        const int d = sdest[j];
        if (d < 0)
            continue;
        if (d >= R_cap) {
            raise_status(status, kDevErrCapacity);
            continue;
        }
        uint8_t *row = buf + (int64_t)d * H + (int64_t)q * 32;
        st16(row, make_uint4(o[0], o[1], o[2], o[3]));
        st16(row + 16, make_uint4(o[4], o[5], o[6], o[7]));
        if (!wordwise)
            scales[(int64_t)d * (H / 32) + q] = (uint8_t)sbyte;
        else if ((q & 3) == 0)
            *reinterpret_cast<uint32_t *>(scales + (int64_t)d * (H / 32) + q) = sw;
    }
}

// MXFP8 pack, one CTA per token (H / 32 > kMaxThreads: several blocks per thread).
__global__ void __launch_bounds__(kMaxThreads)
mxfp8_pack_kernel(const uint16_t *__restrict__ tokens, int T, int H, const int32_t *__restrict__ dest,
                  int k, const int32_t *__restrict__ offsets, const int32_t *__restrict__ counts, int E,
                  uint8_t *__restrict__ buf, int R_cap, uint32_t *__restrict__ status, int pad_ctas,
                  int cpt)
{
    __shared__ int sdest[32];
    pdl_launch_dependents();
    pdl_wait();
    if ((int)blockIdx.x >= T) {
        fill_padding(1, blockIdx.x - T, pad_ctas, offsets, counts, E, R_cap, buf, 0, H, status);
        return;
    }
    const int t = blockIdx.x;
    const int nq = H / 32;
    const uint8_t *src = reinterpret_cast<const uint8_t *>(tokens) + (int64_t)t * H * 2;
    if (threadIdx.x < k)
        sdest[threadIdx.x] = dest[(int64_t)t * k + threadIdx.x];
    __syncthreads();
    uint8_t *scales = buf + (int64_t)R_cap * H;
    for (int c = 0; c < cpt; ++c) {
        const int q = threadIdx.x + c * blockDim.x;
        if (q >= nq)
            break;
        uint32_t w[16];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint4 v = ld_stream16(src + (int64_t)q * 64 + p * 16);
            w[4 * p + 0] = v.x; w[4 * p + 1] = v.y; w[4 * p + 2] = v.z; w[4 * p + 3] = v.w;
        }
        uint32_t o[8], sbyte;
        mxfp8_encode32(w, o, sbyte);
        mxfp8_store_block(o, sbyte, q, nq, H, sdest, k, buf, scales, R_cap, status);
    }
}

// MXFP8 pack, persistent (H / 32 <= the block size: one block per thread):
// the resident token CTAs walk the tokens, each issuing the next token's loads
// (and reading its destinations) before it encodes and stores the current one;
// CTAs past the token CTAs write the padding rows.
__global__ void __launch_bounds__(kMaxThreads)
mxfp8_pack_persistent_kernel(const uint16_t *__restrict__ tokens, int T, int H, const int32_t *__restrict__ dest,
                             int k, const int32_t *__restrict__ offsets, const int32_t *__restrict__ counts, int E,
                             uint8_t *__restrict__ buf, int R_cap, uint32_t *__restrict__ status, int pad_ctas,
                             int n_tok_ctas)
{
    __shared__ int sdest[2][32];
    pdl_launch_dependents();
    pdl_wait();
    if ((int)blockIdx.x >= n_tok_ctas) {
        fill_padding(1, blockIdx.x - n_tok_ctas, pad_ctas, offsets, counts, E, R_cap, buf, 0, H, status);
        return;
    }
    const int nq = H / 32;
    const int q = threadIdx.x;
    const bool mine = q < nq;
    const uint8_t *base = reinterpret_cast<const uint8_t *>(tokens);
    uint8_t *scales = buf + (int64_t)R_cap * H;
    auto load = [&](int t, uint32_t(&w)[16]) {
        const uint8_t *src = base + (int64_t)t * H * 2 + (int64_t)q * 64;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint4 v = ld_stream16(src + p * 16);
            w[4 * p + 0] = v.x; w[4 * p + 1] = v.y; w[4 * p + 2] = v.z; w[4 * p + 3] = v.w;
        }
    };
    int t = blockIdx.x;
    uint32_t w[16];
    if (t < T) {
        if (mine)
            load(t, w);
        if (threadIdx.x < k)
            sdest[0][threadIdx.x] = dest[(int64_t)t * k + threadIdx.x];
    }
    for (int i = 0; t < T; t += n_tok_ctas, ++i) {
        __syncthreads();   // this token's destinations are in sdest[i & 1]
        const int tn = t + n_tok_ctas;
        uint32_t wn[16];
        if (tn < T) {
            if (mine)
                load(tn, wn);
            if (threadIdx.x < k)
                sdest[(i + 1) & 1][threadIdx.x] = dest[(int64_t)tn * k + threadIdx.x];
        }
        if (mine) {
            uint32_t o[8], sbyte;
            mxfp8_encode32(w, o, sbyte);
            mxfp8_store_block(o, sbyte, q, nq, H, sdest[i & 1], k, buf, scales, R_cap, status);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j)
            w[j] = wn[j];
    }
}

static int pack_threads(int H, int cpt)
{
    const int nq = H / 32;
    int th = (nq + cpt - 1) / cpt;
    th = (th + 31) / 32 * 32;
    return th < 32 ? 32 : th;
}

static int padding_ctas(const LaunchCtx &c, int E)
{
    // padding rows total at most E * (A - 1); enough CTAs to spread them
    const int p = 2 * c.num_sms;
    return E < 8 ? 8 : (p < 8 ? 8 : p);
}

static RcpTable make_rcp_table()
{
    RcpTable t;
    for (int code = 0; code < 128; ++code) {
        const int e = code >> 3, m = code & 7;
        const float v = e == 0 ? (float)m * (1.0f / 512.0f) : (1.0f + (float)m / 8.0f) * ldexpf(1.0f, e - 7);
        t.v[code] = (v == 0.0f || code == 127) ? 0.0f : 1.0f / v;
    }
    return t;
}

template <int CPT>
static cudaError_t launch_nvfp4_cpt(const LaunchCtx &c, const uint16_t *tokens, int T, int H,
                                    const int32_t *dest, int k, const int32_t *offsets,
                                    const int32_t *counts, int E, uint8_t *rows, int R_cap,
                                    int rounding, uint64_t seed, uint32_t *status, PackAmax am)
{
    static const RcpTable rcp = make_rcp_table();
    const int th = pack_threads(H, CPT);
    const int pc = padding_ctas(c, E);
    const int64_t S = row_bytes(H);
    // enough resident CTAs to keep a few tokens per SM in flight
    int per_sm = (2048 / th) < 16 ? (2048 / th) : 16;
    int tc = c.num_sms * per_sm;
    if (tc > T)
        tc = T;
    if (tc < 1)
        tc = 1;
    if (rounding == 1)
        return launch_pdl(nvfp4_pack_kernel<CPT, true>, dim3(tc + pc), dim3(th), 0, c.stream, tokens, T, H, dest,
                          k, offsets, counts, E, rows, S, R_cap, philox_key(seed), status, tc, pc, rcp, am.topk,
                          am.amax);
    return launch_pdl(nvfp4_pack_kernel<CPT, false>, dim3(tc + pc), dim3(th), 0, c.stream, tokens, T, H, dest, k,
                      offsets, counts, E, rows, S, R_cap, philox_key(seed), status, tc, pc, rcp, am.topk, am.amax);
}

template <int NB>
static cudaError_t launch_nvfp4_warp(const LaunchCtx &c, const uint16_t *tokens, int T, int H,
                                     const int32_t *dest, int k, const int32_t *offsets,
                                     const int32_t *counts, int E, uint8_t *rows, int R_cap,
                                     int rounding, uint64_t seed, uint32_t *status, int early, PackAmax am)
{
    static const RcpTable rcp = make_rcp_table();
    const int pc = padding_ctas(c, E);
    const int64_t S = row_bytes(H);
    const int th = 32 * kPackWarps, wpb = kPackWarps;
    const size_t smem = (size_t)kPackWarps * kBuf * 2 * (size_t)H;
    static std::atomic<uint32_t> done_rn[2] = {}, done_sr[2] = {};
    cudaError_t err = rounding == 1 ? ensure_smem_limit(nvfp4_pack_warp_kernel<NB, true>, c.device, (int)smem, done_sr)
                                    : ensure_smem_limit(nvfp4_pack_warp_kernel<NB, false>, c.device, (int)smem, done_rn);
    if (err != cudaSuccess)
        return err;
    // one wave of resident CTAs walks all tokens
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, rounding == 1 ? nvfp4_pack_warp_kernel<NB, true> : nvfp4_pack_warp_kernel<NB, false>, th, smem);
    if (err != cudaSuccess)
        return err;
    if (per_sm < 1)
        per_sm = 1;
    int tc = c.num_sms * per_sm;
    const int need = (T + wpb - 1) / wpb;
    if (tc > need)
        tc = need;
    if (tc < 1)
        tc = 1;
    if (rounding == 1)
        return launch_pdl(nvfp4_pack_warp_kernel<NB, true>, dim3(tc + pc), dim3(th), smem, c.stream, tokens, T, H,
                          dest, k, offsets, counts, E, rows, S, R_cap, philox_key(seed), status, tc, pc, rcp, early,
                          am.topk, am.amax);
    return launch_pdl(nvfp4_pack_warp_kernel<NB, false>, dim3(tc + pc), dim3(th), smem, c.stream, tokens, T, H,
                      dest, k, offsets, counts, E, rows, S, R_cap, philox_key(seed), status, tc, pc, rcp, early,
                      am.topk, am.amax);
}

cudaError_t launch_nvfp4_pack(const LaunchCtx &c, const uint16_t *tokens, int T, int H,
                              const int32_t *dest, int k, const int32_t *offsets,
                              const int32_t *counts, int E, uint8_t *rows, int R_cap,
                              int rounding, uint64_t seed, uint32_t *status, bool early, PackAmax am)
{
    if (H % 512 == 0 && H <= 8192) {
        switch (H / 512) {
#define EPQ_NB(n) case n: return launch_nvfp4_warp<n>(c, tokens, T, H, dest, k, offsets, counts, E, rows, R_cap, rounding, seed, status, early ? 1 : 0, am);
            EPQ_NB(1) EPQ_NB(2) EPQ_NB(3) EPQ_NB(4) EPQ_NB(5) EPQ_NB(6) EPQ_NB(7) EPQ_NB(8)
            EPQ_NB(9) EPQ_NB(10) EPQ_NB(11) EPQ_NB(12) EPQ_NB(13) EPQ_NB(14) EPQ_NB(15) EPQ_NB(16)
#undef EPQ_NB
        default: break;
        }
    }
    const int nq = H / 32;
    if (nq <= kMaxThreads)
        return launch_nvfp4_cpt<1>(c, tokens, T, H, dest, k, offsets, counts, E, rows, R_cap,
                                   rounding, seed, status, am);
    if (nq <= 2 * kMaxThreads)
        return launch_nvfp4_cpt<2>(c, tokens, T, H, dest, k, offsets, counts, E, rows, R_cap,
                                   rounding, seed, status, am);
    return launch_nvfp4_cpt<4>(c, tokens, T, H, dest, k, offsets, counts, E, rows, R_cap, rounding,
                               seed, status, am);
}

cudaError_t launch_mxfp8_pack(const LaunchCtx &c, const uint16_t *tokens, int T, int H,
                              const int32_t *dest, int k, const int32_t *offsets,
                              const int32_t *counts, int E, uint8_t *buf, int R_cap,
                              uint32_t *status)
{
    const int nq = H / 32;
    const int cpt = (nq + kMaxThreads - 1) / kMaxThreads;
    const int th = pack_threads(H, cpt);
    const int pc = padding_ctas(c, E);
    if (cpt == 1) {
        // one wave of resident CTAs walks all tokens
        int per_sm = 0;
        cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mxfp8_pack_persistent_kernel, th, 0);
        if (err != cudaSuccess)
            return err;
        int64_t tc = (int64_t)c.num_sms * (per_sm < 1 ? 1 : per_sm);
        if (tc > T)
            tc = T;
        if (tc < 1)
            tc = 1;
        return launch_pdl(mxfp8_pack_persistent_kernel, dim3((unsigned)(tc + pc)), dim3(th), 0, c.stream, tokens, T,
                          H, dest, k, offsets, counts, E, buf, R_cap, status, pc, (int)tc);
    }
    return launch_pdl(mxfp8_pack_kernel, dim3(T + pc), dim3(th), 0, c.stream, tokens, T, H,
                      dest, k, offsets, counts, E, buf, R_cap, status, pc, cpt);
}

} // namespace epq
