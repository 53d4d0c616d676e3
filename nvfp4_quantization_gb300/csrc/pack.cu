// Sender-side pack kernels with the routing gather fused in.
//
// NVFP4 (TE PR #3753 "Add NVFP4 EP dispatch and combine backward", PR
// description: each token travels as one packed NVFP4 row of E2M1 codes, E4M3
// block scales and a power-of-two FP32 token scale; the combine backward uses
// stochastic rounding) and MXFP8 (TE PR #3270 "EP dispatch with unfused MXFP8
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
__device__ __forceinline__ uint32_t absmax16_bits(const uint32_t *w)
{
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        m = __vmaxu2(m, w[i] & 0x7fff7fffu);
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
__device__ __forceinline__ float copysign_bits(float v, float s)
{
    return u2f((f2u(v) & 0x7fffffffu) | (f2u(s) & 0x80000000u));
}

// Block of 16 elements (w[0..7]) -> 8 bytes of E2M1 codes.
//  fast: v = x / s correctly rounded via the per-block correctly rounded
//        reciprocal y = RN(1/s) and one Markstein correction step
//        (P. Markstein, "Computation of elementary functions on the IBM
//        RISC System/6000 processor", IBM J. R&D 34(1), 1990):
//        q0 = x*y, r = x - q0*s (exact), v = q0 + r*y.
//  slow: IEEE division (tokens whose scale is outside 2^[-100, 100]).
template <bool kSR>
__device__ __forceinline__ uint2 encode_block16(const uint32_t *w, float s, float y, bool fast,
                                                const uint32_t *rnd)
{
    uint32_t out[2] = {0u, 0u};
    const float2 y2 = make_float2(y, y), ns2 = make_float2(-s, -s);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 x = make_float2(bf16lo(w[i]), bf16hi(w[i]));
        float2 v;
        if (fast) {
            const float2 q0 = mul2(x, y2);
            const float2 r = __ffma2_rn(q0, ns2, x);
            v = __ffma2_rn(r, y2, q0);
        } else {
            v = (s == 0.0f) ? make_float2(0.0f, 0.0f)
                            : make_float2(__fdiv_rn(x.x, s), __fdiv_rn(x.y, s));
        }
        v.x = copysign_bits(v.x, x.x);
        v.y = copysign_bits(v.y, x.y);
        if (kSR) {
            const uint32_t rw = rnd[i >> 1];
            const int sh = (i & 1) * 16;
            v.x = sr_e2m1_value(v.x, (rw >> sh) & 0xffu);
            v.y = sr_e2m1_value(v.y, (rw >> (sh + 8)) & 0xffu);
        }
        out[i >> 2] |= cvt_e2m1x2(v.x, v.y) << (8 * (i & 3));
    }
    return make_uint2(out[0], out[1]);
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

template <int CPT, bool kSR>
__global__ void __launch_bounds__(kMaxThreads)
nvfp4_pack_kernel(const uint16_t *__restrict__ tokens, int T, int H, const int32_t *__restrict__ dest,
                  int k, const int32_t *__restrict__ offsets, const int32_t *__restrict__ counts, int E,
                  uint8_t *__restrict__ rows, int64_t S, int R_cap, uint64_t seed,
                  uint32_t *__restrict__ status, int pad_ctas)
{
    __shared__ uint32_t wmax[kMaxThreads / 32];
    __shared__ int sdest[32];
    pdl_launch_dependents();
    pdl_wait();
    if ((int)blockIdx.x >= T) {
        fill_padding(0, blockIdx.x - T, pad_ctas, offsets, counts, E, R_cap, rows, S, H, status);
        return;
    }
    const int t = blockIdx.x;
    const int nq = H / 32;
    const uint8_t *src = reinterpret_cast<const uint8_t *>(tokens) + (int64_t)t * H * 2;

    uint32_t w[CPT][16];
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
    if (threadIdx.x < k)
        sdest[threadIdx.x] = dest[(int64_t)t * k + threadIdx.x];

    uint32_t bmax[CPT][2];
    uint32_t amax = 0;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        bmax[c][0] = absmax16_bits(&w[c][0]);
        bmax[c][1] = absmax16_bits(&w[c][8]);
        amax = max(amax, max(bmax[c][0], bmax[c][1]));
    }
    const uint32_t a_bits = cta_max(amax, wmax); // includes a __syncthreads (sdest ready)
    const int kt = token_scale_exp(a_bits);
    const float St = exp2i(kt);
    const float six_st = 6.0f * St;
    const bool fast = (kt >= -100 && kt <= 100);

#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int q = threadIdx.x + c * blockDim.x;
        if (q >= nq)
            continue;
        const float b0 = u2f(bmax[c][0] << 16), b1 = u2f(bmax[c][1] << 16);
        const uint32_t sb2 = cvt_e4m3x2(__fdiv_rn(b0, six_st), __fdiv_rn(b1, six_st));
        const float2 sbf = f16x2_to_f32x2(cvt_f16x2_from_e4m3x2(sb2));
        const float s0 = sbf.x * St, s1 = sbf.y * St;
        const float y0 = (fast && s0 != 0.0f) ? __frcp_rn(s0) : 0.0f;
        const float y1 = (fast && s1 != 0.0f) ? __frcp_rn(s1) : 0.0f;
        uint2 c0, c1;
        if (kSR) {
            const uint64_t idx0 = (uint64_t)t * (uint64_t)H + (uint64_t)q * 32u;
            const Philox4 r0 = sr_bytes16(seed, 0u, idx0);
            const Philox4 r1 = sr_bytes16(seed, 0u, idx0 + 16u);
            const uint32_t rr0[4] = {r0.x, r0.y, r0.z, r0.w};
            const uint32_t rr1[4] = {r1.x, r1.y, r1.z, r1.w};
            c0 = encode_block16<true>(&w[c][0], s0, y0, fast, rr0);
            c1 = encode_block16<true>(&w[c][8], s1, y1, fast, rr1);
        } else {
            c0 = encode_block16<false>(&w[c][0], s0, y0, fast, nullptr);
            c1 = encode_block16<false>(&w[c][8], s1, y1, fast, nullptr);
        }
        const uint4 codes = make_uint4(c0.x, c0.y, c1.x, c1.y);
        for (int j = 0; j < k; ++j) {
            const int d = sdest[j];
            if (d < 0)
                continue;
            if (d >= R_cap) {
                raise_status(status, kDevErrCapacity);
                continue;
            }
            uint8_t *row = rows + (int64_t)d * S;
            st16(row + (int64_t)q * 16, codes);
            *reinterpret_cast<uint16_t *>(row + H / 2 + q * 2) = (uint16_t)sb2;
        }
    }
    // trailer and the zero gap between the scales and the trailer
    if (threadIdx.x < 2) {
        for (int j = 0; j < k; ++j) {
            const int d = sdest[j];
            if (d < 0 || d >= R_cap)
                continue;
            uint8_t *row = rows + (int64_t)d * S;
            if (threadIdx.x == 0) {
                st16(row + S - 16, make_uint4(f2u(St), a_bits << 16, (uint32_t)t, 0u));
            } else {
                for (int64_t o = 9 * (int64_t)H / 16; o < S - 16; o += 2)
                    *reinterpret_cast<uint16_t *>(row + o) = 0;
            }
        }
    }
}

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
        const uint32_t b = max(absmax16_bits(&w[0]), absmax16_bits(&w[8]));
        // smallest e in [-127, 127] with B <= 448 * 2^e; 448 = 1.75 * 2^8, i.e.
        // BF16 exponent field 135 with mantissa field 96
        const int ef = (b >> 7) & 0xff, mt = b & 0x7f;
        int e = (ef == 0) ? -127 : ef - 135 + (mt > 96 ? 1 : 0);
        e = max(-127, min(127, e));
        const float f = (e <= 126) ? exp2i(-e) : u2f(0x00400000u); // 2^-e
        const float2 f2 = make_float2(f, f);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 a = mul2(make_float2(bf16lo(w[2 * i]), bf16hi(w[2 * i])), f2);
            const float2 bb = mul2(make_float2(bf16lo(w[2 * i + 1]), bf16hi(w[2 * i + 1])), f2);
            o[i] = cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(bb.x, bb.y) << 16);
        }
        const uint8_t sbyte = (uint8_t)(e + 127);
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
            scales[(int64_t)d * (H / 32) + q] = sbyte;
        }
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
    int p = 2 * c.num_sms;
    return E < 8 ? 8 : (p < 8 ? 8 : p);
}

template <int CPT>
static cudaError_t launch_nvfp4_cpt(const LaunchCtx &c, const uint16_t *tokens, int T, int H,
                                    const int32_t *dest, int k, const int32_t *offsets,
                                    const int32_t *counts, int E, uint8_t *rows, int R_cap,
                                    int rounding, uint64_t seed, uint32_t *status)
{
    const int th = pack_threads(H, CPT);
    const int pc = padding_ctas(c, E);
    const int64_t S = row_bytes(H);
    if (rounding == 1)
        return launch_pdl(nvfp4_pack_kernel<CPT, true>, dim3(T + pc), dim3(th), 0, c.stream, tokens,
                          T, H, dest, k, offsets, counts, E, rows, S, R_cap, seed, status, pc);
    return launch_pdl(nvfp4_pack_kernel<CPT, false>, dim3(T + pc), dim3(th), 0, c.stream, tokens, T,
                      H, dest, k, offsets, counts, E, rows, S, R_cap, seed, status, pc);
}

cudaError_t launch_nvfp4_pack(const LaunchCtx &c, const uint16_t *tokens, int T, int H,
                              const int32_t *dest, int k, const int32_t *offsets,
                              const int32_t *counts, int E, uint8_t *rows, int R_cap,
                              int rounding, uint64_t seed, uint32_t *status)
{
    const int nq = H / 32;
    if (nq <= kMaxThreads)
        return launch_nvfp4_cpt<1>(c, tokens, T, H, dest, k, offsets, counts, E, rows, R_cap,
                                   rounding, seed, status);
    if (nq <= 2 * kMaxThreads)
        return launch_nvfp4_cpt<2>(c, tokens, T, H, dest, k, offsets, counts, E, rows, R_cap,
                                   rounding, seed, status);
    return launch_nvfp4_cpt<4>(c, tokens, T, H, dest, k, offsets, counts, E, rows, R_cap, rounding,
                               seed, status);
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
    return launch_pdl(mxfp8_pack_kernel, dim3(T + pc), dim3(th), 0, c.stream, tokens, T, H,
                      dest, k, offsets, counts, E, buf, R_cap, status, pc, cpt);
}

} // namespace epq
