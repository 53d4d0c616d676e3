// Decode packed NVFP4 rows to BF16: the path taken when direct receive is off
// (TE PR #3753 "Add NVFP4 EP dispatch and combine backward", PR description:
// without direct receive, the received rows go back to BF16; commit "grad
// direct-receive opt-out": the opt-out hands back that BF16 decode).
//
// Unit of work: 8 consecutive elements of a row (4 code bytes, one E4M3
// block scale, 16 bytes of BF16 out).  Consecutive threads take consecutive
// units, so a warp reads 128 contiguous code bytes and writes 512 contiguous
// output bytes per step; each thread keeps four units in flight.  The decode
// is exact (E2M1 x E4M3 in f16, then x the power-of-two token scale in FP32:
// at most six significant bits), so the BF16 conversion is exact except below
// BF16's normal range, where it rounds to nearest even.
#include "epq_device.cuh"
#include "epq_internal.h"

namespace epq {

// n / d for 32-bit n by a multiply-high (Granlund and Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, round-up variant):
// m = floor(2^32 (2^l - d) / d) + 1 with l = ceil(log2 d), then
// t = mulhi(m, n) and n / d = (t + ((n - t) >> 1)) >> (l - 1).
struct Div32 {
    uint32_t m;
    int s;   // l - 1
    uint32_t d;
};

static Div32 make_div32(uint32_t d)
{
    int l = 0;
    while (l < 32 && (1ull << l) < d)
        ++l;
    Div32 v;
    v.m = (uint32_t)((((1ull << l) - d) << 32) / d + 1);
    v.s = l > 0 ? l - 1 : 0;
    v.d = d;
    return v;
}

__device__ __forceinline__ uint32_t div32(uint32_t n, const Div32 &v)
{
    if (v.d == 1)
        return n;
    const uint32_t t = __umulhi(v.m, n);
    return (t + ((n - t) >> 1)) >> v.s;
}

constexpr int kUnpackThreads = 256;
constexpr int kUnpackUnits = 4;   // units in flight per thread

__global__ void __launch_bounds__(kUnpackThreads)
nvfp4_unpack_kernel(const uint8_t *__restrict__ rows, int R_cap, int H, int64_t S,
                    const int32_t *__restrict__ offsets, int E, uint16_t *__restrict__ out,
                    uint32_t *__restrict__ status, Div32 per_row)
{
    pdl_launch_dependents();
    pdl_wait();
    int R = offsets[E];
    if (R > R_cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            raise_status(status, kDevErrCapacity);
        R = R_cap;
    }
    const uint32_t nu = (uint32_t)H / 8;              // units per row
    const uint32_t total = (uint32_t)R * nu;
    const uint32_t stride = gridDim.x * kUnpackThreads;
    for (uint32_t i0 = blockIdx.x * kUnpackThreads + threadIdx.x; i0 < total; i0 += kUnpackUnits * stride) {
        uint32_t cw[kUnpackUnits], sb[kUnpackUnits];
        float st[kUnpackUnits];
        uint32_t ix[kUnpackUnits];
#pragma unroll
        for (int j = 0; j < kUnpackUnits; ++j) {
            const uint32_t i = i0 + j * stride;
            ix[j] = i;
            cw[j] = 0u;
            sb[j] = 0u;
            st[j] = 0.0f;
            if (i < total) {
                const uint32_t r = div32(i, per_row), q = i - r * nu;
                const uint8_t *row = rows + (int64_t)r * S;
                cw[j] = __ldg(reinterpret_cast<const uint32_t *>(row + 4 * q));
                sb[j] = __ldg(row + H / 2 + (q >> 1));
                st[j] = __ldg(reinterpret_cast<const float *>(row + S - 16));
            }
        }
#pragma unroll
        for (int j = 0; j < kUnpackUnits; ++j) {
            if (ix[j] >= total)
                break;
            const float sc = f16x2_to_f32x2(cvt_f16x2_from_e4m3x2(sb[j])).x * st[j];
            const float2 m = make_float2(sc, sc);
            uint32_t o[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float2 qv = f16x2_to_f32x2(cvt_f16x2_from_e2m1x2((cw[j] >> (8 * b)) & 0xffu));
                const float2 v = mul2(qv, m);
                o[b] = cvt_bf16x2(v.x, v.y);
            }
            *reinterpret_cast<uint4 *>(out + (int64_t)ix[j] * 8) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

cudaError_t launch_nvfp4_unpack(const LaunchCtx &c, const uint8_t *rows, int R_cap, int H,
                                const int32_t *offsets, int E, uint16_t *out, uint32_t *status)
{
    const int64_t S = row_bytes(H);
    const int64_t work = (int64_t)R_cap * (H / 8);
    if (work > (int64_t)UINT32_MAX)
        return cudaErrorInvalidValue;
    int64_t blocks = (work + kUnpackThreads * kUnpackUnits - 1) / (kUnpackThreads * kUnpackUnits);
    const int64_t cap = (int64_t)c.num_sms * (2048 / kUnpackThreads);
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    return launch_pdl(nvfp4_unpack_kernel, dim3((unsigned)blocks), dim3(kUnpackThreads), 0, c.stream, rows,
                      R_cap, H, S, offsets, E, out, status, make_div32((uint32_t)(H / 8)));
}

} // namespace epq
