// Decode packed NVFP4 rows to BF16: the path taken when direct receive is off
// (TE PR #3753 "Add NVFP4 EP dispatch and combine backward", PR description:
// "Otherwise the rows are decoded to BF16"; commit "grad direct-receive
// opt-out": the opt-out returns the BF16 decode of the received rows).
//
// Grid-stride over (row, 32-element chunk): a thread reads 16 code bytes and
// 2 scale bytes of one row, decodes them exactly (E2M1 x E4M3 in f16, then x
// the power-of-two token scale in FP32) and writes 64 bytes of BF16.  The
// product has at most six significant bits, so the BF16 conversion is exact
// except below BF16's normal range, where it rounds to nearest even.
#include "epq_device.cuh"
#include "epq_internal.h"

namespace epq {

__global__ void __launch_bounds__(256)
nvfp4_unpack_kernel(const uint8_t *__restrict__ rows, int R_cap, int H, int64_t S,
                    const int32_t *__restrict__ offsets, int E, uint16_t *__restrict__ out,
                    uint32_t *__restrict__ status)
{
    pdl_launch_dependents();
    pdl_wait();
    int R = offsets[E];
    if (R > R_cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            raise_status(status, kDevErrCapacity);
        R = R_cap;
    }
    const int nq = H / 32;
    const int64_t total = (int64_t)R * nq;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / nq;
        const int q = (int)(i - r * nq);
        const uint8_t *row = rows + r * S;
        const uint4 cb = __ldg(reinterpret_cast<const uint4 *>(row + (int64_t)q * 16));
        const uint32_t sc2 = *reinterpret_cast<const uint16_t *>(row + H / 2 + q * 2);
        const float St = __ldg(reinterpret_cast<const float *>(row + S - 16));
        const float2 sb = f16x2_to_f32x2(cvt_f16x2_from_e4m3x2(sc2));
        const float2 m0 = make_float2(sb.x * St, sb.x * St), m1 = make_float2(sb.y * St, sb.y * St);
        const uint32_t cw[4] = {cb.x, cb.y, cb.z, cb.w};
        uint32_t o[16];
#pragma unroll
        for (int b = 0; b < 16; ++b) {
            const uint32_t byte = (cw[b >> 2] >> (8 * (b & 3))) & 0xffu;
            const float2 qv = f16x2_to_f32x2(cvt_f16x2_from_e2m1x2(byte));
            const float2 v = mul2(qv, b < 8 ? m0 : m1);
            o[b] = cvt_bf16x2(v.x, v.y);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(out + r * H + (int64_t)q * 32);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        dst[2] = make_uint4(o[8], o[9], o[10], o[11]);
        dst[3] = make_uint4(o[12], o[13], o[14], o[15]);
    }
}

cudaError_t launch_nvfp4_unpack(const LaunchCtx &c, const uint8_t *rows, int R_cap, int H,
                                const int32_t *offsets, int E, uint16_t *out, uint32_t *status)
{
    const int64_t S = row_bytes(H);
    const int64_t work = (int64_t)R_cap * (H / 32);
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = (int64_t)c.num_sms * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    return launch_pdl(nvfp4_unpack_kernel, dim3((unsigned)blocks), dim3(256), 0, c.stream, rows,
                      R_cap, H, S, offsets, E, out, status);
}

} // namespace epq
