// Host-side declarations shared by the epq translation units: kernel
// launchers (one per kernel family) and launch helpers.  The extern "C"
// boundary that validates arguments lives in api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace epq {

struct LaunchCtx {
    cudaStream_t stream;
    int device;
    int num_sms;
};

// Launch `kernel` with programmatic stream serialization (PDL) so that its
// launch latency overlaps the tail of the preceding kernel; every epq kernel
// calls griddepcontrol.wait before it reads memory another kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Sets the dynamic shared-memory limit of `kernel` once per device (it is a
// per-function attribute; setting it again inside a stream capture is avoided).
// The per-device flags are atomic: calls from several host threads may race to
// set the same attribute, which is harmless.
template <typename K>
cudaError_t ensure_smem_limit(K kernel, int device, int bytes, std::atomic<uint32_t> *done_mask_words /*[2]*/)
{
    const int w = device >> 5;
    const uint32_t bit = 1u << (device & 31);
    if (device >= 0 && device < 64 && (done_mask_words[w].load(std::memory_order_acquire) & bit))
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && device >= 0 && device < 64)
        done_mask_words[w].fetch_or(bit, std::memory_order_release);
    return e;
}

size_t route_workspace_bytes(int64_t T, int E);
// Launched without programmatic dependency: it starts only once every earlier
// kernel on the stream has finished (launch_nvfp4_pack's `early` relies on it).
// amax_zero (optional, f32 [E]): set to 0 by the kernel, for a pack that
// max-reduces the per-expert amax into it.
cudaError_t launch_route_plan(const LaunchCtx &c, const int32_t *topk, int T, int k, int E, int A,
                              int32_t *offsets, int32_t *counts, int32_t *dest, int32_t *hist,
                              uint32_t *status, float *amax_zero = nullptr);

// The pack's optional per-expert amax: every written row's token amax A_t is
// max-reduced into amax[e] of its expert e (the array holds zeros, or an
// earlier partial max, when the pack starts).  topk, when given, names the
// expert of each (token, slot) directly; otherwise it is found from the row
// index and the expert offsets.
struct PackAmax {
    const int32_t *topk = nullptr;
    float *amax = nullptr;
};

// early: the launch directly follows launch_route_plan on the same stream,
// so the tokens may be read before the wait for the routing kernel.
cudaError_t launch_nvfp4_pack(const LaunchCtx &c, const uint16_t *tokens, int T, int H,
                              const int32_t *dest, int k, const int32_t *offsets,
                              const int32_t *counts, int E, uint8_t *rows, int R_cap,
                              int rounding, uint64_t seed, uint32_t *status, bool early = false,
                              PackAmax am = PackAmax());

cudaError_t launch_mxfp8_pack(const LaunchCtx &c, const uint16_t *tokens, int T, int H,
                              const int32_t *dest, int k, const int32_t *offsets,
                              const int32_t *counts, int E, uint8_t *buf, int R_cap,
                              uint32_t *status);

cudaError_t launch_nvfp4_unpack(const LaunchCtx &c, const uint8_t *rows, int R_cap, int H,
                                const int32_t *offsets, int E, uint16_t *out, uint32_t *status);

struct GroupedOut {
    uint8_t *rw_codes;
    uint8_t *rw_scales;
    float *rw_row_scale;
    uint8_t *cw_codes;
    uint8_t *cw_scales;
    float *amax_row;
    float *amax_col;
    float *scale_enc;
};

cudaError_t launch_colwise_rht_bf16(const LaunchCtx &c, const uint16_t *x, int R_cap, int H, const int32_t *offsets,
                                    int E, const float *amax_in, uint8_t *cw_codes, uint8_t *cw_scales,
                                    float *amax_row, float *amax_col, float *scale_enc, int rounding, uint64_t seed,
                                    uint32_t sign_mask, uint32_t *status);

cudaError_t launch_mxfp8_colwise(const LaunchCtx &c, const uint16_t *x, int R_cap, int H, const int32_t *offsets,
                                 int E, uint8_t *buf, uint32_t *status);

// swz: both scale tensors in the tiled layout of block-scaled GEMM operands
// (H % 128 == 0, checked by the caller).
cudaError_t launch_direct_receive(const LaunchCtx &c, const uint8_t *rows, int R_cap, int H,
                                  const int32_t *offsets, int E, const GroupedOut &out,
                                  int rounding, uint64_t seed, uint32_t sign_mask,
                                  uint32_t *status, bool swz = false, const float *amax_in = nullptr);

// Tensor map of a 2-D byte tensor [outer][inner] with a row pitch of `pitch`
// bytes and a box of box_outer rows x box_inner bytes (no swizzle, L2
// promotion 256 B); false if the driver refuses it.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t pitch,
              uint32_t box_inner, uint32_t box_outer);

// Bytes of a packed NVFP4 row: roundup16(9H/16 + 16).
inline int64_t row_bytes(int64_t H) { return (9 * H / 16 + 16 + 15) / 16 * 16; }

} // namespace epq
