// extern "C" boundary of libepq.so (declared and documented in include/epq.h):
// argument validation on the host, the device guard, and the kernel launches.
// Nothing here allocates, frees or synchronises.
#include <stdint.h>
#include <string.h>

#include "../../include/epq.h"
#include "epq_internal.h"

namespace {

using epq::LaunchCtx;

// Makes `dev` current for the lifetime of the guard and restores the caller's
// current device afterwards (TE PR #3753, commit "guard the NVFP4 EP bindings
// with the input tensor's device").
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess)
            return;
        ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard()
    {
        if (ok && prev >= 0)
            cudaSetDevice(prev);
    }
};

// Device that owns `p`, or -1 if `p` is not device (or managed) memory.
int device_of(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
        return -1;
    return a.device;
}

bool on_device(const void *p, int dev) { return p == nullptr || device_of(p) == dev; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count(int dev)
{
    static std::atomic<int> cache[64] = {};
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0)
            return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 1;
    if (dev >= 0 && dev < 64)
        cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

ep_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess)
        return EP_OK;
    (void)cudaGetLastError();
    return EP_ERR_CUDA;
}

bool shape_ok(int64_t T, int64_t H, int k, int E)
{
    if (T < 0 || T > (int64_t)INT32_MAX / 32 || H < 32 || H % 32 != 0 || H > (1 << 20))
        return false;
    if (k < 1 || k > 32 || E < 1 || E > 1024)
        return false;
    return true;
}

} // namespace

extern "C" {

size_t ep_nvfp4_row_bytes(int64_t H) { return H > 0 ? (size_t)epq::row_bytes(H) : 0; }

int64_t ep_rows_capacity(int64_t T, int k, int E, int A)
{
    if (T < 0 || k < 1 || E < 1 || A < 1)
        return 0;
    return T * (int64_t)k + (int64_t)E * (int64_t)(A - 1);
}

size_t ep_route_workspace_bytes(int64_t T, int k, int E)
{
    (void)k;
    return epq::route_workspace_bytes(T < 0 ? 0 : T, E < 1 ? 1 : E);
}

const char *ep_status_string(int s)
{
    switch (s) {
    case EP_OK: return "EP_OK";
    case EP_ERR_NULL: return "EP_ERR_NULL: a required pointer is NULL";
    case EP_ERR_SHAPE: return "EP_ERR_SHAPE: size out of range (H % 32, k in [1,32], E in [1,1024])";
    case EP_ERR_ALIGN: return "EP_ERR_ALIGN: alignment A must be a positive multiple of 128 and buffers 16-byte aligned";
    case EP_ERR_CAPACITY: return "EP_ERR_CAPACITY: R_cap or workspace too small";
    case EP_ERR_ARG: return "EP_ERR_ARG: bad argument";
    case EP_ERR_DEVICE: return "EP_ERR_DEVICE: pointer is not device memory of the input's device";
    case EP_ERR_CUDA: return "EP_ERR_CUDA: a CUDA call failed";
    default: return "unknown ep_status";
    }
}

ep_status ep_route_plan(const int32_t *topk_idx, int64_t T, int k, int E, int A, int64_t R_cap,
                        int32_t *expert_offsets, int32_t *expert_counts, int32_t *dest,
                        void *workspace, size_t ws_bytes, uint32_t *dev_status, void *stream)
{
    if (!expert_offsets || !expert_counts || !workspace || !dev_status || (T > 0 && (!topk_idx || !dest)))
        return EP_ERR_NULL;
    if (T < 0 || T * (int64_t)k > (int64_t)INT32_MAX || k < 1 || k > 32 || E < 1 || E > 1024)
        return EP_ERR_SHAPE;
    if (A <= 0 || A % 128 != 0)
        return EP_ERR_ALIGN;
    if (R_cap < ep_rows_capacity(T, k, E, A) || R_cap > (int64_t)INT32_MAX)
        return EP_ERR_CAPACITY;
    if (ws_bytes < ep_route_workspace_bytes(T, k, E))
        return EP_ERR_CAPACITY;
    const int dev = device_of(expert_offsets);
    if (dev < 0 || !on_device(topk_idx, dev) || !on_device(expert_counts, dev) || !on_device(dest, dev) ||
        !on_device(workspace, dev) || !on_device(dev_status, dev))
        return EP_ERR_DEVICE;
    DeviceGuard g(dev);
    if (!g.ok)
        return EP_ERR_DEVICE;
    LaunchCtx c{(cudaStream_t)stream, dev, sm_count(dev)};
    return cuda_status(epq::launch_route_plan(c, topk_idx, (int)T, k, E, A, expert_offsets, expert_counts,
                                              dest, (int32_t *)workspace, dev_status));
}

static ep_status pack_common_checks(const void *tokens, int64_t T, int64_t H, const int32_t *dest, int k,
                                    const int32_t *offsets, const int32_t *counts, int E, const uint8_t *out,
                                    int64_t R_cap, const uint32_t *dev_status, int *dev_out)
{
    if (!offsets || !counts || !out || !dev_status || (T > 0 && (!tokens || !dest)))
        return EP_ERR_NULL;
    if (!shape_ok(T, H, k, E))
        return EP_ERR_SHAPE;
    if (R_cap < 0 || R_cap > (int64_t)INT32_MAX)
        return EP_ERR_CAPACITY;
    if (!aligned16(tokens) || !aligned16(out))
        return EP_ERR_ALIGN;
    const int dev = device_of(T > 0 ? tokens : (const void *)offsets);
    if (dev < 0 || !on_device(dest, dev) || !on_device(offsets, dev) || !on_device(counts, dev) ||
        !on_device(out, dev) || !on_device(dev_status, dev))
        return EP_ERR_DEVICE;
    *dev_out = dev;
    return EP_OK;
}

ep_status ep_nvfp4_pack(const void *tokens_bf16, int64_t T, int64_t H, const int32_t *dest, int k,
                        const int32_t *expert_offsets, const int32_t *expert_counts, int E, uint8_t *rows,
                        int64_t R_cap, float *expert_amax, int rounding, uint64_t seed, uint32_t *dev_status,
                        void *stream)
{
    int dev = -1;
    ep_status st = pack_common_checks(tokens_bf16, T, H, dest, k, expert_offsets, expert_counts, E, rows,
                                      R_cap, dev_status, &dev);
    if (st != EP_OK)
        return st;
    if (!on_device(expert_amax, dev))
        return EP_ERR_DEVICE;
    if ((reinterpret_cast<uintptr_t>(expert_amax) & 3u) != 0)
        return EP_ERR_ALIGN;
    if (rounding != EP_ROUND_RNE && rounding != EP_ROUND_SR)
        return EP_ERR_ARG;
    DeviceGuard g(dev);
    if (!g.ok)
        return EP_ERR_DEVICE;
    LaunchCtx c{(cudaStream_t)stream, dev, sm_count(dev)};
    epq::PackAmax am;
    am.amax = expert_amax;
    return cuda_status(epq::launch_nvfp4_pack(c, (const uint16_t *)tokens_bf16, (int)T, (int)H, dest, k,
                                              expert_offsets, expert_counts, E, rows, (int)R_cap, rounding,
                                              seed, dev_status, false, am));
}

ep_status ep_nvfp4_dispatch(const int32_t *topk_idx, const void *tokens_bf16, int64_t T, int64_t H, int k, int E,
                            int A, int64_t R_cap, int32_t *expert_offsets, int32_t *expert_counts, int32_t *dest,
                            void *workspace, size_t ws_bytes, uint8_t *rows, float *expert_amax, int rounding,
                            uint64_t seed, uint32_t *dev_status, void *stream)
{
    if (!expert_offsets || !expert_counts || !workspace || !dev_status || !rows ||
        (T > 0 && (!topk_idx || !dest || !tokens_bf16)))
        return EP_ERR_NULL;
    if (T < 0 || T * (int64_t)k > (int64_t)INT32_MAX || k < 1 || k > 32 || E < 1 || E > 1024 ||
        !shape_ok(T, H, k, E))
        return EP_ERR_SHAPE;
    if (A <= 0 || A % 128 != 0 || !aligned16(tokens_bf16) || !aligned16(rows) ||
        (reinterpret_cast<uintptr_t>(expert_amax) & 3u) != 0)
        return EP_ERR_ALIGN;
    if (R_cap < ep_rows_capacity(T, k, E, A) || R_cap > (int64_t)INT32_MAX)
        return EP_ERR_CAPACITY;
    if (ws_bytes < ep_route_workspace_bytes(T, k, E))
        return EP_ERR_CAPACITY;
    if (rounding != EP_ROUND_RNE && rounding != EP_ROUND_SR)
        return EP_ERR_ARG;
    const int dev = device_of(expert_offsets);
    if (dev < 0 || !on_device(topk_idx, dev) || !on_device(tokens_bf16, dev) || !on_device(expert_counts, dev) ||
        !on_device(dest, dev) || !on_device(workspace, dev) || !on_device(rows, dev) || !on_device(dev_status, dev) ||
        !on_device(expert_amax, dev))
        return EP_ERR_DEVICE;
    DeviceGuard g(dev);
    if (!g.ok)
        return EP_ERR_DEVICE;
    LaunchCtx c{(cudaStream_t)stream, dev, sm_count(dev)};
    // the routing kernel zeroes expert_amax; the pack max-reduces into it,
    // taking each slot's expert straight from topk_idx
    cudaError_t err = epq::launch_route_plan(c, topk_idx, (int)T, k, E, A, expert_offsets, expert_counts, dest,
                                             (int32_t *)workspace, dev_status, expert_amax);
    epq::PackAmax am;
    am.topk = topk_idx;
    am.amax = expert_amax;
    if (err == cudaSuccess)
        err = epq::launch_nvfp4_pack(c, (const uint16_t *)tokens_bf16, (int)T, (int)H, dest, k, expert_offsets,
                                     expert_counts, E, rows, (int)R_cap, rounding, seed, dev_status, true, am);
    return cuda_status(err);
}

ep_status ep_nvfp4_colwise_rht_bf16(const void *x_bf16, int64_t R_cap, int64_t H, const int32_t *expert_offsets,
                                    int E, const float *amax_in, uint8_t *cw_codes, uint8_t *cw_scales,
                                    float *amax_row, float *amax_col, float *cw_scale_enc, int rounding,
                                    uint64_t seed, uint16_t rht_sign_mask, uint32_t *dev_status, void *stream)
{
    if (!x_bf16 || !expert_offsets || !amax_in || !cw_codes || !cw_scales || !amax_row || !amax_col ||
        !cw_scale_enc || !dev_status)
        return EP_ERR_NULL;
    if (!shape_ok(0, H, 1, E))
        return EP_ERR_SHAPE;
    if (R_cap < 0 || R_cap > (int64_t)INT32_MAX || R_cap * H / 2 > (int64_t)INT32_MAX * 16)
        return EP_ERR_CAPACITY;
    if (rounding != EP_ROUND_RNE && rounding != EP_ROUND_SR)
        return EP_ERR_ARG;
    if (!aligned16(x_bf16) || !aligned16(cw_codes) || !aligned16(cw_scales))
        return EP_ERR_ALIGN;
    const int dev = device_of(x_bf16);
    if (dev < 0 || !on_device(expert_offsets, dev) || !on_device(amax_in, dev) || !on_device(cw_codes, dev) ||
        !on_device(cw_scales, dev) || !on_device(amax_row, dev) || !on_device(amax_col, dev) ||
        !on_device(cw_scale_enc, dev) || !on_device(dev_status, dev))
        return EP_ERR_DEVICE;
    DeviceGuard g(dev);
    if (!g.ok)
        return EP_ERR_DEVICE;
    LaunchCtx c{(cudaStream_t)stream, dev, sm_count(dev)};
    return cuda_status(epq::launch_colwise_rht_bf16(c, (const uint16_t *)x_bf16, (int)R_cap, (int)H, expert_offsets,
                                                    E, amax_in, cw_codes, cw_scales, amax_row, amax_col,
                                                    cw_scale_enc, rounding, seed, rht_sign_mask, dev_status));
}

ep_status ep_mxfp8_colwise(const void *x_bf16, int64_t R_cap, int64_t H, const int32_t *expert_offsets, int E,
                           uint8_t *buf, uint32_t *dev_status, void *stream)
{
    if (!x_bf16 || !expert_offsets || !buf || !dev_status)
        return EP_ERR_NULL;
    if (!shape_ok(0, H, 1, E))
        return EP_ERR_SHAPE;
    if (R_cap < 0 || R_cap > (int64_t)INT32_MAX || R_cap * H > (int64_t)INT32_MAX * 32)
        return EP_ERR_CAPACITY;
    if (!aligned16(x_bf16) || !aligned16(buf))
        return EP_ERR_ALIGN;
    const int dev = device_of(x_bf16);
    if (dev < 0 || !on_device(expert_offsets, dev) || !on_device(buf, dev) || !on_device(dev_status, dev))
        return EP_ERR_DEVICE;
    DeviceGuard g(dev);
    if (!g.ok)
        return EP_ERR_DEVICE;
    LaunchCtx c{(cudaStream_t)stream, dev, sm_count(dev)};
    return cuda_status(epq::launch_mxfp8_colwise(c, (const uint16_t *)x_bf16, (int)R_cap, (int)H, expert_offsets, E,
                                                 buf, dev_status));
}

ep_status ep_mxfp8_pack(const void *tokens_bf16, int64_t T, int64_t H, const int32_t *dest, int k,
                        const int32_t *expert_offsets, const int32_t *expert_counts, int E, uint8_t *buf,
                        int64_t R_cap, uint32_t *dev_status, void *stream)
{
    int dev = -1;
    ep_status st = pack_common_checks(tokens_bf16, T, H, dest, k, expert_offsets, expert_counts, E, buf,
                                      R_cap, dev_status, &dev);
    if (st != EP_OK)
        return st;
    DeviceGuard g(dev);
    if (!g.ok)
        return EP_ERR_DEVICE;
    LaunchCtx c{(cudaStream_t)stream, dev, sm_count(dev)};
    return cuda_status(epq::launch_mxfp8_pack(c, (const uint16_t *)tokens_bf16, (int)T, (int)H, dest, k,
                                              expert_offsets, expert_counts, E, buf, (int)R_cap, dev_status));
}

ep_status ep_nvfp4_unpack(const uint8_t *rows, int64_t R_cap, int64_t H, const int32_t *expert_offsets, int E,
                          void *out_bf16, uint32_t *dev_status, void *stream)
{
    if (!rows || !expert_offsets || !out_bf16 || !dev_status)
        return EP_ERR_NULL;
    if (!shape_ok(0, H, 1, E))
        return EP_ERR_SHAPE;
    if (R_cap < 0 || R_cap > (int64_t)INT32_MAX)
        return EP_ERR_CAPACITY;
    if (!aligned16(rows) || !aligned16(out_bf16))
        return EP_ERR_ALIGN;
    const int dev = device_of(rows);
    if (dev < 0 || !on_device(expert_offsets, dev) || !on_device(out_bf16, dev) || !on_device(dev_status, dev))
        return EP_ERR_DEVICE;
    DeviceGuard g(dev);
    if (!g.ok)
        return EP_ERR_DEVICE;
    LaunchCtx c{(cudaStream_t)stream, dev, sm_count(dev)};
    return cuda_status(epq::launch_nvfp4_unpack(c, rows, (int)R_cap, (int)H, expert_offsets, E,
                                                (uint16_t *)out_bf16, dev_status));
}

static ep_status direct_receive_common(const uint8_t *rows, int64_t R_cap, int64_t H,
                                       const int32_t *expert_offsets, int E, const float *expert_amax,
                                       const ep_nvfp4_grouped *out,
                                       int rounding, uint64_t seed, uint16_t rht_sign_mask, uint32_t *dev_status,
                                       void *stream, bool swz)
{
    if (!rows || !expert_offsets || !out || !dev_status)
        return EP_ERR_NULL;
    if (!out->cw_codes || !out->cw_scales || !out->amax_row || !out->amax_col || !out->cw_scale_enc)
        return EP_ERR_NULL;
    const bool rw_any = out->rw_codes || out->rw_scales || out->rw_row_scale;
    const bool rw_all = out->rw_codes && out->rw_scales && out->rw_row_scale;
    if (rw_any && !rw_all)
        return EP_ERR_NULL;
    if (!shape_ok(0, H, 1, E) || (swz && H % 128 != 0))
        return EP_ERR_SHAPE;
    // element positions (the SR counters) below 2^36
    if (R_cap < 0 || R_cap > (int64_t)INT32_MAX || R_cap * H > ((int64_t)1 << 36))
        return EP_ERR_CAPACITY;
    if (rounding != EP_ROUND_RNE && rounding != EP_ROUND_SR)
        return EP_ERR_ARG;
    if (!aligned16(rows) || !aligned16(out->cw_codes) || !aligned16(out->cw_scales) ||
        (rw_all && (!aligned16(out->rw_codes) || !aligned16(out->rw_scales))) ||
        (reinterpret_cast<uintptr_t>(expert_amax) & 3u) != 0)
        return EP_ERR_ALIGN;
    const int dev = device_of(rows);
    if (dev < 0 || !on_device(expert_offsets, dev) || !on_device(dev_status, dev) ||
        !on_device(out->rw_codes, dev) || !on_device(out->rw_scales, dev) || !on_device(out->rw_row_scale, dev) ||
        !on_device(out->cw_codes, dev) || !on_device(out->cw_scales, dev) || !on_device(out->amax_row, dev) ||
        !on_device(out->amax_col, dev) || !on_device(out->cw_scale_enc, dev) || !on_device(expert_amax, dev))
        return EP_ERR_DEVICE;
    DeviceGuard g(dev);
    if (!g.ok)
        return EP_ERR_DEVICE;
    LaunchCtx c{(cudaStream_t)stream, dev, sm_count(dev)};
    epq::GroupedOut o{out->rw_codes, out->rw_scales, out->rw_row_scale, out->cw_codes,
                      out->cw_scales, out->amax_row, out->amax_col, out->cw_scale_enc};
    return cuda_status(epq::launch_direct_receive(c, rows, (int)R_cap, (int)H, expert_offsets, E, o, rounding,
                                                  seed, rht_sign_mask, dev_status, swz, expert_amax));
}

ep_status ep_nvfp4_direct_receive(const uint8_t *rows, int64_t R_cap, int64_t H, const int32_t *expert_offsets,
                                  int E, const float *expert_amax, const ep_nvfp4_grouped *out, int rounding,
                                  uint64_t seed, uint16_t rht_sign_mask, uint32_t *dev_status, void *stream)
{
    return direct_receive_common(rows, R_cap, H, expert_offsets, E, expert_amax, out, rounding, seed, rht_sign_mask,
                                 dev_status, stream, false);
}

ep_status ep_nvfp4_direct_receive_swizzled(const uint8_t *rows, int64_t R_cap, int64_t H,
                                           const int32_t *expert_offsets, int E, const float *expert_amax,
                                           const ep_nvfp4_grouped *out, int rounding, uint64_t seed,
                                           uint16_t rht_sign_mask, uint32_t *dev_status, void *stream)
{
    return direct_receive_common(rows, R_cap, H, expert_offsets, E, expert_amax, out, rounding, seed, rht_sign_mask,
                                 dev_status, stream, true);
}

} // extern "C"
