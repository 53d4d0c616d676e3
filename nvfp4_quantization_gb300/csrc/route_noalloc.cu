// ep_route_plan_noalloc: the routing plan for callers that cannot hand the
// library a workspace buffer.
//
// Who needs it: a caller whose device memory is owned entirely by someone
// else -- an inference runtime or plugin host that reserves the GPU's memory
// up front in its own pool and gives an extension only its input and output
// tensors, or a latency-critical loop where a cudaMalloc would synchronise
// the device and stall the step.  ep_route_plan wants a caller-provided
// workspace; this entry point uses a fixed scratch array that lives inside
// the library instead, and allocates nothing on any call.
//
// The scratch is a file-scope __device__ array.  Every GPU that loads the
// library holds its EP_ROUTE_STATIC_SCRATCH_BYTES until the process exits,
// and every call on a device shares that device's copy, so two calls whose
// kernels overlap on one GPU (two streams, or two host threads) race on it.
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "../../include/epq.h"
#include "epq_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Barrier words, then one row of per-expert totals per CTA, exactly as the
// workspace of ep_route_plan.  Zero at module load; each call clears the
// barrier words again before its launch (a call that timed out may have left
// them non-zero).  The totals need no clearing: every CTA writes its own row
// before any CTA reads it.
static __device__ __align__(256) uint32_t g_route_scratch[EP_ROUTE_STATIC_SCRATCH_BYTES / 4];

// In host code `g_route_scratch` names a host-side stand-in, not device
// memory: only the address cudaGetSymbolAddress returns (per device, with
// that device current) may be handed to a kernel.  The address belongs to the
// device's current context: after that context is destroyed and a new one
// made (cudaDeviceReset, for one), the module is loaded again, possibly
// elsewhere.  So each cached address carries the unique id of the context it
// was looked up in, and a different current context looks it up again.
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};

// Unique id of the calling thread's current context (driver entry points,
// found through the runtime so that nothing links libcuda directly).
cudaError_t current_context_id(unsigned long long *id)
{
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    if (!get_current || !get_id) {
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &r1) != cudaSuccess ||
            r1 != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) != cudaSuccess ||
            r2 != cudaDriverEntryPointSuccess)
            return cudaErrorNotSupported;
        get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(q);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, id) != CUDA_SUCCESS)
        return cudaErrorDeviceUninitialized;
    return cudaSuccess;
}

// The scratch address of device `dev` (current) in its current context.  The
// look-up is set-up work that must not run inside a stream capture: if the
// address is not known yet for this context and `stream` is capturing, the
// call fails (EP_ERR_ARG) instead.
ep_status scratch_address(int dev, cudaStream_t stream, void **out)
{
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    unsigned long long ctx = 0;
    if (current_context_id(&ctx) != cudaSuccess)
        return EP_ERR_CUDA;
    if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess)
            return EP_ERR_CUDA;
        if (cs != cudaStreamCaptureStatusNone)
            return EP_ERR_ARG;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess)
            return EP_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return EP_OK;
}

int owning_device(const void *p)
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

bool same_device(const void *p, int dev) { return p == nullptr || owning_device(p) == dev; }

} // namespace

extern "C" ep_status ep_route_plan_noalloc(const int32_t *topk_idx, int64_t T, int k, int E, int A,
                                           int64_t R_cap, int32_t *expert_offsets, int32_t *expert_counts,
                                           int32_t *dest, uint32_t *dev_status, void *stream)
{
    if (!expert_offsets || !expert_counts || !dev_status || (T > 0 && (!topk_idx || !dest)))
        return EP_ERR_NULL;
    if (T < 0 || T * (int64_t)k > (int64_t)INT32_MAX || k < 1 || k > 32 || E < 1 || E > 1024)
        return EP_ERR_SHAPE;
    if (A <= 0 || A % 128 != 0)
        return EP_ERR_ALIGN;
    if (R_cap < ep_rows_capacity(T, k, E, A) || R_cap > (int64_t)INT32_MAX)
        return EP_ERR_CAPACITY;
    // the one limit this variant adds: its plan must fit the fixed scratch
    if (ep_route_workspace_bytes(T, k, E) > (size_t)EP_ROUTE_STATIC_SCRATCH_BYTES)
        return EP_ERR_CAPACITY;
    const int dev = owning_device(expert_offsets);
    if (dev < 0 || dev >= kMaxDevices || !same_device(topk_idx, dev) || !same_device(expert_counts, dev) ||
        !same_device(dest, dev) || !same_device(dev_status, dev))
        return EP_ERR_DEVICE;

    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) {
        (void)cudaGetLastError();
        return EP_ERR_CUDA;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return EP_ERR_DEVICE;
    }
    void *scratch = nullptr;
    int nsm = 0;
    const ep_status se = scratch_address(dev, (cudaStream_t)stream, &scratch);
    if (se != EP_OK) {
        (void)cudaGetLastError();
        if (prev != dev)
            cudaSetDevice(prev);
        return se;
    }
    cudaError_t e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(scratch, 0, 16, (cudaStream_t)stream);   // barrier count and generation
    if (e == cudaSuccess) {
        const epq::LaunchCtx c{(cudaStream_t)stream, dev, nsm > 0 ? nsm : 1};
        e = epq::launch_route_plan(c, topk_idx, (int)T, k, E, A, expert_offsets, expert_counts, dest,
                                   static_cast<int32_t *>(scratch), dev_status);
    }
    if (prev != dev)
        cudaSetDevice(prev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return EP_ERR_CUDA;
    }
    return EP_OK;
}
