// Route plan: expert-contiguous, alignment-padded placement of every
// (token, routing slot) -- the one-GPU stand-in for the expert-parallel
// dispatch of TE PR #3270 "EP dispatch with unfused MXFP8 quantization"
// (description: expert-major received rows returned as a per-expert grouped
// tensor; review thread: each expert slot aligned to a multiple of 128 rows).
//
// One cooperative launch (every CTA resident), two phases around one grid
// barrier:
//  1. each CTA takes a contiguous run of 512-token chunks (one thread per
//     token), validates the ids and ranks every slot among the CTA's earlier
//     slots of the same expert: per chunk, each warp owns one 32-bit word of
//     every expert's token mask (each lane ORs its bit into the word of its
//     slot's expert, a shared-memory atomic; no warp-synchronous match),
//     the words are prefix-counted, and a running per-expert count carries
//     over to the next chunk; the CTA's per-expert totals go to the workspace.
//  2. after the barrier every CTA sums the totals of the CTAs before it (its
//     base inside each expert) and of all CTAs, scans the aligned totals into
//     expert offsets and turns its slots' ranks into row indices.  Rows of an
//     expert follow ascending token order because CTAs, chunks and ranks are
//     all in token order.
// The barrier waits are bounded: on timeout EP_DEV_ERR_TIMEOUT is raised and
// the outputs are invalid.
// Batches of at most 16 chunks (8192 tokens) with k <= 8 run as one
// thread-block cluster instead, when the device can place it: the totals stay
// in shared memory, the hardware cluster barrier replaces the grid barrier and
// phase 2 reads the other CTAs' totals through distributed shared memory.
#include "epq_device.cuh"
#include "epq_internal.h"

#include <map>
#include <mutex>
#include <tuple>

namespace epq {

constexpr int kChunk = 512;              // tokens per chunk, one thread each
constexpr int kWords = kChunk / 32;      // mask words per expert

// The token masks live as [word][expert] rows of an odd pitch (E, or E + 1
// when E is even): the 16 words of one expert (the per-expert prefix) fall on
// 16 different banks, and the lanes of a warp looking up their own experts'
// word `warp` collide only where two experts meet modulo 32 (with [expert]
// [word] rows, every expert's word `warp` lay on one of two banks).
__host__ __device__ inline int mask_pitch(int E) { return E | 1; }
constexpr int kRankBits = 21;            // temp encoding: expert << 21 | rank in CTA
constexpr int kWsHeader = 4;             // workspace words before the totals: barrier count, generation

// In-place exclusive scan of a[0, n) in shared memory (n <= 1024); every thread
// of the block calls it; returns the total.
__device__ int block_exclusive_scan(int *a, int n, int *wtmp)
{
    const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = (nt + 31) / 32;
    const int per = (n + nt - 1) / nt;
    const int b = min(tid * per, n), en = min(b + per, n);
    int sum = 0;
    for (int i = b; i < en; ++i)
        sum += a[i];
    int x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        wtmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int v = (lane < nwarps) ? wtmp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o)
                v += y;
        }
        wtmp[lane] = v;
    }
    __syncthreads();
    int run = (warp ? wtmp[warp - 1] : 0) + x - sum;
    const int total = wtmp[nwarps - 1];
    for (int i = b; i < en; ++i) {
        const int v = a[i];
        a[i] = run;
        run += v;
    }
    __syncthreads();
    return total;
}

// Grid-wide barrier over a cooperative launch.  Self-resetting: the last CTA
// to arrive zeroes the count and bumps the generation the others wait on, so
// the two workspace words are back to a usable state after every call (they
// must be zero before the first call).  `g` is the generation thread 0 read
// at kernel start: it cannot change before this CTA arrives.  Arrival is one
// acquire-release atomic (it publishes this CTA's writes, and the last CTA
// acquires everyone's before its release of the generation), so no separate
// fences are needed.  Bounded: gives up after ~1 s.
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ bool grid_barrier(uint32_t *count, uint32_t *gen, uint32_t g, uint32_t n, int *flag)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        uint32_t old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(count) : "memory");
        if (old + 1u == n) {
            asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(count), "r"(0u) : "memory");
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(gen) : "memory");
        } else {
            ok = 0;
            for (uint32_t i = 0; i < (1u << 23); ++i) {
                if (ld_acquire_gpu(gen) != g) {
                    ok = 1;
                    break;
                }
                if (i > 4096)
                    __nanosleep(128);
            }
        }
        *flag = ok;
    }
    __syncthreads();
    return *flag != 0;
}

// Fast path: one 512-token chunk per CTA and k <= 8: the validated ids and
// the ranks of a thread's slots stay in registers between the phases.
constexpr int kRegSlots = 8;
constexpr int kMaxClusterCtas = 16;   // largest (non-portable) thread-block cluster

// kCluster: the whole grid is one thread-block cluster (at most 16 CTAs):
// the per-CTA totals stay in shared memory, the grid barrier is the cluster
// barrier and phase 2 reads the other CTAs' totals through distributed shared
// memory, so no global round trip separates the phases.
template <bool kCluster>
__global__ void __launch_bounds__(kChunk, 1)
route_plan_reg_kernel(const int32_t *__restrict__ topk, int T, int k, int E, int A,
                      int32_t *__restrict__ offsets, int32_t *__restrict__ counts, int32_t *__restrict__ dest,
                      uint32_t *__restrict__ ws, uint32_t *__restrict__ status, float *__restrict__ amax_zero)
{
    extern __shared__ uint32_t sm[];
    // the per-expert amax the pack that follows max-reduces into starts at 0
    if (amax_zero && blockIdx.x == 0)
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            amax_zero[e] = 0.0f;
    const int P = mask_pitch(E);
    uint32_t *mask = sm;                         // [kWords][P]
    uint32_t *pre = mask + (size_t)kWords * P;   // [kWords][P]
    int *tot = reinterpret_cast<int *>(pre + (size_t)kWords * P);  // [E]
    int *base = tot + E;                         // [E]
    int *off = base + E;                         // [E]
    int *myhist = off + E;                       // [E] this CTA's totals (cluster variant)
    __shared__ int wtmp[32];
    __shared__ int flag;

    // the next kernel may be scheduled now: it waits for this grid's
    // completion (griddepcontrol.wait) before it reads anything
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cta = blockIdx.x, nctas = gridDim.x;
    int32_t *hist = reinterpret_cast<int32_t *>(ws + kWsHeader);   // [nctas][E]
    const uint32_t g0 = (!kCluster && tid == 0) ? ld_relaxed_gpu(ws + 1) : 0u;  // barrier generation before arrival
    const int64_t t = (int64_t)cta * kChunk + tid;

    int raw[kRegSlots], ev[kRegSlots], rk[kRegSlots];
#pragma unroll
    for (int j = 0; j < kRegSlots; ++j)
        raw[j] = (t < T && j < k) ? topk[t * k + j] : -1;
    for (int i = tid; i < kWords * P; i += kChunk)
        mask[i] = 0u;
    __syncthreads();

    uint32_t bad = 0;
#pragma unroll
    for (int j = 0; j < kRegSlots; ++j) {
        int e = -1;
        const int v = raw[j];
        if (j < k && v != -1) {
            if (v < 0 || v >= E) {
                bad |= kDevErrBadExpert;
            } else {
                bool dup = false;
#pragma unroll
                for (int jj = 0; jj < j; ++jj)
                    dup |= (raw[jj] == v);
                if (dup)
                    bad |= kDevErrDupExpert;
                else
                    e = v;
            }
        }
        ev[j] = e;
        if (e >= 0)
            atomicOr(&mask[warp * P + e], 1u << lane);
    }
    if (bad)
        raise_status(status, bad);
    __syncthreads();
    for (int e = warp; e < E; e += kChunk / 32) {
        const uint32_t c = (lane < kWords) ? __popc(mask[lane * P + e]) : 0u;
        uint32_t x = c;
#pragma unroll
        for (int o = 1; o < kWords; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        if (lane < kWords)
            pre[lane * P + e] = x - c;
        if (lane == kWords - 1) {
            if (kCluster)
                myhist[e] = (int)x;
            else
                hist[(int64_t)cta * E + e] = (int)x;
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kRegSlots; ++j) {
        const int e = ev[j];
        rk[j] = e >= 0 ? (int)(pre[warp * P + e] + __popc(mask[warp * P + e] & ((1u << lane) - 1u))) : 0;
    }

    if (kCluster) {
        cluster_sync();   // every CTA's totals written
        for (int e = tid; e < E; e += kChunk) {
            int p = 0, all = 0;
#pragma unroll 16
            for (int c = 0; c < nctas; ++c) {
                const int h = (int)ld_dsmem_u32(myhist + e, (uint32_t)c);
                p += (c < cta) ? h : 0;
                all += h;
            }
            base[e] = p;
            tot[e] = all;
            off[e] = (all + A - 1) / A * A;
        }
        cluster_sync();   // every CTA done reading the others' totals
    } else {
        if (!grid_barrier(ws, ws + 1, g0, (uint32_t)nctas, &flag)) {
            if (tid == 0)
                raise_status(status, kDevErrTimeout);
            return;
        }
        for (int e = tid; e < E; e += kChunk) {
            int p = 0, all = 0;
            // 32 totals in flight per thread
#pragma unroll 32
            for (int c = 0; c < nctas; ++c) {
                const int h = __ldcg(hist + (int64_t)c * E + e);
                p += (c < cta) ? h : 0;
                all += h;
            }
            base[e] = p;
            tot[e] = all;
            off[e] = (all + A - 1) / A * A;
        }
    }
    __syncthreads();
    const int total = block_exclusive_scan(off, E, wtmp);
    if (cta == 0) {
        for (int e = tid; e < E; e += kChunk) {
            offsets[e] = off[e];
            counts[e] = tot[e];
        }
        if (tid == 0)
            offsets[E] = total;
    }
    for (int e = tid; e < E; e += kChunk)
        base[e] += off[e];
    __syncthreads();
    if (t < T) {
#pragma unroll
        for (int j = 0; j < kRegSlots; ++j)
            if (j < k)
                dest[t * k + j] = ev[j] >= 0 ? base[ev[j]] + rk[j] : -1;
    }
}

__global__ void __launch_bounds__(kChunk)
route_plan_kernel(const int32_t *__restrict__ topk, int T, int k, int E, int A, int chunks_per_cta,
                  int32_t *__restrict__ offsets, int32_t *__restrict__ counts, int32_t *__restrict__ dest,
                  uint32_t *__restrict__ ws, uint32_t *__restrict__ status, float *__restrict__ amax_zero)
{
    extern __shared__ uint32_t sm[];
    if (amax_zero && blockIdx.x == 0)
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            amax_zero[e] = 0.0f;
    const int P = mask_pitch(E);
    uint32_t *mask = sm;                         // [kWords][P]
    uint32_t *pre = mask + (size_t)kWords * P;   // [kWords][P]
    int *run = reinterpret_cast<int *>(pre + (size_t)kWords * P);  // [E]
    int *base = run + E;                         // [E]
    int *off = base + E;                         // [E]
    __shared__ int wtmp[32];
    __shared__ int flag;

    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cta = blockIdx.x, nctas = gridDim.x;
    int32_t *hist = reinterpret_cast<int32_t *>(ws + kWsHeader);   // [nctas][E]
    const uint32_t g0 = tid == 0 ? ld_relaxed_gpu(ws + 1) : 0u;  // barrier generation before arrival
    for (int e = tid; e < E; e += kChunk)
        run[e] = 0;

    // ---- phase 1: ranks inside the CTA's run of chunks
    uint32_t bad = 0;
    for (int ch = 0; ch < chunks_per_cta; ++ch) {
        const int64_t t = ((int64_t)cta * chunks_per_cta + ch) * kChunk + tid;
        for (int i = tid; i < kWords * P; i += kChunk)
            mask[i] = 0u;
        __syncthreads();
        for (int j = 0; j < k; ++j) {
            int e = -1;
            if (t < T) {
                const int v = topk[t * k + j];
                if (v != -1) {
                    if (v < 0 || v >= E) {
                        bad |= kDevErrBadExpert;
                    } else {
                        bool dup = false;
                        for (int jj = 0; jj < j; ++jj)
                            dup |= (topk[t * k + jj] == v);
                        if (dup)
                            bad |= kDevErrDupExpert;
                        else
                            e = v;
                    }
                }
                dest[t * k + j] = e; // validated expert id, consumed below
            }
            // each lane owns its bit of word `warp` of its expert's mask
            if (e >= 0)
                atomicOr(&mask[warp * P + e], 1u << lane);
        }
        __syncthreads();
        // exclusive prefix over the chunk's words of every expert (+ the run)
        for (int e = warp; e < E; e += kChunk / 32) {
            const uint32_t c = (lane < kWords) ? __popc(mask[lane * P + e]) : 0u;
            uint32_t x = c;
#pragma unroll
            for (int o = 1; o < kWords; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o)
                    x += y;
            }
            const int r0 = run[e];
            if (lane < kWords)
                pre[lane * P + e] = (uint32_t)r0 + x - c;
            __syncwarp();
            if (lane == kWords - 1)
                run[e] = r0 + (int)x;
        }
        __syncthreads();
        if (t < T) {
            for (int j = 0; j < k; ++j) {
                const int e = dest[t * k + j];
                if (e >= 0) {
                    const uint32_t below = mask[warp * P + e] & ((1u << lane) - 1u);
                    const int rank = (int)(pre[warp * P + e] + __popc(below));
                    dest[t * k + j] = (e << kRankBits) | rank;
                }
            }
        }
        __syncthreads();
    }
    if (bad)
        raise_status(status, bad);
    for (int e = tid; e < E; e += kChunk)
        hist[(int64_t)cta * E + e] = run[e];

    if (!grid_barrier(ws, ws + 1, g0, (uint32_t)nctas, &flag)) {
        if (tid == 0)
            raise_status(status, kDevErrTimeout);
        return;
    }

    // ---- phase 2: offsets, and global rows of this CTA's slots
    for (int e = tid; e < E; e += kChunk) {
        int p = 0, tot = 0;
#pragma unroll 8
        for (int c = 0; c < nctas; ++c) {
            const int h = __ldcg(hist + (int64_t)c * E + e);
            p += (c < cta) ? h : 0;
            tot += h;
        }
        base[e] = p;
        run[e] = tot;
        off[e] = (tot + A - 1) / A * A;
    }
    __syncthreads();
    const int total = block_exclusive_scan(off, E, wtmp);
    if (cta == 0) {
        for (int e = tid; e < E; e += kChunk) {
            offsets[e] = off[e];
            counts[e] = run[e];
        }
        if (tid == 0)
            offsets[E] = total;
    }
    for (int e = tid; e < E; e += kChunk)
        base[e] += off[e];
    __syncthreads();
    for (int ch = 0; ch < chunks_per_cta; ++ch) {
        const int64_t t = ((int64_t)cta * chunks_per_cta + ch) * kChunk + tid;
        if (t >= T)
            break;
        for (int j = 0; j < k; ++j) {
            const int v = dest[t * k + j];
            if (v >= 0)
                dest[t * k + j] = base[v >> kRankBits] + (v & ((1 << kRankBits) - 1));
        }
    }
}

size_t route_workspace_bytes(int64_t T, int E)
{
    // header + per-CTA totals for at most one CTA per 512-token chunk
    const int64_t nch = (T + kChunk - 1) / kChunk;
    return (size_t)kWsHeader * 4u + (size_t)(nch > 0 ? nch : 1) * (size_t)E * 4u;
}

cudaError_t launch_route_plan(const LaunchCtx &c, const int32_t *topk, int T, int k, int E, int A,
                              int32_t *offsets, int32_t *counts, int32_t *dest, int32_t *hist,
                              uint32_t *status, float *amax_zero)
{
    const size_t smem = (size_t)mask_pitch(E) * kWords * 4u * 2u + (size_t)E * 4u * 4u;
    static std::atomic<uint32_t> done[2] = {}, done_reg[2] = {}, done_cl[2] = {};
    cudaError_t err = ensure_smem_limit(route_plan_kernel, c.device, 1025 * kWords * 8 + 1024 * 16, done);
    if (err == cudaSuccess)
        err = ensure_smem_limit(route_plan_reg_kernel<false>, c.device, 1025 * kWords * 8 + 1024 * 16, done_reg);
    if (err == cudaSuccess)
        err = ensure_smem_limit(route_plan_reg_kernel<true>, c.device, 1025 * kWords * 8 + 1024 * 16, done_cl);
    if (err != cudaSuccess)
        return err;
    // each cooperative form is sized by its own kernel's residency
    int per_sm = 0, per_sm_reg = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_plan_kernel, kChunk, smem);
    if (err == cudaSuccess)
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_reg, route_plan_reg_kernel<false>, kChunk, smem);
    if (err != cudaSuccess)
        return err;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    const int nch = (T + kChunk - 1) / kChunk;
    // one chunk per CTA with the slots in registers when k <= 8 and every
    // chunk's CTA can be resident; else runs of chunks per CTA
    const bool reg = k <= kRegSlots && nch <= per_sm_reg * c.num_sms;
    const int max_ctas = per_sm * c.num_sms;
    int nctas = nch < 1 ? 1 : nch;
    int cpc = 1;
    if (!reg && nctas > max_ctas) {
        cpc = (nch + max_ctas - 1) / max_ctas;
        nctas = (nch + cpc - 1) / cpc;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nctas);
    cfg.blockDim = dim3(kChunk);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (reg && nctas <= kMaxClusterCtas) {
        // one cluster of all CTAs, if the device can place it
        // (placement answer cached per device, cluster size and shared-memory size class)
        static std::mutex mu;
        static std::map<std::tuple<int, int, size_t>, bool> fits;
        cudaLaunchAttribute cl[1];
        cl[0].id = cudaLaunchAttributeClusterDimension;
        cl[0].val.clusterDim.x = (unsigned)nctas;
        cl[0].val.clusterDim.y = 1;
        cl[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t ccfg = cfg;
        ccfg.attrs = cl;
        ccfg.numAttrs = 1;
        bool ok;
        {
            std::lock_guard<std::mutex> g(mu);
            const auto key = std::make_tuple(c.device, nctas, smem);
            auto it = fits.find(key);
            if (it == fits.end()) {
                if (nctas > 8 &&
                    cudaFuncSetAttribute(route_plan_reg_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                         1) != cudaSuccess)
                    (void)cudaGetLastError();
                int nclusters = 0;
                ok = cudaOccupancyMaxActiveClusters(&nclusters, route_plan_reg_kernel<true>, &ccfg) == cudaSuccess &&
                     nclusters >= 1;
                if (!ok)
                    (void)cudaGetLastError();
                fits.emplace(key, ok);
            } else {
                ok = it->second;
            }
        }
        if (ok)
            return cudaLaunchKernelEx(&ccfg, route_plan_reg_kernel<true>, topk, T, k, E, A, offsets, counts, dest,
                                      reinterpret_cast<uint32_t *>(hist), status, amax_zero);
    }
    if (reg)
        return cudaLaunchKernelEx(&cfg, route_plan_reg_kernel<false>, topk, T, k, E, A, offsets, counts, dest,
                                  reinterpret_cast<uint32_t *>(hist), status, amax_zero);
    return cudaLaunchKernelEx(&cfg, route_plan_kernel, topk, T, k, E, A, cpc, offsets, counts, dest,
                              reinterpret_cast<uint32_t *>(hist), status, amax_zero);
}

} // namespace epq
