// Route plan: expert-contiguous, alignment-padded placement of every
// (token, routing slot) -- the one-GPU stand-in for the expert-parallel
// dispatch of TE PR #3270 "EP dispatch with unfused MXFP8 quantization"
// (description: expert-major received rows returned as a per-expert grouped
// tensor; review thread: each expert slot aligned to a multiple of 128 rows).
//
// Two kernels, both over chunks of 512 tokens (one thread per token):
//  1. route_count: validate ids, build per-expert token bitmasks of the chunk
//     (each warp owns one 32-bit word of every expert's mask, filled with
//     __match_any_sync so no atomics are needed), write the chunk's
//     per-expert histogram and each slot's stable rank inside the chunk.
//  2. route_assign: every chunk sums the histograms of the chunks before it
//     (its base inside each expert) and of all chunks (the totals), scans
//     the aligned totals into expert offsets, and rewrites its slots' ranks
//     into global row indices.  Rows of an expert follow ascending token
//     order because chunks and ranks are both in token order.
#include "epq_device.cuh"
#include "epq_internal.h"

namespace epq {

constexpr int kChunk = 512;              // tokens per CTA
constexpr int kWords = kChunk / 32;      // mask words per expert
constexpr int kRankBits = 10;            // temp encoding: expert << 10 | rank

__global__ void __launch_bounds__(kChunk)
route_count_kernel(const int32_t *__restrict__ topk, int T, int k, int E,
                   int32_t *__restrict__ hist, int32_t *__restrict__ dest,
                   uint32_t *__restrict__ status)
{
    extern __shared__ uint32_t sm[];
    uint32_t *mask = sm;                       // [E][kWords]
    uint32_t *pre = sm + (size_t)E * kWords;   // [E][kWords]
    pdl_launch_dependents();
    pdl_wait();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int chunk = blockIdx.x;
    const int64_t t = (int64_t)chunk * kChunk + tid;
    for (int i = tid; i < E * kWords; i += kChunk)
        mask[i] = 0u;
    __syncthreads();

    uint32_t bad = 0;
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
        // lanes routed to the same expert in this slot: their bits of word
        // `warp` of that expert's mask; the lowest such lane writes them
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (peers & ((1u << lane) - 1u)) == 0u)
            mask[e * kWords + warp] |= peers;
    }
    if (bad)
        raise_status(status, bad);
    __syncthreads();

    // exclusive prefix over the chunk's words of every expert, and totals
    for (int e = warp; e < E; e += kChunk / 32) {
        const uint32_t c = (lane < kWords) ? __popc(mask[e * kWords + lane]) : 0u;
        uint32_t x = c;
#pragma unroll
        for (int o = 1; o < kWords; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        if (lane < kWords)
            pre[e * kWords + lane] = x - c;
        if (lane == kWords - 1)
            hist[(int64_t)chunk * E + e] = (int32_t)x;
    }
    __syncthreads();

    if (t < T) {
        for (int j = 0; j < k; ++j) {
            const int e = dest[t * k + j];
            if (e >= 0) {
                const uint32_t below = mask[e * kWords + warp] & ((1u << lane) - 1u);
                const int rank = (int)(pre[e * kWords + warp] + __popc(below));
                dest[t * k + j] = (e << kRankBits) | rank;
            }
        }
    }
}

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

__global__ void __launch_bounds__(kChunk)
route_assign_kernel(int T, int k, int E, int A, int nchunks, const int32_t *__restrict__ hist,
                    int32_t *__restrict__ offsets, int32_t *__restrict__ counts,
                    int32_t *__restrict__ dest)
{
    __shared__ int base[1024];
    __shared__ int off[1024];
    __shared__ int cnt[1024];
    __shared__ int wtmp[32];
    pdl_launch_dependents();
    pdl_wait();

    const int tid = threadIdx.x, chunk = blockIdx.x;
    for (int e = tid; e < E; e += kChunk) {
        int pre = 0, tot = 0;
        int c = 0;
        for (; c + 4 <= nchunks; c += 4) {
            const int h0 = hist[(int64_t)(c + 0) * E + e], h1 = hist[(int64_t)(c + 1) * E + e];
            const int h2 = hist[(int64_t)(c + 2) * E + e], h3 = hist[(int64_t)(c + 3) * E + e];
            pre += (c + 0 < chunk ? h0 : 0) + (c + 1 < chunk ? h1 : 0) + (c + 2 < chunk ? h2 : 0) +
                   (c + 3 < chunk ? h3 : 0);
            tot += h0 + h1 + h2 + h3;
        }
        for (; c < nchunks; ++c) {
            const int h = hist[(int64_t)c * E + e];
            pre += (c < chunk) ? h : 0;
            tot += h;
        }
        base[e] = pre;
        cnt[e] = tot;
        off[e] = (tot + A - 1) / A * A;
    }
    __syncthreads();
    const int total = block_exclusive_scan(off, E, wtmp);
    if (chunk == 0) {
        for (int e = tid; e < E; e += kChunk) {
            offsets[e] = off[e];
            counts[e] = cnt[e];
        }
        if (tid == 0)
            offsets[E] = total;
    }
    for (int e = tid; e < E; e += kChunk)
        base[e] += off[e];
    __syncthreads();

    const int64_t t = (int64_t)chunk * kChunk + tid;
    if (t < T) {
        for (int j = 0; j < k; ++j) {
            const int v = dest[t * k + j];
            if (v >= 0)
                dest[t * k + j] = base[v >> kRankBits] + (v & ((1 << kRankBits) - 1));
        }
    }
}

size_t route_workspace_bytes(int64_t T, int E)
{
    const int64_t nch = (T + kChunk - 1) / kChunk;
    const size_t b = (size_t)nch * (size_t)E * 4u;
    return b < 16 ? 16 : b;
}

cudaError_t launch_route_plan(const LaunchCtx &c, const int32_t *topk, int T, int k, int E, int A,
                              int32_t *offsets, int32_t *counts, int32_t *dest, int32_t *hist,
                              uint32_t *status)
{
    const int nch = (T + kChunk - 1) / kChunk;
    const size_t smem = (size_t)E * kWords * 4u * 2u;
    cudaError_t err;
    if (nch > 0) {
        // the largest request (E = 1024) is set once per device
        static int done[2] = {0, 0};
        err = ensure_smem_limit(route_count_kernel, c.device, 1024 * kWords * 4 * 2, done);
        if (err != cudaSuccess)
            return err;
        err = launch_pdl(route_count_kernel, dim3(nch), dim3(kChunk), smem, c.stream, topk, T, k, E,
                         hist, dest, status);
        if (err != cudaSuccess)
            return err;
    }
    return launch_pdl(route_assign_kernel, dim3(nch > 0 ? nch : 1), dim3(kChunk), 0, c.stream, T, k,
                      E, A, nch, (const int32_t *)hist, offsets, counts, dest);
}

} // namespace epq
