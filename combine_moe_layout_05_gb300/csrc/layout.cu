// layout.cu -- routing histogram, exclusive scan and stable slot map.
//
// Perplexity, "Enabling trillion-parameter models on AWS EFA", section
// "Dispatch and Combine": dispatch-send counts tokens per expert by
// accumulating in shared memory inside a block, then takes the cumulative
// sum of the counts to obtain the offsets at which tokens are packed into
// contiguous per-destination buffers.  Here the counts, offsets, per-rank
// offsets and the slot of every (token, k) entry are all produced on the GPU.
//
// Order inside an expert's range: token ascending, then k (a stable counting
// sort of the flat topk_ids array).  Shared-memory atomics alone give the
// right counts but an arbitrary order, so every warp owns a contiguous
// segment of the entries and keeps a private per-expert counter row:
//   1. each warp counts its segment (warp match + one add per distinct id);
//   2. per expert, the warp rows are scanned in warp order, the expert
//      totals are scanned across experts (warp-shuffle block scan), and each
//      warp's row becomes the first free slot of each expert for that warp;
//   3. each warp walks its segment again 32 entries at a time; an entry's
//      slot is its warp's counter plus the number of lower lanes holding the
//      same id, and the highest such lane advances the counter.
// Small batches (up to kFusedMaxEntries entries) run as one block.  Larger
// ones split the tokens into chunks: a counting kernel writes each chunk's
// histogram to the workspace, then the ranking kernel's block for chunk c
// adds the histograms of chunks before c to its per-expert bases.  No block
// ever waits for another block.
#include "common.cuh"
#include "internal.h"
#include "moe_layout.h"

#include <mutex>

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kFusedMaxEntries = 8192;
constexpr int kChunkEntries = 4096;
constexpr int kMaxChunks = 128;

// The warp's share [lo, hi) of a block's n entries: contiguous, 32-aligned.
__device__ __forceinline__ void warp_segment(int n, int w, int &lo, int &hi)
{
    const int seg = ((n + kWarps - 1) / kWarps + 31) & ~31;
    lo = min(n, w * seg);
    hi = min(n, lo + seg);
}

// Adds the ids in ids[lo, hi) to hist[id].  With kAtomic the row is shared
// by all warps of the block; without, it belongs to this warp alone.
template <bool kAtomic>
__device__ __forceinline__ uint32_t warp_count(const int32_t *__restrict__ ids,
                                               int lo, int hi, int E,
                                               int lane, int32_t *hist)
{
    uint32_t err = 0;
    for (int b = lo; b < hi; b += 32) {
        const int i = b + lane;
        const bool valid = i < hi;
        const int id = valid ? __ldg(ids + i) : 0;
        const bool ok = valid && (unsigned)id < (unsigned)E;
        if (valid && !ok) err |= MOE_DEV_ERR_EXPERT_RANGE;
        const unsigned m = __match_any_sync(kFullMask, ok ? id : -1 - lane);
        if (ok && lane == 31 - __clz(m)) {
            if (kAtomic) atomicAdd(hist + id, __popc(m));
            else hist[id] += __popc(m);
        }
    }
    return err;
}

// A token that lists one valid expert twice.
__device__ uint32_t check_duplicates(const int32_t *__restrict__ ids,
                                     int ntok, int K, int E)
{
    uint32_t err = 0;
    for (int t = threadIdx.x; t < ntok; t += blockDim.x) {
        const int32_t *row = ids + (size_t)t * K;
        for (int a = 0; a < K; ++a) {
            const int ea = __ldg(row + a);
            if ((unsigned)ea >= (unsigned)E) continue;
            for (int b = a + 1; b < K; ++b)
                if (__ldg(row + b) == ea) err |= MOE_DEV_ERR_DUPLICATE;
        }
    }
    return err;
}

// Exclusive prefix sum of one value per thread over the whole block (all
// kThreads threads must call).  `total` receives the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int32_t *warp_sums,
                                                    int &total)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(kFullMask, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = warp_sums[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(kFullMask, s, d);
            if (lane >= d) s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    total = warp_sums[kWarps - 1];
    return (w ? warp_sums[w - 1] : 0) + x - v;
}

// Multi-block path, pass 1: histogram of chunk blockIdx.x into the workspace.
__global__ void __launch_bounds__(kThreads)
layout_count_kernel(const int32_t *__restrict__ ids, int T, int K, int E,
                    int tpc, int32_t *__restrict__ ws_hist,
                    uint32_t *__restrict__ ws_err)
{
    extern __shared__ int32_t hist[];       // [E]
    __shared__ uint32_t s_err;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int c = blockIdx.x;
    const int t0 = min(T, c * tpc), t1 = min(T, t0 + tpc);
    const int first = t0 * K, n = (t1 - t0) * K;

    for (int e = tid; e < E; e += kThreads) hist[e] = 0;
    if (tid == 0) s_err = 0;
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    int lo, hi;
    warp_segment(n, w, lo, hi);
    uint32_t err = warp_count<true>(ids + first, lo, hi, E, lane, hist);
    err |= check_duplicates(ids + first, t1 - t0, K, E);
    if (err) atomicOr(&s_err, err);
    __syncthreads();

    for (int e = tid; e < E; e += kThreads) ws_hist[(size_t)c * E + e] = hist[e];
    if (tid == 0) ws_err[c] = s_err;
}

// Ranking pass.  kFused: one block covers all T tokens and also produces the
// counts and errors.  Otherwise block c covers chunk c and takes the counts
// of every chunk from the workspace; block 0 writes the shared outputs.
template <bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
layout_rank_kernel(const int32_t *__restrict__ ids, int T, int K, int E, int R,
                   int tpc, int chunks, const int32_t *__restrict__ ws_hist,
                   const uint32_t *__restrict__ ws_err,
                   int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                   int32_t *__restrict__ rank_offsets,
                   int32_t *__restrict__ src_token,
                   int32_t *__restrict__ dst_row, uint32_t *__restrict__ dev_error)
{
    extern __shared__ int32_t smem[];
    int32_t *hist = smem;                    // [kWarps][E]
    int32_t *ebase = hist + kWarps * E;      // [E + 1]
    int32_t *warp_sums = ebase + E + 1;      // [32]
    int32_t *part = warp_sums + 32;          // [2][kThreads], multi-block only
    __shared__ uint32_t s_err;

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int c = blockIdx.x;
    const int t0 = min(T, c * tpc), t1 = min(T, t0 + tpc);
    const int first = t0 * K, n = (t1 - t0) * K;

    for (int i = tid; i < kWarps * E; i += kThreads) hist[i] = 0;
    if (tid == 0) s_err = 0;
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    // 1. per-warp counts of this block's entries
    int lo, hi;
    warp_segment(n, w, lo, hi);
    uint32_t err = warp_count<false>(ids + first, lo, hi, E, lane, hist + w * E);
    if (kFused) {
        err |= check_duplicates(ids, T, K, E);
        if (err) atomicOr(&s_err, err);
    } else {
        // totals over all chunks and over the chunks before this one,
        // P threads per expert
        const int P = max(1, kThreads / E);
        const int e = tid % E, p = tid / E;
        int tot = 0, pre = 0;
        if (p < P)
            for (int cc = p; cc < chunks; cc += P) {
                const int v = __ldg(ws_hist + (size_t)cc * E + e);
                tot += v;
                if (cc < c) pre += v;
            }
        part[tid] = tot;
        part[kThreads + tid] = pre;
    }
    __syncthreads();

    // 2. scans: warps within the block, then experts across the block
    int cnt = 0, prefix = 0;
    if (tid < E) {
        int run = 0;
        for (int ww = 0; ww < kWarps; ++ww) {
            const int v = hist[ww * E + tid];
            hist[ww * E + tid] = run;
            run += v;
        }
        cnt = run;
        if (!kFused) {
            const int P = max(1, kThreads / E);
            int tot = 0, pre = 0;
            for (int p = 0; p < P; ++p) {
                tot += part[p * E + tid];
                pre += part[kThreads + p * E + tid];
            }
            cnt = tot;
            prefix = pre;
        }
    }
    int total;
    const int off = block_exclusive_scan(cnt, warp_sums, total);
    if (tid < E) {
        ebase[tid] = off;
        if (c == 0) {
            counts[tid] = cnt;
            offsets[tid] = off;
        }
        for (int ww = 0; ww < kWarps; ++ww) hist[ww * E + tid] += off + prefix;
    }
    if (tid == 0) {
        ebase[E] = total;
        if (c == 0) offsets[E] = total;
    }
    __syncthreads();
    if (c == 0) {
        const int epr = E / R;
        for (int r = tid; r <= R; r += kThreads) rank_offsets[r] = ebase[r * epr];
        if (tid == 0 && dev_error) {
            uint32_t e = s_err;
            if (!kFused)
                for (int cc = 0; cc < chunks; ++cc) e |= __ldg(ws_err + cc);
            *dev_error = e;
        }
    }

    // 3. slots, in entry order
    for (int b = lo; b < hi; b += 32) {
        const int i = b + lane;
        const bool valid = i < hi;
        const int id = valid ? __ldg(ids + first + i) : 0;
        const bool ok = valid && (unsigned)id < (unsigned)E;
        const unsigned m = __match_any_sync(kFullMask, ok ? id : -1 - lane);
        if (ok) {
            const int slot = hist[w * E + id] + __popc(m & ((1u << lane) - 1u));
            dst_row[first + i] = slot;
            src_token[slot] = (first + i) / K;
        } else if (valid) {
            dst_row[first + i] = -1;
        }
        __syncwarp();
        if (ok && lane == 31 - __clz(m)) hist[w * E + id] += __popc(m);
        __syncwarp();
    }
}

size_t rank_smem_bytes(int E, bool fused)
{
    return sizeof(int32_t) * ((size_t)kWarps * E + E + 1 + 32 + (fused ? 0 : 2 * kThreads));
}

// Raises a kernel's dynamic shared memory limit once per device.
cudaError_t allow_smem(const void *fn, size_t bytes)
{
    if (bytes <= 48 * 1024) return cudaSuccess;
    static std::mutex mu;
    static int done[2][64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int which = (fn == (const void *)layout_rank_kernel<true>) ? 0 : 1;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && done[which][dev]) return cudaSuccess;
    int max_optin = 0;
    e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    const size_t need = (size_t)sizeof(int32_t) * (kWarps * MOE_MAX_EXPERTS + MOE_MAX_EXPERTS + 1 + 32 + 2 * kThreads);
    const int set = (int)(need < (size_t)max_optin ? need : (size_t)max_optin);
    if ((size_t)set < bytes) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, set);
    if (e == cudaSuccess && dev < 64) done[which][dev] = 1;
    return e;
}

}  // namespace

LayoutPlan plan_layout(int T, int K, int E)
{
    (void)E;
    const long long n = (long long)T * K;
    if (n <= kFusedMaxEntries) return {true, T, 1};
    int tpc = kChunkEntries / K > 1 ? kChunkEntries / K : 1;
    int chunks = ceil_div(T, tpc);
    if (chunks > kMaxChunks) {
        tpc = ceil_div(T, kMaxChunks);
        chunks = ceil_div(T, tpc);
    }
    return {false, tpc, chunks};
}

size_t layout_workspace_bytes(const LayoutPlan &plan, int E)
{
    if (plan.fused) return 0;
    const size_t b = sizeof(int32_t) * (size_t)plan.chunks * ((size_t)E + 1);
    return (b + 255) & ~(size_t)255;
}

cudaError_t launch_layout(const int32_t *topk_ids, int T, int K, int E, int R,
                          int32_t *expert_counts, int32_t *expert_offsets,
                          int32_t *rank_offsets, int32_t *src_token,
                          int32_t *dst_row, uint32_t *dev_error,
                          void *workspace, cudaStream_t stream)
{
    const LayoutPlan plan = plan_layout(T, K, E);
    if (plan.fused) {
        const size_t smem = rank_smem_bytes(E, true);
        cudaError_t e = allow_smem((const void *)layout_rank_kernel<true>, smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(layout_rank_kernel<true>, dim3(1), dim3(kThreads), smem,
                          stream, topk_ids, T, K, E, R, T, 1,
                          (const int32_t *)nullptr, (const uint32_t *)nullptr,
                          expert_counts, expert_offsets, rank_offsets, src_token,
                          dst_row, dev_error);
    }
    int32_t *ws_hist = static_cast<int32_t *>(workspace);
    uint32_t *ws_err = reinterpret_cast<uint32_t *>(ws_hist + (size_t)plan.chunks * E);
    cudaError_t e = launch_pdl(layout_count_kernel, dim3(plan.chunks), dim3(kThreads),
                               sizeof(int32_t) * E, stream, topk_ids, T, K, E,
                               plan.tokens_per_chunk, ws_hist, ws_err);
    if (e != cudaSuccess) return e;
    const size_t smem = rank_smem_bytes(E, false);
    e = allow_smem((const void *)layout_rank_kernel<false>, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(layout_rank_kernel<false>, dim3(plan.chunks), dim3(kThreads),
                      smem, stream, topk_ids, T, K, E, R, plan.tokens_per_chunk,
                      plan.chunks, (const int32_t *)ws_hist, (const uint32_t *)ws_err,
                      expert_counts, expert_offsets, rank_offsets, src_token,
                      dst_row, dev_error);
}

}  // namespace moe
