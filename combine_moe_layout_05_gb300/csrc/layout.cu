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
// right counts but an arbitrary order, so the entries are split into
// contiguous chunks (one per block) and, inside a block, contiguous
// segments (one per warp); a slot is
//     offsets[e] + (entries of e in earlier chunks)
//                + (entries of e in earlier segments of this chunk)
//                + (entries of e earlier in this warp's segment),
// the last term counted 32 entries at a time with a warp match.
//
// Every block first copies its ids into shared memory with asynchronous
// copies, so it waits for memory once instead of once per loop trip.
//
// Small batches (T*K <= kSelfMaxEntries) take one launch: each block stages
// all T*K ids and counts the totals and the entries before its chunk itself.
// Larger batches take a workspace and, where the ranking blocks' plan fits
// (layout_ranked), two launches: this file's counting kernel in clusters of
// blocks, which sum their histograms through distributed shared memory,
// then the ranking blocks of the large-batch layout + dispatch grid alone
// (layout_dispatch_prefill.cu).  Otherwise (large batches with E near 1024)
// three: the counting kernel writes each chunk's histogram, a one-block
// kernel turns the histograms into each chunk's first slot per expert and
// writes the expert offsets, and the ranking kernel assigns the slots.  In
// no form does a block wait for another block of its own grid.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"
#include "layout_common.cuh"
#include "moe_layout.h"

namespace cg = cooperative_groups;

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
// Most threads of a counting-kernel block; launch_layout_count picks 256 or
// this many (its `threads`).
constexpr int kCountThreads = 512;
constexpr int kSelfMaxEntries = 4096;
constexpr int kSelfChunk = 256;
constexpr int kChunk = 1024;
constexpr int kScanCells = 16 * 1024;    // chunks x E staged by the scan (64 KB)
constexpr int kScanThreads = 1024;

// Multi-launch path, kernel 1: histogram and error bits of chunk c.
// ws_cnt is chunk-major: ws_cnt[c * E + e] (the clustered form writes
// prefixes within each cluster there instead, see below).  Each warp takes 32 entries at a
// time and matches equal ids, so one lane adds each distinct id's count (a
// hot expert costs one shared atomic per warp step, not one per entry); when
// K divides 32 the tokens' entries are whole lane groups and the same match
// shows a duplicated id within a token.
template <bool kCluster>
__global__ void __launch_bounds__(kCountThreads)
layout_count_kernel(const int32_t *__restrict__ ids, int T, int K, int E, int tpc,
                    int chunks, int32_t *__restrict__ ws_cnt,
                    uint32_t *__restrict__ ws_err, uint32_t *__restrict__ dev_error,
                    int32_t *__restrict__ dst_row_fill, int32_t *__restrict__ ws_ctot)
{
    extern __shared__ __align__(16) int32_t sm[];
    int32_t *hist = sm;                      // [E]
    int32_t *ids_s = hist + align4(E);       // [tpc * K], 16-byte aligned
    __shared__ uint32_t s_err;
    const int tid = threadIdx.x, lane = tid & 31, nthr = blockDim.x;
    const int c = blockIdx.x;
    const int t0 = min(T, c * tpc), t1 = min(T, t0 + tpc);
    const int m = (t1 - t0) * K;

    for (int e = tid; e < E; e += nthr) hist[e] = 0;
    if (tid == 0) s_err = 0;
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    // the error word starts at zero; the kernels after this one OR into it
    if (c == 0 && tid == 0 && dev_error) *dev_error = 0;
    // dst_row_fill: the chunk's slots start as kSlotPending, which the
    // kernel that ranks the chunk overwrites
    if (dst_row_fill)
        for (int i = tid; i < m; i += nthr) dst_row_fill[(size_t)t0 * K + i] = kSlotPending;
    stage_i32(ids_s, ids + (size_t)t0 * K, m);
    cp_async_wait_all();
    __syncthreads();

    const bool groups = (32 % K) == 0;
    const unsigned group = K >= 32 ? kFullMask : (((1u << K) - 1u) << (lane - lane % K));
    uint32_t err = 0;
    for (int b = tid - lane; b < m; b += nthr) {
        const int i = b + lane;
        const int id = i < m ? ids_s[i] : -1;
        const bool ok = (unsigned)id < (unsigned)E;
        const unsigned same = __match_any_sync(kFullMask, ok ? id : -1 - lane);
        if (ok && lane == __ffs(same) - 1) atomicAdd(hist + id, __popc(same));
        if (i < m && !ok) err |= MOE_DEV_ERR_EXPERT_RANGE;
        if (groups && ok && (same & group) != (1u << lane)) err |= MOE_DEV_ERR_DUPLICATE;
    }
    if (!groups) err |= token_errors(ids_s, t1 - t0, K, E);
    if (err) atomicOr(&s_err, err);
    if constexpr (!kCluster) {
        __syncthreads();
        for (int e = tid; e < E; e += nthr) ws_cnt[(size_t)c * E + e] = hist[e];
        if (tid == 0) ws_err[c] = s_err;
    } else {
        // Clustered form: block r of cluster g takes the expert slice
        // [r * es, (r + 1) * es) of the cluster's kCountCluster histograms,
        // read from the other blocks' shared memory.  Lane j of each group of
        // kCountCluster lanes holds chunk kCountCluster * g + j of one expert;
        // a scan across the group gives the chunk's prefix within the cluster,
        // and the group's last lane the cluster's total.
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();                      // every histogram of the cluster is complete
        if (tid == 0 && c < chunks) ws_err[c] = s_err;
        const int r = (int)cluster.block_rank(), g = c / kCountCluster;
        const int j = tid % kCountCluster;
        const int es = ceil_div(E, kCountCluster);
        const int e_lo = min(E, r * es), n = (min(E, e_lo + es) - e_lo) * kCountCluster;
        const int32_t *peer = cluster.map_shared_rank(hist, j);
        const int q = g * kCountCluster + j;
        const size_t ep = (size_t)align4(E);     // row stride: rows start 16-byte aligned
        // every read of the other blocks' histograms first (n <= 1024 <=
        // kPeerReads * nthr), then this block announces that it is done
        // with them, and waits for the others only before it leaves
        constexpr int kPeerReads = 4;
        int v[kPeerReads];
#pragma unroll
        for (int it = 0; it < kPeerReads; ++it) {
            const int i = it * nthr + tid;
            v[it] = i < n ? peer[e_lo + i / kCountCluster] : 0;
        }
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
#pragma unroll
        for (int it = 0; it < kPeerReads; ++it) {
            if (it * nthr >= n) break;           // whole warps take the shuffles
            const int i = it * nthr + tid;
            const int e = e_lo + i / kCountCluster;
            int x = v[it];
#pragma unroll
            for (int d = 1; d < kCountCluster; d <<= 1) {
                const int y = __shfl_up_sync(kFullMask, x, d, kCountCluster);
                if (j >= d) x += y;
            }
            if (i < n) {
                if (q < chunks) ws_cnt[q * ep + e] = x - v[it];
                if (j == kCountCluster - 1) ws_ctot[g * ep + e] = x;
            }
        }
        // no block leaves while another may still read its histogram
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    }
}

// Multi-launch path, kernel 2 (one block): turns the chunk histograms into
// each chunk's first slot per expert, in place:
//     ws_cnt[c * E + e] <- offsets[e] + sum of ws_cnt[c' * E + e], c' < c
// and writes the counts, offsets, rank offsets and the OR of the error bits.
// The histograms are staged in shared memory (one memory latency); P
// threads share each expert's chunks, and the threads of a warp hold
// consecutive experts, so shared-memory accesses never conflict.
__global__ void __launch_bounds__(kScanThreads)
layout_scan_kernel(int E, int R, int chunks, int32_t *__restrict__ ws_cnt,
                   const uint32_t *__restrict__ ws_err, int32_t *__restrict__ counts,
                   int32_t *__restrict__ offsets, int32_t *__restrict__ rank_offsets,
                   uint32_t *__restrict__ dev_error)
{
    extern __shared__ __align__(16) int32_t cnt[];   // [chunks][E]
    __shared__ int32_t part[kScanThreads];           // [P][E] partial sums, then prefixes
    __shared__ int32_t tot[MOE_MAX_EXPERTS];
    __shared__ int32_t off[MOE_MAX_EXPERTS + 1];
    __shared__ int32_t warp_sums[32];
    __shared__ uint32_t s_err;
    const int tid = threadIdx.x;
    const int P = E < kScanThreads ? kScanThreads / E : 1;
    const int e = tid % E, p = tid / E;
    const bool mine = p < P;
    const int per = ceil_div(chunks, P);
    const int c0 = min(chunks, p * per), c1 = min(chunks, c0 + per);
    if (tid == 0) s_err = 0;
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    stage_i32(cnt, ws_cnt, E * chunks);
    uint32_t err = 0;
    for (int c = tid; c < chunks; c += kScanThreads) err |= ws_err[c];
    if (err) atomicOr(&s_err, err);
    cp_async_wait_all();
    __syncthreads();

    int sum = 0;
    if (mine)
        for (int c = c0; c < c1; ++c) sum += cnt[c * E + e];
    if (mine) part[p * E + e] = sum;
    __syncthreads();
    if (tid < E) {
        int run = 0;
        for (int q = 0; q < P; ++q) {
            const int v = part[q * E + tid];
            part[q * E + tid] = run;
            run += v;
        }
        tot[tid] = run;
    }
    __syncthreads();
    scan_experts<kScanThreads>(tot, off, E, warp_sums);
    if (mine) {
        int run = off[e] + part[p * E + e];
        for (int c = c0; c < c1; ++c) {
            const int v = cnt[c * E + e];
            ws_cnt[(size_t)c * E + e] = run;
            run += v;
        }
    }
    for (int x = tid; x < E; x += kScanThreads) {
        counts[x] = tot[x];
        offsets[x] = off[x];
    }
    if (tid == 0) {
        offsets[E] = off[E];
        if (dev_error) *dev_error = s_err;
    }
    const int epr = E / R;
    for (int r = tid; r <= R; r += kScanThreads) rank_offsets[r] = off[r * epr];
}

// Ranking.  kSelf: one launch; every block stages all T*K ids, counts the
// totals and the entries before its chunk itself, and block 0 writes the
// counts, offsets, rank offsets and error word.  Otherwise the block's
// per-expert base comes from the scan kernel's offsets and prefixes.
template <bool kSelf>
__global__ void __launch_bounds__(kThreads)
layout_rank_kernel(const int32_t *__restrict__ ids, int T, int K, int E, int R,
                   int tpc, int chunks, const int32_t *__restrict__ ws_cnt,
                   int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                   int32_t *__restrict__ rank_offsets,
                   int32_t *__restrict__ src_token,
                   int32_t *__restrict__ dst_row, uint32_t *__restrict__ dev_error)
{
    extern __shared__ __align__(16) int32_t sm[];
    int32_t *rows = sm;                          // [kWarps][E] running slots
    int32_t *base = rows + kWarps * E;           // [E + 1]
    int32_t *total = base + E + 1;               // [E]      (kSelf)
    int32_t *before = total + E;                 // [E]      (kSelf)
    // all entries (kSelf) or the chunk's, 16-byte aligned for the staging copy
    int32_t *ids_s = sm + align4(kWarps * E + E + 1 + (kSelf ? 2 * E : 0));
    __shared__ int32_t warp_sums[32];
    __shared__ uint32_t s_err;

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int c = blockIdx.x;
    const int t0 = min(T, c * tpc), t1 = min(T, t0 + tpc);
    const int first = t0 * K, m = (t1 - t0) * K, n = T * K;

    for (int i = tid; i < kWarps * E; i += kThreads) rows[i] = 0;
    if (kSelf)
        for (int e = tid; e < E; e += kThreads) total[e] = before[e] = 0;
    if (tid == 0) s_err = 0;
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    if (kSelf) {
        stage_i32(ids_s, ids, n);
    } else {
        stage_i32(ids_s, ids + first, m);
        for (int e = tid; e < E; e += kThreads) base[e] = __ldg(ws_cnt + (size_t)c * E + e);
    }
    cp_async_wait_all();
    __syncthreads();
    const int32_t *mine = kSelf ? ids_s + first : ids_s;

    if (kSelf) {
        for (int i = tid; i < n; i += kThreads) {
            const int e = ids_s[i];
            if ((unsigned)e < (unsigned)E) {
                atomicAdd(total + e, 1);
                if (i < first) atomicAdd(before + e, 1);
            }
        }
        if (c == 0) {
            const uint32_t err = token_errors(ids_s, T, K, E);
            if (err) atomicOr(&s_err, err);
        }
    }
    int lo, hi;
    warp_segment<kWarps>(m, w, lo, hi);
    warp_count<kSelf>(mine, lo, hi, E, lane, rows + w * E);
    __syncthreads();

    if (kSelf) {
        scan_experts<kThreads>(total, base, E, warp_sums);
        if (c == 0) {
            for (int e = tid; e < E; e += kThreads) {
                counts[e] = total[e];
                offsets[e] = base[e];
            }
            if (tid == 0) {
                offsets[E] = base[E];
                if (dev_error) *dev_error = s_err;
            }
            const int epr = E / R;
            for (int r = tid; r <= R; r += kThreads) rank_offsets[r] = base[r * epr];
        }
    }
    for (int e = tid; e < E; e += kThreads) {
        int run = base[e] + (kSelf ? before[e] : 0);
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) {
            const int v = rows[ww * E + e];
            rows[ww * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    warp_rank<kSelf>(mine, lo, hi, E, K, first, lane, rows + w * E, dst_row, src_token);
}

size_t rank_smem_bytes(const LayoutPlan &p, int T, int K, int E)
{
    const size_t ids = p.single_launch ? (size_t)T * K : (size_t)p.tokens_per_chunk * K;
    const int extra = p.single_launch ? 2 * E : 0;
    return sizeof(int32_t) * ((size_t)align4(kWarps * E + E + 1 + extra) + ids);
}

}  // namespace

LayoutPlan plan_layout(int T, int K, int E)
{
    (void)E;
    const long long n = (long long)T * K;
    if (n <= kSelfMaxEntries) {
        const int tpc = kSelfChunk / K > 1 ? kSelfChunk / K : 1;
        const int chunks = T > 0 ? ceil_div(T, tpc) : 1;
        return {true, tpc, chunks};
    }
    // chunks of kChunk entries, fewer (larger) when the scan's staged
    // histograms (chunks x E ints) would not fit kScanCells
    int tpc = kChunk / K > 1 ? kChunk / K : 1;
    int chunks = ceil_div(T, tpc);
    const int max_chunks = kScanCells / E;
    if (chunks > max_chunks) {
        tpc = ceil_div(T, max_chunks);
        chunks = ceil_div(T, tpc);
    }
    return {false, tpc, chunks};
}

bool layout_supported(int T, int K, int E)
{
    // every kernel's dynamic shared memory must fit next to its static part
    constexpr size_t kLimit = 200 * 1024;
    const LayoutPlan p = plan_layout(T, K, E);
    if (rank_smem_bytes(p, T, K, E) > kLimit) return false;
    if (p.single_launch) return true;
    const size_t count = sizeof(int32_t) * ((size_t)align4(E) + (size_t)p.tokens_per_chunk * K);
    const size_t scan = sizeof(int32_t) * (size_t)E * p.chunks;
    return count <= kLimit && scan <= kLimit;
}

size_t layout_workspace_bytes(int T, int K, int E)
{
    const LayoutPlan plan = plan_layout(T, K, E);
    if (plan.single_launch) return 0;
    size_t bytes = workspace_layout(plan.chunks, E).bytes;
    const size_t ranked = ranked_workspace_bytes(T, K, E);
    if (ranked > bytes) bytes = ranked;
    return (bytes + 255) & ~(size_t)255;
}

WorkspaceLayout workspace_layout(int chunks, int E)
{
    WorkspaceLayout w;
    w.err = (size_t)chunks * E;
    w.bytes = sizeof(int32_t) * (w.err + (size_t)chunks);
    return w;
}

cudaError_t launch_layout_count(const int32_t *topk_ids, int T, int K, int E,
                                const LayoutPlan &p, int32_t *ws_cnt, uint32_t *ws_err,
                                uint32_t *dev_error, int32_t *dst_row_fill,
                                cudaStream_t stream, int threads, int32_t *ws_ctot)
{
    if (threads != 256 && threads != kCountThreads) return cudaErrorInvalidValue;
    const size_t csmem = sizeof(int32_t) * ((size_t)align4(E) + (size_t)p.tokens_per_chunk * K);
    if (ws_ctot) {
        const unsigned grid = (unsigned)(ceil_div(p.chunks, kCountCluster) * kCountCluster);
        cudaError_t e = allow_dynamic_smem((const void *)layout_count_kernel<true>, csmem);
        if (e != cudaSuccess) return e;
        return launch_pdl_clusters(layout_count_kernel<true>, dim3(grid), dim3(threads), csmem,
                                   stream, (unsigned)kCountCluster, topk_ids, T, K, E,
                                   p.tokens_per_chunk, p.chunks, ws_cnt, ws_err, dev_error,
                                   dst_row_fill, ws_ctot);
    }
    cudaError_t e = allow_dynamic_smem((const void *)layout_count_kernel<false>, csmem);
    if (e != cudaSuccess) return e;
    return launch_pdl(layout_count_kernel<false>, dim3(p.chunks), dim3(threads), csmem, stream,
                      topk_ids, T, K, E, p.tokens_per_chunk, p.chunks, ws_cnt, ws_err,
                      dev_error, dst_row_fill, (int32_t *)nullptr);
}

cudaError_t launch_layout(const int32_t *topk_ids, int T, int K, int E, int R,
                          int32_t *expert_counts, int32_t *expert_offsets,
                          int32_t *rank_offsets, int32_t *src_token,
                          int32_t *dst_row, uint32_t *dev_error,
                          void *workspace, cudaStream_t stream)
{
    const LayoutPlan p = plan_layout(T, K, E);
    const size_t rsmem = rank_smem_bytes(p, T, K, E);
    if (p.single_launch) {
        cudaError_t e = allow_dynamic_smem((const void *)layout_rank_kernel<true>, rsmem);
        if (e != cudaSuccess) return e;
        return launch_pdl(layout_rank_kernel<true>, dim3(p.chunks), dim3(kThreads), rsmem,
                          stream, topk_ids, T, K, E, R, p.tokens_per_chunk, p.chunks,
                          (const int32_t *)nullptr, expert_counts, expert_offsets,
                          rank_offsets, src_token, dst_row, dev_error);
    }
    if (layout_ranked(T, K, E))
        return launch_layout_ranked(topk_ids, T, K, E, R, expert_counts, expert_offsets,
                                    rank_offsets, src_token, dst_row, dev_error, workspace,
                                    stream);
    int32_t *ws_cnt = static_cast<int32_t *>(workspace);
    uint32_t *ws_err = reinterpret_cast<uint32_t *>(ws_cnt + (size_t)p.chunks * E);
    cudaError_t e = launch_layout_count(topk_ids, T, K, E, p, ws_cnt, ws_err, dev_error,
                                        nullptr, stream);
    if (e != cudaSuccess) return e;
    const size_t ssmem = sizeof(int32_t) * (size_t)E * p.chunks;
    e = allow_dynamic_smem((const void *)layout_scan_kernel, ssmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(layout_scan_kernel, dim3(1), dim3(kScanThreads), ssmem, stream, E, R,
                   p.chunks, ws_cnt, (const uint32_t *)ws_err, expert_counts,
                   expert_offsets, rank_offsets, dev_error);
    if (e != cudaSuccess) return e;
    e = allow_dynamic_smem((const void *)layout_rank_kernel<false>, rsmem);
    if (e != cudaSuccess) return e;
    return launch_pdl(layout_rank_kernel<false>, dim3(p.chunks), dim3(kThreads), rsmem,
                      stream, topk_ids, T, K, E, R, p.tokens_per_chunk, p.chunks,
                      (const int32_t *)ws_cnt, expert_counts, expert_offsets,
                      rank_offsets, src_token, dst_row, dev_error);
}

}  // namespace moe
