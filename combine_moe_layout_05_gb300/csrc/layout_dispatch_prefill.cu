// layout_dispatch_prefill.cu -- layout and dispatch of large batches in two
// launches: the chunk-counting kernel, then one grid that ranks every chunk
// and packs every token row, each row as soon as its chunk is ranked.
//
// Perplexity, "Enabling trillion-parameter models on AWS EFA", section
// "Dispatch and Combine": dispatch-send counts the tokens of every expert,
// takes the cumulative sum of the counts and packs the tokens into
// contiguous per-destination buffers.  For prefill batches the packing is an
// HBM-bound copy of hundreds of megabytes; what the layout adds is latency
// in front of it, which this path hides under the copy's own reads:
//
//  * layout_count_kernel (layout.cu), in clusters of kCountCluster blocks,
//    counts each chunk's experts and, through distributed shared memory,
//    writes each chunk's prefix within its cluster and each cluster's
//    totals to the workspace, with the chunks' error bits; it sets every
//    dst_row entry to kSlotPending and zeroes the error word;
//  * rank_dispatch_kernel: its first C blocks (C <= kMaxRankBlocks) each
//    rank one chunk of tokens.  A ranking block ranks its chunk's entries
//    (from the ids alone) before its wait for the counting kernel; then it
//    reads the clusters' totals and its chunk's prefix in one round of
//    copies, scans the totals into expert_offsets and writes the dst_row
//    and src_token entries of its chunk in the same stable order as
//    moe_layout.  No ranking block waits for another.
//    Every other block packs 256 consecutive 16-byte pieces of the flat
//    sequence of all token rows, like moe_dispatch: its first threads read
//    the K slots of each token it touches while all of them load their
//    pieces; a slot still kSlotPending is read again until its chunk's
//    ranking block has written it; then the pieces are (in the FP8 form
//    quantised and) stored.  So the token rows stream in while the chunks
//    are ranked, a packing block whose chunk is ranked pays one memory round
//    trip as in moe_dispatch, and no separate scan, ranking or dispatch
//    launch sits between the counts and the copy.
//
// The ranking blocks come first in the grid, so they are scheduled before
// any packing block that waits for them.  Each wait is bounded: past its
// deadline a packing block marks the chunk of the slot it waited for
// abandoned in the workspace (so the chunk's other blocks stop waiting at
// once) and sets MOE_DEV_ERR_TIMEOUT in the error word; the rows of the
// slots that could not be read stay unwritten.
#include "common.cuh"
#include "internal.h"
#include "layout_common.cuh"
#include "moe_layout.h"
#include "rowops.cuh"

namespace moe {
namespace {

constexpr uint32_t kAbandonedBit = 0x80000000u;  // ws_err[c]: a wait for chunk c expired
constexpr unsigned long long kWaitNs = 1000000000ull;   // 1 s
constexpr size_t kMaxRankSmem = 28 * 1024;       // keeps packing blocks at full occupancy
constexpr size_t kSmemPerSm = 228 * 1024;        // shared memory of one SM (sm_100 family)
constexpr int kSmPerBlockLimit = 32;             // resident blocks per SM
constexpr int kMaxRankBlocks = 128;              // ranking blocks (chunks) per grid
// moe_layout's ranking-only grid: measured 7.7 us at Qwen3 prefill sizes
// with 64 chunks against 10.2 with 128 (and 10.6 with 32); with packing
// blocks behind them 128 stays the fastest
constexpr int kMaxRankOnlyBlocks = 64;
constexpr size_t kMaxRankOnlySmem = 96 * 1024;   // ranking blocks of moe_layout alone

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Loads that observe other blocks' writes made during this kernel (device
// scope, no stale first-level cache line).
__device__ __forceinline__ int32_t ld_relaxed(const int32_t *p)
{
    int32_t v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Exclusive scan of hist[0..E) into off[0..E] (off[E] = total) by the whole
// block (any multiple of 32 threads up to 1024).  Ends with a barrier.
__device__ __forceinline__ void block_scan(const int32_t *hist, int32_t *off, int E,
                                           int32_t *warp_sums)
{
    const int n = blockDim.x, tid = threadIdx.x;
    const int per = (E + n - 1) / n;
    const int lane = tid & 31, w = tid >> 5, nw = n >> 5;
    int s = 0;
    for (int j = 0; j < per; ++j) {
        const int e = tid * per + j;
        s += e < E ? hist[e] : 0;
    }
    int x = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(kFullMask, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        int q = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(kFullMask, q, d);
            if (lane >= d) q += y;
        }
        if (lane < nw) warp_sums[lane] = q;
    }
    __syncthreads();
    int run = (w ? warp_sums[w - 1] : 0) + x - s;
    for (int j = 0; j < per; ++j) {
        const int e = tid * per + j;
        if (e < E) {
            off[e] = run;
            run += hist[e];
        }
    }
    if (tid == 0) off[E] = warp_sums[nw - 1];
    __syncthreads();
}


constexpr int kIdBits = 11;               // ids below 2^11 > MOE_MAX_EXPERTS
constexpr int kRankWarps = kRowThreads / 32;

// Stable rank of each valid entry of ids[lo, hi) among the equal ids of this
// warp's segment, 32 entries at a time (a warp match gives the lanes with
// the same id): ids[i] becomes (rank << kIdBits) | id, or -1 for an id
// outside [0, E); cnt[e] (this warp's row of counters) ends as the
// segment's count of e.
__device__ __forceinline__ void warp_local_rank(int32_t *ids, int lo, int hi, int E, int lane,
                                                int32_t *cnt)
{
    for (int b = lo; b < hi; b += 32) {
        const int i = b + lane;
        const bool valid = i < hi;
        const int id = valid ? ids[i] : -1;
        const bool ok = (unsigned)id < (unsigned)E;
        const unsigned m = match_ids<false>(id, ok, 0, lane);
        const int r = ok ? cnt[id] + __popc(m & ((1u << lane) - 1u)) : 0;
        __syncwarp();
        if (ok && lane == 31 - __clz(m)) cnt[id] = r + 1;
        if (valid) ids[i] = ok ? (r << kIdBits) | id : -1;
        __syncwarp();
    }
}

// Shared memory of a ranking block, in int32 elements: the clusters' totals
// [clusters][E] (row 0 becomes the expert totals), the chunk's prefix row
// [E], the offsets [E + 1], the per-warp counters [kRankWarps][E] and the
// chunk's ids.
__host__ __device__ inline size_t rank_smem_words(int chunks, int tpc, int K, int E)
{
    const int nc = (chunks + kCountCluster - 1) / kCountCluster;
    return (size_t)nc * align4(E) + align4(E) + align4(E + 1) + (size_t)kRankWarps * E +
           (size_t)tpc * K;
}

// Block c (< chunks) of rank_dispatch_kernel: ranks chunk c and publishes it.
//
//  0. Before the grid's wait (the ids are an input of the call, complete
//     when the grid starts) it stages the chunk's ids, ranks each entry
//     among the equal ids of its warp's segment and turns the per-warp
//     counts into per-warp starts.
//  1. After the wait (for the counting kernel, which ran in clusters of
//     kCountCluster chunks) it copies every cluster's totals and its chunk's
//     prefix within its own cluster to shared memory, in one round of
//     copies, and sums them into each expert's total and each expert's
//     entries in the chunks before this one.
//  2. It scans the totals into expert_offsets and writes every entry's slot,
//         offsets[e] + (entries of e in earlier chunks)
//                    + (warp's start for e) + rank in warp,
//     each entry on its own.  No ranking block waits for another.
__device__ __forceinline__ void rank_chunk(const int32_t *__restrict__ ids, int T, int K, int E,
                                        int R, int tpc, int chunks, int c,
                                        const int32_t *__restrict__ ws_pre,
                                        const uint32_t *__restrict__ ws_err,
                                        const int32_t *__restrict__ ws_ctot,
                                        int32_t *__restrict__ counts,
                                        int32_t *__restrict__ offsets,
                                        int32_t *__restrict__ rank_offsets,
                                        int32_t *__restrict__ src_token,
                                        int32_t *__restrict__ dst_row,
                                        uint32_t *__restrict__ dev_error, int stall_chunk)
{
    extern __shared__ __align__(16) int32_t sm[];
    constexpr int nthr = kRowThreads;
    const int nc = ceil_div(chunks, kCountCluster), cl = c / kCountCluster;
    const int ep = align4(E);                    // workspace rows start 16-byte aligned
    int32_t *tot = sm;                           // [nc][ep]: the clusters' totals; row 0 the sums
    int32_t *pre = tot + nc * ep;                // [ep]
    int32_t *base = pre + align4(E);             // [E + 1]
    int32_t *cnt = base + align4(E + 1);         // [kRankWarps][E], 16-byte aligned
    int32_t *ids_s = cnt + E * kRankWarps;       // [tpc * K], 16-byte aligned
    __shared__ int32_t warp_sums[32];
    __shared__ uint32_t s_err;

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int t0 = min(T, c * tpc), t1 = min(T, t0 + tpc);
    const int first = t0 * K, m = (t1 - t0) * K;
    for (int i = tid; i < E * kRankWarps / 4; i += nthr)
        reinterpret_cast<int4 *>(cnt)[i] = make_int4(0, 0, 0, 0);
    if (tid == 0) s_err = 0;
    // The chunk's ids are an input of the call, complete before this grid
    // started: the counting kernel's blocks let it start only after their own
    // wait for the kernel before the call.  So they are staged and ranked,
    // and the warps' starts computed, before this grid's wait, which is for
    // the counting kernel's histograms only.
    stage_i32(ids_s, ids + first, m);
    cp_async_wait_all();
    __syncthreads();
    const int seg = ((m + kRankWarps - 1) / kRankWarps + 31) & ~31;
    const int lo = min(m, w * seg), hi = min(m, lo + seg);
    warp_local_rank(ids_s, lo, hi, E, lane, cnt + w * E);
    __syncthreads();
    for (int e = tid; e < E; e += nthr) {
        int32_t v[kRankWarps];
#pragma unroll
        for (int ww = 0; ww < kRankWarps; ++ww) v[ww] = cnt[ww * E + e];
        int run = 0;
#pragma unroll
        for (int ww = 0; ww < kRankWarps; ++ww) {
            cnt[ww * E + e] = run;
            run += v[ww];
        }
    }
    pdl_wait();
    pdl_trigger();

    // 1. every cluster's totals and this chunk's prefix within its cluster
    //    (a cluster's first chunk has none) in one round of copies; then
    //    each expert's total, and its entries in the chunks before this one
    const bool own_pre = c % kCountCluster != 0;
    stage_i32(tot, ws_ctot, nc * ep);
    if (own_pre) stage_i32(pre, ws_pre + (size_t)c * ep, ep);
    if (c == 0) {
        uint32_t err = 0;
        for (int q = tid; q < chunks; q += nthr) err |= ld_relaxed(ws_err + q) & ~kAbandonedBit;
        if (err) atomicOr(&s_err, err);
    }
    cp_async_wait_all();
    __syncthreads();
    for (int e = tid; e < E; e += nthr) {
        int t = 0, b = own_pre ? pre[e] : 0;
        for (int k = 0; k < nc; ++k) {
            const int v = tot[k * ep + e];
            t += v;
            if (k < cl) b += v;
        }
        tot[e] = t;
        pre[e] = b;
    }
    __syncthreads();

    // 2. expert offsets, then every entry's slot (chunk 0 has no earlier
    //    entries)
    block_scan(tot, base, E, warp_sums);
    if (c == 0) {
        for (int e = tid; e < E; e += nthr) {
            counts[e] = tot[e];
            offsets[e] = base[e];
        }
        if (tid == 0) {
            offsets[E] = base[E];
            if (dev_error && s_err) atomicOr(dev_error, s_err);
        }
        const int epr = E / R;
        for (int r = tid; r <= R; r += nthr) rank_offsets[r] = base[r * epr];
    } else {
        for (int e = tid; e < E; e += nthr) base[e] += pre[e];
        __syncthreads();
    }
    if (c == stall_chunk) return;           // test hook: the chunk's slots stay pending
    for (int i = lo + lane; i < hi; i += 32) {
        const int v = ids_s[i];
        if (v >= 0) {
            const int id = v & ((1 << kIdBits) - 1);
            const int slot = base[id] + cnt[w * E + id] + (v >> kIdBits);
            dst_row[first + i] = slot;
            src_token[slot] = (first + i) / K;
        } else {
            dst_row[first + i] = -1;
        }
    }
}

// At 40 registers both forms keep 6 blocks of 256 threads (48 warps) per SM.
// The packing blocks stay within them without spilling because the FP8 form
// quantises after its slots are known (quantising before the wait kept the
// block's position and slots live across the division calls and spilled).
#ifndef MOE_RANK_DISPATCH_MIN_BLOCKS
#define MOE_RANK_DISPATCH_MIN_BLOCKS 6
#endif

// KT > 0: K known at compile time.  Blocks [0, chunks) rank; block
// chunks + q packs pieces [q * kRowThreads, (q + 1) * kRowThreads) of the
// flat sequence of all rows' pieces.
template <int KT, bool kFp8>
__global__ void __launch_bounds__(kRowThreads, MOE_RANK_DISPATCH_MIN_BLOCKS)
rank_dispatch_kernel(const int32_t *__restrict__ ids, const uint4 *__restrict__ tokens, int T,
                     int H, int K, int E, int R, int tpc, int chunks,
                     const int32_t *__restrict__ ws_pre, uint32_t *__restrict__ ws_err,
                     const int32_t *__restrict__ ws_ctot,
                     int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                     int32_t *__restrict__ rank_offsets, int32_t *__restrict__ src_token,
                     int32_t *__restrict__ dst_row, uint32_t *__restrict__ dev_error,
                     uint8_t *__restrict__ packed, float *__restrict__ scales,
                     unsigned long long wait_ns, int stall_chunk)
{
    const int k_count = KT > 0 ? KT : K;
    const int b = blockIdx.x;
    if (b < chunks) {
        rank_chunk(ids, T, k_count, E, R, tpc, chunks, b, ws_pre, ws_err, ws_ctot, counts,
                   offsets, rank_offsets, src_token, dst_row, dev_error, stall_chunk);
        return;
    }
    // packing block q covers kRowThreads consecutive pieces of the flat
    // sequence of all rows: tokens t_first .. t_first + n_tok - 1
    __shared__ int32_t s_slots[kRowThreads];
    const int tid = threadIdx.x;
    const int units = kFp8 ? (H >> 4) : (H >> 3);
    const unsigned q = (unsigned)(b - chunks);
    const RowPiece start = flat_block_start(q, units);
    const size_t vrow = (size_t)(H >> 3);
    pdl_wait();
    pdl_trigger();

    // the row piece and the block's slots are requested together; the
    // piece arrives while the chunk is being ranked
    uint4 a = make_uint4(0, 0, 0, 0), bv = make_uint4(0, 0, 0, 0);
    bool active, has_slot;
    {
        const int dt = (start.u + tid) / units, u = start.u + tid - dt * units;
        active = start.t + dt < T;
        if (active) {
            const uint4 *row = tokens + (size_t)(start.t + dt) * vrow;
            if (kFp8) {
                a = ld_stream_v4(row + 2 * u);
                bv = ld_stream_v4(row + 2 * u + 1);
            } else {
                a = ld_stream_v4(row + u);
            }
        }
        // the K slots of each token the block touches, contiguous in dst_row
        const int n_slots = min(T - start.t, (start.u + kRowThreads - 1) / units + 1) * k_count;
        has_slot = tid < n_slots;
        if (has_slot) s_slots[tid] = ld_relaxed(dst_row + (size_t)start.t * k_count + tid);
    }
    // a slot still pending is read again until its chunk's ranking block has
    // written it (bounded; an expired wait abandons the chunk and the slot's
    // row is not written)
    if (has_slot && s_slots[tid] == kSlotPending) {
        const int t_first = flat_block_start(q, units).t;
        const int32_t *my_slot = dst_row + (size_t)t_first * k_count + tid;
        uint32_t *chunk_err = ws_err + (t_first + tid / k_count) / tpc;
        const unsigned long long deadline = global_ns() + wait_ns;
        unsigned sleep = 16;
        int32_t slot;
        while (true) {
            __nanosleep(sleep);
            sleep = sleep < 128 ? 2 * sleep : 128;
            slot = ld_relaxed(my_slot);
            if (slot != kSlotPending) break;
            if ((ld_relaxed(chunk_err) & kAbandonedBit) || global_ns() > deadline) {
                atomicOr(chunk_err, kAbandonedBit);
                if (dev_error) atomicOr(dev_error, MOE_DEV_ERR_TIMEOUT);
                slot = -1;
                break;
            }
        }
        s_slots[tid] = slot;
    }
    __syncthreads();
    Fp8Piece p;
    if (kFp8) p = quantize16(a, bv);     // every lane takes part (shuffles)
    if (!active) return;
    const int rows = T * k_count;
    const RowPiece rp = flat_piece(q, units, tid);
    const int32_t *slots = s_slots + (rp.t - flat_block_start(q, units).t) * k_count;
    if (kFp8)
        store_fp8_to_slots<KT>(slots, k_count, rows, packed, scales, H, rp.u, p);
    else
        store_to_slots<KT>(slots, k_count, rows, packed, vrow * 16, (size_t)rp.u * 16, a);
}

// The ranking blocks' plan: the layout's chunks, made larger where there
// would be more than max_chunks (fewer chunks also need less workspace than
// the layout's plan), and larger again, a cluster at a time, until the
// ranking blocks' shared memory fits smem_limit (the clusters' totals
// shrink with fewer chunks while each chunk's ids grow).
struct RankPlan {
    bool ok;
    LayoutPlan lp;
    size_t smem;
};

RankPlan plan_rank(int T, int K, int E, int max_chunks, size_t smem_limit)
{
    RankPlan rp{};
    rp.lp = plan_layout(T, K, E);
    if (T <= 0 || rp.lp.single_launch) return rp;
    int tpc = rp.lp.tokens_per_chunk, chunks = rp.lp.chunks;
    if (chunks > max_chunks) {
        tpc = ceil_div(T, max_chunks);
        chunks = ceil_div(T, tpc);
    }
    while (true) {
        const size_t smem = sizeof(int32_t) * rank_smem_words(chunks, tpc, K, E);
        if (smem <= smem_limit) {
            rp.ok = true;
            rp.lp.tokens_per_chunk = tpc;
            rp.lp.chunks = chunks;
            rp.smem = smem;
            return rp;
        }
        if (chunks <= kCountCluster) return rp;
        tpc = ceil_div(T, chunks - kCountCluster);
        chunks = ceil_div(T, tpc);
    }
}

// Where the ranking blocks' form keeps its state in the workspace, in int32
// elements from its start, rows of align4(E) elements (16-byte aligned):
// ws_pre[chunks][E] (each chunk's prefix within its cluster),
// ws_ctot[clusters][E] (each cluster's totals), then ws_err[chunks].
struct RankedWorkspaceLayout {
    size_t ctot, err;
    size_t bytes;
};

RankedWorkspaceLayout ranked_workspace_layout(int chunks, int E)
{
    RankedWorkspaceLayout w;
    w.ctot = (size_t)chunks * align4(E);
    w.err = w.ctot + (size_t)ceil_div(chunks, kCountCluster) * align4(E);
    w.bytes = sizeof(int32_t) * (w.err + (size_t)chunks);
    return w;
}

struct PrefillPlan {
    bool use;
    LayoutPlan lp;          // this path's chunks (at most kMaxRankBlocks)
    long long pack_blocks;
    size_t smem;
};

PrefillPlan plan_prefill(int T, int H, int K, int E, bool fp8)
{
    PrefillPlan pp{};
    const RankPlan rp = plan_rank(T, K, E, kMaxRankBlocks, kMaxRankSmem);
    pp.lp = rp.lp;
    pp.smem = rp.smem;
    if (!rp.ok) return pp;
    const int units = fp8 ? H / 16 : H / 8;
    pp.pack_blocks = ((long long)T * units + kRowThreads - 1) / kRowThreads;
    // a packing block's tokens' slots, one per thread at most
    const long long max_slots = (long long)((units - 1 + kRowThreads - 1) / units + 1) * K;
    const long long grid = (long long)pp.lp.chunks + pp.pack_blocks;
    // every block carries the ranking blocks' shared memory: take this path
    // only while the packing blocks still fill at least 3/4 of an SM
    const long long per_sm = min((long long)kSmPerBlockLimit, (long long)(kSmemPerSm / (pp.smem + 1024)));
    pp.use = units < kMaxRowPieces && max_slots <= kRowThreads && pp.smem <= kMaxRankSmem &&
             per_sm * kRowThreads >= 1536 && grid <= 0x7fffffffll;
    return pp;
}

struct PrefillWorkspace {
    int32_t *pre;
    uint32_t *err;
    int32_t *ctot;
};

PrefillWorkspace prefill_workspace(void *workspace, int chunks, int E)
{
    const RankedWorkspaceLayout wl = ranked_workspace_layout(chunks, E);
    int32_t *base = static_cast<int32_t *>(workspace);
    return {base, reinterpret_cast<uint32_t *>(base + wl.err), base + wl.ctot};
}

template <int KT, bool kFp8>
cudaError_t run_prefill(const PrefillPlan &pp, const int32_t *ids, const void *tokens, int T,
                        int H, int K, int E, int R, const PrefillWorkspace &ws,
                        int32_t *counts, int32_t *offsets, int32_t *rank_offsets,
                        int32_t *src_token, int32_t *dst_row, uint32_t *dev_error,
                        void *packed, float *scales, unsigned long long wait_ns,
                        int stall_chunk, cudaStream_t s)
{
    auto *fn = rank_dispatch_kernel<KT, kFp8>;
    cudaError_t e = allow_dynamic_smem((const void *)fn, pp.smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(pp.lp.chunks + pp.pack_blocks);   // no packing blocks: layout only
    return launch_pdl(fn, dim3(grid), dim3(kRowThreads), pp.smem, s, ids,
                      static_cast<const uint4 *>(tokens), T, H, K, E, R,
                      pp.lp.tokens_per_chunk, pp.lp.chunks, (const int32_t *)ws.pre, ws.err,
                      (const int32_t *)ws.ctot, counts, offsets, rank_offsets, src_token,
                      dst_row, dev_error,
                      static_cast<uint8_t *>(packed), scales, wait_ns, stall_chunk);
}

template <bool kFp8>
cudaError_t run_prefill_k(const PrefillPlan &pp, const int32_t *ids, const void *tokens, int T,
                          int H, int K, int E, int R, const PrefillWorkspace &ws,
                          int32_t *counts, int32_t *offsets, int32_t *rank_offsets,
                          int32_t *src_token, int32_t *dst_row, uint32_t *dev_error,
                          void *packed, float *scales, unsigned long long wait_ns,
                          int stall_chunk, cudaStream_t s)
{
#define MOE_PREFILL_CASE(KV)                                                                   \
    return run_prefill<KV, kFp8>(pp, ids, tokens, T, H, K, E, R, ws, counts, offsets,          \
                                 rank_offsets, src_token, dst_row, dev_error, packed, scales,  \
                                 wait_ns, stall_chunk, s)
    switch (K) {
    case 1: MOE_PREFILL_CASE(1);
    case 2: MOE_PREFILL_CASE(2);
    case 4: MOE_PREFILL_CASE(4);
    case 6: MOE_PREFILL_CASE(6);
    case 8: MOE_PREFILL_CASE(8);
    default: MOE_PREFILL_CASE(0);
    }
#undef MOE_PREFILL_CASE
}

}  // namespace

bool layout_dispatch_prefill(int T, int H, int K, int E, int fp8)
{
    return plan_prefill(T, H, K, E, fp8 != 0).use;
}

bool layout_ranked(int T, int K, int E)
{
    return plan_rank(T, K, E, kMaxRankOnlyBlocks, kMaxRankOnlySmem).ok;
}

size_t ranked_workspace_bytes(int T, int K, int E)
{
    // both forms' chunks: moe_layout's ranking-only grid and
    // moe_layout_dispatch's rank-and-pack grid
    size_t bytes = 0;
    for (const RankPlan &rp : {plan_rank(T, K, E, kMaxRankOnlyBlocks, kMaxRankOnlySmem),
                               plan_rank(T, K, E, kMaxRankBlocks, kMaxRankSmem)}) {
        if (rp.ok) {
            const size_t b = ranked_workspace_layout(rp.lp.chunks, E).bytes;
            if (b > bytes) bytes = b;
        }
    }
    return bytes;
}

cudaError_t launch_layout_ranked(const int32_t *topk_ids, int T, int K, int E, int R,
                                 int32_t *expert_counts, int32_t *expert_offsets,
                                 int32_t *rank_offsets, int32_t *src_token, int32_t *dst_row,
                                 uint32_t *dev_error, void *workspace, cudaStream_t stream)
{
    const RankPlan rp = plan_rank(T, K, E, kMaxRankOnlyBlocks, kMaxRankOnlySmem);
    if (!rp.ok) return cudaErrorInvalidValue;
    PrefillPlan pp{};
    pp.use = true;
    pp.lp = rp.lp;
    pp.smem = rp.smem;
    pp.pack_blocks = 0;                 // the grid is the ranking blocks alone
    const PrefillWorkspace ws = prefill_workspace(workspace, pp.lp.chunks, E);
    // no packing blocks poll dst_row, so it needs no pending marks
    cudaError_t e = launch_layout_count(topk_ids, T, K, E, pp.lp, ws.pre, ws.err, dev_error,
                                        nullptr, stream, 256, ws.ctot);
    if (e != cudaSuccess) return e;
    return run_prefill_k<false>(pp, topk_ids, nullptr, T, 8, K, E, R, ws, expert_counts,
                                expert_offsets, rank_offsets, src_token, dst_row, dev_error,
                                nullptr, nullptr, kWaitNs, -1, stream);
}

cudaError_t launch_layout_dispatch_prefill(const int32_t *topk_ids, const void *tokens, int T,
                                           int H, int K, int E, int R, int fp8,
                                           int32_t *expert_counts, int32_t *expert_offsets,
                                           int32_t *rank_offsets, int32_t *src_token,
                                           int32_t *dst_row, uint32_t *dev_error, void *packed,
                                           float *scales, void *workspace,
                                           unsigned long long wait_ns, int stall_chunk,
                                           cudaStream_t stream)
{
    const PrefillPlan pp = plan_prefill(T, H, K, E, fp8 != 0);
    if (!pp.use) return cudaErrorInvalidValue;
    const PrefillWorkspace ws = prefill_workspace(workspace, pp.lp.chunks, E);
    cudaError_t e = launch_layout_count(topk_ids, T, K, E, pp.lp, ws.pre, ws.err, dev_error,
                                        dst_row, stream, 512, ws.ctot);
    if (e != cudaSuccess) return e;
    if (wait_ns == 0) wait_ns = kWaitNs;
    if (fp8)
        return run_prefill_k<true>(pp, topk_ids, tokens, T, H, K, E, R, ws, expert_counts,
                                   expert_offsets, rank_offsets, src_token, dst_row, dev_error,
                                   packed, scales, wait_ns, stall_chunk, stream);
    return run_prefill_k<false>(pp, topk_ids, tokens, T, H, K, E, R, ws, expert_counts,
                                expert_offsets, rank_offsets, src_token, dst_row, dev_error,
                                packed, scales, wait_ns, stall_chunk, stream);
}

}  // namespace moe

// Test hook, deliberately absent from the public header: the large-batch
// path of moe_layout_dispatch with a chosen bound on every wait for a
// ranked chunk and
//  * stall_chunk >= 0: that chunk never ranked (its ranking block stops
//    before writing the slots, which stay pending).  The chunk's packing
//    blocks' waits expire: they set MOE_DEV_ERR_TIMEOUT and skip its rows;
//    every other row is packed;
//  * stall_chunk == -1: the normal call.
// Tests use it to see the bounded waits expire with the context still
// usable.  Arguments are checked by the caller (tests only).
extern "C" __attribute__((visibility("default"))) int32_t
moe_testing_layout_dispatch_prefill(const int32_t *topk_ids, const void *tokens, int32_t T,
                                    int32_t H, int32_t K, int32_t E, int32_t R, int32_t fp8,
                                    int32_t *expert_counts, int32_t *expert_offsets,
                                    int32_t *rank_offsets, int32_t *src_token, int32_t *dst_row,
                                    uint32_t *dev_error, void *packed, float *scales,
                                    void *workspace, uint64_t wait_ns, int32_t stall_chunk,
                                    cudaStream_t stream)
{
    if (!moe::layout_dispatch_prefill(T, H, K, E, fp8)) return MOE_ERR_INVALID_ARG;
    const cudaError_t e = moe::launch_layout_dispatch_prefill(
        topk_ids, tokens, T, H, K, E, R, fp8, expert_counts, expert_offsets, rank_offsets,
        src_token, dst_row, dev_error, packed, scales, workspace, wait_ns, stall_chunk, stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
