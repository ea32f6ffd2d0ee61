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
//  * layout_count_kernel (layout.cu) writes each chunk's histogram and error
//    bits to the workspace, sets every dst_row entry to kSlotPending and
//    zeroes the error word;
//  * rank_dispatch_kernel: its first C blocks each rank one chunk of tokens.
//    Block c sums the chunk histograms column by column (the per-expert
//    totals, whose exclusive scan is expert_offsets, and the entries of each
//    expert in chunks before c), ranks its chunk's entries in the same stable
//    order as moe_layout (per-warp counters, warp match) and writes dst_row
//    and src_token.  Every other block packs one slice of one token row, like
//    moe_dispatch: its first threads read the token's K slots while all of
//    them load their 16-byte pieces (and in the FP8 form quantise them); a
//    slot still kSlotPending is read again until its chunk's ranking block
//    has written it; then the pieces are stored.  So the token rows stream in
//    while the chunks are ranked, a packing block whose chunk is ranked pays
//    one memory round trip as in moe_dispatch, and no separate scan, ranking
//    or dispatch launch sits between the counts and the copy.
//
// The ranking blocks come first in the grid, so they are scheduled before
// any packing block that waits for them.  Each wait is bounded: past its
// deadline the block marks the chunk abandoned in the workspace (so the
// chunk's other blocks stop waiting at once), sets MOE_DEV_ERR_TIMEOUT in the
// error word and returns without storing.
#include "common.cuh"
#include "internal.h"
#include "layout_common.cuh"
#include "moe_layout.h"
#include "rowops.cuh"

namespace moe {
namespace {

constexpr uint32_t kAbandonedBit = 0x80000000u;  // ws_err[c]: a wait for chunk c expired
constexpr unsigned long long kWaitNs = 1000000000ull;   // 1 s
constexpr size_t kMaxRankSmem = 24 * 1024;       // keeps packing blocks at full occupancy
constexpr size_t kSmemPerSm = 228 * 1024;        // shared memory of one SM (sm_100 family)
constexpr int kSmPerBlockLimit = 32;             // resident blocks per SM

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

// Block c (< chunks) of rank_dispatch_kernel: ranks chunk c and publishes it.
__device__ __forceinline__ void rank_chunk(const int32_t *__restrict__ ids, int T, int K, int E,
                                           int R, int tpc, int chunks, int c,
                                           const int32_t *__restrict__ ws_cnt,
                                           uint32_t *__restrict__ ws_err,
                                           int32_t *__restrict__ counts,
                                           int32_t *__restrict__ offsets,
                                           int32_t *__restrict__ rank_offsets,
                                           int32_t *__restrict__ src_token,
                                           int32_t *__restrict__ dst_row,
                                           uint32_t *__restrict__ dev_error, int stall_chunk)
{
    extern __shared__ __align__(16) int32_t sm[];
    const int nthr = blockDim.x, nw = nthr >> 5;
    int32_t *tot = sm;                          // [E]
    int32_t *pre = tot + align4(E);             // [E]
    int32_t *base = pre + align4(E);            // [E + 1]
    int32_t *rows = base + align4(E + 1);       // [nw][E]
    int32_t *ids_s = rows + align4(nw * E);     // [tpc * K], 16-byte aligned
    __shared__ int32_t warp_sums[32];
    __shared__ uint32_t s_err;

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int t0 = min(T, c * tpc), t1 = min(T, t0 + tpc);
    const int first = t0 * K, m = (t1 - t0) * K;
    for (int e = tid; e < E; e += nthr) {
        tot[e] = 0;
        pre[e] = 0;
    }
    for (int i = tid; i < nw * E; i += nthr) rows[i] = 0;
    if (tid == 0) s_err = 0;
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    stage_i32(ids_s, ids + first, m);

    // per-expert totals and entries in earlier chunks: column sums of the
    // chunk histograms, four experts per 16-byte load where rows allow
    if ((E & 3) == 0) {
        const int E4 = E >> 2;
        const int G = nthr >= E4 ? nthr / E4 : 1;
        for (int idx = tid; idx < G * E4; idx += nthr) {
            const int e4 = idx % E4, g = idx / E4;
            int4 tt = make_int4(0, 0, 0, 0), pp = make_int4(0, 0, 0, 0);
#pragma unroll 16
            for (int q = g; q < chunks; q += G) {
                const int4 v = __ldg(reinterpret_cast<const int4 *>(ws_cnt + (size_t)q * E) + e4);
                tt.x += v.x;
                tt.y += v.y;
                tt.z += v.z;
                tt.w += v.w;
                if (q < c) {
                    pp.x += v.x;
                    pp.y += v.y;
                    pp.z += v.z;
                    pp.w += v.w;
                }
            }
            atomicAdd(tot + 4 * e4, tt.x);
            atomicAdd(tot + 4 * e4 + 1, tt.y);
            atomicAdd(tot + 4 * e4 + 2, tt.z);
            atomicAdd(tot + 4 * e4 + 3, tt.w);
            atomicAdd(pre + 4 * e4, pp.x);
            atomicAdd(pre + 4 * e4 + 1, pp.y);
            atomicAdd(pre + 4 * e4 + 2, pp.z);
            atomicAdd(pre + 4 * e4 + 3, pp.w);
        }
    } else {
        const int G = nthr >= E ? nthr / E : 1;
        for (int idx = tid; idx < G * E; idx += nthr) {
            const int e = idx % E, g = idx / E;
            int tt = 0, pp = 0;
#pragma unroll 8
            for (int q = g; q < chunks; q += G) {
                const int v = __ldg(ws_cnt + (size_t)q * E + e);
                tt += v;
                pp += q < c ? v : 0;
            }
            atomicAdd(tot + e, tt);
            atomicAdd(pre + e, pp);
        }
    }
    if (c == 0) {
        uint32_t err = 0;
        for (int q = tid; q < chunks; q += nthr) err |= ld_relaxed(ws_err + q) & ~kAbandonedBit;
        if (err) atomicOr(&s_err, err);
    }
    cp_async_wait_all();
    __syncthreads();
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
    }

    // stable ranking of the chunk: warp w owns a contiguous segment
    const int seg = ((m + nw - 1) / nw + 31) & ~31;
    const int lo = min(m, w * seg), hi = min(m, lo + seg);
    warp_count<false>(ids_s, lo, hi, E, lane, rows + w * E);
    __syncthreads();
    for (int e = tid; e < E; e += nthr) {
        int run = base[e] + pre[e];
        for (int ww = 0; ww < nw; ++ww) {
            const int v = rows[ww * E + e];
            rows[ww * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    if (c == stall_chunk) return;           // test hook: the chunk's slots stay pending
    warp_rank<false>(ids_s, lo, hi, E, K, first, lane, rows + w * E, dst_row, src_token);
}

// The FP8 form at 40 registers keeps 6 blocks of 256 threads per SM (46
// registers, 5 blocks, without the bound): 56.5 against 57.0 us at the
// Kimi-K2 prefill shape, no spills, unchanged at the Qwen3 shape.
#ifndef MOE_RANK_DISPATCH_FP8_MIN_BLOCKS
#define MOE_RANK_DISPATCH_FP8_MIN_BLOCKS 6
#endif

// KT > 0: K known at compile time.  Blocks [0, chunks) rank; block
// chunks + t * slices + s packs slice s of token t.
template <int KT, bool kFp8>
__global__ void __launch_bounds__(256, kFp8 ? MOE_RANK_DISPATCH_FP8_MIN_BLOCKS : 1)
rank_dispatch_kernel(const int32_t *__restrict__ ids, const uint4 *__restrict__ tokens, int T,
                     int H, int K, int E, int R, int tpc, int chunks, int slices,
                     const int32_t *__restrict__ ws_cnt, uint32_t *__restrict__ ws_err,
                     int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                     int32_t *__restrict__ rank_offsets, int32_t *__restrict__ src_token,
                     int32_t *__restrict__ dst_row, uint32_t *__restrict__ dev_error,
                     uint8_t *__restrict__ packed, float *__restrict__ scales,
                     unsigned long long wait_ns, int stall_chunk)
{
    const int k_count = KT > 0 ? KT : K;
    const int b = blockIdx.x;
    if (b < chunks) {
        rank_chunk(ids, T, k_count, E, R, tpc, chunks, b, ws_cnt, ws_err, counts, offsets,
                   rank_offsets, src_token, dst_row, dev_error, stall_chunk);
        return;
    }
    __shared__ int32_t s_slots[MOE_MAX_TOPK];
    const int q = b - chunks;
    const int t = q / slices, sl = q - (q / slices) * slices;
    const int tid = threadIdx.x;
    const int units = kFp8 ? (H >> 4) : (H >> 3);
    const int u = sl * blockDim.x + tid;
    const bool active = u < units;
    const size_t vrow = (size_t)(H >> 3);
    pdl_wait();
    pdl_trigger();

    // the row piece and the token's K slots are requested together; the
    // piece arrives while the chunk is being ranked
    uint4 a = make_uint4(0, 0, 0, 0), bv = make_uint4(0, 0, 0, 0);
    if (active) {
        if (kFp8) {
            a = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u);
            bv = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u + 1);
        } else {
            a = ld_stream_v4(tokens + (size_t)t * vrow + u);
        }
    }
    const int32_t *my_slot = dst_row + (size_t)t * k_count + tid;
    int32_t slot = tid < k_count ? ld_relaxed(my_slot) : 0;
    Fp8Piece p;
    if (kFp8) p = quantize16(a, bv);     // every lane takes part (shuffles)

    // a slot still pending is read again until its chunk's ranking block has
    // written it (bounded; an expired wait abandons the chunk)
    int ok = 1;
    if (tid < k_count && slot == kSlotPending) {
        uint32_t *chunk_err = ws_err + t / tpc;
        const unsigned long long deadline = global_ns() + wait_ns;
        unsigned sleep = 16;
        while (true) {
            __nanosleep(sleep);
            sleep = sleep < 128 ? 2 * sleep : 128;
            slot = ld_relaxed(my_slot);
            if (slot != kSlotPending) break;
            if ((ld_relaxed(chunk_err) & kAbandonedBit) || global_ns() > deadline) {
                atomicOr(chunk_err, kAbandonedBit);
                if (dev_error) atomicOr(dev_error, MOE_DEV_ERR_TIMEOUT);
                ok = 0;
                break;
            }
        }
    }
    if (tid < k_count) s_slots[tid] = slot;
    if (!__syncthreads_and(ok) || !active) return;
    const int rows = T * k_count;
    if (kFp8)
        store_fp8_to_slots<KT>(s_slots, k_count, rows, packed, scales, H, u, p);
    else
        store_to_slots<KT>(s_slots, k_count, rows, packed, vrow * 16, (size_t)u * 16, a);
}

struct PrefillPlan {
    bool use;
    LayoutPlan lp;
    int threads;
    int slices;
    size_t smem;
};

PrefillPlan plan_prefill(int T, int H, int K, int E, bool fp8)
{
    PrefillPlan pp{};
    pp.lp = plan_layout(T, K, E);
    if (T <= 0 || pp.lp.single_launch) return pp;
    const int units = fp8 ? H / 16 : H / 8;
    pp.threads = pick_row_block(units);
    pp.slices = ceil_div(units, pp.threads);
    const int nw = pp.threads / 32;
    pp.smem = sizeof(int32_t) * ((size_t)2 * align4(E) + align4(E + 1) + align4(nw * E) +
                                 (size_t)pp.lp.tokens_per_chunk * K);
    const long long grid = (long long)pp.lp.chunks + (long long)T * pp.slices;
    // every block carries the ranking blocks' shared memory: take this path
    // only while the packing blocks still fill at least 3/4 of an SM
    const long long per_sm = min((long long)kSmPerBlockLimit, (long long)(kSmemPerSm / (pp.smem + 1024)));
    pp.use = pp.threads >= 64 && pp.smem <= kMaxRankSmem && per_sm * pp.threads >= 1536 &&
             grid <= 0x7fffffffll;
    return pp;
}

template <int KT, bool kFp8>
cudaError_t run_prefill(const PrefillPlan &pp, const int32_t *ids, const void *tokens, int T,
                        int H, int K, int E, int R, const int32_t *ws_cnt, uint32_t *ws_err,
                        int32_t *counts, int32_t *offsets, int32_t *rank_offsets,
                        int32_t *src_token, int32_t *dst_row, uint32_t *dev_error,
                        void *packed, float *scales, unsigned long long wait_ns,
                        int stall_chunk, cudaStream_t s)
{
    auto *fn = rank_dispatch_kernel<KT, kFp8>;
    cudaError_t e = allow_dynamic_smem((const void *)fn, pp.smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(pp.lp.chunks + (long long)T * pp.slices);
    return launch_pdl(fn, dim3(grid), dim3(pp.threads), pp.smem, s, ids,
                      static_cast<const uint4 *>(tokens), T, H, K, E, R,
                      pp.lp.tokens_per_chunk, pp.lp.chunks, pp.slices, ws_cnt, ws_err, counts,
                      offsets, rank_offsets, src_token, dst_row, dev_error,
                      static_cast<uint8_t *>(packed), scales, wait_ns, stall_chunk);
}

template <bool kFp8>
cudaError_t run_prefill_k(const PrefillPlan &pp, const int32_t *ids, const void *tokens, int T,
                          int H, int K, int E, int R, const int32_t *ws_cnt, uint32_t *ws_err,
                          int32_t *counts, int32_t *offsets, int32_t *rank_offsets,
                          int32_t *src_token, int32_t *dst_row, uint32_t *dev_error,
                          void *packed, float *scales, unsigned long long wait_ns,
                          int stall_chunk, cudaStream_t s)
{
#define MOE_PREFILL_CASE(KV)                                                                   \
    return run_prefill<KV, kFp8>(pp, ids, tokens, T, H, K, E, R, ws_cnt, ws_err, counts,       \
                                 offsets, rank_offsets, src_token, dst_row, dev_error, packed, \
                                 scales, wait_ns, stall_chunk, s)
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
    int32_t *ws_cnt = static_cast<int32_t *>(workspace);
    uint32_t *ws_err = reinterpret_cast<uint32_t *>(ws_cnt + (size_t)pp.lp.chunks * E);
    cudaError_t e = launch_layout_count(topk_ids, T, K, E, pp.lp, ws_cnt, ws_err, dev_error,
                                        dst_row, stream);
    if (e != cudaSuccess) return e;
    if (wait_ns == 0) wait_ns = kWaitNs;
    if (fp8)
        return run_prefill_k<true>(pp, topk_ids, tokens, T, H, K, E, R, ws_cnt, ws_err,
                                   expert_counts, expert_offsets, rank_offsets, src_token,
                                   dst_row, dev_error, packed, scales, wait_ns, stall_chunk,
                                   stream);
    return run_prefill_k<false>(pp, topk_ids, tokens, T, H, K, E, R, ws_cnt, ws_err,
                                expert_counts, expert_offsets, rank_offsets, src_token, dst_row,
                                dev_error, packed, scales, wait_ns, stall_chunk, stream);
}

}  // namespace moe

// Test hook, deliberately absent from the public header: the large-batch
// path of moe_layout_dispatch with a chosen bound on every wait for a
// ranked chunk and, when stall_chunk >= 0, that chunk never ranked (its
// ranking block stops before writing the slots, which stay pending).  A test
// uses it to see the bounded wait expire: the chunk's packing blocks set
// MOE_DEV_ERR_TIMEOUT and return, every other row is packed, and the context
// stays usable.  Arguments are checked by the caller (tests only).
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
