// layout_dispatch_persistent.cu -- a persistent form of the large-batch
// layout + dispatch, kept for comparison (reachable only through a test
// hook; moe_layout_dispatch uses layout_dispatch_prefill.cu).
//
// Perplexity, "Enabling trillion-parameter models on AWS EFA", section
// "Dispatch and Combine": dispatch-send counts, takes the cumulative sum and
// packs the tokens into contiguous per-destination buffers.  This form
// stages the token rows in shared memory with the copy engine:
//
//  * layout_count_kernel (layout.cu) writes each chunk's histogram and error
//    bits to the workspace and zeroes the error word;
//  * rank_pack_kernel runs one CTA per SM; CTA p owns a contiguous token
//    range [t0, t1).  Its warp 0 is the producer: one lane asks the copy
//    engine (bulk asynchronous copies) for the token rows of the range, one
//    row per stage of a shared-memory ring, and refills a stage as soon as
//    its consumers release it.  The other warps are the consumers.  While the
//    first rows arrive they sum the chunk histograms column by column, rank
//    the CTA's entries in the same stable order as moe_layout and write
//    dst_row / src_token.  Then they form groups of 8 warps; group g takes
//    the tokens j = g, g + G, ... of the range and writes each row to its K
//    slots: bf16 rows with 16-byte stores or, in the bulk-store form, by bulk
//    copies straight out of the ring; FP8 rows quantised per 1x128 block.
//
// Measured on one GB300 (CUDA graphs, cold L2) it is slower than the
// two-launch form of layout_dispatch_prefill.cu, whose packing blocks stage
// through registers: at the Kimi-K2 prefill shape (bf16) 102 us with 16-byte
// stores and 98 us with bulk stores, against 90 us; at the Qwen3 prefill
// shape (FP8) 139 us against 112 us.  One CTA per SM keeps too few stores
// in flight (ncu: 62 % DRAM throughput, 14 % issue slots, warps throttled
// on the store queue), and a persistent copy of the same rows from
// registers, without the ring, was 10 % slower than many small blocks too.
//
// No CTA waits for another.  Every wait on a barrier is bounded by a
// deadline; when one expires the CTA raises an abort flag that ends every
// other wait at once, waits (bounded again) for the row loads it has in
// flight, sets MOE_DEV_ERR_TIMEOUT in the error word and finishes.
#include "bulk.cuh"
#include "common.cuh"
#include "internal.h"
#include "layout_common.cuh"
#include "moe_layout.h"
#include "rowops.cuh"

namespace moe {
namespace {

constexpr int kGroupThreads = 256;         // consumer threads per group (8 warps)
constexpr int kRankWarps = 8;              // consumer warps that rank (the first group)
constexpr int kPieceEntries = 2048;        // entries ranked per pass over the ids
constexpr int kMaxStages = 16;
constexpr int kBarBytes = 512;             // full[], empty[] and the test barrier
constexpr size_t kSmemBudget = 220 * 1024; // dynamic shared memory per CTA
constexpr unsigned long long kWaitNs = 1000000000ull;   // 1 s
constexpr int kConsumerBarrier = 1;        // named barrier of the consumer warps
#ifndef MOE_PACK_GROUPS
#define MOE_PACK_GROUPS 3
#endif
constexpr int kPackGroups = MOE_PACK_GROUPS;   // consumer groups per CTA

// Bytes of the integer arrays: tot[E], pre[E], base[E+1], rows[kRankWarps][E],
// ids[kPieceEntries], slots[kPieceEntries]; a multiple of 128.
__host__ __device__ inline size_t ints_bytes(int E)
{
    const size_t n = 2 * (size_t)align4(E) + (size_t)align4(E + 1) + (size_t)kRankWarps * E +
                     2 * (size_t)kPieceEntries;
    return (4 * n + 127) & ~(size_t)127;
}

__device__ __forceinline__ uint4 ld_shared_v4(const void *p)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(smem_addr(p)));
    return r;
}

// Exclusive scan of hist[0..E) into off[0..E] (off[E] = total) by the n
// consumer threads ct = 0 .. n-1 (n a multiple of 32, at most 1024).
__device__ __forceinline__ void consumer_scan(const int32_t *hist, int32_t *off, int E,
                                              int32_t *warp_sums, int ct, int n)
{
    const int per = (E + n - 1) / n;
    const int lane = ct & 31, w = ct >> 5, nw = n >> 5;
    int s = 0;
    for (int j = 0; j < per; ++j) {
        const int e = ct * per + j;
        s += e < E ? hist[e] : 0;
    }
    int x = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(kFullMask, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    named_barrier(kConsumerBarrier, n);
    if (w == 0) {
        int q = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(kFullMask, q, d);
            if (lane >= d) q += y;
        }
        if (lane < nw) warp_sums[lane] = q;
    }
    named_barrier(kConsumerBarrier, n);
    int run = (w ? warp_sums[w - 1] : 0) + x - s;
    for (int j = 0; j < per; ++j) {
        const int e = ct * per + j;
        if (e < E) {
            off[e] = run;
            run += hist[e];
        }
    }
    if (ct == 0) off[E] = warp_sums[nw - 1];
    named_barrier(kConsumerBarrier, n);
}

// kMode: 0 = bf16 rows with 16-byte stores, 1 = bf16 rows by bulk stores out
// of the ring, 2 = FP8 (quantised by the consumers, 16-byte stores).
template <int KT, int kMode, int kGroups>
__global__ void __launch_bounds__(32 + kGroups * kGroupThreads, 1)
rank_pack_kernel(const int32_t *__restrict__ ids, const uint8_t *__restrict__ tokens,
                 int T, int H, int K, int E, int R, int tpc, int chunks,
                 const int32_t *__restrict__ ws_cnt, const uint32_t *__restrict__ ws_err,
                 int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                 int32_t *__restrict__ rank_offsets, int32_t *__restrict__ src_token,
                 int32_t *__restrict__ dst_row, uint32_t *__restrict__ dev_error,
                 uint8_t *__restrict__ packed, float *__restrict__ scales, int stages,
                 unsigned long long wait_ns, int stall_cta)
{
    constexpr int NC = kGroups * kGroupThreads;             // consumer threads
    extern __shared__ __align__(128) uint8_t sm[];
    uint64_t *full = reinterpret_cast<uint64_t *>(sm);     // [kMaxStages]: row landed
    uint64_t *empty = full + kMaxStages;                     // [kMaxStages]: row consumed
    uint64_t *never = empty + kMaxStages;                    // signalled by nothing
    int32_t *tot = reinterpret_cast<int32_t *>(sm + kBarBytes);
    int32_t *pre = tot + align4(E);
    int32_t *base = pre + align4(E);
    int32_t *rows = base + align4(E + 1);
    int32_t *ids_s = rows + kRankWarps * E;                  // 16-byte aligned
    int32_t *slots_s = ids_s + kPieceEntries;
    uint8_t *ring = sm + kBarBytes + ints_bytes(E);
    __shared__ int32_t warp_sums[32];
    __shared__ uint32_t s_err;
    __shared__ int s_abort;
    volatile int *abort = &s_abort;

    const int tid = threadIdx.x;
    const int k_count = KT > 0 ? KT : K;
    const int P = gridDim.x, p = blockIdx.x;
    const int per = T / P, extra = T % P;
    const int t0 = p * per + min(p, extra);
    const int t1 = t0 + per + (p < extra ? 1 : 0);
    const int n_own = t1 - t0;
    const uint32_t row_in = 2u * (uint32_t)H;               // bytes of a bf16 token row
    const int rows_total = T * k_count;

    if (tid == 0) {
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kGroupThreads / 32);
        }
        mbar_init(never, 1);
        s_err = 0;
        s_abort = 0;
        fence_barrier_init();
        fence_async_shared();
    }
    for (int e = tid; e < E; e += blockDim.x) {
        tot[e] = 0;
        pre[e] = 0;
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    if (tid < 32) {
        // ---- producer: one lane streams the rows of [t0, t1) through the ring
        if (tid == 0) {
            int last[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) last[s] = -1;
            for (int x = 0; x < n_own; ++x) {
                const int s = x % stages;
                if (x >= stages &&
                    !mbar_wait_or_abort(empty + s, (uint32_t)(x / stages - 1) & 1u,
                                        global_ns() + wait_ns, abort)) {
                    *abort = 1;
                    break;
                }
                mbar_arrive_expect(full + s, row_in);
                bulk_load(ring + (size_t)s * row_in, tokens + (size_t)(t0 + x) * row_in, row_in,
                          full + s);
                last[s] = x;
            }
            // every row load issued lands before the CTA's shared memory is released
            const unsigned long long until = global_ns() + wait_ns;
            for (int s = 0; s < stages; ++s)
                if (last[s] >= 0)
                    mbar_wait_until(full + s, (uint32_t)(last[s] / stages) & 1u, until);
            if (*abort && dev_error) atomicOr(dev_error, MOE_DEV_ERR_TIMEOUT);
        }
        return;
    }

    // ---- consumers
    const int ct = tid - 32;
    const int lane = ct & 31, cw = ct >> 5;

    // totals per expert, and the entries of each expert before t0: whole
    // chunks before t0's chunk from the histograms, then the ids of t0's
    // chunk up to t0
    const int c0 = t0 / tpc;
    {
        const int G = E < NC ? NC / E : 1;
        for (int idx = ct; idx < G * E; idx += NC) {
            const int e = idx % E, g = idx / E;
            int tt = 0, pp = 0;
#pragma unroll 4
            for (int c = g; c < chunks; c += G) {
                const int v = __ldg(ws_cnt + (size_t)c * E + e);
                tt += v;
                pp += c < c0 ? v : 0;
            }
            atomicAdd(tot + e, tt);
            atomicAdd(pre + e, pp);
        }
        for (int i = c0 * tpc * k_count + ct; i < t0 * k_count; i += NC) {
            const int e = __ldg(ids + i);
            if ((unsigned)e < (unsigned)E) atomicAdd(pre + e, 1);
        }
        if (p == 0) {
            uint32_t err = 0;
            for (int c = ct; c < chunks; c += NC) err |= __ldg(ws_err + c);
            if (err) atomicOr(&s_err, err);
        }
    }
    named_barrier(kConsumerBarrier, NC);
    consumer_scan(tot, base, E, warp_sums, ct, NC);
    if (p == 0) {
        for (int e = ct; e < E; e += NC) {
            counts[e] = tot[e];
            offsets[e] = base[e];
        }
        if (ct == 0) {
            offsets[E] = base[E];
            if (dev_error && s_err) atomicOr(dev_error, s_err);
        }
        const int epr = E / R;
        for (int r = ct; r <= R; r += NC) rank_offsets[r] = base[r * epr];
    }

    const int g = ct / kGroupThreads, r = ct % kGroupThreads;
    const int piece_tokens = kPieceEntries / k_count;
    for (int pt0 = t0; pt0 < t1; pt0 += piece_tokens) {
        // rank the piece's entries (the first kRankWarps consumer warps)
        const int pt1 = min(t1, pt0 + piece_tokens);
        const int first = pt0 * k_count, m = (pt1 - pt0) * k_count;
        stage_i32(ids_s, ids + first, m, ct, NC);
        for (int i = ct; i < kRankWarps * E; i += NC) rows[i] = 0;
        cp_async_wait_all();
        named_barrier(kConsumerBarrier, NC);
        int lo = 0, hi = 0;
        if (cw < kRankWarps) {
            warp_segment<kRankWarps>(m, cw, lo, hi);
            warp_count<false>(ids_s, lo, hi, E, lane, rows + cw * E);
        }
        named_barrier(kConsumerBarrier, NC);
        for (int e = ct; e < E; e += NC) {
            int run = base[e] + pre[e];
#pragma unroll
            for (int ww = 0; ww < kRankWarps; ++ww) {
                const int v = rows[ww * E + e];
                rows[ww * E + e] = run;
                run += v;
            }
            pre[e] = run - base[e];
        }
        named_barrier(kConsumerBarrier, NC);
        if (cw < kRankWarps)
            warp_rank<false>(ids_s, lo, hi, E, k_count, first, lane, rows + cw * E, dst_row,
                             src_token, slots_s);
        named_barrier(kConsumerBarrier, NC);

        // pack: group g takes own tokens j = g (mod kGroups)
        const int jp0 = pt0 - t0, jp1 = pt1 - t0;
        for (int j = jp0 + ((g - jp0 % kGroups) + kGroups) % kGroups; j < jp1; j += kGroups) {
            const int s = j % stages;
            const uint32_t par = (uint32_t)(j / stages) & 1u;
            uint64_t *bar = (stall_cta == p && j == 0) ? never : full + s;
            // every lane observes the phase itself (that orders the copy engine's
            // writes before its reads); the warp then acts on one common decision
            const bool ok = mbar_wait_or_abort(bar, par, global_ns() + wait_ns, abort);
            if (!__all_sync(kFullMask, ok)) {
                *abort = 1;
                continue;        // nothing is read or released; the loops run out
            }
            const uint8_t *src = ring + (size_t)s * row_in;
            const int32_t *sl = slots_s + (size_t)(j - jp0) * k_count;
            if (kMode == 0) {
                for (int u = r; u < (int)(row_in >> 4); u += kGroupThreads)
                    store_to_slots<KT>(sl, k_count, rows_total, packed, row_in, 16 * (size_t)u,
                                       ld_shared_v4(src + 16 * (size_t)u));
            } else if (kMode == 1) {
                if (r == 0) {
                    for (int k = 0; k < k_count; ++k) {
                        const int q = sl[k];
                        if ((unsigned)q < (unsigned)rows_total)
                            bulk_store(packed + (size_t)q * row_in, src, row_in);
                    }
                    bulk_commit();
                    bulk_wait_read<0>();
                }
            } else {
                const int groups16 = H >> 4;
                for (int u0 = 0; u0 < groups16; u0 += kGroupThreads) {   // uniform per warp
                    const int u = u0 + r;
                    const bool active = u < groups16;
                    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
                    if (active) {
                        a = ld_shared_v4(src + 32 * (size_t)u);
                        b = ld_shared_v4(src + 32 * (size_t)u + 16);
                    }
                    const Fp8Piece q = quantize16(a, b);
                    if (active)
                        store_fp8_to_slots<KT>(sl, k_count, rows_total, packed, scales, H, u, q);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + s);
        }
        named_barrier(kConsumerBarrier, NC);     // slots_s is rewritten by the next piece
    }
    if (kMode == 1 && r == 0) bulk_wait_all();
}

struct PackPlan {
    bool use;
    int stages;
    size_t smem;
};

PackPlan plan_pack(int T, int H, int K, int E)
{
    const LayoutPlan lp = plan_layout(T, K, E);
    if (T <= 0 || lp.single_launch) return {false, 0, 0};
    const size_t fixed = kBarBytes + ints_bytes(E);
    const size_t row = 2 * (size_t)H;
    constexpr int kMinStages = 4;
    if (fixed + kMinStages * row > kSmemBudget) return {false, 0, 0};
    const int stages = (int)min((size_t)kMaxStages, (kSmemBudget - fixed) / row);
    return {true, stages, fixed + (size_t)stages * row};
}

template <int KT, int kMode, int kGroups>
cudaError_t run_pack(const PackPlan &pp, const LayoutPlan &lp, const int32_t *ids,
                     const void *tokens, int T, int H, int K, int E, int R,
                     const int32_t *ws_cnt, const uint32_t *ws_err, int32_t *counts,
                     int32_t *offsets, int32_t *rank_offsets, int32_t *src_token,
                     int32_t *dst_row, uint32_t *dev_error, void *packed, float *scales,
                     unsigned long long wait_ns, int stall_cta, cudaStream_t s)
{
    auto *fn = rank_pack_kernel<KT, kMode, kGroups>;
    cudaError_t e = allow_dynamic_smem((const void *)fn, pp.smem);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    const int grid = min(sms, T);
    return launch_pdl(fn, dim3(grid), dim3(32 + kGroups * kGroupThreads), pp.smem, s, ids,
                      static_cast<const uint8_t *>(tokens), T, H, K, E, R,
                      lp.tokens_per_chunk, lp.chunks, ws_cnt, ws_err, counts, offsets,
                      rank_offsets, src_token, dst_row, dev_error,
                      static_cast<uint8_t *>(packed), scales, pp.stages, wait_ns, stall_cta);
}

template <int kMode, int kGroups>
cudaError_t run_pack_k(const PackPlan &pp, const LayoutPlan &lp, const int32_t *ids,
                       const void *tokens, int T, int H, int K, int E, int R,
                       const int32_t *ws_cnt, const uint32_t *ws_err, int32_t *counts,
                       int32_t *offsets, int32_t *rank_offsets, int32_t *src_token,
                       int32_t *dst_row, uint32_t *dev_error, void *packed, float *scales,
                       unsigned long long wait_ns, int stall_cta, cudaStream_t s)
{
#define MOE_PACK_CASE(KV)                                                                   \
    return run_pack<KV, kMode, kGroups>(pp, lp, ids, tokens, T, H, K, E, R, ws_cnt, ws_err,  \
                                        counts, offsets, rank_offsets, src_token, dst_row,   \
                                        dev_error, packed, scales, wait_ns, stall_cta, s)
    switch (K) {
    case 1: MOE_PACK_CASE(1);
    case 2: MOE_PACK_CASE(2);
    case 4: MOE_PACK_CASE(4);
    case 6: MOE_PACK_CASE(6);
    case 8: MOE_PACK_CASE(8);
    default: MOE_PACK_CASE(0);
    }
#undef MOE_PACK_CASE
}

}  // namespace

bool layout_dispatch_persistent(int T, int H, int K, int E)
{
    return plan_pack(T, H, K, E).use;
}

cudaError_t launch_layout_dispatch_persistent(const int32_t *topk_ids, const void *tokens, int T, int H,
                               int K, int E, int R, int fp8, int32_t *expert_counts,
                               int32_t *expert_offsets, int32_t *rank_offsets,
                               int32_t *src_token, int32_t *dst_row, uint32_t *dev_error,
                               void *packed, float *scales, void *workspace,
                               unsigned long long wait_ns, int stall_cta, int bulk_store,
                               cudaStream_t stream)
{
    const PackPlan pp = plan_pack(T, H, K, E);
    if (!pp.use) return cudaErrorInvalidValue;
    const LayoutPlan lp = plan_layout(T, K, E);
    int32_t *ws_cnt = static_cast<int32_t *>(workspace);
    uint32_t *ws_err = reinterpret_cast<uint32_t *>(ws_cnt + (size_t)lp.chunks * E);
    cudaError_t e = launch_layout_count(topk_ids, T, K, E, lp, ws_cnt, ws_err, dev_error,
                                        nullptr, stream);
    if (e != cudaSuccess) return e;
    if (wait_ns == 0) wait_ns = kWaitNs;
#define MOE_PACK_ARGS                                                                     \
    pp, lp, topk_ids, tokens, T, H, K, E, R, ws_cnt, ws_err, expert_counts, expert_offsets, \
        rank_offsets, src_token, dst_row, dev_error, packed, scales, wait_ns, stall_cta, stream
    if (fp8) return run_pack_k<2, kPackGroups>(MOE_PACK_ARGS);
    if (bulk_store) return run_pack_k<1, kPackGroups>(MOE_PACK_ARGS);
    return run_pack_k<0, kPackGroups>(MOE_PACK_ARGS);
#undef MOE_PACK_ARGS
}

}  // namespace moe

// Test hook, deliberately absent from the public header: this persistent
// form of the large-batch layout + dispatch, with a chosen bound on every
// barrier wait (0: the default),
// the bf16 rows written by bulk stores when bulk_store != 0, and, when
// stall_cta >= 0, that CTA waiting for its first row on a barrier that
// nothing signals.  A test uses it to see the bounded wait expire: the
// kernel sets MOE_DEV_ERR_TIMEOUT and finishes, and the context stays
// usable.  Arguments are checked by the caller (tests only).
extern "C" __attribute__((visibility("default"))) int32_t
moe_testing_layout_pack(const int32_t *topk_ids, const void *tokens, int32_t T, int32_t H,
                        int32_t K, int32_t E, int32_t R, int32_t fp8, int32_t *expert_counts,
                        int32_t *expert_offsets, int32_t *rank_offsets, int32_t *src_token,
                        int32_t *dst_row, uint32_t *dev_error, void *packed, float *scales,
                        void *workspace, uint64_t wait_ns, int32_t stall_cta,
                        int32_t bulk_store, cudaStream_t stream)
{
    if (!moe::layout_dispatch_persistent(T, H, K, E)) return MOE_ERR_INVALID_ARG;
    const cudaError_t e = moe::launch_layout_dispatch_persistent(
        topk_ids, tokens, T, H, K, E, R, fp8, expert_counts, expert_offsets, rank_offsets,
        src_token, dst_row, dev_error, packed, scales, workspace, wait_ns, stall_cta,
        bulk_store, stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
