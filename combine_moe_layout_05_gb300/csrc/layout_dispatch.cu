// layout_dispatch.cu -- layout and dispatch in one launch for small batches.
//
// Perplexity, "Enabling trillion-parameter models on AWS EFA", section
// "Dispatch and Combine": one dispatch-send kernel counts tokens per expert,
// takes the cumulative sum of the counts and packs the tokens into the
// contiguous send buffers.  For decode-sized batches the whole step is a few
// microseconds of data movement, so launch latency and the dependency
// between a layout kernel and a dispatch kernel cost as much as the copy.
// This kernel does both in one launch without any block waiting for another:
//
//  * block (t, c) packs slice c of token t's row;
//  * before that, every block copies all T*K ids into its shared memory
//    (asynchronous copies, one memory latency) and recomputes there the
//    expert histogram of all entries, the histogram of the entries that
//    come before token t, and the exclusive scan of the totals.  The slot of
//    entry (t, k) is offsets[e] + (entries of e before token t) + (earlier
//    k' of token t with the same e), the same stable order as moe_layout;
//  * the row slice is loaded before the histogram work, so the HBM latency
//    of the token row overlaps it;
//  * slice 0 of each token writes its dst_row / src_token entries and block
//    0 writes the counts, offsets, rank offsets and error word.
// The redundant histogram costs T*K shared-memory atomics per block, so this
// path is used only while blocks x entries stays small (decode shapes); the
// C ABI falls back to moe_layout + moe_dispatch otherwise.
#include "common.cuh"
#include "internal.h"
#include "layout_common.cuh"
#include "moe_layout.h"
#include "rowops.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxEntries = 8192;
constexpr long long kMaxRedundantEntries = 1ll << 22;

template <int KT, bool kFp8>
__global__ void __launch_bounds__(kThreads)
layout_dispatch_kernel(const int32_t *__restrict__ ids, const uint4 *__restrict__ tokens,
                       int T, int H, int K, int E, int R, int chunks, int upc,
                       int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                       int32_t *__restrict__ rank_offsets,
                       int32_t *__restrict__ src_token, int32_t *__restrict__ dst_row,
                       uint32_t *__restrict__ dev_error, uint8_t *__restrict__ packed,
                       float *__restrict__ scales)
{
    extern __shared__ __align__(16) int32_t sm[];
    int32_t *hist = sm;                   // [E] all entries
    int32_t *before = hist + E;           // [E] entries of tokens before t
    int32_t *off = before + E;            // [E + 1]
    int32_t *ids_s = sm + align4(3 * E + 1);  // [T*K], 16-byte aligned
    __shared__ int32_t slots[MOE_MAX_TOPK];
    __shared__ int32_t warp_sums[32];
    __shared__ uint32_t s_err;

    const int tid = threadIdx.x;
    const int t = blockIdx.x / chunks, c = blockIdx.x - (blockIdx.x / chunks) * chunks;
    const int k_count = KT > 0 ? KT : K;
    const int n = T * k_count;
    const int mine = t * k_count;
    const int units = kFp8 ? (H >> 4) : (H >> 3);
    const int u0 = c * upc, u1 = min(units, u0 + upc);
    const size_t vrow = (size_t)(H >> 3);

    for (int e = tid; e < E; e += kThreads) {
        hist[e] = 0;
        before[e] = 0;
    }
    if (tid == 0) s_err = 0;
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    // the first piece of this thread's share of the row, loaded early
    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
    {
        const int u = u0 + tid;
        if (u < u1) {
            if (kFp8) {
                a = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u);
                b = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u + 1);
            } else {
                a = ld_stream_v4(tokens + (size_t)t * vrow + u);
            }
        }
    }

    stage_i32(ids_s, ids, n);
    cp_async_wait_all();
    __syncthreads();

    for (int i = tid; i < n; i += kThreads) {
        const int e = ids_s[i];
        if ((unsigned)e < (unsigned)E) {
            atomicAdd(hist + e, 1);
            if (i < mine) atomicAdd(before + e, 1);
        }
    }
    if (blockIdx.x == 0) {
        const uint32_t err = token_errors(ids_s, T, k_count, E);
        if (err) atomicOr(&s_err, err);
    }
    __syncthreads();
    scan_experts<kThreads>(hist, off, E, warp_sums);

    if (tid < k_count) {
        const int e = ids_s[mine + tid];
        int slot = -1;
        if ((unsigned)e < (unsigned)E) {
            int dup = 0;
            for (int x = 0; x < tid; ++x) dup += ids_s[mine + x] == e;
            slot = off[e] + before[e] + dup;
        }
        slots[tid] = slot;
        if (c == 0) {
            dst_row[mine + tid] = slot;
            if (slot >= 0) src_token[slot] = t;
        }
    }
    if (blockIdx.x == 0) {
        for (int e = tid; e < E; e += kThreads) {
            counts[e] = hist[e];
            offsets[e] = off[e];
        }
        if (tid == 0) {
            offsets[E] = off[E];
            if (dev_error) *dev_error = s_err;
        }
        const int epr = E / R;
        for (int r = tid; r <= R; r += kThreads) rank_offsets[r] = off[r * epr];
    }
    __syncthreads();

    const int rows = n;
    for (int base = u0; base < u1; base += kThreads) {     // uniform per block
        const int u = base + tid;
        const bool active = u < u1;
        if (base != u0 && active) {
            if (kFp8) {
                a = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u);
                b = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u + 1);
            } else {
                a = ld_stream_v4(tokens + (size_t)t * vrow + u);
            }
        }
        if (kFp8) {
            const Fp8Piece p = quantize16(a, b);    // every lane takes part
            if (active)
                store_fp8_to_slots<KT>(slots, k_count, rows, packed, scales, H, u, p);
        } else if (active) {
            store_to_slots<KT>(slots, k_count, rows, packed, vrow * 16, (size_t)u * 16, a);
        }
    }
}

struct FusedPlan {
    bool use;
    int chunks;
    int upc;
};

FusedPlan plan_fused(int T, int H, int K, bool fp8)
{
    const long long n = (long long)T * K;
    const int units = fp8 ? H / 16 : H / 8;
    int chunks = ceil_div(units, kThreads);
    int upc = ceil_div(ceil_div(units, chunks), 32) * 32;
    chunks = ceil_div(units, upc);
    const long long blocks = (long long)T * chunks;
    const bool use = T > 0 && n <= kMaxEntries && blocks * n <= kMaxRedundantEntries &&
                     blocks <= 0x7fffffffll;
    return {use, chunks, upc};
}

template <int KT, bool kFp8>
cudaError_t run_fused(const FusedPlan &p, const int32_t *ids, const void *tokens,
                      int T, int H, int K, int E, int R, int32_t *counts,
                      int32_t *offsets, int32_t *rank_offsets, int32_t *src_token,
                      int32_t *dst_row, uint32_t *dev_error, void *packed,
                      float *scales, cudaStream_t s)
{
    const size_t smem = sizeof(int32_t) * ((size_t)align4(3 * E + 1) + (size_t)T * K);
    return launch_pdl(layout_dispatch_kernel<KT, kFp8>, dim3(T * p.chunks), dim3(kThreads),
                      smem, s, ids, static_cast<const uint4 *>(tokens), T, H, K, E, R,
                      p.chunks, p.upc, counts, offsets, rank_offsets, src_token,
                      dst_row, dev_error, static_cast<uint8_t *>(packed), scales);
}

template <bool kFp8>
cudaError_t run_fused_k(const FusedPlan &p, const int32_t *ids, const void *tokens,
                        int T, int H, int K, int E, int R, int32_t *counts,
                        int32_t *offsets, int32_t *rank_offsets, int32_t *src_token,
                        int32_t *dst_row, uint32_t *dev_error, void *packed,
                        float *scales, cudaStream_t s)
{
#define MOE_FUSED_CASE(KV)                                                          \
    return run_fused<KV, kFp8>(p, ids, tokens, T, H, K, E, R, counts, offsets,      \
                               rank_offsets, src_token, dst_row, dev_error, packed, \
                               scales, s)
    switch (K) {
    case 1: MOE_FUSED_CASE(1);
    case 2: MOE_FUSED_CASE(2);
    case 4: MOE_FUSED_CASE(4);
    case 6: MOE_FUSED_CASE(6);
    case 8: MOE_FUSED_CASE(8);
    default: MOE_FUSED_CASE(0);
    }
#undef MOE_FUSED_CASE
}

}  // namespace

bool layout_dispatch_fused(int T, int H, int K, int fp8)
{
    return plan_fused(T, H, K, fp8 != 0).use;
}

cudaError_t launch_layout_dispatch(const int32_t *topk_ids, const void *tokens,
                                   int T, int H, int K, int E, int R, int fp8,
                                   int32_t *expert_counts, int32_t *expert_offsets,
                                   int32_t *rank_offsets, int32_t *src_token,
                                   int32_t *dst_row, uint32_t *dev_error,
                                   void *packed, float *scales, void *workspace,
                                   cudaStream_t stream)
{
    const FusedPlan p = plan_fused(T, H, K, fp8 != 0);
    if (p.use) {
        if (fp8)
            return run_fused_k<true>(p, topk_ids, tokens, T, H, K, E, R, expert_counts,
                                     expert_offsets, rank_offsets, src_token, dst_row,
                                     dev_error, packed, scales, stream);
        return run_fused_k<false>(p, topk_ids, tokens, T, H, K, E, R, expert_counts,
                                  expert_offsets, rank_offsets, src_token, dst_row,
                                  dev_error, packed, scales, stream);
    }
    cudaError_t e = launch_layout(topk_ids, T, K, E, R, expert_counts, expert_offsets,
                                  rank_offsets, src_token, dst_row, dev_error,
                                  workspace, stream);
    if (e != cudaSuccess || T == 0) return e;
    if (fp8) return launch_dispatch_fp8(tokens, T, H, K, dst_row, packed, scales, stream);
    return launch_dispatch_bf16(tokens, T, H, K, dst_row, packed, stream);
}

}  // namespace moe
