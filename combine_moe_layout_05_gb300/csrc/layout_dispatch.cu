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
//    (asynchronous copies, one memory latency) and counts there, for each of
//    its token's K entries (t, k) with expert e, the valid ids below e (that
//    is offsets[e]), the entries of e before token t and the earlier k' of
//    token t with id e; their sum is the slot, the same stable order as
//    moe_layout.  One pass over the ids with K predicated counters per
//    thread and one block reduction; no histogram, no scan, no atomics;
//  * the row slice is loaded before the histogram work, so the HBM latency
//    of the token row overlaps it;
//  * slice 0 of each token writes its dst_row / src_token entries; block b
//    also counts expert b (count and offset, and the rank offset when b
//    starts a rank), and block 0 writes the error word.
// Each block reads all T*K ids, so this path is used only while blocks x
// entries stays small (decode shapes); the C ABI falls back to moe_layout +
// moe_dispatch otherwise.
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

// Sum over the block of N per-thread counters; the totals land in out[0..N)
// (shared memory) and are visible to every thread on return.
template <int N>
__device__ __forceinline__ void block_sum(const int (&v)[N], int32_t (*red)[16],
                                          int32_t *out)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < N; ++j) {
        const int s = __reduce_add_sync(kFullMask, v[j]);
        if (lane == 0) red[w][j] = s;
    }
    __syncthreads();
    if (threadIdx.x < N) {
        int s = 0;
#pragma unroll
        for (int q = 0; q < kThreads / 32; ++q) s += red[q][threadIdx.x];
        out[threadIdx.x] = s;
    }
    __syncthreads();
}

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
    extern __shared__ __align__(16) int32_t ids_s[];   // [T*K]
    __shared__ int32_t red[kThreads / 32][16];
    __shared__ int32_t sums[16];
    __shared__ int32_t slots[MOE_MAX_TOPK];
    __shared__ uint32_t s_err;

    const int tid = threadIdx.x;
    const int nb = gridDim.x, b = blockIdx.x;
    const int t = b / chunks, c = b - (b / chunks) * chunks;
    const int k_count = KT > 0 ? KT : K;
    const int n = T * k_count;
    const int mine = t * k_count;
    const int units = kFp8 ? (H >> 4) : (H >> 3);
    const int u0 = c * upc, u1 = min(units, u0 + upc);
    const size_t vrow = (size_t)(H >> 3);
    const int epr = E / R;

    if (tid == 0) s_err = 0;
    pdl_wait();
    pdl_trigger();

    // the first piece of this thread's share of the row, loaded early
    uint4 a = make_uint4(0, 0, 0, 0), bv = make_uint4(0, 0, 0, 0);
    {
        const int u = u0 + tid;
        if (u < u1) {
            if (kFp8) {
                a = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u);
                bv = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u + 1);
            } else {
                a = ld_stream_v4(tokens + (size_t)t * vrow + u);
            }
        }
    }
    stage_i32(ids_s, ids, n);
    cp_async_wait_all();
    __syncthreads();

    // Slots of this token's entries, 8 at a time:
    //   slot(t,k) = #{valid ids < e} + #{entries before token t with id e}
    //             + #{k' < k of token t with id e},  e = ids[t,k].
    // The first pass also gives block b the count and offset of expert b
    // (offsets[e] = #{valid ids < e}), so these outputs are spread over the
    // grid; experts beyond the grid take further passes below.
    for (int k0 = 0; k0 < k_count; k0 += 8) {
        int tg[8], v[10];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            tg[j] = k0 + j < k_count ? ids_s[mine + k0 + j] : -1;
            v[j] = 0;
        }
        const int role = (k0 == 0 && b <= E) ? b : -1;
        v[8] = v[9] = 0;
        for (int i = tid; i < n; i += kThreads) {
            const int x = ids_s[i];
            if ((unsigned)x >= (unsigned)E) continue;
            const bool before = i < mine;
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] += (x < tg[j]) | ((x == tg[j]) & before);
            v[8] += x < role;
            v[9] += x == role;
        }
        block_sum<10>(v, red, sums);
        if (tid < 8 && k0 + tid < k_count) {
            const int e = ids_s[mine + k0 + tid];
            int slot = -1;
            if ((unsigned)e < (unsigned)E) {
                int dup = 0;
                for (int x = 0; x < k0 + tid; ++x) dup += ids_s[mine + x] == e;
                slot = sums[tid] + dup;
            }
            slots[k0 + tid] = slot;
            if (c == 0) {
                dst_row[mine + k0 + tid] = slot;
                if (slot >= 0) src_token[slot] = t;
            }
        }
        if (role >= 0 && tid == 0) {
            offsets[role] = sums[8];
            if (role < E) counts[role] = sums[9];
            if (role % epr == 0) rank_offsets[role / epr] = sums[8];
        }
        __syncthreads();    // sums is reused by the next pass
    }
    // experts not covered by the first pass (grids smaller than E + 1)
    for (int r0 = b + nb; r0 <= E; r0 += 8 * nb) {
        int v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0;
        for (int i = tid; i < n; i += kThreads) {
            const int x = ids_s[i];
            if ((unsigned)x >= (unsigned)E) continue;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[2 * j] += x < r0 + j * nb;
                v[2 * j + 1] += x == r0 + j * nb;
            }
        }
        block_sum<16>(v, red, sums);
        if (tid < 8) {
            const int e = r0 + tid * nb;
            if (e <= E) {
                offsets[e] = sums[2 * tid];
                if (e < E) counts[e] = sums[2 * tid + 1];
                if (e % epr == 0) rank_offsets[e / epr] = sums[2 * tid];
            }
        }
        __syncthreads();
    }
    if (b == 0) {
        const uint32_t err = token_errors(ids_s, T, k_count, E);
        if (err) atomicOr(&s_err, err);
        __syncthreads();
        if (tid == 0 && dev_error) *dev_error = s_err;
    }

    const int rows = n;
    for (int base = u0; base < u1; base += kThreads) {     // uniform per block
        const int u = base + tid;
        const bool active = u < u1;
        if (base != u0 && active) {
            if (kFp8) {
                a = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u);
                bv = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u + 1);
            } else {
                a = ld_stream_v4(tokens + (size_t)t * vrow + u);
            }
        }
        if (kFp8) {
            const Fp8Piece p = quantize16(a, bv);   // every lane takes part
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
    const size_t smem = sizeof(int32_t) * (size_t)T * K;
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
