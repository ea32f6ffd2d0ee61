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
//  * before that, every block reads all T*K ids (16-byte loads into
//    registers) and counts, for each of its token's K entries (t, k) with
//    expert e, the valid ids below e (that is offsets[e]), the entries of e
//    before token t and the earlier k' of token t with id e; their sum is
//    the slot, the same stable order as moe_layout.  One pass over the ids
//    with the counters packed two to a word (two fp16 lanes per compare for
//    larger batches), a warp reduction and one barrier, after which every
//    thread adds the warps' partial sums itself and holds the slots in
//    registers; no histogram, no scan, no atomics;
//  * the row slice is requested first, so its HBM latency overlaps the
//    counting; in the FP8 form it is quantised just before the block
//    barrier, filling the time warps wait there;
//  * slice 0 of each token writes its dst_row / src_token entries; block b
//    also counts expert b (count and offset, and the rank offset when b
//    starts a rank), and block 0 writes the error word.
// Each block reads all T*K ids, so this path is used only while blocks x
// entries stays small (decode shapes); larger batches take the two-launch
// path of layout_dispatch_prefill.cu (or moe_layout + moe_dispatch where that
// path's shared memory would cost too much occupancy).  (A form for larger
// batches, in which each packing block counted only its layout chunk's
// earlier ids after the counting and scan kernels, replacing the ranking
// kernel, measured 25-50 % slower.)
#include "bulk.cuh"
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

// Adds, for the 8 targets tg[] (and the block's expert role), this entry's
// contributions to the packed 16-bit counters (two per 32-bit word; every
// count is at most T*K <= kMaxEntries < 2^16, so halves never carry).
__device__ __forceinline__ void count_entry(int x, int i, int mine, int E, int role,
                                            const int (&tg)[8], uint32_t (&v)[5])
{
    if ((unsigned)x >= (unsigned)E) return;
    const bool before = i < mine;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        v[j >> 1] += (uint32_t)((x < tg[j]) | ((x == tg[j]) & before)) << (16 * (j & 1));
    v[4] += (uint32_t)(x < role) | ((uint32_t)(x == role) << 16);
}

// Batches of at least kHalfCountMin entries count on packed fp16 pairs
// instead: an id x (0 <= x < E <= 1024) is the fp16 value 1024 + x, exact
// and ordered like the ids, and an invalid id is 2048, above every valid one,
// so one half2 compare tests two targets.  The fp16 sums stay exact: a
// thread sees at most kMaxEntries / kThreads = 32 entries.  (With fewer
// entries per thread the integer form is as fast.)
constexpr int kHalfCountMin = 2048;

__device__ __forceinline__ uint32_t enc_id(int x, int E)
{
    return 0x6400u + ((unsigned)x < (unsigned)E ? (uint32_t)x : 1024u);
}

__device__ __forceinline__ __half2 bits_h2(uint32_t u)
{
    return *reinterpret_cast<const __half2 *>(&u);
}

// count_entry on fp16 pairs: target pair q gains, per half,
// (x < tg) | (x == tg & before); the role pair gains (x < role, x == role).
__device__ __forceinline__ void count_entry_h2(int x, bool before, int E,
                                               const __half2 (&tg2)[4], __half2 role2,
                                               __half2 (&acc)[5])
{
    const __half2 xh = bits_h2(enc_id(x, E) * 0x10001u);
    const __half2 bm = before ? __float2half2_rn(1.0f) : __float2half2_rn(0.0f);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        acc[q] = __hadd2(acc[q], __hfma2(__heq2(xh, tg2[q]), bm, __hlt2(xh, tg2[q])));
    const __half2 lt = __hlt2(xh, role2), eq = __heq2(xh, role2);
    acc[4] = __hadd2(acc[4], __halves2half2(__low2half(lt), __high2half(eq)));
}

// Counting modes, fixed at compile time so each kernel holds one path:
// integer counters or fp16 pairs.
enum CountMode { kCountInt, kCountHalf };

// kBulk: the block's row slice is staged in shared memory and one thread
// writes it to every slot with bulk copies.  Measured at the DeepSeek-V3
// decode shape: 5.73 us against 5.12 with 16-byte stores (FP8: 6.76 against
// 6.55), so it is kept only for comparison, behind the test hook below.
template <int KT, bool kFp8, int kMode, bool kBulk = false>
__global__ void __launch_bounds__(kThreads)
layout_dispatch_kernel(const int32_t *__restrict__ ids, const uint4 *__restrict__ tokens,
                       int T, int H, int K, int E, int R, int chunks, int upc,
                       int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                       int32_t *__restrict__ rank_offsets,
                       int32_t *__restrict__ src_token, int32_t *__restrict__ dst_row,
                       uint32_t *__restrict__ dev_error, uint8_t *__restrict__ packed,
                       float *__restrict__ scales)
{
    __shared__ uint32_t red[kThreads / 32][8];
    __shared__ int32_t slots_s[MOE_MAX_TOPK];
    __shared__ uint32_t s_err;

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nb = gridDim.x, b = blockIdx.x;
    const int t = b / chunks, c = b - (b / chunks) * chunks;
    const int k_count = KT > 0 ? KT : K;
    const int n = T * k_count;
    const int mine = t * k_count;
    const int units = kFp8 ? (H >> 4) : (H >> 3);
    const int u0 = c * upc, u1 = min(units, u0 + upc);
    const size_t vrow = (size_t)(H >> 3);
    const int epr = E / R;
    constexpr bool kRegSlots = KT > 0 && KT <= 8;   // slots live in registers
    const bool vec_ids = ((reinterpret_cast<uintptr_t>(ids) & 15) == 0) && (n & 3) == 0;

    if (tid == 0) s_err = 0;
    pdl_wait();
    pdl_trigger();

    // this thread's first piece of the row; it arrives while slots are counted
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

    // Slots of this token's entries, 8 at a time:
    //   slot(t,k) = #{valid ids < e} + #{entries before token t with id e}
    //             + #{k' < k of token t with id e},  e = ids[t,k].
    // Each thread counts its share of the ids straight from global memory
    // (16-byte loads), each warp reduces its packed counters, and after one
    // barrier every thread adds up the warps' partial sums itself, so the
    // whole block holds the slots without further synchronisation.  The same
    // pass gives block b the count and offset of expert b
    // (offsets[e] = #{valid ids < e}), spreading those outputs over the grid.
    int sl[8];
    Fp8Piece q0;                        // the first row piece, quantised before the barrier
    for (int k0 = 0; k0 < k_count; k0 += 8) {
        int tg[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) tg[j] = k0 + j < k_count ? __ldg(ids + mine + k0 + j) : -1;
        const int role = (k0 == 0 && b <= E) ? b : -1;
        uint32_t v[5] = {0, 0, 0, 0, 0};
        if (kMode == kCountHalf) {
            __half2 tg2[4], acc[5];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                tg2[q] = bits_h2(enc_id(tg[2 * q], E) | enc_id(tg[2 * q + 1], E) << 16);
            const __half2 role2 = bits_h2(role >= 0 ? (0x6400u + (uint32_t)role) * 0x10001u : 0u);
#pragma unroll
            for (int q = 0; q < 5; ++q) acc[q] = __float2half2_rn(0.0f);
            if (vec_ids) {
                for (int i = 4 * tid; i < n; i += 4 * kThreads) {
                    const int4 q = __ldg(reinterpret_cast<const int4 *>(ids + i));
                    count_entry_h2(q.x, i < mine, E, tg2, role2, acc);
                    count_entry_h2(q.y, i + 1 < mine, E, tg2, role2, acc);
                    count_entry_h2(q.z, i + 2 < mine, E, tg2, role2, acc);
                    count_entry_h2(q.w, i + 3 < mine, E, tg2, role2, acc);
                }
            } else {
                for (int i = tid; i < n; i += kThreads)
                    count_entry_h2(__ldg(ids + i), i < mine, E, tg2, role2, acc);
            }
            // counts c <= 32 to packed 16-bit integers: 1024 + c has bits 0x6400 + c
#pragma unroll
            for (int q = 0; q < 5; ++q) {
                const __half2 h = __hadd2(acc[q], __float2half2_rn(1024.0f));
                v[q] = *reinterpret_cast<const uint32_t *>(&h) - 0x64006400u;
            }
        } else if (vec_ids) {
            for (int i = 4 * tid; i < n; i += 4 * kThreads) {
                const int4 q = __ldg(reinterpret_cast<const int4 *>(ids + i));
                count_entry(q.x, i, mine, E, role, tg, v);
                count_entry(q.y, i + 1, mine, E, role, tg, v);
                count_entry(q.z, i + 2, mine, E, role, tg, v);
                count_entry(q.w, i + 3, mine, E, role, tg, v);
            }
        } else {
            for (int i = tid; i < n; i += kThreads) count_entry(__ldg(ids + i), i, mine, E, role, tg, v);
        }
#pragma unroll
        for (int j = 0; j < 5; ++j) {
            const uint32_t sum = __reduce_add_sync(kFullMask, v[j]);
            if (lane == 0) red[w][j] = sum;
        }
        if (kFp8 && k0 == 0) q0 = quantize16(a, bv);   // fills the wait at the barrier
        __syncthreads();
        uint32_t tot[5] = {0, 0, 0, 0, 0};
#pragma unroll
        for (int q = 0; q < kThreads / 32; ++q)
#pragma unroll
            for (int j = 0; j < 5; ++j) tot[j] += red[q][j];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int dup = 0;
#pragma unroll
            for (int x = 0; x < j; ++x) dup += tg[x] == tg[j];
            for (int x = 0; x < k0; ++x) dup += __ldg(ids + mine + x) == tg[j];
            const int below = (int)((tot[j >> 1] >> (16 * (j & 1))) & 0xffffu);
            sl[j] = (unsigned)tg[j] < (unsigned)E ? below + dup : -1;
        }
        // the index-map and offset writes go to the block's last warp, which
        // has the least (at decode sizes often no) copying to do
        const int wl = tid - (kThreads - 32);
        if (wl >= 0 && wl < 8 && k0 + wl < k_count) {
            int mine_slot = sl[0];
#pragma unroll
            for (int j = 1; j < 8; ++j)
                if (wl == j) mine_slot = sl[j];
            if (!kRegSlots) slots_s[k0 + wl] = mine_slot;
            if (c == 0) {
                dst_row[mine + k0 + wl] = mine_slot;
                if (mine_slot >= 0) src_token[mine_slot] = t;
            }
        }
        if (role >= 0 && wl == 8) {
            const int lt = (int)(tot[4] & 0xffffu), eq = (int)(tot[4] >> 16);
            offsets[role] = lt;
            if (role < E) counts[role] = eq;
            if (role % epr == 0) rank_offsets[role / epr] = lt;
        }
        if (!kRegSlots) __syncthreads();   // red is reused; slots_s complete
    }

    const int rows = n;
    if (kBulk) {
        // one slice per block (upc <= kThreads): stage it, then one thread copies
        // it to every slot straight out of shared memory
        __shared__ __align__(128) uint4 stage[kThreads];
        const int u = u0 + tid;
        const int32_t *slots = kRegSlots ? sl : slots_s;
        if (u < u1) {
            if (kFp8) {
                stage[tid] = q0.codes;
                if ((u & 7) == 0)
                    for (int k = 0; k < k_count; ++k)
                        if ((unsigned)slots[k] < (unsigned)rows)
                            scales[(size_t)slots[k] * (H >> 7) + (u >> 3)] = q0.scale;
            } else {
                stage[tid] = a;
            }
        }
        fence_async_shared();
        __syncthreads();
        if (tid == 0) {
            const size_t row_bytes = kFp8 ? (size_t)H : vrow * 16;
            const uint32_t bytes = 16u * (uint32_t)(u1 - u0);
            for (int k = 0; k < k_count; ++k)
                if ((unsigned)slots[k] < (unsigned)rows)
                    bulk_store(packed + (size_t)slots[k] * row_bytes + 16 * (size_t)u0, stage, bytes);
            bulk_commit();
            bulk_wait_all();
        }
    }
    for (int base = u0; base < (kBulk ? u0 : u1); base += kThreads) {     // uniform per block
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
        const int32_t *slots = kRegSlots ? sl : slots_s;
        if (kFp8) {
            const Fp8Piece p = base == u0 ? q0 : quantize16(a, bv);   // every lane takes part
            if (active)
                store_fp8_to_slots<KT>(slots, k_count, rows, packed, scales, H, u, p);
        } else if (active) {
            store_to_slots<KT>(slots, k_count, rows, packed, vrow * 16, (size_t)u * 16, a);
        }
    }

    // experts not covered by the first pass (grids smaller than E + 1), in
    // groups of 8: plain 32-bit counters here, these passes are rare
    if (kRegSlots) __syncthreads();        // red is reused below
    for (int r0 = b + nb; r0 <= E; r0 += 4 * nb) {
        uint32_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int i = tid; i < n; i += kThreads) {
            const int x = __ldg(ids + i);
            if ((unsigned)x >= (unsigned)E) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[2 * j] += x < r0 + j * nb;
                v[2 * j + 1] += x == r0 + j * nb;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t sum = __reduce_add_sync(kFullMask, v[j]);
            if (lane == 0) red[w][j] = sum;
        }
        __syncthreads();
        if (tid < 4) {
            const int e = r0 + tid * nb;
            int lt = 0, eq = 0;
            for (int q = 0; q < kThreads / 32; ++q) {
                lt += red[q][2 * tid];
                eq += red[q][2 * tid + 1];
            }
            if (e <= E) {
                offsets[e] = lt;
                if (e < E) counts[e] = eq;
                if (e % epr == 0) rank_offsets[e / epr] = lt;
            }
        }
        __syncthreads();
    }
    if (b == 0) {
        const uint32_t err = token_errors(ids, T, k_count, E);
        if (err) atomicOr(&s_err, err);
        __syncthreads();
        if (tid == 0 && dev_error) *dev_error = s_err;
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

template <int KT, bool kFp8, int kMode, bool kBulk = false>
cudaError_t run_fused(const FusedPlan &p, const int32_t *ids, const void *tokens,
                      int T, int H, int K, int E, int R, int32_t *counts,
                      int32_t *offsets, int32_t *rank_offsets, int32_t *src_token,
                      int32_t *dst_row, uint32_t *dev_error, void *packed,
                      float *scales, cudaStream_t s)
{
    return launch_pdl(layout_dispatch_kernel<KT, kFp8, kMode, kBulk>, dim3(T * p.chunks),
                      dim3(kThreads), 0, s, ids, static_cast<const uint4 *>(tokens), T, H, K,
                      E, R, p.chunks, p.upc, counts, offsets, rank_offsets, src_token,
                      dst_row, dev_error, static_cast<uint8_t *>(packed), scales);
}

template <bool kFp8, int kMode>
cudaError_t run_fused_k(const FusedPlan &p, const int32_t *ids, const void *tokens,
                        int T, int H, int K, int E, int R, int32_t *counts,
                        int32_t *offsets, int32_t *rank_offsets, int32_t *src_token,
                        int32_t *dst_row, uint32_t *dev_error, void *packed,
                        float *scales, cudaStream_t s)
{
#define MOE_FUSED_CASE(KV)                                                             \
    return run_fused<KV, kFp8, kMode>(p, ids, tokens, T, H, K, E, R, counts, offsets,    \
                                         rank_offsets, src_token, dst_row, dev_error,    \
                                         packed, scales, s)
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

cudaError_t launch_layout_dispatch_fused(const int32_t *topk_ids, const void *tokens, int T,
                                         int H, int K, int E, int R, int fp8,
                                         int32_t *expert_counts, int32_t *expert_offsets,
                                         int32_t *rank_offsets, int32_t *src_token,
                                         int32_t *dst_row, uint32_t *dev_error, void *packed,
                                         float *scales, cudaStream_t stream)
{
    const FusedPlan p = plan_fused(T, H, K, fp8 != 0);
    if (!p.use) return cudaErrorInvalidValue;
#define MOE_FUSED_RUN(F, M)                                                                 \
    return run_fused_k<F, M>(p, topk_ids, tokens, T, H, K, E, R, expert_counts, expert_offsets, \
                             rank_offsets, src_token, dst_row, dev_error, packed, scales,       \
                             stream)
    const bool half = (long long)T * K >= kHalfCountMin;
    if (fp8) {
        if (half) MOE_FUSED_RUN(true, kCountHalf);
        MOE_FUSED_RUN(true, kCountInt);
    }
    if (half) MOE_FUSED_RUN(false, kCountHalf);
    MOE_FUSED_RUN(false, kCountInt);
#undef MOE_FUSED_RUN
}

cudaError_t launch_layout_dispatch_fused_bulk(const int32_t *topk_ids, const void *tokens,
                                              int T, int H, int K, int E, int R, int fp8,
                                              int32_t *expert_counts, int32_t *expert_offsets,
                                              int32_t *rank_offsets, int32_t *src_token,
                                              int32_t *dst_row, uint32_t *dev_error,
                                              void *packed, float *scales, cudaStream_t stream)
{
    const FusedPlan p = plan_fused(T, H, K, fp8 != 0);
    // the staged form copies one slice per block out of a kThreads-piece stage
    if (!p.use || K != 8 || p.upc > kThreads) return cudaErrorInvalidValue;
    const bool half = (long long)T * K >= kHalfCountMin;
#define MOE_BULK_RUN(F, M)                                                                   \
    return run_fused<8, F, M, true>(p, topk_ids, tokens, T, H, K, E, R, expert_counts,        \
                                    expert_offsets, rank_offsets, src_token, dst_row, dev_error, \
                                    packed, scales, stream)
    if (fp8) {
        if (half) MOE_BULK_RUN(true, kCountHalf);
        MOE_BULK_RUN(true, kCountInt);
    }
    if (half) MOE_BULK_RUN(false, kCountHalf);
    MOE_BULK_RUN(false, kCountInt);
#undef MOE_BULK_RUN
}

cudaError_t launch_layout_dispatch(const int32_t *topk_ids, const void *tokens,
                                   int T, int H, int K, int E, int R, int fp8,
                                   int32_t *expert_counts, int32_t *expert_offsets,
                                   int32_t *rank_offsets, int32_t *src_token,
                                   int32_t *dst_row, uint32_t *dev_error,
                                   void *packed, float *scales, void *workspace,
                                   cudaStream_t stream)
{
    // (the cluster form, layout_dispatch_cluster.cu, measured slower at every
    // decode shape and is reachable only through the test hook below)
    if (plan_fused(T, H, K, fp8 != 0).use)
        return launch_layout_dispatch_fused(topk_ids, tokens, T, H, K, E, R, fp8, expert_counts,
                                            expert_offsets, rank_offsets, src_token, dst_row,
                                            dev_error, packed, scales, stream);
    if (layout_dispatch_prefill(T, H, K, E, fp8))
        return launch_layout_dispatch_prefill(topk_ids, tokens, T, H, K, E, R, fp8,
                                              expert_counts, expert_offsets, rank_offsets,
                                              src_token, dst_row, dev_error, packed, scales,
                                              workspace, 0, -1, stream);
    cudaError_t e = launch_layout(topk_ids, T, K, E, R, expert_counts, expert_offsets,
                                  rank_offsets, src_token, dst_row, dev_error,
                                  workspace, stream);
    if (e != cudaSuccess || T == 0) return e;
    if (fp8) return launch_dispatch_fp8(tokens, T, H, K, dst_row, packed, scales, stream);
    return launch_dispatch_bf16(tokens, T, H, K, dst_row, packed, stream);
}

}  // namespace moe

// Test hook, deliberately absent from the public header: moe_layout_dispatch
// for a decode batch in a chosen form (0: every block counts all ids, the
// form the library uses; 1: the cluster form; 2: form 0 writing its rows by
// bulk copies out of shared memory, K = 8 only), for comparisons.
// Arguments are checked by the caller (tests only).
extern "C" __attribute__((visibility("default"))) int32_t
moe_testing_layout_dispatch_decode(const int32_t *topk_ids, const void *tokens, int32_t T,
                                   int32_t H, int32_t K, int32_t E, int32_t R, int32_t fp8,
                                   int32_t *expert_counts, int32_t *expert_offsets,
                                   int32_t *rank_offsets, int32_t *src_token, int32_t *dst_row,
                                   uint32_t *dev_error, void *packed, float *scales,
                                   int32_t variant, cudaStream_t stream)
{
    cudaError_t e;
    if (variant == 2) {
        if (!moe::layout_dispatch_fused(T, H, K, fp8) || K != 8) return MOE_ERR_INVALID_ARG;
        e = moe::launch_layout_dispatch_fused_bulk(topk_ids, tokens, T, H, K, E, R, fp8,
                                                   expert_counts, expert_offsets, rank_offsets,
                                                   src_token, dst_row, dev_error, packed, scales,
                                                   stream);
    } else if (variant == 1) {
        if (!moe::layout_dispatch_clustered(T, H, K, E, fp8)) return MOE_ERR_INVALID_ARG;
        e = moe::launch_layout_dispatch_cluster(topk_ids, tokens, T, H, K, E, R, fp8,
                                                expert_counts, expert_offsets, rank_offsets,
                                                src_token, dst_row, dev_error, packed, scales,
                                                stream);
    } else {
        if (!moe::layout_dispatch_fused(T, H, K, fp8)) return MOE_ERR_INVALID_ARG;
        e = moe::launch_layout_dispatch_fused(topk_ids, tokens, T, H, K, E, R, fp8,
                                              expert_counts, expert_offsets, rank_offsets,
                                              src_token, dst_row, dev_error, packed, scales,
                                              stream);
    }
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
