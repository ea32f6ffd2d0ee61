// layout_common.cuh -- block-level pieces of the layout kernels: the
// per-expert block scan, per-warp stable counting and duplicate detection.
#pragma once

#include "common.cuh"
#include "moe_layout.h"

namespace moe {

// Exclusive scan of hist[0..E) into off[0..E] (off[E] = total) by a block
// of kBlock threads, MOE_MAX_EXPERTS / kBlock experts per thread, warp
// shuffles inside warps.  All threads must call; ends with a barrier.
template <int kBlock>
__device__ __forceinline__ void scan_experts(const int32_t *hist, int32_t *off,
                                             int E, int32_t *warp_sums)
{
    static_assert(kBlock % 32 == 0 && kBlock <= 1024, "block size");
    constexpr int kPer = (MOE_MAX_EXPERTS + kBlock - 1) / kBlock;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    int v[kPer];
    int s = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = tid * kPer + j;
        v[j] = e < E ? hist[e] : 0;
        s += v[j];
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
        int q = lane < kBlock / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(kFullMask, q, d);
            if (lane >= d) q += y;
        }
        if (lane < kBlock / 32) warp_sums[lane] = q;
    }
    __syncthreads();
    int run = (w ? warp_sums[w - 1] : 0) + x - s;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = tid * kPer + j;
        if (e < E) off[e] = run;
        run += v[j];
    }
    if (tid == 0) off[E] = warp_sums[kBlock / 32 - 1];
    __syncthreads();
}

// The share [lo, hi) of warp w among kWarps warps splitting n entries:
// contiguous and 32-aligned, in entry order.
template <int kWarps>
__device__ __forceinline__ void warp_segment(int n, int w, int &lo, int &hi)
{
    const int seg = ((n + kWarps - 1) / kWarps + 31) & ~31;
    lo = min(n, w * seg);
    hi = min(n, lo + seg);
}

// Bits that tell the ids 0 .. E-1 apart.
__device__ __forceinline__ int id_bits(int E) { return 32 - __clz(E > 1 ? E - 1 : 1); }

// The lanes of this warp whose valid id equals this lane's (0 for an invalid
// id).  kBallot: from one ballot per id bit -- a lane stays in the set while
// it agrees with this lane on every bit -- which measured faster in the
// single-kernel layout; otherwise the warp match instruction, faster in the
// ranking kernel of the multi-kernel layout.  Every lane of the warp must
// call.
template <bool kBallot>
__device__ __forceinline__ unsigned match_ids(int id, bool ok, int bits, int lane)
{
    if (!kBallot) {
        const unsigned m = __match_any_sync(kFullMask, ok ? id : -1 - lane);
        return ok ? m : 0u;
    }
    unsigned m = __ballot_sync(kFullMask, ok);
    for (int b = 0; b < bits; ++b) {
        const bool set = (id >> b) & 1;
        const unsigned v = __ballot_sync(kFullMask, set);
        m &= set ? v : ~v;
    }
    return ok ? m : 0u;
}

// Adds the valid ids of ids[lo, hi) to this warp's private counter row:
// one add per distinct id of each 32-entry batch.
template <bool kBallot>
__device__ __forceinline__ void warp_count(const int32_t *ids, int lo, int hi,
                                           int E, int lane, int32_t *row)
{
    const int bits = id_bits(E);
    for (int b = lo; b < hi; b += 32) {
        const int i = b + lane;
        const int id = i < hi ? ids[i] : -1;
        const bool ok = (unsigned)id < (unsigned)E;
        const unsigned m = match_ids<kBallot>(id, ok, bits, lane);
        if (ok && lane == 31 - __clz(m)) row[id] += __popc(m);
    }
}

// Gives every valid entry of ids[lo, hi) its slot: the warp's running
// counter of its id plus the number of lower lanes holding the same id;
// the highest such lane then advances the counter.  Writes dst_row[first +
// i] and src_token[slot]; an invalid id gets dst_row -1.  With slots_out,
// slot i also goes to slots_out[i].
template <bool kBallot>
__device__ __forceinline__ void warp_rank(const int32_t *ids, int lo, int hi, int E,
                                          int K, int first, int lane, int32_t *row,
                                          int32_t *dst_row, int32_t *src_token,
                                          int32_t *slots_out = nullptr)
{
    const int bits = id_bits(E);
    for (int b = lo; b < hi; b += 32) {
        const int i = b + lane;
        const bool valid = i < hi;
        const int id = valid ? ids[i] : -1;
        const bool ok = (unsigned)id < (unsigned)E;
        const unsigned m = match_ids<kBallot>(id, ok, bits, lane);
        if (ok) {
            const int slot = row[id] + __popc(m & ((1u << lane) - 1u));
            dst_row[first + i] = slot;
            src_token[slot] = (first + i) / K;
            if (slots_out) slots_out[i] = slot;
        } else if (valid) {
            dst_row[first + i] = -1;
            if (slots_out) slots_out[i] = -1;
        }
        __syncwarp();
        if (ok && lane == 31 - __clz(m)) row[id] += __popc(m);
        __syncwarp();
    }
}

// Error bits of tokens [0, ntok) whose K ids start at ids (any memory):
// an id outside [0,E), or one valid id listed twice.
__device__ __forceinline__ uint32_t token_errors(const int32_t *ids, int ntok, int K,
                                                 int E)
{
    uint32_t err = 0;
    for (int t = threadIdx.x; t < ntok; t += blockDim.x) {
        const int32_t *row = ids + (size_t)t * K;
        for (int a = 0; a < K; ++a) {
            const int ea = row[a];
            if ((unsigned)ea >= (unsigned)E) {
                err |= MOE_DEV_ERR_EXPERT_RANGE;
                continue;
            }
            for (int b = a + 1; b < K; ++b)
                if (row[b] == ea) err |= MOE_DEV_ERR_DUPLICATE;
        }
    }
    return err;
}

}  // namespace moe
