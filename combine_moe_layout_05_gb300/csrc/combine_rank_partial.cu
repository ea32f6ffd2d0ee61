// combine_rank_partial.cu -- combine with sender-side per-rank partial sums.
//
// Perplexity, "Enabling trillion-parameter models on AWS EFA", section
// "Evaluation": the page accumulates only on the receiving side and
// contrasts this with DeepEP, which sums in the sender to cut the bytes
// transferred, at some cost in accuracy.  This kernel computes that scheme:
// each token's entries are grouped by destination rank r = e / (E/R); each
// group is an fp32 FMA chain in k order from +0 rounded to bf16 (the
// transfer format), and the groups are added as fp32 in ascending rank order
// from +0, then rounded to bf16.
#include "combine_common.cuh"
#include "common.cuh"
#include "internal.h"
#include "moe_layout.h"

namespace moe {
namespace {

// Every warp orders the token's valid entries by (rank, k) itself, with no
// shared memory and no barrier: lane k (< K) loads entry k's slot, expert and
// weight, its position in that order is the number of lanes with a smaller
// key (rank << 5 | k), and a lane whose rank no higher lane shares ends its
// rank's group.  The order is the same for every warp of the block (one
// token), so every loop below is warp-uniform.  Each thread then gathers its
// 8 values of every entry in that order -- the source lane of position p is
// found with a ballot and the slot and weight are shuffled from it -- and
// makes a single pass: fused multiply-adds into the group's partial, and at
// each group's end the partial rounded to bf16 is added into the fp32 total.
// Up to KT (or kBatch) gathers are in flight before any arithmetic.
template <int KT>
__global__ void __launch_bounds__(256, 4)   // 4 blocks per SM: the decode grid in one wave
combine_rank_partial_kernel(const uint4 *__restrict__ y, const float *__restrict__ weights,
                            const int32_t *__restrict__ ids, const int32_t *__restrict__ dst_row,
                            int K, int vpr, int rows, int E, int epr, uint4 *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int v = blockIdx.y * blockDim.x + threadIdx.x;
    const bool active = v < vpr;            // inactive lanes still take part in the collectives
    const int lane = threadIdx.x & 31;
    const int k_count = KT > 0 ? KT : K;

    int row = 0, key = 0x7fffffff, group = 0x40000000 | lane;
    float wt = 0.0f;
    bool valid = false;
    if (lane < k_count) {
        row = __ldg(dst_row + (size_t)t * k_count + lane);
        const int e = __ldg(ids + (size_t)t * k_count + lane);
        wt = __ldg(weights + (size_t)t * k_count + lane);
        valid = (unsigned)row < (unsigned)rows && (unsigned)e < (unsigned)E;
        if (valid) {
            group = e / epr;
            key = (group << 5) | lane;      // rank major, then k
        }
    }
    int pos = 0;
    if (KT > 0) {
#pragma unroll
        for (int j = 0; j < (KT > 0 ? KT : 1); ++j) pos += __shfl_sync(kFullMask, key, j) < key;
    } else {
        for (int j = 0; j < k_count; ++j) pos += __shfl_sync(kFullMask, key, j) < key;
    }
    const uint32_t valid_mask = __ballot_sync(kFullMask, valid);
    const int n = __popc(valid_mask);
    const uint32_t same = __match_any_sync(kFullMask, group);
    const bool ends = valid && (same & ~((2u << lane) - 1u)) == 0u;
    const uint32_t last = __reduce_or_sync(kFullMask, ends ? 1u << pos : 0u);

    float total[8], part[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) total[j] = part[j] = 0.0f;
    constexpr int B = KT > 0 ? KT : kBatch;
    // source lane of position p (0 when p >= n)
    auto lane_of = [&](int p) {
        const uint32_t at = __ballot_sync(kFullMask, valid && pos == p);
        return at ? __ffs(at) - 1 : 0;
    };
    for (int p0 = 0; p0 < n; p0 += B) {
        uint4 val[B];
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const int p = p0 + i;
            const int r = __shfl_sync(kFullMask, row, lane_of(p));
            val[i] = (p < n && active) ? ld_stream_v4(y + (size_t)r * vpr + v)
                                       : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const int p = p0 + i;
            if (p < n) {                    // warp-uniform
                fma8(part, __shfl_sync(kFullMask, wt, lane_of(p)), val[i]);
                if ((last >> p) & 1u) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        total[j] = __fadd_rn(total[j],
                                             __bfloat162float(__float2bfloat16_rn(part[j])));
                        part[j] = 0.0f;
                    }
                }
            }
        }
    }
    if (!active) return;
    uint4 o;
    o.x = pack_bf16x2_rn(total[0], total[1]);
    o.y = pack_bf16x2_rn(total[2], total[3]);
    o.z = pack_bf16x2_rn(total[4], total[5]);
    o.w = pack_bf16x2_rn(total[6], total[7]);
    st_v4(out + (size_t)t * vpr + v, o);
}

template <int KT>
cudaError_t run_rank_partial(const void *y, const float *w, const int32_t *ids,
                             const int32_t *dst_row, int T, int H, int K, int E, int R,
                             void *out, cudaStream_t s)
{
    const int vpr = H / 8;
    const int threads = pick_row_block(vpr);
    return launch_pdl(combine_rank_partial_kernel<KT>, dim3(T, ceil_div(vpr, threads)),
                      dim3(threads), 0, s, static_cast<const uint4 *>(y), w, ids, dst_row,
                      K, vpr, T * K, E, E / R, static_cast<uint4 *>(out));
}

}  // namespace

cudaError_t launch_combine_rank_partial(const void *expert_out, const float *topk_weights,
                                        const int32_t *topk_ids, const int32_t *dst_row,
                                        int T, int H, int K, int E, int R, void *out,
                                        cudaStream_t stream)
{
#define MOE_RP_CASE(KV) \
    return run_rank_partial<KV>(expert_out, topk_weights, topk_ids, dst_row, T, H, K, E, R, out, stream)
    switch (K) {
    case 1: MOE_RP_CASE(1);
    case 2: MOE_RP_CASE(2);
    case 4: MOE_RP_CASE(4);
    case 6: MOE_RP_CASE(6);
    case 8: MOE_RP_CASE(8);
    default: MOE_RP_CASE(0);
    }
#undef MOE_RP_CASE
}

}  // namespace moe
