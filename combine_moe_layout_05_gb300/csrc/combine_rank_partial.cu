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

// lo += f32(low bf16 of h), hi += f32(high bf16 of h), each an IEEE fp32 add
// rounded to nearest even: the mixed-precision add widens the bf16 operand
// exactly, so this equals __fadd_rn on the widened value, in one instruction.
__device__ __forceinline__ void add_bf16x2_rn(float &lo, float &hi, uint32_t h)
{
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, u, %1;\n\t}"
        : "+f"(lo), "+f"(hi) : "r"(h));
}

// Every warp orders the token's valid entries by (rank, k) itself, with no
// shared memory and no barrier: lane k (< K) loads entry k's slot, expert and
// weight, its position in that order is the number of lanes with a smaller
// key (rank << 5 | k), and a lane whose rank no higher lane shares ends its
// rank's group.  Lane p then fetches the slot and weight of the entry at
// position p, so each position costs two shuffles later.  The order is the
// same for every warp of the block (one token), so every loop below is
// warp-uniform.  Each thread gathers its 8 values of every entry in that
// order and makes a single pass: fused multiply-adds into the group's
// partial, and at each group's end the partial rounded to bf16 (two values
// per conversion) is added into the fp32 total with a mixed bf16 + fp32
// add.  Up to KT (or kBatch) gathers are in flight before any arithmetic.
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
#pragma unroll
    for (int j = 0; j < (KT > 0 ? KT : MOE_MAX_TOPK); ++j)
        if (KT > 0 || j < k_count) pos += __shfl_sync(kFullMask, key, j) < key;
    const int n = __popc(__ballot_sync(kFullMask, valid));
    const uint32_t same = __match_any_sync(kFullMask, group);
    const bool ends = valid && (same & ~((2u << lane) - 1u)) == 0u;
    const uint32_t last = __reduce_or_sync(kFullMask, ends ? 1u << pos : 0u);
    // lane p <- the entry at position p (lanes p >= n keep lane 0's, unused)
    const int at = valid ? pos : -1;
    int src = 0;
#pragma unroll
    for (int j = 0; j < (KT > 0 ? KT : MOE_MAX_TOPK); ++j)
        if (KT > 0 || j < k_count) src = __shfl_sync(kFullMask, at, j) == lane ? j : src;
    const int row_p = __shfl_sync(kFullMask, row, src);
    const float wt_p = __shfl_sync(kFullMask, wt, src);

    float total[8], part[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) total[j] = part[j] = 0.0f;
    constexpr int B = KT > 0 ? KT : kBatch;
    for (int p0 = 0; p0 < n; p0 += B) {
        uint4 val[B];
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const int p = p0 + i;
            const int r = __shfl_sync(kFullMask, row_p, p & 31);
            val[i] = (p < n && active) ? ld_stream_v4(y + (size_t)r * vpr + v)
                                       : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const int p = p0 + i;
            if (p < n) {                    // warp-uniform
                fma8(part, __shfl_sync(kFullMask, wt_p, p & 31), val[i]);
                if ((last >> p) & 1u) {
#pragma unroll
                    for (int j = 0; j < 8; j += 2) {
                        add_bf16x2_rn(total[j], total[j + 1],
                                      pack_bf16x2_rn(part[j], part[j + 1]));
                        part[j] = part[j + 1] = 0.0f;
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
