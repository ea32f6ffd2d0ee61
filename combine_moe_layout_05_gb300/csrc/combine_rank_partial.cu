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

// One thread per block orders the token's valid entries by (rank, k) in
// shared memory -- slot, weight, and a bit marking the last entry of each
// rank's group -- so every thread then gathers its 8 values per entry in that
// order and makes a single pass: fused multiply-adds into the group's
// partial, and at each group's end the partial rounded to bf16 is added into
// the fp32 total.  KT > 0: all gathers are issued before any arithmetic.
template <int KT>
__global__ void __launch_bounds__(256)
combine_rank_partial_kernel(const uint4 *__restrict__ y, const float *__restrict__ weights,
                            const int32_t *__restrict__ ids, const int32_t *__restrict__ dst_row,
                            int K, int vpr, int rows, int E, int epr, uint4 *__restrict__ out)
{
    __shared__ int32_t s_row[MOE_MAX_TOPK];
    __shared__ float s_w[MOE_MAX_TOPK];
    __shared__ uint32_t s_last;
    __shared__ int32_t s_n;
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int v = blockIdx.y * blockDim.x + threadIdx.x;
    const int k_count = KT > 0 ? KT : K;
    if (threadIdx.x == 0) {
        int key[MOE_MAX_TOPK];
        int n = 0;
        for (int k = 0; k < k_count; ++k) {
            const int r = __ldg(dst_row + (size_t)t * k_count + k);
            const int e = __ldg(ids + (size_t)t * k_count + k);
            if ((unsigned)r < (unsigned)rows && (unsigned)e < (unsigned)E)
                key[n++] = ((e / epr) << 5) | k;          // rank major, then k
        }
        for (int i = 1; i < n; ++i) {                     // insertion sort, n <= 32
            const int x = key[i];
            int j = i - 1;
            while (j >= 0 && key[j] > x) {
                key[j + 1] = key[j];
                --j;
            }
            key[j + 1] = x;
        }
        uint32_t last = 0;
        for (int i = 0; i < n; ++i) {
            const int k = key[i] & 31;
            s_row[i] = __ldg(dst_row + (size_t)t * k_count + k);
            s_w[i] = __ldg(weights + (size_t)t * k_count + k);
            if (i == n - 1 || (key[i] >> 5) != (key[i + 1] >> 5)) last |= 1u << i;
        }
        s_last = last;
        s_n = n;
    }
    __syncthreads();
    if (v >= vpr) return;
    const int n = s_n;
    const uint32_t last = s_last;

    float total[8], part[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) total[j] = part[j] = 0.0f;
    auto step = [&](int i, const uint4 &val) {
        fma8(part, s_w[i], val);
        if ((last >> i) & 1u) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                total[j] = __fadd_rn(total[j], __bfloat162float(__float2bfloat16_rn(part[j])));
                part[j] = 0.0f;
            }
        }
    };
    constexpr int B = KT > 0 ? KT : kBatch;
    for (int i0 = 0; i0 < n; i0 += B) {
        uint4 val[B];
#pragma unroll
        for (int i = 0; i < B; ++i)
            val[i] = i0 + i < n ? ld_stream_v4(y + (size_t)s_row[i0 + i] * vpr + v)
                                : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < B; ++i)
            if (i0 + i < n) step(i0 + i, val[i]);
    }
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
