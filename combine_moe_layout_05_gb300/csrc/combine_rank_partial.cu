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

__device__ __forceinline__ void fma4(float acc[4], float w, const uint2 &y)
{
    acc[0] = __fmaf_rn(w, bf16_lo(y.x), acc[0]);
    acc[1] = __fmaf_rn(w, bf16_hi(y.x), acc[1]);
    acc[2] = __fmaf_rn(w, bf16_lo(y.y), acc[2]);
    acc[3] = __fmaf_rn(w, bf16_hi(y.y), acc[3]);
}

// A thread owns 4 hidden values (8 bytes): the per-rank pass keeps all K
// gathered pieces, one partial and one total live, which fits the register
// budget of a fully occupied SM.  KT > 0: every gather is issued before any
// arithmetic; a runtime K loads inside the rank loop.
template <int KT>
__global__ void __launch_bounds__(256)
combine_rank_partial_kernel(const uint2 *__restrict__ y, const float *__restrict__ weights,
                            const int32_t *__restrict__ ids, const int32_t *__restrict__ dst_row,
                            int K, int vpr, int rows, int E, int epr, uint2 *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int v = blockIdx.y * blockDim.x + threadIdx.x;
    if (v >= vpr) return;
    const int k_count = KT > 0 ? KT : K;
    const int32_t *d = dst_row + (size_t)t * k_count;
    const int32_t *ex = ids + (size_t)t * k_count;
    const float *wt = weights + (size_t)t * k_count;

    // rank of each entry (-1 when its expert or slot is invalid)
    auto rank_of = [&](int k, int &r) {
        r = __ldg(d + k);
        const int e = __ldg(ex + k);
        const bool ok = (unsigned)r < (unsigned)rows && (unsigned)e < (unsigned)E;
        return ok ? e / epr : -1;
    };
    float total[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    auto flush = [&](const float part[4]) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            total[j] = __fadd_rn(total[j], __bfloat162float(__float2bfloat16_rn(part[j])));
    };

    if constexpr (KT > 0) {
        int rk[KT], row[KT];
        float wk[KT];
        uint2 val[KT];
#pragma unroll
        for (int k = 0; k < KT; ++k) {
            rk[k] = rank_of(k, row[k]);
            wk[k] = __ldg(wt + k);
            val[k] = rk[k] >= 0 ? ld_stream_v2(y + (size_t)row[k] * vpr + v) : make_uint2(0, 0);
        }
        int prev = -1;
        for (;;) {
            int cur = 0x7fffffff;
#pragma unroll
            for (int k = 0; k < KT; ++k)
                if (rk[k] > prev && rk[k] < cur) cur = rk[k];
            if (cur == 0x7fffffff) break;
            float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int k = 0; k < KT; ++k)
                if (rk[k] == cur) fma4(part, wk[k], val[k]);
            flush(part);
            prev = cur;
        }
    } else {
        int prev = -1;
        for (;;) {
            int cur = 0x7fffffff, row;
            for (int k = 0; k < k_count; ++k) {
                const int r = rank_of(k, row);
                if (r > prev && r < cur) cur = r;
            }
            if (cur == 0x7fffffff) break;
            float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int k = 0; k < k_count; ++k)
                if (rank_of(k, row) == cur)
                    fma4(part, __ldg(wt + k), ld_stream_v2(y + (size_t)row * vpr + v));
            flush(part);
            prev = cur;
        }
    }
    uint2 o;
    o.x = pack_bf16x2_rn(total[0], total[1]);
    o.y = pack_bf16x2_rn(total[2], total[3]);
    st_v2(out + (size_t)t * vpr + v, o);
}

template <int KT>
cudaError_t run_rank_partial(const void *y, const float *w, const int32_t *ids,
                             const int32_t *dst_row, int T, int H, int K, int E, int R,
                             void *out, cudaStream_t s)
{
    const int vpr = H / 4;
    const int threads = pick_row_block(vpr);
    return launch_pdl(combine_rank_partial_kernel<KT>, dim3(T, ceil_div(vpr, threads)),
                      dim3(threads), 0, s, static_cast<const uint2 *>(y), w, ids, dst_row,
                      K, vpr, T * K, E, E / R, static_cast<uint2 *>(out));
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
