// combine.cu -- routing-weighted sum of each token's K expert outputs.
//
// Perplexity, "Enabling trillion-parameter models on AWS EFA": combine
// receives the processed rows of each token and forms their weighted average
// ("MoE all-to-all over EFA", "Dispatch and Combine"); the accumulation is
// done on the receiving side only ("Evaluation").  With normalised router
// weights the weighted sum is that average; nothing is divided.
//
// acc = +0; acc = fma(w[t,k], y[dst_row[t,k], j], acc) for k = 0..K-1 in
// order (fp32, round to nearest); out[t, j] = bf16 round-to-nearest-even.
//
// HBM-bound gather.  A block covers one token and a slice of its row; each
// thread owns 8 hidden values (one 16-byte vector), issues all K gathers of
// its vector before using any of them, then runs the fused multiply-add
// chain and writes one 16-byte vector.  A warp's K loads each cover 512
// contiguous bytes of one expert-output row.
#include "combine_common.cuh"
#include "common.cuh"
#include "internal.h"
#include "moe_layout.h"

namespace moe {
namespace {

// KT > 0 is a compile-time K; otherwise up to kBatch gathers are in flight.
template <int KT>
__global__ void __launch_bounds__(256)
combine_kernel(const uint4 *__restrict__ y, const float *__restrict__ weights,
               const int32_t *__restrict__ dst_row, int K, int vpr, int rows,
               uint4 *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int v = blockIdx.y * blockDim.x + threadIdx.x;
    if (v >= vpr) return;
    const int k_count = KT > 0 ? KT : K;
    const int32_t *d = dst_row + (size_t)t * k_count;
    const float *wt = weights + (size_t)t * k_count;

    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;

    constexpr int B = KT > 0 ? KT : kBatch;
    for (int k0 = 0; k0 < k_count; k0 += B) {
        uint4 val[B];
        float wk[B];
        bool ok[B];
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const int k = k0 + i;
            const int r = k < k_count ? __ldg(d + k) : -1;
            ok[i] = (unsigned)r < (unsigned)rows;
            wk[i] = k < k_count ? __ldg(wt + k) : 0.0f;
            val[i] = ok[i] ? ld_stream_v4(y + (size_t)r * vpr + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < B; ++i)
            if (ok[i]) fma8(acc, wk[i], val[i]);
    }
    uint4 o;
    o.x = pack_bf16x2_rn(acc[0], acc[1]);
    o.y = pack_bf16x2_rn(acc[2], acc[3]);
    o.z = pack_bf16x2_rn(acc[4], acc[5]);
    o.w = pack_bf16x2_rn(acc[6], acc[7]);
    st_v4(out + (size_t)t * vpr + v, o);
}

template <int KT>
cudaError_t run_combine(const void *y, const float *w, const int32_t *dst_row,
                        int T, int H, int K, void *out, cudaStream_t s)
{
    const int vpr = H / 8;
    const int threads = pick_row_block(vpr);
    return launch_pdl(combine_kernel<KT>, dim3(T, ceil_div(vpr, threads)),
                      dim3(threads), 0, s, static_cast<const uint4 *>(y), w,
                      dst_row, K, vpr, T * K, static_cast<uint4 *>(out));
}

}  // namespace

cudaError_t launch_combine(const void *expert_out, const float *topk_weights,
                           const int32_t *dst_row, int T, int H, int K,
                           void *out, cudaStream_t stream)
{
    switch (K) {
    case 1: return run_combine<1>(expert_out, topk_weights, dst_row, T, H, K, out, stream);
    case 2: return run_combine<2>(expert_out, topk_weights, dst_row, T, H, K, out, stream);
    case 4: return run_combine<4>(expert_out, topk_weights, dst_row, T, H, K, out, stream);
    case 6: return run_combine<6>(expert_out, topk_weights, dst_row, T, H, K, out, stream);
    case 8: return run_combine<8>(expert_out, topk_weights, dst_row, T, H, K, out, stream);
    default: return run_combine<0>(expert_out, topk_weights, dst_row, T, H, K, out, stream);
    }
}

}  // namespace moe
