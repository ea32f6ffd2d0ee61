// combine_fp8.cu -- combine reading block-scaled e4m3 expert outputs.
//
// Perplexity, "Enabling trillion-parameter models on AWS EFA", section
// "Evaluation": the evaluated setting dispatches block-scaled FP8.  When the
// expert outputs stay in that form (e4m3 codes and one fp32 scale per 1x128
// block), combine reads them directly: each value is f32(code) * scale
// (fp32, round to nearest; the code widens exactly through f16), then the
// same fp32 FMA chain in k order as the bf16 combine, rounded to bf16.  It
// moves about half the bytes of the bf16 combine.
#include "combine_common.cuh"
#include "common.cuh"
#include "internal.h"
#include "moe_layout.h"

namespace moe {
namespace {

// Combine from FP8 expert outputs: a thread owns 16 values of one 1x128
// block (one 16-byte vector of codes); per k it gathers the codes and the
// block's scale, issues every gather before using any, then for each value
// y = f32(code) * scale (fp32, round to nearest; the code widens exactly via
// f16) and acc = fma(w, y, acc) in k order; two 16-byte bf16 stores.
template <int KT>
__global__ void __launch_bounds__(256)
combine_fp8_kernel(const uint4 *__restrict__ codes, const float *__restrict__ scales,
                   const float *__restrict__ weights, const int32_t *__restrict__ dst_row,
                   int K, int H, int rows, uint4 *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int g = blockIdx.y * blockDim.x + threadIdx.x;   // 16-value group
    const int groups = H >> 4;
    if (g >= groups) return;
    const int k_count = KT > 0 ? KT : K;
    const int nb = H >> 7, blk = g >> 3;
    const int32_t *d = dst_row + (size_t)t * k_count;
    const float *wt = weights + (size_t)t * k_count;

    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.0f;

    constexpr int B = KT > 0 ? KT : kBatch;
    for (int k0 = 0; k0 < k_count; k0 += B) {
        uint4 q[B];
        float sc[B], wk[B];
        bool ok[B];
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const int k = k0 + i;
            const int r = k < k_count ? __ldg(d + k) : -1;
            ok[i] = (unsigned)r < (unsigned)rows;
            wk[i] = k < k_count ? __ldg(wt + k) : 0.0f;
            q[i] = ok[i] ? ld_stream_v4(codes + (size_t)r * groups + g) : make_uint4(0, 0, 0, 0);
            sc[i] = ok[i] ? __ldg(scales + (size_t)r * nb + blk) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < B; ++i) {
            if (!ok[i]) continue;
            const uint32_t wq[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float2 lo = e4m3x2_to_f32x2((uint16_t)(wq[m] & 0xffffu));
                const float2 hi = e4m3x2_to_f32x2((uint16_t)(wq[m] >> 16));
                acc[4 * m + 0] = __fmaf_rn(wk[i], __fmul_rn(lo.x, sc[i]), acc[4 * m + 0]);
                acc[4 * m + 1] = __fmaf_rn(wk[i], __fmul_rn(lo.y, sc[i]), acc[4 * m + 1]);
                acc[4 * m + 2] = __fmaf_rn(wk[i], __fmul_rn(hi.x, sc[i]), acc[4 * m + 2]);
                acc[4 * m + 3] = __fmaf_rn(wk[i], __fmul_rn(hi.y, sc[i]), acc[4 * m + 3]);
            }
        }
    }
    uint4 o0, o1;
    o0.x = pack_bf16x2_rn(acc[0], acc[1]);
    o0.y = pack_bf16x2_rn(acc[2], acc[3]);
    o0.z = pack_bf16x2_rn(acc[4], acc[5]);
    o0.w = pack_bf16x2_rn(acc[6], acc[7]);
    o1.x = pack_bf16x2_rn(acc[8], acc[9]);
    o1.y = pack_bf16x2_rn(acc[10], acc[11]);
    o1.z = pack_bf16x2_rn(acc[12], acc[13]);
    o1.w = pack_bf16x2_rn(acc[14], acc[15]);
    uint4 *dst = out + (size_t)t * (H >> 3) + 2 * g;
    st_v4(dst, o0);
    st_v4(dst + 1, o1);
}

template <int KT>
cudaError_t run_combine_fp8(const void *codes, const float *scales, const float *w,
                            const int32_t *dst_row, int T, int H, int K, void *out,
                            cudaStream_t s)
{
    const int groups = H / 16;
    const int threads = pick_row_block(groups);
    return launch_pdl(combine_fp8_kernel<KT>, dim3(T, ceil_div(groups, threads)),
                      dim3(threads), 0, s, static_cast<const uint4 *>(codes), scales, w,
                      dst_row, K, H, T * K, static_cast<uint4 *>(out));
}

}  // namespace

cudaError_t launch_combine_fp8(const void *codes, const float *scales,
                               const float *topk_weights, const int32_t *dst_row,
                               int T, int H, int K, void *out, cudaStream_t stream)
{
    switch (K) {
    case 1: return run_combine_fp8<1>(codes, scales, topk_weights, dst_row, T, H, K, out, stream);
    case 2: return run_combine_fp8<2>(codes, scales, topk_weights, dst_row, T, H, K, out, stream);
    case 4: return run_combine_fp8<4>(codes, scales, topk_weights, dst_row, T, H, K, out, stream);
    case 6: return run_combine_fp8<6>(codes, scales, topk_weights, dst_row, T, H, K, out, stream);
    case 8: return run_combine_fp8<8>(codes, scales, topk_weights, dst_row, T, H, K, out, stream);
    default: return run_combine_fp8<0>(codes, scales, topk_weights, dst_row, T, H, K, out, stream);
    }
}

}  // namespace moe
