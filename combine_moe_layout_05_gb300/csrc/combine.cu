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
// HBM-bound gather.  A block of kRowThreads threads covers kRowThreads
// consecutive 16-byte pieces of the flat sequence of all output rows (so it
// may span a row boundary); each thread owns 8 hidden values (one 16-byte
// vector), issues all K gathers of its vector before using any of them,
// then runs the fused multiply-add chain and writes one 16-byte vector.  A
// warp's K loads each cover up to 512 contiguous bytes of one expert-output
// row.
#include "combine_common.cuh"
#include "common.cuh"
#include "internal.h"
#include "moe_layout.h"
#include "rowops.cuh"

namespace moe {
namespace {

// KT > 0 is a compile-time K; otherwise up to kBatch gathers are in flight.
// kShfl (KT <= 32 only): lanes 0 .. K-1 of each warp load the token's slots
// and weights (one coalesced request each) and shuffles hand them to the
// warp, instead of every thread loading all K of each (a form kept for
// comparison, reachable only through the test hook below).
// kFlat: blocks walk flat pieces (grid row_blocks(T, vpr)); otherwise one
// token per block (grid T x row slices), which the shuffle form needs.
template <int KT, bool kFlat, bool kShfl = false>
__global__ void __launch_bounds__(256)
combine_kernel(const uint4 *__restrict__ y, const float *__restrict__ weights,
               const int32_t *__restrict__ dst_row, int T, int K, int vpr, int rows,
               uint4 *__restrict__ out)
{
    static_assert(!(kFlat && kShfl), "the shuffle form takes one token per block");
    pdl_wait();
    pdl_trigger();
    int t, v;
    if (!kFlat) {
        t = blockIdx.x;
        v = blockIdx.y * blockDim.x + threadIdx.x;
    } else {
        const RowPiece rp = flat_piece(blockIdx.x, vpr, threadIdx.x);
        if (rp.t >= T) return;
        t = rp.t;
        v = rp.u;
    }
    const int k_count = KT > 0 ? KT : K;
    const int32_t *d = dst_row + (size_t)t * k_count;
    const float *wt = weights + (size_t)t * k_count;

    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;

    if (kShfl) {
        static_assert(!kShfl || (KT > 0 && KT <= 32), "the shuffle form takes a compile-time K <= 32");
        const int lane = threadIdx.x & 31;
        const int my_r = lane < KT ? __ldg(d + lane) : -1;
        const float my_w = lane < KT ? __ldg(wt + lane) : 0.0f;
        uint4 val[KT > 0 ? KT : 1];
        float wk[KT > 0 ? KT : 1];
        bool ok[KT > 0 ? KT : 1];
#pragma unroll
        for (int i = 0; i < KT; ++i) {
            const int r = __shfl_sync(kFullMask, my_r, i);
            wk[i] = __shfl_sync(kFullMask, my_w, i);
            ok[i] = (unsigned)r < (unsigned)rows && v < vpr;
            val[i] = ok[i] ? ld_stream_v4(y + (size_t)r * vpr + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < KT; ++i)
            if (ok[i]) fma8(acc, wk[i], val[i]);
        if (v >= vpr) return;
        uint4 o;
        o.x = pack_bf16x2_rn(acc[0], acc[1]);
        o.y = pack_bf16x2_rn(acc[2], acc[3]);
        o.z = pack_bf16x2_rn(acc[4], acc[5]);
        o.w = pack_bf16x2_rn(acc[6], acc[7]);
        st_v4(out + (size_t)t * vpr + v, o);
        return;
    }
    if (v >= vpr) return;

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
    if (flat_rows(T, vpr)) {
        const unsigned blocks = row_blocks(T, vpr);
        if (blocks == 0) return cudaErrorInvalidValue;
        return launch_pdl(combine_kernel<KT, true>, dim3(blocks), dim3(kRowThreads), 0, s,
                          static_cast<const uint4 *>(y), w, dst_row, T, K, vpr, T * K,
                          static_cast<uint4 *>(out));
    }
    const int threads = pick_row_block(vpr);
    return launch_pdl(combine_kernel<KT, false>, dim3(T, ceil_div(vpr, threads)), dim3(threads),
                      0, s, static_cast<const uint4 *>(y), w, dst_row, T, K, vpr, T * K,
                      static_cast<uint4 *>(out));
}

}  // namespace

cudaError_t launch_combine_shfl(const void *expert_out, const float *topk_weights,
                                const int32_t *dst_row, int T, int H, int K, void *out,
                                cudaStream_t stream)
{
    if (K != 8) return cudaErrorInvalidValue;
    const int vpr = H / 8;
    const int threads = pick_row_block(vpr);
    return launch_pdl(combine_kernel<8, false, true>, dim3(T, ceil_div(vpr, threads)), dim3(threads), 0,
                      stream, static_cast<const uint4 *>(expert_out), topk_weights, dst_row, T,
                      K, vpr, T * K, static_cast<uint4 *>(out));
}

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

// Test hook, deliberately absent from the public header: moe_combine in the
// form whose lanes 0 .. 7 load the token's slots and weights and shuffle them
// to the warp (K = 8 only), for comparison with the library's form.
// Arguments are checked by the caller (tests only).
extern "C" __attribute__((visibility("default"))) int32_t
moe_testing_combine_shfl(const void *expert_out, const float *topk_weights,
                         const int32_t *dst_row, int32_t T, int32_t H, int32_t K, void *out,
                         cudaStream_t stream)
{
    if (K != 8 || T <= 0 || H % 8 != 0) return MOE_ERR_INVALID_ARG;
    const cudaError_t e = moe::launch_combine_shfl(expert_out, topk_weights, dst_row, T, H, K,
                                                   out, stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
