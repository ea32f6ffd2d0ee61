// dispatch.cu -- pack each token row into its K slots (bf16 copy or
// block-scaled e4m3).
//
// Perplexity, "Enabling trillion-parameter models on AWS EFA": the dispatch
// sender shuffles the tokens into contiguous send buffers, one write per
// destination ("Dispatch and Combine"); the evaluated setting quantises the
// dispatched payload to block-scaled FP8 ("Evaluation").  On one GPU the
// packed buffer is both the send buffer and the grouped-GEMM input, so the
// receive-side copy disappears.
//
// Both kernels are HBM-bound copies.  A block covers one token and a slice
// of its row; each thread reads its 16-byte piece once (read-only path, no
// L1 allocation), keeps it in registers and writes it to all K slots.  A
// warp's stores to one slot cover 512 contiguous bytes, so every write is
// fully coalesced.  The FP8 kernel gives 8 consecutive threads one 1x128
// block (16 values each), see rowops.cuh.
#include "common.cuh"
#include "internal.h"
#include "moe_layout.h"
#include "rowops.cuh"

namespace moe {
namespace {

// KT > 0: K known at compile time (fully unrolled); KT == 0: runtime K.
template <int KT>
__global__ void __launch_bounds__(256)
dispatch_bf16_kernel(const uint4 *__restrict__ tokens, int K, int vpr,
                     const int32_t *__restrict__ dst_row, int rows,
                     uint4 *__restrict__ packed)
{
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int v = blockIdx.y * blockDim.x + threadIdx.x;
    if (v >= vpr) return;
    const int k_count = KT > 0 ? KT : K;
    const uint4 x = ld_stream_v4(tokens + (size_t)t * vpr + v);
    store_to_slots<KT>(dst_row + (size_t)t * k_count, k_count, rows,
                       reinterpret_cast<uint8_t *>(packed), (size_t)vpr * 16,
                       (size_t)v * 16, x);
}

template <int KT>
__global__ void __launch_bounds__(256)
dispatch_fp8_kernel(const uint4 *__restrict__ tokens, int K, int H,
                    const int32_t *__restrict__ dst_row, int rows,
                    uint8_t *__restrict__ packed, float *__restrict__ scales)
{
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int g = blockIdx.y * blockDim.x + threadIdx.x;   // 16-value group
    const bool active = g < (H >> 4);
    const int k_count = KT > 0 ? KT : K;
    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
    if (active) {
        const uint4 *src = tokens + (size_t)t * (H >> 3) + 2 * g;
        a = ld_stream_v4(src);
        b = ld_stream_v4(src + 1);
    }
    // groups per row is a multiple of 8 and blocks start at multiples of 32
    // threads, so the 8 lanes of a 128-value block are always together.
    const Fp8Piece p = quantize16(a, b);
    if (!active) return;
    store_fp8_to_slots<KT>(dst_row + (size_t)t * k_count, k_count, rows, packed,
                           scales, H, g, p);
}

template <int KT>
cudaError_t run_bf16(const void *tokens, int T, int H, int K,
                     const int32_t *dst_row, void *packed, cudaStream_t s)
{
    const int vpr = H / 8;
    const int threads = pick_row_block(vpr);
    return launch_pdl(dispatch_bf16_kernel<KT>, dim3(T, ceil_div(vpr, threads)),
                      dim3(threads), 0, s, static_cast<const uint4 *>(tokens), K,
                      vpr, dst_row, T * K, static_cast<uint4 *>(packed));
}

template <int KT>
cudaError_t run_fp8(const void *tokens, int T, int H, int K,
                    const int32_t *dst_row, void *packed, float *scales,
                    cudaStream_t s)
{
    const int groups = H / 16;
    const int threads = pick_row_block(groups);
    return launch_pdl(dispatch_fp8_kernel<KT>, dim3(T, ceil_div(groups, threads)),
                      dim3(threads), 0, s, static_cast<const uint4 *>(tokens), K,
                      H, dst_row, T * K, static_cast<uint8_t *>(packed), scales);
}

}  // namespace

int pick_row_block(int units)
{
    for (int b = 256; b >= 64; b -= 32)
        if (units % b == 0) return b;
    return units < 128 ? ((units + 31) / 32) * 32 : 128;
}

cudaError_t launch_dispatch_bf16(const void *tokens, int T, int H, int K,
                                 const int32_t *dst_row, void *packed,
                                 cudaStream_t stream)
{
    switch (K) {
    case 1: return run_bf16<1>(tokens, T, H, K, dst_row, packed, stream);
    case 2: return run_bf16<2>(tokens, T, H, K, dst_row, packed, stream);
    case 4: return run_bf16<4>(tokens, T, H, K, dst_row, packed, stream);
    case 6: return run_bf16<6>(tokens, T, H, K, dst_row, packed, stream);
    case 8: return run_bf16<8>(tokens, T, H, K, dst_row, packed, stream);
    default: return run_bf16<0>(tokens, T, H, K, dst_row, packed, stream);
    }
}

cudaError_t launch_dispatch_fp8(const void *tokens, int T, int H, int K,
                                const int32_t *dst_row, void *packed,
                                float *scales, cudaStream_t stream)
{
    switch (K) {
    case 1: return run_fp8<1>(tokens, T, H, K, dst_row, packed, scales, stream);
    case 2: return run_fp8<2>(tokens, T, H, K, dst_row, packed, scales, stream);
    case 4: return run_fp8<4>(tokens, T, H, K, dst_row, packed, scales, stream);
    case 6: return run_fp8<6>(tokens, T, H, K, dst_row, packed, scales, stream);
    case 8: return run_fp8<8>(tokens, T, H, K, dst_row, packed, scales, stream);
    default: return run_fp8<0>(tokens, T, H, K, dst_row, packed, scales, stream);
    }
}

}  // namespace moe
