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
// Both kernels are HBM-bound copies.  A block of kRowThreads threads covers
// kRowThreads consecutive 16-byte pieces of the flat sequence of all token
// rows (so it may span a row boundary); each thread reads its piece once
// (read-only path, no L1 allocation), keeps it in registers and writes it to
// all K slots of its token.  A warp's stores to one slot cover up to 512
// contiguous bytes, so every write is coalesced.  The FP8 kernel gives 8
// consecutive threads one 1x128 block (16 values each), see rowops.cuh; rows
// hold a multiple of 8 pieces, so those 8 threads always share a token.
#include "common.cuh"
#include "internal.h"
#include "moe_layout.h"
#include "rowops.cuh"

namespace moe {
namespace {

// KT > 0: K known at compile time (fully unrolled); KT == 0: runtime K.
template <int KT>
__global__ void __launch_bounds__(kRowThreads)
dispatch_bf16_kernel(const uint4 *__restrict__ tokens, int T, int K, int vpr,
                     const int32_t *__restrict__ dst_row, int rows,
                     uint4 *__restrict__ packed)
{
    pdl_wait();
    pdl_trigger();
    const RowPiece rp = flat_piece(blockIdx.x, vpr, threadIdx.x);
    if (rp.t >= T) return;
    const int k_count = KT > 0 ? KT : K;
    const uint4 x = ld_stream_v4(tokens + (size_t)rp.t * vpr + rp.u);
    store_to_slots<KT>(dst_row + (size_t)rp.t * k_count, k_count, rows,
                       reinterpret_cast<uint8_t *>(packed), (size_t)vpr * 16,
                       (size_t)rp.u * 16, x);
}

// 40 registers keep 6 blocks (48 warps) per SM; 44 without the bound.
template <int KT>
__global__ void __launch_bounds__(kRowThreads, 6)
dispatch_fp8_kernel(const uint4 *__restrict__ tokens, int T, int K, int H,
                    const int32_t *__restrict__ dst_row, int rows,
                    uint8_t *__restrict__ packed, float *__restrict__ scales)
{
    pdl_wait();
    pdl_trigger();
    const RowPiece rp = flat_piece(blockIdx.x, H >> 4, threadIdx.x);
    const bool active = rp.t < T;
    const int k_count = KT > 0 ? KT : K;
    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
    if (active) {
        const uint4 *src = tokens + (size_t)rp.t * (H >> 3) + 2 * rp.u;
        a = ld_stream_v4(src);
        b = ld_stream_v4(src + 1);
    }
    // every lane takes part in the block's shuffles; the threads past the
    // last row are whole groups of 8
    const Fp8Piece p = quantize16(a, b);
    if (!active) return;
    store_fp8_to_slots<KT>(dst_row + (size_t)rp.t * k_count, k_count, rows, packed,
                           scales, H, rp.u, p);
}

template <int KT>
cudaError_t run_bf16(const void *tokens, int T, int H, int K,
                     const int32_t *dst_row, void *packed, cudaStream_t s)
{
    const int vpr = H / 8;
    if (row_blocks(T, vpr) == 0) return cudaErrorInvalidValue;
    return launch_pdl(dispatch_bf16_kernel<KT>, dim3(row_blocks(T, vpr)), dim3(kRowThreads), 0,
                      s, static_cast<const uint4 *>(tokens), T, K, vpr, dst_row, T * K,
                      static_cast<uint4 *>(packed));
}

template <int KT>
cudaError_t run_fp8(const void *tokens, int T, int H, int K,
                    const int32_t *dst_row, void *packed, float *scales,
                    cudaStream_t s)
{
    if (row_blocks(T, H / 16) == 0) return cudaErrorInvalidValue;
    return launch_pdl(dispatch_fp8_kernel<KT>, dim3(row_blocks(T, H / 16)), dim3(kRowThreads),
                      0, s, static_cast<const uint4 *>(tokens), T, K, H, dst_row, T * K,
                      static_cast<uint8_t *>(packed), scales);
}

}  // namespace

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
