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
// block (16 values each): amax is reduced with three xor-shuffles, the scale
// is amax / 448 (IEEE divide), each value is divided by the scale (IEEE
// divide) and converted with cvt.rn.satfinite.e4m3x2; a thread then stores
// 16 code bytes per slot and the group's first thread stores the scale.
#include "common.cuh"
#include "internal.h"
#include "moe_layout.h"

namespace moe {
namespace {

// KT > 0: K known at compile time (fully unrolled); KT == 0: runtime K.
template <int KT>
__global__ void __launch_bounds__(256)
dispatch_bf16_kernel(const uint4 *__restrict__ tokens, int K, int vpr,
                     const int32_t *__restrict__ dst_row, int rows,
                     uint4 *__restrict__ packed)
{
    const int t = blockIdx.x;
    const int v = blockIdx.y * blockDim.x + threadIdx.x;
    if (v >= vpr) return;
    const int k_count = KT > 0 ? KT : K;
    const uint4 x = ld_stream_v4(tokens + (size_t)t * vpr + v);
    const int32_t *d = dst_row + (size_t)t * k_count;
#pragma unroll
    for (int k = 0; k < (KT > 0 ? KT : MOE_MAX_TOPK); ++k) {
        if (KT == 0 && k >= k_count) break;
        const int r = __ldg(d + k);
        if ((unsigned)r < (unsigned)rows) st_v4(packed + (size_t)r * vpr + v, x);
    }
}

template <int KT>
__global__ void __launch_bounds__(256)
dispatch_fp8_kernel(const uint4 *__restrict__ tokens, int K, int H,
                    const int32_t *__restrict__ dst_row, int rows,
                    uint4 *__restrict__ packed, float *__restrict__ scales)
{
    const int t = blockIdx.x;
    const int g = blockIdx.y * blockDim.x + threadIdx.x;   // 16-value group
    const int groups = H >> 4;
    const bool active = g < groups;
    const int k_count = KT > 0 ? KT : K;

    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
    if (active) {
        const uint4 *src = tokens + (size_t)t * (H >> 3) + 2 * g;
        a = ld_stream_v4(src);
        b = ld_stream_v4(src + 1);
    }
    float x[16];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        x[2 * i] = bf16_lo(w[i]);
        x[2 * i + 1] = bf16_hi(w[i]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    // 8 consecutive lanes hold one 128-value block (groups per row is a
    // multiple of 8 and blocks start at multiples of 32 threads).
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 4));
    if (!active) return;

    const float scale = __fdiv_rn(amax, 448.0f);
    uint32_t q[4];
    if (amax == 0.0f) {
        // all values are zeros: keep each sign, divide nothing
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t s = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                s |= (__float_as_uint(x[4 * i + j]) >> 31) << (8 * j + 7);
            q[i] = s;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = cvt_e4m3x2_satfinite(__fdiv_rn(x[4 * i], scale),
                                                     __fdiv_rn(x[4 * i + 1], scale));
            const uint32_t hi = cvt_e4m3x2_satfinite(__fdiv_rn(x[4 * i + 2], scale),
                                                     __fdiv_rn(x[4 * i + 3], scale));
            q[i] = lo | (hi << 16);
        }
    }
    const uint4 codes = make_uint4(q[0], q[1], q[2], q[3]);
    const int nb = H >> 7;
    const int blk = g >> 3;
    const bool leader = (g & 7) == 0;
    const int32_t *d = dst_row + (size_t)t * k_count;
#pragma unroll
    for (int k = 0; k < (KT > 0 ? KT : MOE_MAX_TOPK); ++k) {
        if (KT == 0 && k >= k_count) break;
        const int r = __ldg(d + k);
        if ((unsigned)r >= (unsigned)rows) continue;
        st_v4(reinterpret_cast<uint8_t *>(packed) + (size_t)r * H + 16 * (size_t)g, codes);
        if (leader) scales[(size_t)r * nb + blk] = scale;
    }
}

template <template <int> class Launch, typename... Args>
cudaError_t dispatch_on_k(int K, Args... args)
{
    switch (K) {
    case 1: return Launch<1>::run(args...);
    case 2: return Launch<2>::run(args...);
    case 4: return Launch<4>::run(args...);
    case 6: return Launch<6>::run(args...);
    case 8: return Launch<8>::run(args...);
    default: return Launch<0>::run(args...);
    }
}

template <int KT>
struct Bf16Launch {
    static cudaError_t run(const void *tokens, int T, int H, int K,
                           const int32_t *dst_row, void *packed, cudaStream_t s)
    {
        const int vpr = H / 8;
        const int threads = pick_row_block(vpr);
        const dim3 grid(T, ceil_div(vpr, threads));
        dispatch_bf16_kernel<KT><<<grid, threads, 0, s>>>(
            static_cast<const uint4 *>(tokens), K, vpr, dst_row, T * K,
            static_cast<uint4 *>(packed));
        return cudaGetLastError();
    }
};

template <int KT>
struct Fp8Launch {
    static cudaError_t run(const void *tokens, int T, int H, int K,
                           const int32_t *dst_row, void *packed, float *scales,
                           cudaStream_t s)
    {
        const int groups = H / 16;
        const int threads = pick_row_block(groups);
        const dim3 grid(T, ceil_div(groups, threads));
        dispatch_fp8_kernel<KT><<<grid, threads, 0, s>>>(
            static_cast<const uint4 *>(tokens), K, H, dst_row, T * K,
            static_cast<uint4 *>(packed), scales);
        return cudaGetLastError();
    }
};

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
    return dispatch_on_k<Bf16Launch>(K, tokens, T, H, K, dst_row, packed, stream);
}

cudaError_t launch_dispatch_fp8(const void *tokens, int T, int H, int K,
                                const int32_t *dst_row, void *packed,
                                float *scales, cudaStream_t stream)
{
    return dispatch_on_k<Fp8Launch>(K, tokens, T, H, K, dst_row, packed, scales,
                                    stream);
}

}  // namespace moe
