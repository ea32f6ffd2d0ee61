// regions.cu -- dispatch into per-destination send regions, and the
// receive step back to the grouped-GEMM input.
//
// Perplexity, "Enabling trillion-parameter models on AWS EFA", section
// "Send/receive buffers": senders lay their writes out contiguously once the
// per-expert counts are known, a small private area per sender on each
// receiver takes the first tokens before that, and the rest go in one write
// per peer.  With one sender and R destination ranks, rank r's rows in slot
// order i = 0 .. n_r - 1 (n_r = rank_offsets[r+1] - rank_offsets[r]) go to
// its private area priv[r, i] for i < P and to its bulk area bulk[r, i - P]
// otherwise; bulk rows at or beyond the capacity C are not written and set
// MOE_DEV_ERR_REGION_OVERFLOW.  The receive step puts every region row back
// at its slot, so send + receive gives exactly what moe_dispatch gives.
//
// send: like the dispatch kernels (block = one token x a slice of its row,
// each token piece read once), but each of the K stores goes to the region
// row of its slot.  recv: block = one packed row x a slice, 4 vectors of 16
// bytes per thread; the row's rank is found by binary search of
// rank_offsets, staged in shared memory first.
#include "common.cuh"
#include "internal.h"
#include "moe_layout.h"
#include "rowops.cuh"

namespace moe {
namespace {

constexpr int kRecvVecs = 4;

// Region row of slot s whose expert e is valid, as (base, row); false when
// the slot falls past the bulk capacity.
struct RegionDst {
    uint8_t *base;
    float *scale_base;
    size_t row;
};

__device__ __forceinline__ bool region_of(int s, int e, int epr, const int32_t *rank_offsets,
                                          int P, int C, uint8_t *priv, float *priv_sc,
                                          uint8_t *bulk, float *bulk_sc, RegionDst &d)
{
    const int r = e / epr;
    const int i = s - rank_offsets[r];
    if (i < P) {
        d = {priv, priv_sc, (size_t)r * P + i};
        return true;
    }
    if (i - P < C) {
        d = {bulk, bulk_sc, (size_t)r * C + (i - P)};
        return true;
    }
    return false;
}

// KT > 0: K known at compile time.  The row piece, the block's copy of
// rank_offsets (shared memory) and a token's slots and experts are all
// requested before the first store, so a block waits for memory once.
template <int KT, bool kFp8>
__global__ void __launch_bounds__(256)
dispatch_send_kernel(const uint4 *__restrict__ tokens, int H, int K, int E, int epr,
                     const int32_t *__restrict__ ids, const int32_t *__restrict__ dst_row,
                     const int32_t *__restrict__ rank_offsets, int R, int rows, int P, int C,
                     uint8_t *__restrict__ priv, float *__restrict__ priv_sc,
                     uint8_t *__restrict__ bulk, float *__restrict__ bulk_sc,
                     uint32_t *__restrict__ dev_error)
{
    __shared__ int32_t s_ro[MOE_MAX_EXPERTS + 1];
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int u = blockIdx.y * blockDim.x + threadIdx.x;
    const int units = kFp8 ? (H >> 4) : (H >> 3);
    const bool active = u < units;
    const int k_count = KT > 0 ? KT : K;
    const size_t vrow = (size_t)(H >> 3);
    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
    if (active) {
        if (kFp8) {
            a = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u);
            b = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u + 1);
        } else {
            a = ld_stream_v4(tokens + (size_t)t * vrow + u);
        }
    }
    for (int q = threadIdx.x; q <= R; q += blockDim.x) s_ro[q] = __ldg(rank_offsets + q);
    if (t == 0 && blockIdx.y == 0 && threadIdx.x == 0 && dev_error) {
        uint32_t err = 0;
        for (int r = 0; r < R; ++r)
            if (__ldg(rank_offsets + r + 1) - __ldg(rank_offsets + r) - P > C)
                err |= MOE_DEV_ERR_REGION_OVERFLOW;
        *dev_error = err;
    }
    __syncthreads();
    Fp8Piece p;
    if (kFp8) {
        p = quantize16(a, b);        // every lane takes part (8-lane blocks)
        if (!active) return;
    } else if (!active) {
        return;
    }
    const size_t row_bytes = kFp8 ? (size_t)H : (size_t)H * 2;
    const int nb = H >> 7;
    constexpr int G = KT > 0 && KT < 8 ? KT : 8;
    for (int k0 = 0; k0 < k_count; k0 += G) {
        int sl[G], ex[G];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const bool in = KT > 0 || k0 + j < k_count;
            sl[j] = in ? __ldg(dst_row + (size_t)t * k_count + k0 + j) : -1;
            ex[j] = in ? __ldg(ids + (size_t)t * k_count + k0 + j) : -1;
        }
#pragma unroll
        for (int j = 0; j < G; ++j) {
            if ((unsigned)sl[j] >= (unsigned)rows || (unsigned)ex[j] >= (unsigned)E) continue;
            RegionDst d;
            if (!region_of(sl[j], ex[j], epr, s_ro, P, C, priv, priv_sc, bulk, bulk_sc, d))
                continue;
            st_v4(d.base + d.row * row_bytes + (size_t)u * 16, kFp8 ? p.codes : a);
            if (kFp8 && (u & 7) == 0) d.scale_base[d.row * nb + (u >> 3)] = p.scale;
        }
    }
}

template <bool kFp8>
__global__ void __launch_bounds__(256)
dispatch_recv_kernel(const uint8_t *__restrict__ priv, const float *__restrict__ priv_sc,
                     const uint8_t *__restrict__ bulk, const float *__restrict__ bulk_sc,
                     const int32_t *__restrict__ rank_offsets, int R, int P, int C, int H,
                     uint8_t *__restrict__ packed, float *__restrict__ scales)
{
    __shared__ int32_t s_ro[MOE_MAX_EXPERTS + 1];
    pdl_wait();
    pdl_trigger();
    // rank_offsets in shared memory: one parallel load, then the search
    for (int q = threadIdx.x; q <= R; q += blockDim.x) s_ro[q] = __ldg(rank_offsets + q);
    __syncthreads();
    const int row = blockIdx.x;
    if (row >= s_ro[R]) return;
    int lo = 0, hi = R;                 // largest r with rank_offsets[r] <= row
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_ro[mid] <= row) lo = mid;
        else hi = mid;
    }
    const int r = lo;
    const int i = row - s_ro[r];
    if (i < 0) return;                  // row below rank_offsets[0]: no region row
    const uint8_t *src;
    const float *ssc;
    size_t srow;
    if (i < P) {
        src = priv;
        ssc = priv_sc;
        srow = (size_t)r * P + i;
    } else if (i - P < C) {
        src = bulk;
        ssc = bulk_sc;
        srow = (size_t)r * C + (i - P);
    } else {
        return;
    }
    const size_t row_bytes = kFp8 ? (size_t)H : (size_t)H * 2;
    const int vecs = (int)(row_bytes >> 4);
    // kRecvVecs 16-byte vectors per thread, all loads issued before the stores
    const int v0 = blockIdx.y * blockDim.x * kRecvVecs + threadIdx.x;
    uint4 val[kRecvVecs];
#pragma unroll
    for (int j = 0; j < kRecvVecs; ++j) {
        const int v = v0 + j * blockDim.x;
        if (v < vecs) val[j] = ld_stream_v4(src + srow * row_bytes + (size_t)v * 16);
    }
#pragma unroll
    for (int j = 0; j < kRecvVecs; ++j) {
        const int v = v0 + j * blockDim.x;
        if (v < vecs) st_v4(packed + (size_t)row * row_bytes + (size_t)v * 16, val[j]);
    }
    if (kFp8) {
        const int nb = H >> 7;
        for (int j = blockIdx.y * blockDim.x + threadIdx.x; j < nb; j += gridDim.y * blockDim.x)
            scales[(size_t)row * nb + j] = __ldg(ssc + srow * nb + j);
    }
}

template <int KT, bool kFp8>
cudaError_t run_send(const void *tokens, int T, int H, int K, int E, int R,
                     const int32_t *topk_ids, const int32_t *dst_row,
                     const int32_t *rank_offsets, int P, void *priv, float *priv_scales,
                     int C, void *bulk, float *bulk_scales, uint32_t *dev_error,
                     cudaStream_t stream)
{
    const int units = kFp8 ? H / 16 : H / 8;
    const int threads = pick_row_block(units);
    const dim3 grid(T, ceil_div(units, threads));
    return launch_pdl(dispatch_send_kernel<KT, kFp8>, grid, dim3(threads), 0, stream,
                      static_cast<const uint4 *>(tokens), H, K, E, E / R, topk_ids, dst_row,
                      rank_offsets, R, T * K, P, C, static_cast<uint8_t *>(priv), priv_scales,
                      static_cast<uint8_t *>(bulk), bulk_scales, dev_error);
}

}  // namespace

cudaError_t launch_dispatch_send(const void *tokens, int T, int H, int K, int E, int R,
                                 const int32_t *topk_ids, const int32_t *dst_row,
                                 const int32_t *rank_offsets, int fp8, int P, void *priv,
                                 float *priv_scales, int C, void *bulk, float *bulk_scales,
                                 uint32_t *dev_error, cudaStream_t stream)
{
#define MOE_SEND_CASE(KV)                                                                     \
    return fp8 ? run_send<KV, true>(tokens, T, H, K, E, R, topk_ids, dst_row, rank_offsets, P, \
                                    priv, priv_scales, C, bulk, bulk_scales, dev_error, stream) \
               : run_send<KV, false>(tokens, T, H, K, E, R, topk_ids, dst_row, rank_offsets, P,\
                                     priv, priv_scales, C, bulk, bulk_scales, dev_error, stream)
    switch (K) {
    case 1: MOE_SEND_CASE(1);
    case 2: MOE_SEND_CASE(2);
    case 4: MOE_SEND_CASE(4);
    case 6: MOE_SEND_CASE(6);
    case 8: MOE_SEND_CASE(8);
    default: MOE_SEND_CASE(0);
    }
#undef MOE_SEND_CASE
}

cudaError_t launch_dispatch_recv(const void *priv, const float *priv_scales, int P,
                                 const void *bulk, const float *bulk_scales, int C,
                                 const int32_t *rank_offsets, int R, int T, int H, int K,
                                 int fp8, void *packed, float *scales, cudaStream_t stream)
{
    const int vecs = fp8 ? H / 16 : H / 8;
    const int threads = pick_row_block(ceil_div(vecs, kRecvVecs));
    const dim3 grid(T * K, ceil_div(vecs, threads * kRecvVecs));
    if (fp8)
        return launch_pdl(dispatch_recv_kernel<true>, grid, dim3(threads), 0, stream,
                          static_cast<const uint8_t *>(priv), priv_scales,
                          static_cast<const uint8_t *>(bulk), bulk_scales, rank_offsets, R, P, C,
                          H, static_cast<uint8_t *>(packed), scales);
    return launch_pdl(dispatch_recv_kernel<false>, grid, dim3(threads), 0, stream,
                      static_cast<const uint8_t *>(priv), priv_scales,
                      static_cast<const uint8_t *>(bulk), bulk_scales, rank_offsets, R, P, C, H,
                      static_cast<uint8_t *>(packed), scales);
}

}  // namespace moe
