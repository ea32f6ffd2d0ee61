// layout_dispatch_cluster.cu -- layout and dispatch of a decode batch in one
// launch, the ids counted once per token by a thread-block cluster.
//
// Perplexity, "Enabling trillion-parameter models on AWS EFA", section
// "Dispatch and Combine": one dispatch-send kernel counts tokens per expert,
// takes the cumulative sum and packs the tokens into the contiguous send
// buffers.  The single-kernel form in layout_dispatch.cu gives every block
// (one slice of one token's row) the whole count: each block reads all T*K
// ids and counts them against its token's K experts.  Here the n blocks that
// share a token form one cluster, and the count is split between them:
//
//  * block r of the cluster for token t packs slice r of t's row; it first
//    requests its row piece (and in the FP8 form quantises it while the
//    count runs);
//  * it counts its 1/n share of the ids against t's K <= 8 experts e:
//    (id < e) | (id == e and entry before t's), and against the cluster's
//    expert "roles" (expert t + j*T, j < 4: ids below it and equal to it),
//    as 16-bit counters packed two to a word; the warps' sums go to shared
//    memory;
//  * after a cluster barrier, 8 threads of every block read the n partial
//    sums from the other blocks' shared memory (distributed shared memory)
//    and add them; the slot of (t,k) is that sum plus the earlier k' of t
//    with the same expert, as in moe_layout;
//  * block 0 of the cluster writes dst_row / src_token of t and the counts,
//    offsets and rank offsets of the cluster's roles; grid block 0 checks the
//    ids for range and duplicate errors.
// A second cluster barrier, arrived at right after the remote reads and
// waited on at exit, keeps every block's shared memory alive until the
// others have read it.  Only this GPU's own memory is touched; nothing is
// multicast.
//
// Measured against the single-kernel form on one GB300 (CUDA graphs, cold
// L2): 6.48 us against 4.60 us at the DeepSeek-V3 decode shape (clusters of
// 7 x 128 threads) and 11.68 against 6.22 us in the FP8 form (7 x 64): the
// cluster launch and barriers cost more than the counting they save.  So
// moe_layout_dispatch does not use it; it stays reachable through a test
// hook for that comparison.
#include "common.cuh"
#include "internal.h"
#include "layout_common.cuh"
#include "moe_layout.h"
#include "rowops.cuh"

namespace moe {
namespace {

constexpr int kMaxRoles = 4;       // experts whose count and offset one cluster writes
constexpr int kMaxCluster = 8;     // portable cluster size

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size()
{
    uint32_t n;
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// The 32-bit word at `p` (this block's shared memory) in block `cta` of the
// cluster.
__device__ __forceinline__ uint32_t ld_cluster(const uint32_t *p, uint32_t cta)
{
    uint32_t remote, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(cta));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
    return v;
}

// Adds one id to the packed counters: targets (x < tg) | (x == tg & before)
// in v[0..3], roles (x < role, x == role) in v[4..7].
__device__ __forceinline__ void count_id(int x, bool before, int E, const int (&tg)[8],
                                         const int (&role)[kMaxRoles], uint32_t (&v)[8])
{
    if ((unsigned)x >= (unsigned)E) return;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        v[j >> 1] += (uint32_t)((x < tg[j]) | ((x == tg[j]) & before)) << (16 * (j & 1));
#pragma unroll
    for (int j = 0; j < kMaxRoles; ++j)
        v[4 + j] += (uint32_t)(x < role[j]) | ((uint32_t)(x == role[j]) << 16);
}

template <int KT, bool kFp8, int kThreads>
__global__ void __launch_bounds__(kThreads)
layout_dispatch_cluster_kernel(const int32_t *__restrict__ ids, const uint4 *__restrict__ tokens,
                               int T, int H, int K, int E, int R,
                               int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                               int32_t *__restrict__ rank_offsets,
                               int32_t *__restrict__ src_token, int32_t *__restrict__ dst_row,
                               uint32_t *__restrict__ dev_error, uint8_t *__restrict__ packed,
                               float *__restrict__ scales)
{
    constexpr int kWarps = kThreads / 32;
    __shared__ uint32_t red[kWarps][8];
    __shared__ uint32_t part[8];
    __shared__ uint32_t tot[8];
    __shared__ uint32_t s_err;

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const uint32_t n = cluster_size(), cr = cluster_rank();
    const int t = blockIdx.x / n;
    const int k_count = KT > 0 ? KT : K;
    const int nids = T * k_count, mine = t * k_count;
    const int units = kFp8 ? (H >> 4) : (H >> 3);
    const int u = (int)cr * kThreads + tid;
    const bool active = u < units;
    const size_t vrow = (size_t)(H >> 3);
    const int epr = E / R;

    if (tid == 0) s_err = 0;
    pdl_wait();
    pdl_trigger();

    // this thread's piece of the row; it arrives while the ids are counted
    uint4 a = make_uint4(0, 0, 0, 0), bv = make_uint4(0, 0, 0, 0);
    if (active) {
        if (kFp8) {
            a = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u);
            bv = ld_stream_v4(tokens + (size_t)t * vrow + 2 * u + 1);
        } else {
            a = ld_stream_v4(tokens + (size_t)t * vrow + u);
        }
    }
    int tg[8], role[kMaxRoles];
#pragma unroll
    for (int j = 0; j < 8; ++j) tg[j] = j < k_count ? __ldg(ids + mine + j) : -1;
#pragma unroll
    for (int j = 0; j < kMaxRoles; ++j) {
        const int e = t + j * T;
        role[j] = e <= E ? e : -1;
    }

    // this block's share of the ids, 4 at a time where aligned
    uint32_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const int share = ((nids + (int)n - 1) / (int)n + 3) & ~3;
    const int i0 = min(nids, (int)cr * share), i1 = min(nids, i0 + share);
    if ((reinterpret_cast<uintptr_t>(ids) & 15) == 0) {
        const int i4 = i0 + ((i1 - i0) & ~3);
        for (int i = i0 + 4 * tid; i < i4; i += 4 * kThreads) {
            const int4 q = __ldg(reinterpret_cast<const int4 *>(ids + i));
            count_id(q.x, i < mine, E, tg, role, v);
            count_id(q.y, i + 1 < mine, E, tg, role, v);
            count_id(q.z, i + 2 < mine, E, tg, role, v);
            count_id(q.w, i + 3 < mine, E, tg, role, v);
        }
        for (int i = i4 + tid; i < i1; i += kThreads) count_id(__ldg(ids + i), i < mine, E, tg, role, v);
    } else {
        for (int i = i0 + tid; i < i1; i += kThreads) count_id(__ldg(ids + i), i < mine, E, tg, role, v);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t s = __reduce_add_sync(kFullMask, v[j]);
        if (lane == 0) red[w][j] = s;
    }
    Fp8Piece q;
    if (kFp8) q = quantize16(a, bv);           // fills the wait at the barriers
    __syncthreads();
    if (tid < 8) {
        uint32_t s = 0;
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) s += red[ww][tid];
        part[tid] = s;
    }
    cluster_arrive();                          // every block's partial sums are complete
    cluster_wait();
    if (tid < 8) {
        uint32_t s = 0;
        for (uint32_t c = 0; c < n; ++c) s += ld_cluster(&part[tid], c);
        tot[tid] = s;
    }
    __syncthreads();
    cluster_arrive();                          // done reading the other blocks' memory

    int sl[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        int dup = 0;
#pragma unroll
        for (int x = 0; x < j; ++x) dup += tg[x] == tg[j];
        const int below = (int)((tot[j >> 1] >> (16 * (j & 1))) & 0xffffu);
        sl[j] = (unsigned)tg[j] < (unsigned)E ? below + dup : -1;
    }
    if (cr == 0) {
        // index maps of token t, and the counts and offsets of the cluster's roles
        const int wl = tid - (kThreads - 32);
        if (wl >= 0 && wl < k_count) {
            int my = sl[0];
#pragma unroll
            for (int j = 1; j < 8; ++j)
                if (wl == j) my = sl[j];
            dst_row[mine + wl] = my;
            if (my >= 0) src_token[my] = t;
        }
        if (tid < kMaxRoles && role[tid] >= 0) {
            const uint32_t rv = tot[4 + tid];
            const int lt = (int)(rv & 0xffffu), eq = (int)(rv >> 16);
            offsets[role[tid]] = lt;
            if (role[tid] < E) counts[role[tid]] = eq;
            if (role[tid] % epr == 0) rank_offsets[role[tid] / epr] = lt;
        }
    }

    const int rows = nids;
    if (kFp8) {
        if (active) store_fp8_to_slots<KT>(sl, k_count, rows, packed, scales, H, u, q);
    } else if (active) {
        store_to_slots<KT>(sl, k_count, rows, packed, vrow * 16, (size_t)u * 16, a);
    }
    if (blockIdx.x == 0) {
        const uint32_t err = token_errors(ids, T, k_count, E);
        if (err) atomicOr(&s_err, err);
        __syncthreads();
        if (tid == 0 && dev_error) *dev_error = s_err;
    }
    cluster_wait();
}

struct ClusterPlan {
    bool use;
    int threads;
    int n;
};

ClusterPlan plan_cluster(int T, int H, int K, int E, bool fp8)
{
    ClusterPlan p{false, 0, 0};
    if (!layout_dispatch_fused(T, H, K, fp8) || K > 8) return p;
    if ((long long)kMaxRoles * T < (long long)E + 1) return p;
    const int units = fp8 ? H / 16 : H / 8;
    for (int th : {128, 64}) {
        if (units % th == 0 && units / th >= 2 && units / th <= kMaxCluster) {
            p = {true, th, units / th};
            return p;
        }
    }
    return p;
}

template <int KT, bool kFp8, int kThreads>
cudaError_t run_cluster(const ClusterPlan &p, const int32_t *ids, const void *tokens, int T,
                        int H, int K, int E, int R, int32_t *counts, int32_t *offsets,
                        int32_t *rank_offsets, int32_t *src_token, int32_t *dst_row,
                        uint32_t *dev_error, void *packed, float *scales, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(T * p.n);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = p.n;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, layout_dispatch_cluster_kernel<KT, kFp8, kThreads>,
                                       ids, static_cast<const uint4 *>(tokens), T, H, K, E, R,
                                       counts, offsets, rank_offsets, src_token, dst_row,
                                       dev_error, static_cast<uint8_t *>(packed), scales);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <bool kFp8, int kThreads>
cudaError_t run_cluster_k(const ClusterPlan &p, const int32_t *ids, const void *tokens, int T,
                          int H, int K, int E, int R, int32_t *counts, int32_t *offsets,
                          int32_t *rank_offsets, int32_t *src_token, int32_t *dst_row,
                          uint32_t *dev_error, void *packed, float *scales, cudaStream_t s)
{
#define MOE_CLUSTER_CASE(KV)                                                                  \
    return run_cluster<KV, kFp8, kThreads>(p, ids, tokens, T, H, K, E, R, counts, offsets,    \
                                           rank_offsets, src_token, dst_row, dev_error, packed, \
                                           scales, s)
    switch (K) {
    case 1: MOE_CLUSTER_CASE(1);
    case 2: MOE_CLUSTER_CASE(2);
    case 4: MOE_CLUSTER_CASE(4);
    case 6: MOE_CLUSTER_CASE(6);
    case 8: MOE_CLUSTER_CASE(8);
    default: MOE_CLUSTER_CASE(0);
    }
#undef MOE_CLUSTER_CASE
}

}  // namespace

bool layout_dispatch_clustered(int T, int H, int K, int E, int fp8)
{
    return plan_cluster(T, H, K, E, fp8 != 0).use;
}

cudaError_t launch_layout_dispatch_cluster(const int32_t *topk_ids, const void *tokens, int T,
                                           int H, int K, int E, int R, int fp8,
                                           int32_t *expert_counts, int32_t *expert_offsets,
                                           int32_t *rank_offsets, int32_t *src_token,
                                           int32_t *dst_row, uint32_t *dev_error, void *packed,
                                           float *scales, cudaStream_t stream)
{
    const ClusterPlan p = plan_cluster(T, H, K, E, fp8 != 0);
    if (!p.use) return cudaErrorInvalidValue;
#define MOE_CLUSTER_ARGS                                                                    \
    p, topk_ids, tokens, T, H, K, E, R, expert_counts, expert_offsets, rank_offsets,         \
        src_token, dst_row, dev_error, packed, scales, stream
    if (fp8)
        return p.threads == 128 ? run_cluster_k<true, 128>(MOE_CLUSTER_ARGS)
                                : run_cluster_k<true, 64>(MOE_CLUSTER_ARGS);
    return p.threads == 128 ? run_cluster_k<false, 128>(MOE_CLUSTER_ARGS)
                            : run_cluster_k<false, 64>(MOE_CLUSTER_ARGS);
#undef MOE_CLUSTER_ARGS
}

}  // namespace moe
