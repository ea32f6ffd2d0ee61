// internal.h -- launchers shared between the C-ABI layer and the kernels.
// Every launcher assumes its arguments have already been validated.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// How the layout of T*K entries is split over thread blocks.
struct LayoutPlan {
    bool single_launch;    // one kernel, no workspace
    int tokens_per_chunk;  // tokens per block in the multi-block path
    int chunks;            // number of blocks in the multi-block path
};

LayoutPlan plan_layout(int T, int K, int E);
// False when a batch this large would not fit the kernels' shared memory.
bool layout_supported(int T, int K, int E);
// Bytes of workspace moe_layout and moe_layout_dispatch need for these sizes:
// the larger of the count/scan/rank form's and the ranking blocks' form's.
size_t layout_workspace_bytes(int T, int K, int E);

// Where the count/scan/rank layout keeps its state in the workspace, in
// int32 elements from its start: ws_cnt[chunks][E] (chunk histograms, then
// each chunk's first slot per expert), then ws_err[chunks] (chunk error
// bits).
struct WorkspaceLayout {
    size_t err;              // element offset
    size_t bytes;            // bytes used
};
WorkspaceLayout workspace_layout(int chunks, int E);

// Blocks per thread-block cluster of the counting kernel in its clustered
// form (the largest portable cluster).
constexpr int kCountCluster = 8;

// The counting kernel of the multi-launch layout alone: chunk error bits to
// ws_err[chunks], dev_error zeroed, and when dst_row_fill is not null every
// dst_row entry set to kSlotPending.  With ws_ctot null it writes each
// chunk's histogram to ws_cnt[chunks][E].  With ws_ctot set it runs in
// clusters of kCountCluster blocks (chunks kCountCluster*g .. +7 form
// cluster g; the grid is padded with empty chunks) and writes, through
// distributed shared memory, each chunk's exclusive prefix within its
// cluster, ws_cnt[c][e] = entries of e in the earlier chunks of c's
// cluster, and each cluster's totals, ws_ctot[g][e], both in rows of
// align4(E) elements.  threads: 256 or 512
// per block (one chunk per block).  512 measured 0.2-0.4 us faster inside
// the large-batch moe_layout_dispatch at Kimi-K2 sizes (equal at Qwen3), but
// 5 us slower ahead of moe_layout's ranking-only grid at Qwen3 sizes, where
// 256 is used.
constexpr int32_t kSlotPending = INT32_MIN;
cudaError_t launch_layout_count(const int32_t *topk_ids, int T, int K, int E,
                                const LayoutPlan &plan, int32_t *ws_cnt, uint32_t *ws_err,
                                uint32_t *dev_error, int32_t *dst_row_fill,
                                cudaStream_t stream, int threads = 256,
                                int32_t *ws_ctot = nullptr);

cudaError_t launch_layout(const int32_t *topk_ids, int T, int K, int E, int R,
                          int32_t *expert_counts, int32_t *expert_offsets,
                          int32_t *rank_offsets, int32_t *src_token,
                          int32_t *dst_row, uint32_t *dev_error,
                          void *workspace, cudaStream_t stream);

cudaError_t launch_dispatch_bf16(const void *tokens, int T, int H, int K,
                                 const int32_t *dst_row, void *packed,
                                 cudaStream_t stream);

cudaError_t launch_dispatch_fp8(const void *tokens, int T, int H, int K,
                                const int32_t *dst_row, void *packed,
                                float *scales, cudaStream_t stream);

cudaError_t launch_combine(const void *expert_out, const float *topk_weights,
                           const int32_t *dst_row, int T, int H, int K,
                           void *out, cudaStream_t stream);

// moe_combine with the slots and weights loaded by lanes 0..7 and shuffled
// to the warp (K = 8; reachable only through a test hook).
cudaError_t launch_combine_shfl(const void *expert_out, const float *topk_weights,
                                const int32_t *dst_row, int T, int H, int K, void *out,
                                cudaStream_t stream);

cudaError_t launch_combine_fp8(const void *codes, const float *scales,
                               const float *topk_weights, const int32_t *dst_row,
                               int T, int H, int K, void *out, cudaStream_t stream);

cudaError_t launch_combine_rank_partial(const void *expert_out, const float *topk_weights,
                                        const int32_t *topk_ids, const int32_t *dst_row,
                                        int T, int H, int K, int E, int R, void *out,
                                        cudaStream_t stream);

cudaError_t launch_dispatch_send(const void *tokens, int T, int H, int K, int E, int R,
                                 const int32_t *topk_ids, const int32_t *dst_row,
                                 const int32_t *rank_offsets, int fp8, int P, void *priv,
                                 float *priv_scales, int C, void *bulk, float *bulk_scales,
                                 uint32_t *dev_error, cudaStream_t stream);
cudaError_t launch_dispatch_recv(const void *priv, const float *priv_scales, int P,
                                 const void *bulk, const float *bulk_scales, int C,
                                 const int32_t *rank_offsets, int R, int T, int H, int K,
                                 int fp8, void *packed, float *scales, cudaStream_t stream);

// Layout and dispatch together: one fused kernel when
// layout_dispatch_fused() says the batch is small enough, else the layout
// kernels followed by the dispatch kernel.
bool layout_dispatch_fused(int T, int H, int K, int fp8);
cudaError_t launch_layout_dispatch(const int32_t *topk_ids, const void *tokens,
                                   int T, int H, int K, int E, int R, int fp8,
                                   int32_t *expert_counts, int32_t *expert_offsets,
                                   int32_t *rank_offsets, int32_t *src_token,
                                   int32_t *dst_row, uint32_t *dev_error,
                                   void *packed, float *scales, void *workspace,
                                   cudaStream_t stream);

// Raises fn's dynamic shared memory limit to the most the current device
// allows next to its static shared memory (once per kernel and device) and
// checks that `bytes` fits; cudaErrorInvalidValue when it does not.
cudaError_t allow_dynamic_smem(const void *fn, size_t bytes);

// Number of SMs of the current device (looked up once per device).
cudaError_t device_sm_count(int *count);

// Decode batches in one launch of clusters, the n blocks of a token's row
// sharing the count through distributed shared memory
// (layout_dispatch_cluster.cu; measured slower than the single-kernel form,
// so reachable only through a test hook).
bool layout_dispatch_clustered(int T, int H, int K, int E, int fp8);
cudaError_t launch_layout_dispatch_cluster(const int32_t *topk_ids, const void *tokens, int T,
                                           int H, int K, int E, int R, int fp8,
                                           int32_t *expert_counts, int32_t *expert_offsets,
                                           int32_t *rank_offsets, int32_t *src_token,
                                           int32_t *dst_row, uint32_t *dev_error, void *packed,
                                           float *scales, cudaStream_t stream);
// The single-kernel form in which every block counts all ids itself.
cudaError_t launch_layout_dispatch_fused(const int32_t *topk_ids, const void *tokens, int T,
                                         int H, int K, int E, int R, int fp8,
                                         int32_t *expert_counts, int32_t *expert_offsets,
                                         int32_t *rank_offsets, int32_t *src_token,
                                         int32_t *dst_row, uint32_t *dev_error, void *packed,
                                         float *scales, cudaStream_t stream);

// The single-kernel form writing its rows by bulk copies out of shared
// memory (K = 8; measured slower, reachable only through a test hook).
cudaError_t launch_layout_dispatch_fused_bulk(const int32_t *topk_ids, const void *tokens,
                                              int T, int H, int K, int E, int R, int fp8,
                                              int32_t *expert_counts, int32_t *expert_offsets,
                                              int32_t *rank_offsets, int32_t *src_token,
                                              int32_t *dst_row, uint32_t *dev_error,
                                              void *packed, float *scales, cudaStream_t stream);

// Large batches: the counting kernel, then one grid whose first blocks rank
// the chunks while the others pack the rows of ranked chunks
// (layout_dispatch_prefill.cu).  layout_dispatch_prefill() says whether these
// sizes take that path.  wait_ns bounds every wait for a ranked chunk (0: the
// default); stall_chunk >= 0 leaves that chunk unranked (tests of the
// bounded wait only), otherwise -1.
bool layout_dispatch_prefill(int T, int H, int K, int E, int fp8);
cudaError_t launch_layout_dispatch_prefill(const int32_t *topk_ids, const void *tokens, int T,
                                           int H, int K, int E, int R, int fp8,
                                           int32_t *expert_counts, int32_t *expert_offsets,
                                           int32_t *rank_offsets, int32_t *src_token,
                                           int32_t *dst_row, uint32_t *dev_error, void *packed,
                                           float *scales, void *workspace,
                                           unsigned long long wait_ns, int stall_chunk,
                                           cudaStream_t stream);

// moe_layout's large-batch form when its plan fits (layout_dispatch_prefill.cu):
// the counting kernel, then the ranking blocks of the two-launch
// layout + dispatch grid alone.  layout_ranked() says whether these sizes take
// it; otherwise launch_layout runs count, scan and rank.
bool layout_ranked(int T, int K, int E);
// Workspace bytes of the ranking blocks' form (0 when it does not apply).
size_t ranked_workspace_bytes(int T, int K, int E);
cudaError_t launch_layout_ranked(const int32_t *topk_ids, int T, int K, int E, int R,
                                 int32_t *expert_counts, int32_t *expert_offsets,
                                 int32_t *rank_offsets, int32_t *src_token, int32_t *dst_row,
                                 uint32_t *dev_error, void *workspace, cudaStream_t stream);

// The persistent form (layout_dispatch_persistent.cu): a shared-memory ring
// of token rows fed by bulk copies, one CTA per SM; measured slower, so
// reachable only through a test hook.  bulk_store != 0 writes bf16 rows by
// bulk copies out of the ring.
bool layout_dispatch_persistent(int T, int H, int K, int E);
cudaError_t launch_layout_dispatch_persistent(const int32_t *topk_ids, const void *tokens, int T,
                                              int H, int K, int E, int R, int fp8,
                                              int32_t *expert_counts, int32_t *expert_offsets,
                                              int32_t *rank_offsets, int32_t *src_token,
                                              int32_t *dst_row, uint32_t *dev_error,
                                              void *packed, float *scales, void *workspace,
                                              unsigned long long wait_ns, int stall_cta,
                                              int bulk_store, cudaStream_t stream);

// Threads per block for `units` work items per row: the largest multiple of
// 32 up to 256 that divides `units`, else 128 (last block of a row partial).
int pick_row_block(int units);

}  // namespace moe
