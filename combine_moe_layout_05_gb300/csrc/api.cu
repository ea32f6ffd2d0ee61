// api.cu -- the C ABI: host-side argument checks, then the launchers.
// Nothing here allocates memory or synchronises a stream.
#include "internal.h"
#include "moe_layout.h"

#include <cstdint>
#include <nvtx3/nvToolsExt.h>

namespace {

// An NVTX range named after the C-ABI call, open for the call's host-side
// work (checks and launches), so a profiler can attribute each call's
// kernels (e.g. ncu --nvtx --nvtx-include "moe_combine/").  Without a tool
// attached, a push and a pop cost a few nanoseconds.
struct CallRange {
    explicit CallRange(const char *name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool layout_sizes_ok(int32_t T, int32_t K, int32_t E)
{
    if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS) return false;
    if (K < 1 || K > MOE_MAX_TOPK || K > E) return false;
    if ((int64_t)T * K > (int64_t)INT32_MAX - 1) return false;
    return moe::layout_supported(T, K, E);
}

moe_status_t rows_ok(int32_t T, int32_t H, int32_t K)
{
    if (T < 0 || K < 1 || K > MOE_MAX_TOPK || H < 8 || H % 8 != 0) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * K > (int64_t)INT32_MAX - 1) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace

extern "C" {

const char *moe_status_string(moe_status_t status)
{
    switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_ALIGNMENT: return "misaligned pointer";
    case MOE_ERR_CUDA: return "CUDA launch failed";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

size_t moe_layout_workspace_bytes(int32_t T, int32_t K, int32_t E)
{
    if (!layout_sizes_ok(T, K, E)) return 0;
    return moe::layout_workspace_bytes(T, K, E);
}

moe_status_t moe_layout(const int32_t *topk_ids, int32_t T, int32_t K,
                        int32_t E, int32_t R, int32_t *expert_counts,
                        int32_t *expert_offsets, int32_t *rank_offsets,
                        int32_t *src_token, int32_t *dst_row,
                        uint32_t *dev_error, void *workspace,
                        size_t workspace_bytes, cudaStream_t stream)
{
    const CallRange range("moe_layout");
    if (!layout_sizes_ok(T, K, E) || R < 1 || E % R != 0) return MOE_ERR_INVALID_ARG;
    if (!expert_counts || !expert_offsets || !rank_offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_ids || !src_token || !dst_row)) return MOE_ERR_INVALID_ARG;
    const void *p4[] = {topk_ids, expert_counts, expert_offsets, rank_offsets,
                        src_token, dst_row, dev_error};
    for (const void *p : p4)
        if (!aligned(p, 4)) return MOE_ERR_ALIGNMENT;
    const size_t need = moe::layout_workspace_bytes(T, K, E);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return MOE_ERR_WORKSPACE;
        if (!aligned(workspace, 16)) return MOE_ERR_ALIGNMENT;
    }
    return cuda_status(moe::launch_layout(topk_ids, T, K, E, R, expert_counts,
                                          expert_offsets, rank_offsets,
                                          src_token, dst_row, dev_error,
                                          workspace, stream));
}

moe_status_t moe_dispatch(const void *tokens, int32_t T, int32_t H, int32_t K,
                          const int32_t *dst_row, int32_t fp8, void *packed,
                          float *scales, cudaStream_t stream)
{
    const CallRange range("moe_dispatch");
    moe_status_t s = rows_ok(T, H, K);
    if (s != MOE_OK) return s;
    if (fp8 != 0 && fp8 != 1) return MOE_ERR_INVALID_ARG;
    if (fp8 && H % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!tokens || !dst_row || !packed || (fp8 && !scales)) return MOE_ERR_INVALID_ARG;
    if (!aligned(tokens, 16) || !aligned(packed, 16) || !aligned(dst_row, 4) ||
        (fp8 && !aligned(scales, 4)))
        return MOE_ERR_ALIGNMENT;
    if (fp8)
        return cuda_status(moe::launch_dispatch_fp8(tokens, T, H, K, dst_row,
                                                    packed, scales, stream));
    return cuda_status(moe::launch_dispatch_bf16(tokens, T, H, K, dst_row,
                                                 packed, stream));
}

moe_status_t moe_combine(const void *expert_out, const float *topk_weights,
                         const int32_t *dst_row, int32_t T, int32_t H,
                         int32_t K, void *out, cudaStream_t stream)
{
    const CallRange range("moe_combine");
    moe_status_t s = rows_ok(T, H, K);
    if (s != MOE_OK) return s;
    if (T == 0) return MOE_OK;
    if (!expert_out || !topk_weights || !dst_row || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned(expert_out, 16) || !aligned(out, 16) || !aligned(topk_weights, 4) ||
        !aligned(dst_row, 4))
        return MOE_ERR_ALIGNMENT;
    return cuda_status(moe::launch_combine(expert_out, topk_weights, dst_row, T,
                                           H, K, out, stream));
}

moe_status_t moe_combine_fp8(const void *expert_out, const float *expert_scales,
                             const float *topk_weights, const int32_t *dst_row,
                             int32_t T, int32_t H, int32_t K, void *out,
                             cudaStream_t stream)
{
    const CallRange range("moe_combine_fp8");
    moe_status_t s = rows_ok(T, H, K);
    if (s != MOE_OK) return s;
    if (H % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!expert_out || !expert_scales || !topk_weights || !dst_row || !out)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(expert_out, 16) || !aligned(out, 16) || !aligned(expert_scales, 4) ||
        !aligned(topk_weights, 4) || !aligned(dst_row, 4))
        return MOE_ERR_ALIGNMENT;
    return cuda_status(moe::launch_combine_fp8(expert_out, expert_scales, topk_weights,
                                               dst_row, T, H, K, out, stream));
}

moe_status_t moe_combine_rank_partial(const void *expert_out, const float *topk_weights,
                                      const int32_t *topk_ids, const int32_t *dst_row,
                                      int32_t T, int32_t H, int32_t K, int32_t E,
                                      int32_t R, void *out, cudaStream_t stream)
{
    const CallRange range("moe_combine_rank_partial");
    moe_status_t s = rows_ok(T, H, K);
    if (s != MOE_OK) return s;
    if (E < 1 || E > MOE_MAX_EXPERTS || R < 1 || E % R != 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!expert_out || !topk_weights || !topk_ids || !dst_row || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned(expert_out, 16) || !aligned(out, 16) || !aligned(topk_weights, 4) ||
        !aligned(topk_ids, 4) || !aligned(dst_row, 4))
        return MOE_ERR_ALIGNMENT;
    return cuda_status(moe::launch_combine_rank_partial(expert_out, topk_weights, topk_ids,
                                                        dst_row, T, H, K, E, R, out, stream));
}

moe_status_t moe_dispatch_send(const void *tokens, int32_t T, int32_t H, int32_t K,
                               int32_t E, int32_t R, const int32_t *topk_ids,
                               const int32_t *dst_row, const int32_t *rank_offsets,
                               int32_t fp8, int32_t P, void *priv, float *priv_scales,
                               int32_t C, void *bulk, float *bulk_scales,
                               uint32_t *dev_error, cudaStream_t stream)
{
    const CallRange range("moe_dispatch_send");
    moe_status_t s = rows_ok(T, H, K);
    if (s != MOE_OK) return s;
    if (E < 1 || E > MOE_MAX_EXPERTS || K > E || R < 1 || E % R != 0 || P < 0 || C < 0)
        return MOE_ERR_INVALID_ARG;
    if ((fp8 != 0 && fp8 != 1) || (fp8 && H % 128 != 0)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!tokens || !topk_ids || !dst_row || !rank_offsets || (P > 0 && !priv) ||
        (C > 0 && !bulk) || (fp8 && ((P > 0 && !priv_scales) || (C > 0 && !bulk_scales))))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(tokens, 16) || !aligned(priv, 16) || !aligned(bulk, 16) ||
        !aligned(topk_ids, 4) || !aligned(dst_row, 4) || !aligned(rank_offsets, 4) ||
        !aligned(priv_scales, 4) || !aligned(bulk_scales, 4) || !aligned(dev_error, 4))
        return MOE_ERR_ALIGNMENT;
    return cuda_status(moe::launch_dispatch_send(tokens, T, H, K, E, R, topk_ids, dst_row,
                                                 rank_offsets, fp8, P, priv, priv_scales, C,
                                                 bulk, bulk_scales, dev_error, stream));
}

moe_status_t moe_dispatch_recv(const void *priv, const float *priv_scales, int32_t P,
                               const void *bulk, const float *bulk_scales, int32_t C,
                               const int32_t *rank_offsets, int32_t R, int32_t T, int32_t H,
                               int32_t K, int32_t fp8, void *packed, float *scales,
                               cudaStream_t stream)
{
    const CallRange range("moe_dispatch_recv");
    moe_status_t s = rows_ok(T, H, K);
    if (s != MOE_OK) return s;
    if (R < 1 || R > MOE_MAX_EXPERTS || P < 0 || C < 0) return MOE_ERR_INVALID_ARG;
    if ((fp8 != 0 && fp8 != 1) || (fp8 && H % 128 != 0)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!rank_offsets || !packed || (P > 0 && !priv) || (C > 0 && !bulk) ||
        (fp8 && (!scales || (P > 0 && !priv_scales) || (C > 0 && !bulk_scales))))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(priv, 16) || !aligned(bulk, 16) || !aligned(packed, 16) ||
        !aligned(rank_offsets, 4) || !aligned(scales, 4) || !aligned(priv_scales, 4) ||
        !aligned(bulk_scales, 4))
        return MOE_ERR_ALIGNMENT;
    return cuda_status(moe::launch_dispatch_recv(priv, priv_scales, P, bulk, bulk_scales, C,
                                                 rank_offsets, R, T, H, K, fp8, packed, scales,
                                                 stream));
}

moe_status_t moe_layout_dispatch(const int32_t *topk_ids, const void *tokens,
                                 int32_t T, int32_t H, int32_t K, int32_t E,
                                 int32_t R, int32_t fp8, int32_t *expert_counts,
                                 int32_t *expert_offsets, int32_t *rank_offsets,
                                 int32_t *src_token, int32_t *dst_row,
                                 uint32_t *dev_error, void *packed, float *scales,
                                 void *workspace, size_t workspace_bytes,
                                 cudaStream_t stream)
{
    const CallRange range("moe_layout_dispatch");
    if (!layout_sizes_ok(T, K, E) || R < 1 || E % R != 0) return MOE_ERR_INVALID_ARG;
    moe_status_t s = rows_ok(T, H, K);
    if (s != MOE_OK) return s;
    if (fp8 != 0 && fp8 != 1) return MOE_ERR_INVALID_ARG;
    if (fp8 && H % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (!expert_counts || !expert_offsets || !rank_offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_ids || !src_token || !dst_row || !tokens || !packed ||
                  (fp8 && !scales)))
        return MOE_ERR_INVALID_ARG;
    const void *p4[] = {topk_ids, expert_counts, expert_offsets, rank_offsets,
                        src_token, dst_row, dev_error, fp8 ? scales : nullptr};
    for (const void *p : p4)
        if (!aligned(p, 4)) return MOE_ERR_ALIGNMENT;
    if (!aligned(tokens, 16) || !aligned(packed, 16)) return MOE_ERR_ALIGNMENT;
    if (!moe::layout_dispatch_fused(T, H, K, fp8)) {
        const size_t need = moe::layout_workspace_bytes(T, K, E);
        if (need > 0) {
            if (!workspace || workspace_bytes < need) return MOE_ERR_WORKSPACE;
            if (!aligned(workspace, 16)) return MOE_ERR_ALIGNMENT;
        }
    }
    return cuda_status(moe::launch_layout_dispatch(
        topk_ids, tokens, T, H, K, E, R, fp8, expert_counts, expert_offsets,
        rank_offsets, src_token, dst_row, dev_error, packed, scales, workspace, stream));
}

int32_t moe_layout_dispatch_kernels(int32_t T, int32_t H, int32_t K, int32_t E,
                                    int32_t fp8)
{
    if (!layout_sizes_ok(T, K, E) || rows_ok(T, H, K) != MOE_OK) return 0;
    if ((fp8 != 0 && fp8 != 1) || (fp8 && H % 128 != 0)) return 0;
    if (moe::layout_dispatch_fused(T, H, K, fp8)) return 1;
    if (moe::layout_dispatch_prefill(T, H, K, E, fp8)) return 2;
    const int layout = moe_layout_kernels(T, K, E);
    return T > 0 ? layout + 1 : layout;
}

int32_t moe_layout_kernels(int32_t T, int32_t K, int32_t E)
{
    if (!layout_sizes_ok(T, K, E)) return 0;
    if (moe::plan_layout(T, K, E).single_launch) return 1;
    return moe::layout_ranked(T, K, E) ? 2 : 3;
}

}  // extern "C"
