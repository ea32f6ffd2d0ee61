/*
 * moe_layout.h -- C ABI of the single-GPU MoE layout / dispatch / combine
 * library (libmoe_layout.so, CUDA, sm_103a).
 *
 * The operations follow Perplexity, "Enabling trillion-parameter models on
 * AWS EFA" (2025-11-04).  The page splits MoE routing into a dispatch that
 * takes the tokens and their per-token experts and packs each token into
 * contiguous per-destination buffers, and its dual, combine, that brings the
 * processed rows back and forms their routing-weighted average (sections
 * "MoE all-to-all over EFA" and "Dispatch and Combine").  Here the R
 * expert-parallel destinations are R row ranges of one packed buffer in the
 * GPU's own memory; there is no network, peer or collective.
 *
 * Conventions for every call:
 *  - All pointers are device pointers unless stated otherwise.  The caller
 *    allocates and owns every buffer; the library allocates nothing and
 *    never synchronises, and apart from moe_layout_static's scratch array
 *    (described with that call) it keeps no state between calls.
 *  - moe_layout, moe_dispatch, moe_combine, moe_combine_fp8,
 *    moe_combine_rank_partial, moe_dispatch_send, moe_dispatch_recv and
 *    moe_layout_dispatch are asynchronous on `stream` (0 = legacy default
 *    stream) and may be captured into a CUDA graph.
 *  - Arguments are checked on the host before anything is enqueued.  A
 *    failed check returns an error status and enqueues nothing.
 *  - Matrices are row-major and dense: a [rows, H] matrix has row stride H.
 *  - bf16 means IEEE binary32 truncated to its top 16 bits (stored as 2-byte
 *    words); e4m3 means the 8-bit "fn" float format (bias 7, largest finite
 *    448, no infinities).
 *  - Indices are int32: T*K must stay below 2^31.
 *  - Notation: T tokens, H hidden size, E experts, R destination ranks,
 *    K experts per token, Epr = E/R experts per rank.  Expert e belongs to
 *    rank e / Epr.
 */
#ifndef MOE_LAYOUT_H
#define MOE_LAYOUT_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status returned synchronously by every call. */
typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null pointer, size out of range, E % R != 0 ... */
    MOE_ERR_ALIGNMENT = 2,    /* a pointer misses its required alignment       */
    MOE_ERR_CUDA = 3,         /* the CUDA runtime refused a launch             */
    MOE_ERR_WORKSPACE = 4     /* workspace missing or smaller than required    */
} moe_status_t;

/* Bits of the device error word written by moe_layout (read it after the
 * stream has reached that point). */
#define MOE_DEV_ERR_EXPERT_RANGE 1u  /* some topk_ids entry is outside [0, E)   */
#define MOE_DEV_ERR_DUPLICATE    2u  /* some token lists one expert twice       */
#define MOE_DEV_ERR_REGION_OVERFLOW 4u /* moe_dispatch_send: a rank's rows exceed
                                          its private + bulk capacity          */
#define MOE_DEV_ERR_TIMEOUT 8u       /* moe_layout_dispatch: a bounded wait
                                        between its blocks expired; outputs
                                        unspecified                            */

/* Limits of this implementation. */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 32

/* Human-readable name of a status code (static storage, never NULL). */
MOE_API const char *moe_status_string(moe_status_t status);

/* Bytes of device workspace moe_layout needs for these sizes (0 when the
 * whole layout fits one thread block).  Returns 0 for invalid sizes, which
 * moe_layout then rejects. */
MOE_API size_t moe_layout_workspace_bytes(int32_t T, int32_t K, int32_t E);

/* Number of kernel launches moe_layout makes for these sizes: 1 when the
 * whole layout fits one launch of self-counting blocks, 2 (count in
 * clusters of blocks that sum their histograms together, then one ranking
 * block per chunk) when the ranking blocks' shared memory fits, otherwise 3
 * (count, scan, rank; large batches with E near 1024).  0 for invalid
 * sizes.  A query: nothing is launched. */
MOE_API int32_t moe_layout_kernels(int32_t T, int32_t K, int32_t E);

/*
 * moe_layout -- routing histogram, exclusive scan and stable slot map.
 *
 * The page's dispatch-send first counts tokens per expert in shared memory,
 * then takes the cumulative sum of the counts to find the offsets at which
 * tokens are packed into contiguous per-destination send buffers ("Dispatch
 * and Combine"); the per-expert counts are also the routing information that
 * ranks exchange before writing ("Send/receive buffers").  This call computes
 * that metadata for all T*K (token, k) entries:
 *
 *   expert_counts[e]  = #{(t,k) : topk_ids[t,k] == e}                      [E]
 *   expert_offsets[e] = sum of expert_counts[e'] for e' < e;
 *   expert_offsets[E] = number of valid entries (T*K when no error)       [E+1]
 *   rank_offsets[r]   = expert_offsets[r*Epr]                              [R+1]
 *   dst_row[t,k]      = expert_offsets[e] + #{(t',k') before (t,k) in
 *                       row-major order with topk_ids[t',k'] == e}         [T*K]
 *   src_token[row]    = t for row = dst_row[t,k]                           [T*K]
 *
 * So packed row ranges [expert_offsets[e], expert_offsets[e+1]) hold expert
 * e's tokens in ascending token order, and rank r's region is rows
 * [rank_offsets[r], rank_offsets[r+1]).
 *
 * topk_ids     [T,K] int32, 4-byte aligned.
 * T >= 0, 1 <= K <= min(E, MOE_MAX_TOPK), 1 <= E <= MOE_MAX_EXPERTS,
 * R >= 1 with E % R == 0, T*K < 2^31, and T*K small enough for the kernels'
 * shared memory: at least 6.5 * 10^8 / E entries (671 K for E = 1024, 6.4 M
 * for E = 128); larger batches return MOE_ERR_INVALID_ARG.
 * Outputs (int32, 4-byte aligned): expert_counts, expert_offsets,
 * rank_offsets, src_token, dst_row.  dst_row and src_token may be NULL only
 * when T == 0.
 * dev_error    [1] uint32 or NULL.  Overwritten with MOE_DEV_ERR_* bits.
 *              An id outside [0,E) is not counted, gets dst_row -1 and no
 *              src_token row; src_token rows at or after expert_offsets[E]
 *              are then left untouched.  A duplicated id still gets its own
 *              slot, in k order.
 * workspace    device scratch of at least moe_layout_workspace_bytes(T,K,E)
 *              bytes, 16-byte aligned (may be NULL when that is 0).  Its
 *              contents on entry do not matter; it is in use until the
 *              stream passes this call.
 * T == 0 writes zero counts and offsets.
 */
MOE_API moe_status_t moe_layout(const int32_t *topk_ids, int32_t T, int32_t K,
                                int32_t E, int32_t R,
                                int32_t *expert_counts, int32_t *expert_offsets,
                                int32_t *rank_offsets, int32_t *src_token,
                                int32_t *dst_row, uint32_t *dev_error,
                                void *workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/*
 * moe_dispatch -- pack every token row into each of its K slots.
 *
 * The page's dispatch sender shuffles the tokens into send buffers so that
 * each destination receives one contiguous write ("Dispatch and Combine"),
 * and the evaluated setting quantises that payload to block-scaled FP8
 * ("Evaluation").  For every token t and k with 0 <= dst_row[t,k] < T*K:
 *
 *   fp8 == 0:  packed[dst_row[t,k], :] = tokens[t, :]            (bit copy)
 *   fp8 == 1:  for each 1x128 block b of row t:
 *                amax  = max |tokens[t, 128b .. 128b+127]|       (fp32)
 *                scale = amax / 448                              (fp32, RN)
 *                packed[dst_row[t,k], 128b+j] =
 *                    e4m3_satfinite_rn(tokens[t,128b+j] / scale) (fp32 divide)
 *                scales[dst_row[t,k], b] = scale
 *              a block with amax == 0 stores scale 0 and codes 0x00 / 0x80
 *              (the sign of each zero).
 * Entries with dst_row outside [0, T*K) are skipped.
 *
 * tokens   [T,H] bf16, 16-byte aligned.   dst_row [T,K] int32 (moe_layout).
 * packed   [T*K,H] bf16 (fp8 == 0) or e4m3 bytes (fp8 == 1), 16-byte aligned.
 * scales   [T*K,H/128] fp32, 4-byte aligned; required when fp8 == 1,
 *          ignored otherwise.
 * H >= 8 with H % 8 == 0 (H % 128 == 0 when fp8 == 1).  T == 0 is a no-op.
 */
MOE_API moe_status_t moe_dispatch(const void *tokens, int32_t T, int32_t H, int32_t K,
                                  const int32_t *dst_row, int32_t fp8, void *packed,
                                  float *scales, cudaStream_t stream);

/*
 * moe_combine -- routing-weighted sum of each token's K expert outputs.
 *
 * The page's combine receives the processed rows of every token and computes
 * their weighted average, accumulating only on the receiving side ("MoE
 * all-to-all over EFA", "Dispatch and Combine", "Evaluation").  With router
 * weights that already sum to one the weighted sum is that average, so no
 * division by the weight sum is made:
 *
 *   acc = +0 (fp32);  for k = 0 .. K-1:  acc = fma(topk_weights[t,k],
 *                                              expert_out[dst_row[t,k], j], acc)
 *   out[t, j] = bf16 round-to-nearest-even(acc)
 *
 * Terms whose dst_row is outside [0, T*K) are skipped.
 *
 * expert_out    [T*K,H] bf16, 16-byte aligned (rows in dispatch order).
 * topk_weights  [T,K] fp32, 4-byte aligned.   dst_row [T,K] int32.
 * out           [T,H] bf16, 16-byte aligned; must not overlap expert_out.
 * H >= 8 with H % 8 == 0.  T == 0 is a no-op.
 */
MOE_API moe_status_t moe_combine(const void *expert_out, const float *topk_weights,
                         const int32_t *dst_row, int32_t T, int32_t H,
                         int32_t K, void *out, cudaStream_t stream);

/*
 * moe_combine_fp8 -- moe_combine for expert outputs held as block-scaled e4m3.
 *
 * The evaluated setting dispatches block-scaled FP8 ("Evaluation"); when the
 * expert outputs stay in that form (e4m3 codes plus one fp32 scale per 1x128
 * block, as moe_dispatch with fp8 == 1 writes them), combine can read them
 * directly, moving about half the bytes of a bf16 combine.  Each value is
 * y = f32(code) * scale (fp32, round to nearest), then the same chain:
 *
 *   acc = +0;  for k = 0 .. K-1:  acc = fma(topk_weights[t,k], y[dst_row[t,k], j], acc)
 *   out[t, j] = bf16 round-to-nearest-even(acc)
 *
 * Terms whose dst_row is outside [0, T*K) are skipped.
 *
 * expert_out     [T*K,H] e4m3 bytes, 16-byte aligned.
 * expert_scales  [T*K,H/128] fp32, 4-byte aligned.
 * topk_weights   [T,K] fp32.   dst_row [T,K] int32.
 * out            [T,H] bf16, 16-byte aligned.
 * H >= 128 with H % 128 == 0.  T == 0 is a no-op.
 */
MOE_API moe_status_t moe_combine_fp8(const void *expert_out, const float *expert_scales,
                                     const float *topk_weights, const int32_t *dst_row,
                                     int32_t T, int32_t H, int32_t K, void *out,
                                     cudaStream_t stream);

/*
 * moe_combine_rank_partial -- combine with sender-side partial sums.
 *
 * The page accumulates only on the receiving side and contrasts this with
 * DeepEP, which sums in the sender to cut the bytes transferred, at some cost
 * in accuracy ("Evaluation").  This call computes that scheme on the same
 * data: each token's entries are grouped by the rank r = e / (E/R) hosting
 * their expert; each group is summed as the fp32 FMA chain in k order from
 * +0 and rounded to bf16 (the transfer format); the receiver adds the
 * groups' values as fp32 in ascending rank order from +0 and rounds to bf16.
 * With R == 1 or K == 1 it equals moe_combine.
 *
 * expert_out [T*K,H] bf16 (16-byte aligned), topk_weights [T,K] fp32,
 * topk_ids [T,K] int32 (the layout's input), dst_row [T,K] int32,
 * out [T,H] bf16 (16-byte aligned).  1 <= E <= MOE_MAX_EXPERTS, E % R == 0,
 * H % 8 == 0.  Entries whose expert id or dst_row is invalid are skipped.
 */
MOE_API moe_status_t moe_combine_rank_partial(const void *expert_out,
                                              const float *topk_weights,
                                              const int32_t *topk_ids,
                                              const int32_t *dst_row, int32_t T,
                                              int32_t H, int32_t K, int32_t E, int32_t R,
                                              void *out, cudaStream_t stream);

/*
 * moe_dispatch_send / moe_dispatch_recv -- dispatch through per-destination
 * send regions, then back into the grouped-GEMM input.
 *
 * The page's send-buffer design ("Send/receive buffers"): senders lay their
 * writes out contiguously once the per-expert counts are known; a small
 * private area per sender on each receiver takes the first tokens before
 * that, and the rest travel in one write per peer.  With one sender and R
 * destination ranks (rank r hosts experts r*E/R .. (r+1)*E/R - 1), rank r's
 * rows in slot order i = 0 .. n_r - 1 (n_r = rank_offsets[r+1] -
 * rank_offsets[r], from moe_layout) are written to
 *   priv[r, i]      for i < P          (the private area), or
 *   bulk[r, i - P]  for P <= i < P + C (the contiguous area),
 * and rows at i >= P + C are not written.  Rows are what moe_dispatch writes:
 * bf16 copies (fp8 == 0) or e4m3 codes with their 1x128 block scales
 * (fp8 == 1).  A region of T * min(K, E/R) rows can never overflow.
 * moe_dispatch_recv puts every region row back at its slot of `packed`
 * (and `scales`), so send + recv gives exactly the moe_dispatch output.
 *
 * priv   [R, P, row] and bulk [R, C, row], row = H bf16 or H e4m3 bytes;
 *        16-byte aligned.  priv_scales [R, P, H/128], bulk_scales [R, C, H/128]
 *        fp32 (fp8 == 1 only).  P >= 0, C >= 0.
 * topk_ids, dst_row [T, K] int32 and rank_offsets [R+1] int32 from moe_layout.
 *        rank_offsets must be moe_layout's output (non-decreasing, starting at
 *        0); moe_dispatch_recv skips packed rows outside
 *        [rank_offsets[0], rank_offsets[R]).
 * dev_error (send; may be NULL) is overwritten with
 *        MOE_DEV_ERR_REGION_OVERFLOW when some n_r exceeds P + C, else 0.
 * H % 8 == 0 (H % 128 == 0 for fp8), E % R == 0.  T == 0 is a no-op.
 */
MOE_API moe_status_t moe_dispatch_send(const void *tokens, int32_t T, int32_t H, int32_t K,
                                       int32_t E, int32_t R, const int32_t *topk_ids,
                                       const int32_t *dst_row, const int32_t *rank_offsets,
                                       int32_t fp8, int32_t P, void *priv, float *priv_scales,
                                       int32_t C, void *bulk, float *bulk_scales,
                                       uint32_t *dev_error, cudaStream_t stream);

MOE_API moe_status_t moe_dispatch_recv(const void *priv, const float *priv_scales, int32_t P,
                                       const void *bulk, const float *bulk_scales, int32_t C,
                                       const int32_t *rank_offsets, int32_t R, int32_t T,
                                       int32_t H, int32_t K, int32_t fp8, void *packed,
                                       float *scales, cudaStream_t stream);

/*
 * moe_layout_dispatch -- moe_layout followed by moe_dispatch, as one call.
 *
 * The page's dispatch-send kernel counts, scans and packs in one pass
 * ("Dispatch and Combine").  Every output is bit-identical to calling
 * moe_layout and then moe_dispatch with the same arguments.  For small
 * batches (decode shapes: T*K <= 8192 and a bounded amount of redundant
 * histogram work) it runs as a single kernel launch.  Larger batches run a
 * counting kernel and then one grid in which ranking blocks compute the
 * slots of each chunk of tokens while packing blocks copy every row as soon
 * as its chunk is ranked (two launches); where that grid's shared memory
 * would cost too much occupancy (E near 1024) they run moe_layout's kernels
 * and then the dispatch kernel.  moe_layout_dispatch_kernels() tells which.
 *
 * Arguments are those of moe_layout and moe_dispatch together, with the same
 * layouts, alignment and limits.  workspace: as for moe_layout (a buffer of
 * moe_layout_workspace_bytes(T,K,E) bytes always suffices; the single-kernel
 * path uses none).  dev_error gets moe_layout's bits and, on the two-launch
 * path, MOE_DEV_ERR_TIMEOUT when a bounded wait (1 s) expired: a packing
 * block's wait for its chunk's slots; the outputs are then unspecified.
 */
MOE_API moe_status_t moe_layout_dispatch(const int32_t *topk_ids, const void *tokens,
                                         int32_t T, int32_t H, int32_t K, int32_t E,
                                         int32_t R, int32_t fp8, int32_t *expert_counts,
                                         int32_t *expert_offsets, int32_t *rank_offsets,
                                         int32_t *src_token, int32_t *dst_row,
                                         uint32_t *dev_error, void *packed, float *scales,
                                         void *workspace, size_t workspace_bytes,
                                         cudaStream_t stream);

/* Number of kernel launches moe_layout_dispatch makes for these sizes: 1
 * when it runs as a single kernel, 2 on the two-launch path, otherwise
 * moe_layout_kernels() plus moe_dispatch's one.  0 for invalid sizes. */
MOE_API int32_t moe_layout_dispatch_kernels(int32_t T, int32_t H, int32_t K,
                                            int32_t E, int32_t fp8);

/* Bytes of the fixed scratch array that moe_layout_static uses (96 KiB). */
#define MOE_LAYOUT_STATIC_SCRATCH_BYTES (96u << 10)

/*
 * moe_layout_static -- moe_layout for callers that cannot allocate device
 * memory.  (The paper has no counterpart; this is a library convenience.)
 *
 * Some callers cannot call cudaMalloc where they need the layout: a plugin or
 * custom op run by an inference engine whose memory planner owns every device
 * allocation, or a latency-critical serving loop that must not enter the
 * device allocator once it runs (an allocation can block, synchronise or
 * fail).  This
 * call takes the same arguments and gives the same results as moe_layout, but
 * has no workspace argument: the scratch that large batches need lives in a
 * fixed array of MOE_LAYOUT_STATIC_SCRATCH_BYTES in the library's own device
 * memory, which every GPU that loads the library keeps until the process
 * exits.  The call allocates nothing (no cudaMalloc, no cudaFree).
 *
 * - Limit: a batch whose moe_layout_workspace_bytes(T,K,E) exceeds
 *   MOE_LAYOUT_STATIC_SCRATCH_BYTES is rejected with MOE_ERR_WORKSPACE.
 *   That covers every batch moe_layout accepts with E >= 2; with E = 1,
 *   batches above about 12.5 million entries are rejected.
 * - Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  Set-up failure returns MOE_ERR_CUDA.  The
 *   address is kept for the life of the process: after cudaDeviceReset on a
 *   device the kept address is stale, so do not call moe_layout_static on
 *   that device again in the same process.
 * - Sharing: all calls on a device share the one array, and it keeps the last
 *   call's contents.  Nothing in it needs to start at zero: each call writes
 *   every scratch entry before reading it.  Calls that can run at the same
 *   time on the GPU (different streams with no ordering between them) race
 *   on the array; order them on one stream or with events.
 */
MOE_API moe_status_t moe_layout_static(const int32_t *topk_ids, int32_t T, int32_t K,
                                       int32_t E, int32_t R, int32_t *expert_counts,
                                       int32_t *expert_offsets, int32_t *rank_offsets,
                                       int32_t *src_token, int32_t *dst_row,
                                       uint32_t *dev_error, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LAYOUT_H */
