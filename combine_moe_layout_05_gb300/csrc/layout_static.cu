// layout_static.cu -- moe_layout without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they need the
// layout: a plugin or custom op run by an inference engine whose memory
// planner owns every device allocation, or a latency-critical serving loop
// that must not enter the device allocator once it runs (an allocation can
// block, synchronise or fail).  For them this file
// keeps the large-batch layout's scratch in a fixed-size array in the
// library's own device memory, so the call allocates nothing.
//
// The array is file-scope device memory: every GPU that loads the library
// holds it until the process exits.  Host code cannot use its name as a
// device address, so the address is looked up once per device.
#include "internal.h"
#include "moe_layout.h"

#include <mutex>

namespace {

constexpr size_t kScratchBytes = MOE_LAYOUT_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_layout_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_layout_scratch on the current device, looked up the
// first time this device is seen (with it current).
cudaError_t scratch_address(void **out)
{
    static std::mutex mu;
    static void *addr[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_layout_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" moe_status_t moe_layout_static(const int32_t *topk_ids, int32_t T,
                                          int32_t K, int32_t E, int32_t R,
                                          int32_t *expert_counts,
                                          int32_t *expert_offsets,
                                          int32_t *rank_offsets,
                                          int32_t *src_token, int32_t *dst_row,
                                          uint32_t *dev_error, cudaStream_t stream)
{
    const size_t need = moe_layout_workspace_bytes(T, K, E);
    if (need > kScratchBytes) return MOE_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0 && scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    return moe_layout(topk_ids, T, K, E, R, expert_counts, expert_offsets,
                      rank_offsets, src_token, dst_row, dev_error, scratch,
                      need > 0 ? kScratchBytes : 0, stream);
}
