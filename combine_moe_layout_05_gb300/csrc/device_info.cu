// device_info.cu -- host-side helpers of the launchers: per-device facts
// looked up once per device and kept (the dynamic shared memory limit raised
// for each kernel, the SM count), and the block size of row-slice grids.
#include "internal.h"

#include <mutex>

namespace moe {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxKernels = 128;

struct SmemEntry {
    const void *fn;
    int dev;
    size_t dyn_max;
};

std::mutex g_mu;
SmemEntry g_smem[kMaxKernels];
int g_smem_n = 0;
int g_sms[kMaxDevices];

}  // namespace

cudaError_t allow_dynamic_smem(const void *fn, size_t bytes)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_smem_n; ++i)
        if (g_smem[i].fn == fn && g_smem[i].dev == dev)
            return bytes <= g_smem[i].dyn_max ? cudaSuccess : cudaErrorInvalidValue;
    int max_optin = 0;
    e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    const size_t dyn_max = (size_t)max_optin - fa.sharedSizeBytes;
    if (dyn_max < bytes) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_max);
    if (e == cudaSuccess && g_smem_n < kMaxKernels) g_smem[g_smem_n++] = {fn, dev, dyn_max};
    return e;
}

cudaError_t device_sm_count(int *count)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_sms[dev] == 0) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_sms[dev] = n;
    }
    *count = g_sms[dev];
    return cudaSuccess;
}

int pick_row_block(int units)
{
    for (int b = 256; b >= 64; b -= 32)
        if (units % b == 0) return b;
    return units < 128 ? ((units + 31) / 32) * 32 : 128;
}

}  // namespace moe
