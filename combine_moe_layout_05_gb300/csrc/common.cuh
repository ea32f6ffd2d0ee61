// common.cuh -- small device helpers shared by the layout, dispatch and
// combine kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace moe {

constexpr unsigned kFullMask = 0xffffffffu;

// 16-byte load of data that stays read-only for the kernel's lifetime and is
// touched once: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// 8-byte load of read-only data touched once (no L1 allocation).
__device__ __forceinline__ uint2 ld_stream_v2(const void *p)
{
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
        : "=r"(r.x), "=r"(r.y)
        : "l"(p));
    return r;
}

// 8-byte store.
__device__ __forceinline__ void st_v2(void *p, const uint2 &v)
{
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// 16-byte store.
__device__ __forceinline__ void st_v4(void *p, const uint4 &v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// The two bf16 halves of a 32-bit word, widened exactly to fp32.
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Two fp32 values rounded to bf16 (nearest, ties to even) and packed with
// `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Two fp32 values converted to e4m3 (nearest, ties to even, saturating to
// +-448), `lo` in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2_satfinite(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two e4m3 codes (low byte first) widened exactly to fp32 via f16x2.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t codes)
{
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(codes));
    __half2 v = *reinterpret_cast<__half2 *>(&h);
    return __half22float2(v);
}

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr int align4(int n) { return (n + 3) & ~3; }

// Copies n int32 values from global to shared memory with asynchronous
// copies issued by all threads of the block, or by the `nthreads` threads
// numbered `tid` = 0 .. nthreads-1 (every request is in flight at once, so
// the block pays one memory latency, not one per loop trip).  The caller
// must call cp_async_wait_all() and then synchronise those threads.
__device__ __forceinline__ void stage_i32(int32_t *dst, const int32_t *src, int n,
                                          int tid = -1, int nthreads = 0)
{
    if (tid < 0) {
        tid = threadIdx.x;
        nthreads = blockDim.x;
    }
    const unsigned base = (unsigned)__cvta_generic_to_shared(dst);
    const bool vec = ((reinterpret_cast<uintptr_t>(src) | base) & 15) == 0;
    int done = 0;
    if (vec) {
        const int n4 = n >> 2;
        for (int i = tid; i < n4; i += nthreads)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                         :: "r"(base + 16u * i), "l"(src + 4 * i) : "memory");
        done = n4 << 2;
    }
    for (int i = done + tid; i < n; i += nthreads)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;"
                     :: "r"(base + 4u * i), "l"(src + i) : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Programmatic dependent launch.  Every kernel here is launched with
// programmatic stream serialisation, so it may start while the previous
// kernel in the stream is finishing.  It must not touch global memory before
// pdl_wait(), which returns once that kernel has completed and its writes are
// visible (immediately when there is no such kernel).  pdl_trigger() lets the
// next kernel in the stream start its own prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Host-side launch with programmatic stream serialisation allowed and, when
// cluster > 1, the grid's blocks in thread-block clusters of that many
// (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_clusters(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, unsigned cluster, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                       size_t smem, cudaStream_t stream, Args... args)
{
    return launch_pdl_clusters(kernel, grid, block, smem, stream, 1u, args...);
}

}  // namespace moe
