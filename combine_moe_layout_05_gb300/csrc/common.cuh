// common.cuh -- small device helpers shared by the layout, dispatch and
// combine kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

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

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace moe
