// combine_common.cuh -- the fused multiply-add step shared by the combine
// kernels: eight bf16 values widened exactly, acc = fma(w, y, acc) each.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ void fma8(float acc[8], float w, const uint4 &y)
{
    acc[0] = __fmaf_rn(w, bf16_lo(y.x), acc[0]);
    acc[1] = __fmaf_rn(w, bf16_hi(y.x), acc[1]);
    acc[2] = __fmaf_rn(w, bf16_lo(y.y), acc[2]);
    acc[3] = __fmaf_rn(w, bf16_hi(y.y), acc[3]);
    acc[4] = __fmaf_rn(w, bf16_lo(y.z), acc[4]);
    acc[5] = __fmaf_rn(w, bf16_hi(y.z), acc[5]);
    acc[6] = __fmaf_rn(w, bf16_lo(y.w), acc[6]);
    acc[7] = __fmaf_rn(w, bf16_hi(y.w), acc[7]);
}

// Up to kBatch gathers are in flight per thread when K is a runtime value.
constexpr int kBatch = 8;

}  // namespace moe
