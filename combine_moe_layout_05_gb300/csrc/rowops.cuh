// rowops.cuh -- the per-thread pieces of the row kernels: the flat piece
// indexing shared by dispatch and combine, writing one 16-byte piece of a
// token row to all of its slots, and quantising 16 values of a 1x128 block
// to e4m3 with the block's scale.
#pragma once

#include "common.cuh"
#include "moe_layout.h"

namespace moe {

// Threads per block of the row-copy kernels.  Blocks walk the flat sequence
// of 16-byte pieces of all token rows, so one block may cover the end of one
// row and the start of the next: every block size keeps 8 warps whatever H
// is (a block per row slice would leave 7-warp blocks at H = 7168, and at 40
// registers only 6 of those fit an SM where 6 of 8 warps do).
constexpr int kRowThreads = 256;
constexpr int kMaxRowPieces = 1 << 23;   // pieces per row the flat indexing allows

// Token and piece index within the row.
struct RowPiece {
    int t;
    int u;
};

// Where block q of kRowThreads pieces starts in rows of per_row pieces:
// token t = q * kRowThreads / per_row and piece u within it, with 32-bit
// divisions only (q = A * per_row + B gives q * kRowThreads / per_row =
// A * kRowThreads + B * kRowThreads / per_row).  Needs per_row < 2^23.
__device__ __forceinline__ RowPiece flat_block_start(unsigned q, int per_row)
{
    const unsigned n = (unsigned)per_row;
    const unsigned A = q / n, B = q - A * n;
    const unsigned C = B * kRowThreads, D = C / n;
    return RowPiece{(int)(A * kRowThreads + D), (int)(C - D * n)};
}

// Blocks of kRowThreads pieces covering T rows of per_row pieces; 0 past
// the grid limit (2^31 - 1) or the flat indexing's row length.
inline unsigned row_blocks(int T, int per_row)
{
    const long long n = ((long long)T * per_row + kRowThreads - 1) / kRowThreads;
    return n <= 0x7fffffffll && per_row < kMaxRowPieces ? (unsigned)n : 0u;
}

// Whether the bf16 combine walks flat pieces: for grids of many waves,
// where 8-warp blocks keep more warps resident than row slices of fewer
// threads; single-wave (decode-sized) grids keep one token per block, which
// measured faster there.  (The dispatch kernels always walk flat pieces; the
// FP8 combine keeps one token per block, as flat indexing spilled at its 64
// registers.)
inline bool flat_rows(int T, int per_row)
{
    return (long long)T * per_row >= (1ll << 20) && per_row < kMaxRowPieces;
}

// Token and piece index of piece `tid` of block q (per_row < 2^23).
__device__ __forceinline__ RowPiece flat_piece(unsigned q, int per_row, int tid)
{
    const RowPiece s = flat_block_start(q, per_row);
    const int off = s.u + tid;
    const int dt = off / per_row;
    return RowPiece{s.t + dt, off - dt * per_row};
}

// Writes `x` (16 bytes at byte offset `off` of a packed row) to each slot in
// slots[0 .. k_count); slots outside [0, rows) are skipped.  `slots` may
// point to global or shared memory or to registers.  KT > 0 is a
// compile-time k_count.  All slots of a group of 8 are read before its first
// store (a store is an ordering point for the compiler, so a slot read after
// it would add one memory latency per slot).
template <int KT>
__device__ __forceinline__ void store_to_slots(const int32_t *slots, int k_count,
                                               int rows, uint8_t *packed,
                                               size_t row_bytes, size_t off,
                                               const uint4 &x)
{
    constexpr int G = KT > 0 && KT < 8 ? KT : 8;
    for (int k0 = 0; k0 < k_count; k0 += G) {
        int r[G];
#pragma unroll
        for (int j = 0; j < G; ++j) r[j] = (KT > 0 || k0 + j < k_count) ? slots[k0 + j] : -1;
#pragma unroll
        for (int j = 0; j < G; ++j)
            if ((unsigned)r[j] < (unsigned)rows) st_v4(packed + (size_t)r[j] * row_bytes + off, x);
    }
}

// Block-scaled e4m3 of the 16 bf16 values in (a, b).  The 8 consecutive
// lanes holding one 128-value block must all call this together (xor
// shuffles over lane groups of 8; every lane of the warp participates).
// amax is exact in fp32, scale = amax / 448 and every value is divided by
// the scale with IEEE round-to-nearest division before the saturating
// round-to-nearest-even conversion; an all-zero block keeps only the signs.
struct Fp8Piece {
    uint4 codes;
    float scale;
};

__device__ __forceinline__ Fp8Piece quantize16(const uint4 &a, const uint4 &b)
{
    float x[16];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        x[2 * i] = bf16_lo(w[i]);
        x[2 * i + 1] = bf16_hi(w[i]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 4));

    Fp8Piece p;
    p.scale = __fdiv_rn(amax, 448.0f);
    uint32_t q[4];
    if (amax == 0.0f) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t s = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                s |= (__float_as_uint(x[4 * i + j]) >> 31) << (8 * j + 7);
            q[i] = s;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = cvt_e4m3x2_satfinite(__fdiv_rn(x[4 * i], p.scale),
                                                     __fdiv_rn(x[4 * i + 1], p.scale));
            const uint32_t hi = cvt_e4m3x2_satfinite(__fdiv_rn(x[4 * i + 2], p.scale),
                                                     __fdiv_rn(x[4 * i + 3], p.scale));
            q[i] = lo | (hi << 16);
        }
    }
    p.codes = make_uint4(q[0], q[1], q[2], q[3]);
    return p;
}

// Writes a quantised piece (group g of 16 values) and, from the block's
// first lane, its scale, to each slot (slots read as in store_to_slots).
template <int KT>
__device__ __forceinline__ void store_fp8_to_slots(const int32_t *slots, int k_count,
                                                   int rows, uint8_t *packed,
                                                   float *scales, int H, int g,
                                                   const Fp8Piece &p)
{
    const int nb = H >> 7;
    const bool leader = (g & 7) == 0;
    constexpr int G = KT > 0 && KT < 8 ? KT : 8;
    for (int k0 = 0; k0 < k_count; k0 += G) {
        int r[G];
#pragma unroll
        for (int j = 0; j < G; ++j) r[j] = (KT > 0 || k0 + j < k_count) ? slots[k0 + j] : -1;
#pragma unroll
        for (int j = 0; j < G; ++j) {
            if ((unsigned)r[j] >= (unsigned)rows) continue;
            st_v4(packed + (size_t)r[j] * H + 16 * (size_t)g, p.codes);
            if (leader) scales[(size_t)r[j] * nb + (g >> 3)] = p.scale;
        }
    }
}

}  // namespace moe
