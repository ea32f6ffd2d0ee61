/*
 * moe_oracle.c -- plain, slow, single-threaded CPU oracle for MoE layout,
 * dispatch and combine.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity reference that the CUDA
 * path is checked against.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may build, load or call it; the library's
 * product path never does.  It shares no code, header, table or helper with
 * the CUDA sources.
 *
 * Source of the method: Perplexity, "Enabling trillion-parameter models on
 * AWS EFA" (blog, 2025-11-04), sections "MoE all-to-all over EFA",
 * "Send/receive buffers", "Dispatch and Combine" and "Evaluation".  The page
 * states the problem; the choices it leaves open are written next to the code
 * that makes them.
 *
 * Build: cc -O2 -ffp-contract=off -std=c11 -shared -fPIC -o liboracle.so
 * moe_oracle.c -lm.  -ffp-contract=off matters: GCC fuses a*b+c into an FMA
 * by default on aarch64, and the oracle must round exactly where this code
 * says it rounds (every fused multiply-add below is an explicit fmaf()).
 *
 * Every function here is pinned by CPU tests to something other than itself
 * (library codecs, numpy's stable sort, brute force, exact rational
 * arithmetic, closed-form error bounds); see tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16: IEEE-754 binary32 with the low 16 fraction bits removed.           */
/* ------------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* Widening is exact: the bf16 bits become the top half of a binary32. */
float oracle_bf16_to_f32(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

/* Narrowing keeps the top 16 bits and rounds on the dropped 16 bits to the
 * nearest value, ties to the one whose kept last bit is 0.  NaN stays NaN
 * (quiet, sign kept).  A carry out of the fraction moves into the exponent,
 * which is exactly how the next binade (or infinity) is reached. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u = bits_from_f32(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);           /* NaN */
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* ------------------------------------------------------------------------ */
/* e4m3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 fraction    */
/* bits, no infinities, S.1111.111 is NaN, largest finite 448 = 1.75 * 2^8, */
/* subnormals e=0 with value m * 2^-9.                                       */
/* ------------------------------------------------------------------------ */

float oracle_e4m3_to_f32(uint8_t c)
{
    int s = (c >> 7) & 1, e = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);                 /* subnormal */
    else v = ldexp((double)(8 + m), e - 7 - 3);           /* (1 + m/8) * 2^(e-7) */
    return (float)(s ? -v : v);
}

/* Round-to-nearest-even with saturation to the largest finite value.
 *
 * The magnitude a is placed in its binade 2^E <= a < 2^(E+1), with E clamped
 * to the smallest normal exponent -6 so that subnormals share its spacing.
 * A binade holds 8 steps, so the spacing there is q = 2^(E-3).  a/q is exact
 * in double; it is rounded to an integer n, ties to even, and n*q is the
 * result (n == 16 is the next power of two, still representable below 448).
 * Anything at or above 448 saturates to 448: values in (448, 464) round to
 * 448 anyway, 464 is a tie that goes to the even neighbour 448, and larger
 * values would leave the finite range, which "satfinite" forbids.  NaN input
 * is outside the contract and maps to the NaN code. */
uint8_t oracle_f32_to_e4m3_satfinite(float f)
{
    if (isnan(f)) return 0x7F;
    int neg = signbit(f) ? 1 : 0;
    double a = fabs((double)f);
    uint8_t sign = (uint8_t)(neg << 7);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a == 0.0) return sign;

    int E;
    frexp(a, &E);           /* a = fr * 2^E with 0.5 <= fr < 1 */
    E -= 1;                 /* now 2^E <= a < 2^(E+1) */
    if (E < -6) E = -6;
    double q = ldexp(1.0, E - 3);
    double n = a / q;       /* exact: a has 24 significant bits */
    double fl = floor(n);
    double frac = n - fl;
    double r;
    if (frac > 0.5) r = fl + 1.0;
    else if (frac < 0.5) r = fl;
    else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;      /* tie: even */
    double v = r * q;
    if (v == 0.0) return sign;

    if (v < ldexp(1.0, -6)) {                              /* subnormal */
        int m = (int)(v / ldexp(1.0, -9));
        return (uint8_t)(sign | m);
    }
    int Ev;
    frexp(v, &Ev);
    Ev -= 1;                                               /* 2^Ev <= v */
    int m = (int)(v / ldexp(1.0, Ev - 3)) - 8;
    return (uint8_t)(sign | ((Ev + 7) << 3) | m);
}

/* ------------------------------------------------------------------------ */
/* Layout: per-expert counts, offsets, and the stable slot of every (t,k).  */
/* ------------------------------------------------------------------------ */

/* The page's dispatch-send first counts tokens per expert, then takes the
 * cumulative sum of those counts as the offsets at which tokens are packed
 * into contiguous per-destination buffers ("Dispatch and Combine"; the counts
 * are also what ranks exchange first, "Send/receive buffers").
 *
 * Readings where the page is silent:
 *  - inside an expert's bucket, entries are ordered by token index, then by k
 *    (a stable counting sort of the flat array topk_ids[T*K] keyed by expert);
 *  - expert e lives on destination rank e / (E/R) (contiguous blocks), so
 *    rank_offsets[r] = expert_offsets[r*E/R];
 *  - an id outside [0,E) is an error (bit 1): it is not counted, gets no slot
 *    and its dst_row is -1;
 *  - the same expert twice in one token is reported (bit 2) but each entry
 *    still gets its own slot, in k order.
 *
 * Outputs: counts[E], offsets[E+1], rank_offsets[R+1], src_token[T*K] (rows
 * at or beyond offsets[E] are left untouched), dst_row[T*K].
 * Returns the error bits (bit 31: out of host memory).  Requires
 * E % R == 0 (checked by the caller). */
uint32_t oracle_layout(const int32_t *topk_ids, int32_t T, int32_t K,
                       int32_t E, int32_t R,
                       int32_t *counts, int32_t *offsets,
                       int32_t *rank_offsets, int32_t *src_token,
                       int32_t *dst_row)
{
    uint32_t err = 0;
    int64_t n = (int64_t)T * K;
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    if (!next) return 0x80000000u;

    for (int32_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t i = 0; i < n; ++i) {
        int32_t e = topk_ids[i];
        if (e < 0 || e >= E) { err |= 1u; continue; }
        counts[e] += 1;
    }

    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];

    int32_t per_rank = E / R;
    for (int32_t r = 0; r <= R; ++r) rank_offsets[r] = offsets[r * per_rank];

    for (int32_t e = 0; e < E; ++e) next[e] = offsets[e];
    for (int64_t i = 0; i < n; ++i) {          /* t ascending, then k */
        int32_t e = topk_ids[i];
        if (e < 0 || e >= E) { dst_row[i] = -1; continue; }
        int32_t row = next[e]++;
        dst_row[i] = row;
        src_token[row] = (int32_t)(i / K);
    }

    for (int32_t t = 0; t < T; ++t)
        for (int32_t a = 0; a < K; ++a)
            for (int32_t b = a + 1; b < K; ++b) {
                int32_t ea = topk_ids[(int64_t)t * K + a];
                int32_t eb = topk_ids[(int64_t)t * K + b];
                if (ea == eb && ea >= 0 && ea < E) err |= 2u;
            }
    free(next);
    return err;
}

/* ------------------------------------------------------------------------ */
/* Dispatch: pack every token row into each of its K slots.                 */
/* ------------------------------------------------------------------------ */

/* bf16 dispatch is a bit copy: packed[dst_row[t,k], :] = tokens[t, :]
 * ("Dispatch and Combine": tokens are shuffled into contiguous send buffers).
 * A dst_row outside [0, T*K) is skipped. */
void oracle_dispatch_bf16(const uint16_t *tokens, int32_t T, int32_t H,
                          int32_t K, const int32_t *dst_row, uint16_t *packed)
{
    int64_t rows = (int64_t)T * K;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t k = 0; k < K; ++k) {
            int32_t r = dst_row[(int64_t)t * K + k];
            if (r < 0 || r >= rows) continue;
            for (int32_t j = 0; j < H; ++j)
                packed[(int64_t)r * H + j] = tokens[(int64_t)t * H + j];
        }
}

/* Block-scaled FP8 dispatch ("Evaluation": block-scaled fp8 dispatch, bf16
 * combine).  The page names the scheme only; the readings taken:
 *  - blocks are 1 x 128 along the hidden dimension;
 *  - per block, amax = max |x| over the 128 values widened to fp32 (exact);
 *  - scale = amax / 448 in fp32 (IEEE division, round to nearest);
 *  - each code is e4m3 round-to-nearest-even, saturating, of x / scale
 *    (fp32 IEEE division, not a multiply by a reciprocal);
 *  - a block whose amax is 0 stores scale 0 and codes that keep only the sign
 *    of each zero (0x00 or 0x80); nothing is divided.
 * Codes and scales go to every one of the token's K slots.  scales is
 * [T*K, H/128] fp32, row-major.  Requires H % 128 == 0. */
void oracle_dispatch_fp8(const uint16_t *tokens, int32_t T, int32_t H,
                         int32_t K, const int32_t *dst_row, uint8_t *packed,
                         float *scales)
{
    int64_t rows = (int64_t)T * K;
    int32_t nb = H / 128;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t b = 0; b < nb; ++b) {
            const uint16_t *x = tokens + (int64_t)t * H + (int64_t)b * 128;
            float amax = 0.0f;
            for (int j = 0; j < 128; ++j) {
                float v = fabsf(oracle_bf16_to_f32(x[j]));
                if (v > amax) amax = v;
            }
            float scale = amax / 448.0f;
            uint8_t code[128];
            for (int j = 0; j < 128; ++j) {
                float v = oracle_bf16_to_f32(x[j]);
                if (amax == 0.0f) code[j] = signbit(v) ? 0x80 : 0x00;
                else code[j] = oracle_f32_to_e4m3_satfinite(v / scale);
            }
            for (int32_t k = 0; k < K; ++k) {
                int32_t r = dst_row[(int64_t)t * K + k];
                if (r < 0 || r >= rows) continue;
                memcpy(packed + (int64_t)r * H + (int64_t)b * 128, code, 128);
                scales[(int64_t)r * nb + b] = scale;
            }
        }
}

/* ------------------------------------------------------------------------ */
/* Combine: the routing-weighted sum of each token's K expert outputs.      */
/* ------------------------------------------------------------------------ */

/* "Dispatch and Combine" / "MoE all-to-all over EFA": the receiver gathers
 * the processed rows of each token and forms their weighted average; the
 * accumulation happens only on the receiving side ("Evaluation").
 * Readings: the weights are used as given (router weights are already
 * normalised, so the weighted sum is the weighted average and no division by
 * their sum is made); the sum runs in fp32 in k order as a chain of fused
 * multiply-adds starting from +0; the result is rounded to bf16 to nearest
 * even.  A dst_row outside [0, T*K) contributes nothing. */
void oracle_combine(const uint16_t *y, const float *topk_weights,
                    const int32_t *dst_row, int32_t T, int32_t H, int32_t K,
                    uint16_t *out)
{
    int64_t rows = (int64_t)T * K;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < H; ++j) {
            float acc = 0.0f;
            for (int32_t k = 0; k < K; ++k) {
                int32_t r = dst_row[(int64_t)t * K + k];
                if (r < 0 || r >= rows) continue;
                float w = topk_weights[(int64_t)t * K + k];
                acc = fmaf(w, oracle_bf16_to_f32(y[(int64_t)r * H + j]), acc);
            }
            out[(int64_t)t * H + j] = oracle_f32_to_bf16(acc);
        }
}

/* ------------------------------------------------------------------------ */
/* Array forms of the codecs (loops over the scalar functions above), so     */
/* the tests can sweep millions of values without a call per value.         */
/* ------------------------------------------------------------------------ */

void oracle_f32_to_bf16_n(const float *in, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(in[i]);
}

void oracle_f32_to_e4m3_n(const float *in, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_e4m3_satfinite(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Combine from FP8 expert outputs (codes + per-1x128-block scales).         */
/* ------------------------------------------------------------------------ */

/* The same weighted sum as oracle_combine, but each expert output element is
 * given as an e4m3 code q and its block's fp32 scale s, the form the
 * block-scaled FP8 dispatch produces ("Evaluation": block-scaled fp8).
 * Reading: the element's value is the fp32 product f32(q) * s (rounded to
 * nearest), exactly what dequantising the block means; the chain is then the
 * same fp32 fused multiply-add in k order from +0, rounded once to bf16.
 * codes [T*K, H] bytes, scales [T*K, H/128] fp32; H % 128 == 0. */
void oracle_combine_fp8(const uint8_t *codes, const float *scales,
                        const float *topk_weights, const int32_t *dst_row,
                        int32_t T, int32_t H, int32_t K, uint16_t *out)
{
    int64_t rows = (int64_t)T * K;
    int32_t nb = H / 128;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < H; ++j) {
            float acc = 0.0f;
            for (int32_t k = 0; k < K; ++k) {
                int32_t r = dst_row[(int64_t)t * K + k];
                if (r < 0 || r >= rows) continue;
                float w = topk_weights[(int64_t)t * K + k];
                float y = oracle_e4m3_to_f32(codes[(int64_t)r * H + j]) *
                          scales[(int64_t)r * nb + j / 128];
                acc = fmaf(w, y, acc);
            }
            out[(int64_t)t * H + j] = oracle_f32_to_bf16(acc);
        }
}

/* ------------------------------------------------------------------------ */
/* Combine with sender-side partial sums (per destination rank).            */
/* ------------------------------------------------------------------------ */

/* The page contrasts its receiver-side accumulation with DeepEP, which sums
 * in the sender to cut the bytes transferred and may lose accuracy doing so
 * ("Evaluation").  Reading of that scheme on the same data:
 *  - the sender is the rank r = e / (E/R) that hosts expert e;
 *  - for each token, each rank forms the partial sum of its own entries as
 *    the fp32 fused multiply-add chain over them in k order, from +0, and
 *    rounds it to bf16 (the transfer format) -- the accuracy loss;
 *  - the receiver adds the partials as fp32, in ascending rank order, from
 *    +0, and rounds the total to bf16.
 * Entries with an invalid expert id or dst_row are skipped.  With R == 1, or
 * one entry per token, this equals oracle_combine. */
void oracle_combine_rank_partial(const uint16_t *y, const float *topk_weights,
                                 const int32_t *topk_ids, const int32_t *dst_row,
                                 int32_t T, int32_t H, int32_t K, int32_t E,
                                 int32_t R, uint16_t *out)
{
    int64_t rows = (int64_t)T * K;
    int32_t per_rank = E / R;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < H; ++j) {
            float total = 0.0f;
            for (int32_t r = 0; r < R; ++r) {
                float part = 0.0f;
                int any = 0;
                for (int32_t k = 0; k < K; ++k) {
                    int32_t e = topk_ids[(int64_t)t * K + k];
                    int32_t row = dst_row[(int64_t)t * K + k];
                    if (e < 0 || e >= E || row < 0 || row >= rows) continue;
                    if (e / per_rank != r) continue;
                    part = fmaf(topk_weights[(int64_t)t * K + k],
                                oracle_bf16_to_f32(y[(int64_t)row * H + j]), part);
                    any = 1;
                }
                if (any) total = total + oracle_bf16_to_f32(oracle_f32_to_bf16(part));
            }
            out[(int64_t)t * H + j] = oracle_f32_to_bf16(total);
        }
}

/* ------------------------------------------------------------------------ */
/* Send and receive regions per destination rank.                           */
/* ------------------------------------------------------------------------ */

/* "Send/receive buffers": a receiving rank can get at most a bounded number
 * of tokens; senders write them contiguously once the routing information
 * (the per-expert counts) is known, and a small private area per sender on
 * each receiver takes the first tokens early, before the routing is known;
 * the rest go in one write per peer.  Reading for one sender and R
 * destinations: rank r's rows, in slot order i = 0 .. n_r - 1
 * (n_r = rank_offsets[r+1] - rank_offsets[r]), go to its private area for
 * i < P and to its contiguous bulk area at row i - P otherwise; a bulk row
 * at or beyond the capacity C is not written and sets error bit 4.  Rows
 * are the dispatched rows (bf16 copies, or e4m3 codes plus their block
 * scales), so receive (regions -> slot order) returns exactly the
 * dispatch output.  priv is [R, P, row_bytes], bulk is [R, C, row_bytes];
 * the scale arrays (fp8 only) are [R, P, H/128] and [R, C, H/128]. */
uint32_t oracle_dispatch_send(const uint8_t *packed, const float *scales,
                              const int32_t *rank_offsets, int32_t R,
                              int32_t row_bytes, int32_t nb, int32_t P,
                              int32_t C, uint8_t *priv, float *priv_scales,
                              uint8_t *bulk, float *bulk_scales)
{
    uint32_t err = 0;
    for (int32_t r = 0; r < R; ++r) {
        int32_t n_r = rank_offsets[r + 1] - rank_offsets[r];
        for (int32_t i = 0; i < n_r; ++i) {
            int64_t src = (int64_t)rank_offsets[r] + i;
            uint8_t *dst;
            float *dsc;
            if (i < P) {
                dst = priv + ((int64_t)r * P + i) * row_bytes;
                dsc = priv_scales ? priv_scales + ((int64_t)r * P + i) * nb : 0;
            } else if (i - P < C) {
                dst = bulk + ((int64_t)r * C + (i - P)) * row_bytes;
                dsc = bulk_scales ? bulk_scales + ((int64_t)r * C + (i - P)) * nb : 0;
            } else {
                err |= 4u;
                continue;
            }
            memcpy(dst, packed + src * row_bytes, (size_t)row_bytes);
            if (dsc) memcpy(dsc, scales + src * nb, sizeof(float) * (size_t)nb);
        }
    }
    return err;
}

/* The receiving side: regions back to slot order (the grouped-GEMM input). */
void oracle_dispatch_recv(const uint8_t *priv, const float *priv_scales,
                          const uint8_t *bulk, const float *bulk_scales,
                          const int32_t *rank_offsets, int32_t R, int32_t row_bytes,
                          int32_t nb, int32_t P, int32_t C, uint8_t *packed,
                          float *scales)
{
    for (int32_t r = 0; r < R; ++r) {
        int32_t n_r = rank_offsets[r + 1] - rank_offsets[r];
        for (int32_t i = 0; i < n_r; ++i) {
            int64_t dst = (int64_t)rank_offsets[r] + i;
            const uint8_t *src;
            const float *ssc;
            if (i < P) {
                src = priv + ((int64_t)r * P + i) * row_bytes;
                ssc = priv_scales ? priv_scales + ((int64_t)r * P + i) * nb : 0;
            } else if (i - P < C) {
                src = bulk + ((int64_t)r * C + (i - P)) * row_bytes;
                ssc = bulk_scales ? bulk_scales + ((int64_t)r * C + (i - P)) * nb : 0;
            } else {
                continue;
            }
            memcpy(packed + dst * row_bytes, src, (size_t)row_bytes);
            if (ssc) memcpy(scales + dst * nb, ssc, sizeof(float) * (size_t)nb);
        }
    }
}
