"""Pins for the oracle's dispatch (bf16 and block-scaled FP8) and combine.

* bf16 dispatch: bit identity of every packed row with its source row.
* FP8 dispatch: each code is the nearest e4m3 value of x/scale found by
  exhaustive search over the code table (ties to the even code, saturating);
  the dequantisation error obeys the closed-form bound of the block scale; the
  block's largest element decodes to exactly +-448 * scale.
* combine: exact rational arithmetic (Python fractions) of the defined fp32
  fused-multiply-add chain, including cases built so that a separate
  multiply and add, another k order or a non-zero start would differ; the
  identity round trip combine(dispatch(x)) == x; the closed form
  sum_k w_k * s_e * x for per-expert-scalar experts.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from combine_moe_layout_05_gb300 import workload as wl


def f32(bits_u16):
    return wl.bf16_bits_to_f32(bits_u16)


# ---------------------------------------------------------------- dispatch --

@pytest.mark.parametrize("name", ["tiny", "decode_dsv3", "prefill_kimi_k2"])
def test_dispatch_bf16_bit_identity(oracle, name):
    w = wl.get(name)
    inp = wl.make_inputs(w, T=min(w.T, 512))
    lay = oracle.layout(inp.topk_ids, w.E, w.R)
    packed = oracle.dispatch_bf16(inp.tokens, lay.dst_row)
    assert np.array_equal(packed, inp.tokens[lay.src_token])
    for t in range(0, inp.tokens.shape[0], 37):
        for k in range(w.K):
            assert np.array_equal(packed[lay.dst_row[t, k]], inp.tokens[t])


def _e4m3_table():
    v = torch.from_numpy(np.arange(128, dtype=np.uint8)).view(
        torch.float8_e4m3fn).float().numpy().astype(np.float64)
    return v[:127]


def _nearest_even_code(v_abs):
    table = _e4m3_table()
    codes = np.arange(127)[None, :]
    out = np.empty(v_abs.size, np.int64)
    for s in range(0, v_abs.size, 32768):
        a = np.minimum(v_abs[s:s + 32768], 448.0)
        d = np.abs(a[:, None] - table[None, :])
        cand = d == d.min(axis=1, keepdims=True)
        tie = cand.sum(axis=1) > 1
        even = np.where(cand & (codes % 2 == 0), codes, 999).min(axis=1)
        first = np.where(cand, codes, 999).min(axis=1)
        out[s:s + 32768] = np.where(tie, even, first)
    return out


@pytest.mark.parametrize("name,T", [("tiny", 64), ("decode_dsv3_fp8", 16),
                                    ("prefill_qwen3", 40)])
def test_dispatch_fp8_codes_by_search_and_bound(oracle, name, T):
    w = wl.get(name)
    inp = wl.make_inputs(w, T=T)
    # plant zero blocks (with signed zeros) and a denormal-only block
    x_bits = inp.tokens.copy()
    x_bits[0, :128] = 0
    x_bits[0, 3] = 0x8000
    if T > 1:
        x_bits[1, 128:256] = 0x0001          # smallest bf16 subnormal
    lay = oracle.layout(inp.topk_ids, w.E, w.R)
    codes, scales = oracle.dispatch_fp8(x_bits, lay.dst_row)
    H, nb = w.H, w.H // 128
    x = f32(x_bits).reshape(T, nb, 128)
    amax = np.abs(x).max(axis=2)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    # every slot of a token carries the same codes and scales
    src = lay.src_token
    got_codes = codes.reshape(T * w.K, nb, 128)
    got_scales = scales
    assert np.array_equal(got_scales.view(np.uint32), scale[src].view(np.uint32))

    v = np.zeros_like(x)
    nz = amax > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        v = np.where(nz[:, :, None], x / scale[:, :, None], x)   # fp32 divide
    exp_mag = _nearest_even_code(np.abs(v.astype(np.float64)).ravel())
    exp_mag = np.where(nz[:, :, None].repeat(128, 2).ravel(), exp_mag, 0)
    exp = (exp_mag | (np.signbit(v.ravel()).astype(np.int64) << 7)).astype(np.uint8)
    exp = exp.reshape(T, nb, 128)
    assert np.array_equal(got_codes, exp[src])

    # closed-form bound: |x - q*scale| <= scale * (half spacing at |x/scale|)
    # + |x| * 2^-23 (the rounding of x/scale itself), which is <= amax/28
    q = torch.from_numpy(got_codes.reshape(-1)).view(torch.float8_e4m3fn).float().numpy()
    q = q.reshape(T * w.K, nb, 128).astype(np.float64)
    deq = q * got_scales[:, :, None].astype(np.float64)
    xs = x[src].astype(np.float64)
    err = np.abs(xs - deq)
    sc = got_scales[:, :, None].astype(np.float64)
    vabs = np.abs(xs) / np.maximum(sc, 1e-300)
    e = np.floor(np.log2(np.maximum(vabs, 2.0 ** -6)))
    half = np.exp2(e - 4)
    bound = sc * half * (1 + 2.0 ** -20) + np.abs(xs) * 2.0 ** -23
    assert np.all(err <= bound + 1e-300)
    amax_s = amax[src].astype(np.float64)
    assert np.all(err <= amax_s[:, :, None] / 28 * (1 + 2.0 ** -20))
    # the element holding amax decodes to +-448 * scale exactly
    idx = np.argmax(np.abs(xs), axis=2)
    qa = np.take_along_axis(q, idx[:, :, None], 2)[:, :, 0]
    big = amax_s > 0
    assert np.all(np.abs(qa[big]) == 448.0)


# ----------------------------------------------------------------- combine --

def _round_fraction(q: Fraction, mant_bits: int) -> Fraction:
    """Round a rational to the nearest binary float with `mant_bits` fraction
    bits and fp32's exponent range, ties to even (no overflow here)."""
    if q == 0:
        return Fraction(0)
    s = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)
    step = Fraction(2) ** (e - mant_bits)
    n = a / step
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return s * fl * step


def exact_combine(y_bits, w, dst_row):
    """The defined combine in exact arithmetic: acc starts at +0, each step
    rounds w*y + acc once to fp32, the end result rounds once to bf16."""
    T, K = dst_row.shape
    H = y_bits.shape[1]
    yf = f32(y_bits)
    out = np.zeros((T, H), np.uint16)
    for t in range(T):
        for j in range(H):
            acc = Fraction(0)
            for k in range(K):
                r = dst_row[t, k]
                acc = _round_fraction(Fraction(float(w[t, k])) * Fraction(float(yf[r, j])) + acc, 23)
            b = _round_fraction(acc, 7)
            out[t, j] = wl.to_bf16_bits(np.array([float(b)], np.float32))[0]
            if b == 0:
                out[t, j] = 0            # +0: the chain starts at +0
    return out


def test_combine_exact_rational_random(oracle):
    rng = np.random.default_rng(3)
    for trial in range(6):
        T, H, K = 3, 8, (1, 2, 3, 4, 8, 5)[trial]
        y = wl.to_bf16_bits((rng.standard_normal((T * K, H)) *
                             np.exp2(rng.integers(-20, 20, (T * K, H)))).astype(np.float32))
        w = (rng.standard_normal((T, K)) * np.exp2(rng.integers(-8, 8, (T, K)))).astype(np.float32)
        dst = rng.permutation(T * K).astype(np.int32).reshape(T, K)
        got = oracle.combine(y, w, dst)
        assert np.array_equal(got, exact_combine(y, w, dst)), trial


def test_combine_exact_rational_fma_sensitive(oracle):
    """w0*y0 + w1*y1 with y1 = -y0: the fused chain leaves exactly the
    rounding error of w0*y0; a separate multiply and add would give 0."""
    w0 = np.float32(1 + 2.0 ** -23)
    y0 = np.float32(1 - 2.0 ** -8)
    y = wl.to_bf16_bits(np.array([[y0] * 8, [-y0] * 8], np.float32))
    w = np.array([[w0, w0]], np.float32)
    dst = np.array([[0, 1]], np.int32)
    got = oracle.combine(y, w, dst)
    exp = exact_combine(y, w, dst)
    assert np.array_equal(got, exp)
    assert np.all(f32(got) != 0)          # nonzero only with a fused chain
    # order matters: a large term first then cancelling small terms
    y2 = wl.to_bf16_bits(np.array([[2.0 ** 30] * 8, [1.0] * 8, [-(2.0 ** 30)] * 8],
                                  np.float32))
    w2 = np.array([[1.0, 1.0, 1.0]], np.float32)
    d2 = np.array([[0, 1, 2]], np.int32)
    got2 = oracle.combine(y2, w2, d2)
    assert np.array_equal(got2, exact_combine(y2, w2, d2))
    assert np.all(got2 == 0)              # 2^30 + 1 rounds to 2^30 in fp32
    d3 = np.array([[0, 2, 1]], np.int32)  # other order: exact 1.0
    got3 = oracle.combine(y2, w2, d3)
    assert np.all(f32(got3) == 1.0)


def test_combine_signed_zero_start(oracle):
    """All terms -0: a chain starting at +0 ends at +0."""
    y = np.full((2, 8), 0x8000, np.uint16)
    w = np.array([[1.0, 1.0]], np.float32)
    got = oracle.combine(y, w, np.array([[0, 1]], np.int32))
    assert np.all(got == 0x0000)


@pytest.mark.parametrize("name", ["tiny", "decode_dsv3", "prefill_qwen3"])
def test_identity_round_trip(oracle, name):
    """combine(dispatch(x)) with identity experts and weights summing to one
    returns x: the fp32 sum is within K*2^-24 relative of x, far inside half a
    bf16 step, so rounding lands back on x."""
    w = wl.get(name)
    inp = wl.make_inputs(w, T=min(w.T, 256))
    lay = oracle.layout(inp.topk_ids, w.E, w.R)
    packed = oracle.dispatch_bf16(inp.tokens, lay.dst_row)
    out = oracle.combine(packed, inp.topk_weights, lay.dst_row)
    # equal as numbers; a -0 input comes back as +0 (the chain starts at +0)
    assert np.array_equal(f32(out), f32(inp.tokens))
    nz = f32(inp.tokens) != 0
    assert np.array_equal(out[nz], inp.tokens[nz])


def test_identity_single_expert(oracle):
    rng = np.random.default_rng(9)
    x = wl.to_bf16_bits(rng.standard_normal((32, 64)).astype(np.float32))
    ids = rng.integers(0, 4, (32, 1)).astype(np.int32)
    lay = oracle.layout(ids, 4, 2)
    packed = oracle.dispatch_bf16(x, lay.dst_row)
    out = oracle.combine(packed, np.ones((32, 1), np.float32), lay.dst_row)
    assert np.array_equal(out, x)


def test_per_expert_scalar_closed_form(oracle):
    """y = bf16(x * s_e): out matches sum_k w_k * y_k (exact in fp64) within
    the fp32 chain's error and one bf16 rounding."""
    w = wl.get("decode_dsv3")
    inp = wl.make_inputs(w, T=32)
    lay = oracle.layout(inp.topk_ids, w.E, w.R)
    packed = oracle.dispatch_bf16(inp.tokens, lay.dst_row)
    e_of_row = np.searchsorted(lay.expert_offsets[1:], np.arange(32 * w.K), side="right")
    y = wl.to_bf16_bits(f32(packed) * inp.expert_scale[e_of_row][:, None])
    out = oracle.combine(y, inp.topk_weights, lay.dst_row)
    yd = f32(y).astype(np.float64)
    exact = np.einsum("tk,tkh->th", inp.topk_weights.astype(np.float64),
                      yd[lay.dst_row])
    mag = np.einsum("tk,tkh->th", np.abs(inp.topk_weights.astype(np.float64)),
                    np.abs(yd[lay.dst_row]))
    err = np.abs(f32(out).astype(np.float64) - exact)
    assert np.all(err <= np.abs(exact) * 2.0 ** -8 + mag * w.K * 2.0 ** -23 + 1e-30)


# ------------------------------------------------------ combine, FP8 input --

def exact_combine_fp8(codes, scales, w, dst_row):
    """Exact rationals: value = round_f32(f32(code) * scale), then the fp32
    FMA chain from +0 and one bf16 rounding."""
    T, K = dst_row.shape
    H = codes.shape[1]
    dec = torch.from_numpy(codes.reshape(-1)).view(torch.float8_e4m3fn).float().numpy().reshape(codes.shape)
    out = np.zeros((T, H), np.uint16)
    for t in range(T):
        for j in range(H):
            acc = Fraction(0)
            for k in range(K):
                r = dst_row[t, k]
                y = _round_fraction(Fraction(float(dec[r, j])) * Fraction(float(scales[r, j // 128])), 23)
                acc = _round_fraction(Fraction(float(w[t, k])) * y + acc, 23)
            b = _round_fraction(acc, 7)
            out[t, j] = 0 if b == 0 else wl.to_bf16_bits(np.array([float(b)], np.float32))[0]
    return out


def test_combine_fp8_exact_rational(oracle):
    rng = np.random.default_rng(21)
    for K in (1, 3, 8):
        T, H = 2, 128
        codes = rng.integers(0, 256, (T * K, H)).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x3C               # no NaN codes
        scales = (rng.random((T * K, 1)) * np.exp2(rng.integers(-20, 20, (T * K, 1)))).astype(np.float32)
        w = rng.standard_normal((T, K)).astype(np.float32)
        dst = rng.permutation(T * K).astype(np.int32).reshape(T, K)
        got = oracle.combine_fp8(codes, scales, w, dst)
        assert np.array_equal(got, exact_combine_fp8(codes, scales, w, dst)), K


def test_combine_fp8_equals_bf16_combine_when_exact(oracle):
    """With power-of-two scales the dequantised values are exact in bf16, so
    the FP8-input combine equals the (pinned) bf16 combine of those values."""
    rng = np.random.default_rng(22)
    T, H, K = 16, 256, 4
    codes = rng.integers(0, 256, (T * K, H)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x40
    scales = np.exp2(rng.integers(-10, 10, (T * K, H // 128))).astype(np.float32)
    w = rng.standard_normal((T, K)).astype(np.float32)
    dst = rng.permutation(T * K).astype(np.int32).reshape(T, K)
    dec = torch.from_numpy(codes.reshape(-1)).view(torch.float8_e4m3fn).float().numpy().reshape(codes.shape)
    y = wl.to_bf16_bits(dec * np.repeat(scales, 128, axis=1))
    assert np.array_equal(f32(y), dec * np.repeat(scales, 128, axis=1))   # exact
    assert np.array_equal(oracle.combine_fp8(codes, scales, w, dst), oracle.combine(y, w, dst))


def test_combine_fp8_round_trip(oracle):
    """FP8 dispatch then FP8-input combine returns x within the block bound."""
    w = wl.get("prefill_qwen3")
    inp = wl.make_inputs(w, T=24)
    lay = oracle.layout(inp.topk_ids, w.E, w.R)
    codes, scales = oracle.dispatch_fp8(inp.tokens, lay.dst_row)
    out = f32(oracle.combine_fp8(codes, scales, inp.topk_weights, lay.dst_row)).astype(np.float64)
    x = f32(inp.tokens).astype(np.float64).reshape(24, -1, 128)
    amax = np.abs(x).max(axis=2, keepdims=True)
    err = np.abs(out.reshape(24, -1, 128) - x)
    assert np.all(err <= amax / 28 * 1.01 + np.abs(x) * 2.0 ** -7)


def test_combine_fp8_rounding_sensitive(oracle):
    """Token i: w_i * (q_i * s_i) - 1 * (q_i * 1) with w_i, s_i = 1 + small
    multiples of 2^-23: the result is a few fp32 ulps of q_i, exact in bf16,
    so it shows whether the value is round(q*s) before the FMA (the reading)
    or the scale folded into the weight, or the product left unrounded."""
    dec = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).float().numpy()
    cases = []
    for code in range(0x38, 0x40):                      # 1 + m/8, m = 0..7
        for a in range(-6, 7):
            for b in range(-6, 7):
                w = np.float32(1 + a * 2.0 ** -23)
                s = np.float32(1 + b * 2.0 ** -23)
                q = np.float32(dec[code])
                reading = np.float32(w * np.float32(q * s))
                folded = np.float32(np.float32(w * s) * q)
                exact = np.float32(float(w) * float(q) * float(s))
                cases.append((code, w, s, reading != folded or reading != exact))
    assert sum(c[3] for c in cases) >= 20               # the set separates the orders
    T, H, K = len(cases), 128, 2
    codes = np.zeros((T * K, H), np.uint8)
    scales = np.ones((T * K, 1), np.float32)
    wts = np.zeros((T, K), np.float32)
    dst = np.arange(T * K, dtype=np.int32).reshape(T, K)
    for i, (code, w, s, _) in enumerate(cases):
        codes[2 * i] = code
        codes[2 * i + 1] = code
        scales[2 * i] = s
        wts[i] = (w, -1.0)
    got = oracle.combine_fp8(codes, scales, wts, dst)
    assert np.array_equal(got, got[:, :1].repeat(H, 1))  # every column is the same sum
    for i in range(T):                                   # column 0, exact rationals
        acc = Fraction(0)
        for k in range(K):
            y = _round_fraction(Fraction(float(dec[codes[2 * i + k, 0]])) *
                                Fraction(float(scales[2 * i + k, 0])), 23)
            acc = _round_fraction(Fraction(float(wts[i, k])) * y + acc, 23)
        b = _round_fraction(acc, 7)
        e = 0 if b == 0 else wl.to_bf16_bits(np.array([float(b)], np.float32))[0]
        assert got[i, 0] == e, i
    assert np.count_nonzero(got[:, 0]) > T // 2        # outputs carry the low bits


# ----------------------------------------- combine, sender-side partial sums --

def exact_rank_partial(y_bits, w, ids, dst_row, E, R):
    """Exact rationals of the reading: per rank an fp32 FMA chain in k order
    from +0 rounded to bf16, then the fp32 add chain over ranks in ascending
    order from +0 and a final bf16 rounding."""
    T, K = dst_row.shape
    H = y_bits.shape[1]
    yf = f32(y_bits)
    out = np.zeros((T, H), np.uint16)
    for t in range(T):
        ranks = sorted({int(ids[t, k]) // (E // R) for k in range(K)})
        for j in range(H):
            total = Fraction(0)
            for r in ranks:
                part = Fraction(0)
                for k in range(K):
                    if int(ids[t, k]) // (E // R) == r:
                        part = _round_fraction(Fraction(float(w[t, k])) * Fraction(float(yf[dst_row[t, k], j])) + part, 23)
                total = _round_fraction(total + _round_fraction(part, 7), 23)
            b = _round_fraction(total, 7)
            out[t, j] = 0 if b == 0 else wl.to_bf16_bits(np.array([float(b)], np.float32))[0]
    return out


def test_rank_partial_exact_rational(oracle):
    rng = np.random.default_rng(41)
    for (T, K, E, R) in [(3, 4, 8, 2), (2, 8, 16, 4), (4, 3, 6, 3), (2, 6, 12, 12)]:
        H = 8
        ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
        lay = oracle.layout(ids, E, R)
        y = wl.to_bf16_bits((rng.standard_normal((T * K, H)) *
                             np.exp2(rng.integers(-6, 6, (T * K, H)))).astype(np.float32))
        w = rng.standard_normal((T, K)).astype(np.float32)
        got = oracle.combine_rank_partial(y, w, ids, lay.dst_row, E, R)
        assert np.array_equal(got, exact_rank_partial(y, w, ids, lay.dst_row, E, R)), (T, K, E, R)


def test_rank_partial_reduces_to_combine(oracle):
    """One rank (R = 1), or one entry per token: no intermediate rounding is
    added, so the result is the (pinned) receiver-side combine's."""
    w = wl.get("decode_dsv3")
    inp = wl.make_inputs(w, T=32)
    for R in (1,):
        lay = oracle.layout(inp.topk_ids, w.E, R)
        y = oracle.dispatch_bf16(inp.tokens, lay.dst_row)
        assert np.array_equal(oracle.combine_rank_partial(y, inp.topk_weights, inp.topk_ids, lay.dst_row, w.E, R),
                              oracle.combine(y, inp.topk_weights, lay.dst_row))
    ids1 = inp.topk_ids[:, :1].copy()
    lay = oracle.layout(ids1, w.E, w.R)
    y = oracle.dispatch_bf16(inp.tokens, lay.dst_row)
    w1 = inp.topk_weights[:, :1].copy()
    assert np.array_equal(oracle.combine_rank_partial(y, w1, ids1, lay.dst_row, w.E, w.R),
                          oracle.combine(y, w1, lay.dst_row))


def test_rank_partial_accuracy_cost(oracle):
    """The sender-side scheme is within its extra rounding bound of the exact
    sum, and it does differ from the receiver-side result on real routing."""
    w = wl.get("decode_dsv3")
    inp = wl.make_inputs(w, T=64)
    lay = oracle.layout(inp.topk_ids, w.E, w.R)
    y = wl.to_bf16_bits(f32(oracle.dispatch_bf16(inp.tokens, lay.dst_row)) *
                        inp.expert_scale[np.searchsorted(lay.expert_offsets[1:], np.arange(64 * w.K), side="right")][:, None])
    part = f32(oracle.combine_rank_partial(y, inp.topk_weights, inp.topk_ids, lay.dst_row, w.E, w.R)).astype(np.float64)
    recv = f32(oracle.combine(y, inp.topk_weights, lay.dst_row)).astype(np.float64)
    yd = f32(y).astype(np.float64)
    terms = inp.topk_weights.astype(np.float64)[:, :, None] * yd[lay.dst_row]
    exact = terms.sum(axis=1)
    mag = np.abs(terms).sum(axis=1)
    # each of <= K partials rounds to bf16 (2^-9 relative), plus the final rounding
    assert np.all(np.abs(part - exact) <= mag * (w.K + 1) * 2.0 ** -8 + 1e-30)
    assert np.count_nonzero(part != recv) > 0


def test_rank_partial_order_sensitive(oracle):
    """Terms 2^30, -2^30, 1 (2^30 + 1 rounds to 2^30 in fp32): in the defined
    orders the sum is exactly 1, any other order gives 0."""
    big = 2.0 ** 30
    # ranks in ascending order: experts 0, 2, 4 on ranks 0, 1, 2 (E=6, R=3)
    ids_a = np.array([[4, 2, 0]], np.int32)
    lay_a = oracle.layout(ids_a, 6, 3)
    y_a = np.zeros((3, 8), np.float32)
    y_a[lay_a.dst_row[0, 2]] = big         # expert 0, rank 0
    y_a[lay_a.dst_row[0, 1]] = -big        # expert 2, rank 1
    y_a[lay_a.dst_row[0, 0]] = 1.0         # expert 4, rank 2
    w = np.ones((1, 3), np.float32)
    got_a = oracle.combine_rank_partial(wl.to_bf16_bits(y_a), w, ids_a, lay_a.dst_row, 6, 3)
    assert np.all(f32(got_a) == 1.0)
    # k order inside one rank: experts 0, 1, 2 all on rank 0 (E=6, R=2)
    ids_b = np.array([[0, 1, 2]], np.int32)
    lay_b = oracle.layout(ids_b, 6, 2)
    y_b = np.zeros((3, 8), np.float32)
    for k, v in enumerate((big, -big, 1.0)):
        y_b[lay_b.dst_row[0, k]] = v
    got_b = oracle.combine_rank_partial(wl.to_bf16_bits(y_b), w, ids_b, lay_b.dst_row, 6, 2)
    assert np.all(f32(got_b) == 1.0)
    for yb, ids, lay, R in ((y_a, ids_a, lay_a, 3), (y_b, ids_b, lay_b, 2)):
        yb16 = wl.to_bf16_bits(yb)
        assert np.array_equal(oracle.combine_rank_partial(yb16, w, ids, lay.dst_row, 6, R),
                              exact_rank_partial(yb16, w, ids, lay.dst_row, 6, R))


# ------------------------------------------ send / receive regions per rank --

@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("P", [0, 3, 1000])
def test_regions_round_trip_and_contents(oracle, fp8, P):
    """Receive(send(x)) is the dispatch output, and every region row is the
    matching slice of it: private rows first, then the bulk rows."""
    w = wl.get("decode_dsv3")
    inp = wl.make_inputs(w, T=40)
    lay = oracle.layout(inp.topk_ids, w.E, w.R)
    if fp8:
        packed, scales = oracle.dispatch_fp8(inp.tokens, lay.dst_row)
    else:
        packed, scales = oracle.dispatch_bf16(inp.tokens, lay.dst_row), None
    n = np.diff(lay.rank_offsets)
    C = 40 * min(w.K, w.E // w.R)                  # worst case per region
    priv, ps, bulk, bs, err = oracle.dispatch_send(packed, scales, lay.rank_offsets, P, C)
    assert err == 0
    rows = packed.view(np.uint8).reshape(packed.shape[0], -1)
    for r in range(w.R):
        base, nr = lay.rank_offsets[r], n[r]
        k = min(P, nr)
        assert np.array_equal(priv[r, :k], rows[base:base + k])
        assert np.array_equal(bulk[r, :nr - k], rows[base + k:base + nr])
        if fp8:
            assert np.array_equal(ps[r, :k], scales[base:base + k])
            assert np.array_equal(bs[r, :nr - k], scales[base + k:base + nr])
    back, back_sc = oracle.dispatch_recv(priv, ps, bulk, bs, lay.rank_offsets, packed.shape[0])
    assert np.array_equal(back, rows)
    if fp8:
        assert np.array_equal(back_sc.view(np.uint32), scales.view(np.uint32))


def test_regions_overflow(oracle):
    """A bulk area smaller than a rank's rows keeps what fits, flags bit 4 and
    writes nothing past its capacity (rank 1's bulk area stays untouched)."""
    ids = np.array([[0, 1], [0, 1], [0, 1], [2, 0]], np.int32)   # rank 0: 7 rows, rank 1: 1
    lay = oracle.layout(ids, 4, 2)
    assert lay.rank_offsets.tolist() == [0, 7, 8]
    x = wl.to_bf16_bits(np.arange(1, 33, dtype=np.float32).reshape(4, 8))
    packed = oracle.dispatch_bf16(x, lay.dst_row)
    priv, _, bulk, _, err = oracle.dispatch_send(packed, None, lay.rank_offsets, 1, 3)
    assert err == 4
    rows = packed.view(np.uint8).reshape(8, -1)
    assert np.array_equal(priv[0, 0], rows[0]) and np.array_equal(bulk[0], rows[1:4])
    assert np.array_equal(priv[1, 0], rows[7]) and not bulk[1].any()
    back, _ = oracle.dispatch_recv(priv, None, bulk, None, lay.rank_offsets, 8)
    assert np.array_equal(back[:4], rows[:4]) and not back[4:7].any()   # dropped rows
    assert np.array_equal(back[7], rows[7])
