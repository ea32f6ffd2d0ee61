"""GPU parity: the CUDA path, called through the C ABI, against the CPU
oracle, element by element on the same seeded inputs.

The bar (bit-exact everywhere) is the one the method's fixed arithmetic
allows: counts, offsets and index maps are integers; bf16 dispatch is a bit
copy; FP8 codes and scales come from the same IEEE fp32 divides and the same
round-to-nearest-even saturating conversion; combine runs the same fp32
fused-multiply-add chain in the same k order and rounds once to bf16.
All five workloads run at their full sizes, in the launch configuration the
benchmark uses, plus ragged and degenerate shapes.
"""
import numpy as np
import pytest
import torch

import combine_moe_layout_05_gb300 as moe
from combine_moe_layout_05_gb300 import experts as ex
from combine_moe_layout_05_gb300 import workload as wl

from gpu_util import (bf16_dev, bf16_host, f32_dev, gpu_combine,
                      gpu_dispatch_bf16, gpu_dispatch_fp8, gpu_layout, i32_dev)

pytestmark = pytest.mark.gpu

ALL = list(wl.WORKLOADS)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_layout_05_gb300 import build
    build.build()
    moe.load()


def assert_layout_equal(buf, ref, T, K, E, R):
    assert int(buf.dev_error.item()) == ref.error
    assert np.array_equal(buf.expert_counts.cpu().numpy(), ref.expert_counts)
    assert np.array_equal(buf.expert_offsets.cpu().numpy(), ref.expert_offsets)
    assert np.array_equal(buf.rank_offsets.cpu().numpy(), ref.rank_offsets)
    assert np.array_equal(buf.dst_row.cpu().numpy(), ref.dst_row)
    n = int(ref.expert_offsets[E])
    assert np.array_equal(buf.src_token.cpu().numpy()[:n], ref.src_token[:n])


# ------------------------------------------------------------------ layout --

@pytest.mark.parametrize("name", ALL)
def test_layout_full_size(oracle, name):
    w = wl.get(name)
    inp = wl.make_inputs(w)
    ref = oracle.layout(inp.topk_ids, w.E, w.R)
    buf = gpu_layout(inp.topk_ids, w.E, w.R)
    assert_layout_equal(buf, ref, w.T, w.K, w.E, w.R)


SHAPES = [  # T, K, E, R: single kernel, count + ranking, count/scan/rank, ragged tails, limits
    (0, 4, 16, 4), (1, 1, 1, 1), (1, 8, 256, 32), (3, 2, 4, 2), (33, 3, 7, 7),
    (1000, 6, 64, 8), (1024, 8, 256, 32), (1025, 8, 256, 32),
    (1500, 5, 40, 5), (4097, 2, 1024, 16), (5000, 8, 1024, 1024),
    (20000, 8, 384, 48), (70001, 4, 96, 12), (3000, 32, 64, 4),
    (300000, 1, 1, 1), (500, 8, 256, 32), (1365, 3, 5, 5), (3000, 3, 16, 4),
    (4096, 1, 1024, 2), (130000, 8, 128, 16), (30000, 8, 1024, 64),
    # just above one kernel's size, T = 129 at K = 32, Qwen3-sized
    (1025, 4, 16, 4), (129, 32, 64, 8), (16384, 8, 128, 16),
]


def test_layout_shapes_cover_every_launch_plan():
    assert {moe.moe_layout_kernels(T, K, E) for T, K, E, _ in SHAPES} == {1, 2, 3}


@pytest.mark.parametrize("T,K,E,R", SHAPES)
def test_layout_shapes(oracle, T, K, E, R):
    rng = np.random.default_rng(T * 131 + K * 7 + E)
    ids = wl.routing_zipf(T, E, K, 1.1, rng) if T else np.zeros((0, K), np.int32)
    ref = oracle.layout(ids, E, R)
    buf = gpu_layout(ids, E, R)
    assert_layout_equal(buf, ref, T, K, E, R)


@pytest.mark.parametrize("T", [40, 9000])
def test_layout_bad_ids(oracle, T):
    """Out-of-range ids and duplicates: the kernel's bounds checks turn them
    into error bits and -1 slots, exactly as the oracle does."""
    rng = np.random.default_rng(T)
    E, K, R = 32, 4, 4
    ids = wl.routing_uniform(T, E, K, rng)
    ids[3, 1] = E
    ids[5, 0] = -1
    ids[7, 2] = ids[7, 0]
    ids[T - 1, 3] = 1 << 30
    ref = oracle.layout(ids, E, R)
    assert ref.error == 3
    buf = gpu_layout(ids, E, R)
    assert_layout_equal(buf, ref, T, K, E, R)


# ---------------------------------------------------------------- dispatch --

_cache = {}


def _setup(oracle, name, T=None):
    key = (name, T)
    if key not in _cache:
        w = wl.get(name)
        inp = wl.make_inputs(w, T=T)
        ref = oracle.layout(inp.topk_ids, w.E, w.R)
        _cache.clear()
        _cache[key] = (w, inp, ref)
    return _cache[key]


@pytest.mark.parametrize("name", ALL)
def test_dispatch_bf16_full_size(oracle, name):
    w, inp, ref = _setup(oracle, name)
    packed = gpu_dispatch_bf16(bf16_dev(inp.tokens), i32_dev(ref.dst_row))
    exp = oracle.dispatch_bf16(inp.tokens, ref.dst_row)
    assert np.array_equal(bf16_host(packed), exp)


@pytest.mark.parametrize("name", ALL)
def test_dispatch_fp8_full_size(oracle, name):
    w, inp, ref = _setup(oracle, name)
    codes, scales = gpu_dispatch_fp8(bf16_dev(inp.tokens), i32_dev(ref.dst_row))
    exp_codes, exp_scales = oracle.dispatch_fp8(inp.tokens, ref.dst_row)
    got = codes.view(torch.uint8).cpu().numpy()
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), exp_scales.view(np.uint32))
    assert np.array_equal(got, exp_codes)


def test_dispatch_fp8_special_blocks(oracle):
    """Zero blocks with signed zeros, subnormal-only blocks (scale underflow),
    exact ties, values that saturate, and negative values rounding to -0."""
    T, H, K = 6, 512, 2
    rng = np.random.default_rng(0)
    x = wl.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    x[0, :128] = 0
    x[0, 5::7] = 0x8000
    x[1, :128] = 0x0001                      # 2^-133 everywhere
    x[1, 128:256] = 0x8001
    x[2, :128] = wl.to_bf16_bits(np.float32(1.0) * np.ones(128, np.float32))
    x[2, 7] = wl.to_bf16_bits(np.array([448.0], np.float32))[0]
    x[2, 8] = wl.to_bf16_bits(np.array([-17.0], np.float32))[0]   # tie
    x[3, 256:384] = wl.to_bf16_bits(np.float32(1e-30) * rng.standard_normal(128).astype(np.float32))
    x[3, 300] = wl.to_bf16_bits(np.array([3e30], np.float32))[0]  # tiny ones -> +-0
    x[4] = wl.to_bf16_bits(rng.standard_normal(H).astype(np.float32) * np.float32(1e35))
    ids = np.stack([rng.permutation(4)[:K] for _ in range(T)]).astype(np.int32)
    ref = oracle.layout(ids, 4, 2)
    codes, scales = gpu_dispatch_fp8(bf16_dev(x), i32_dev(ref.dst_row))
    exp_codes, exp_scales = oracle.dispatch_fp8(x, ref.dst_row)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), exp_scales.view(np.uint32))
    assert np.array_equal(codes.view(torch.uint8).cpu().numpy(), exp_codes)


@pytest.mark.parametrize("T,H,K", [(1, 8, 1), (7, 24, 3), (5, 128, 5),
                                   (130, 1032, 7), (65, 4096, 16), (3, 2048, 32),
                                   (300, 24, 3), (1000, 1032, 8)])
def test_dispatch_bf16_shapes(oracle, T, H, K):
    rng = np.random.default_rng(H + K)
    x = wl.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    ids = wl.routing_uniform(T, max(K, 40), K, rng)
    ref = oracle.layout(ids, max(K, 40), 1)
    packed = gpu_dispatch_bf16(bf16_dev(x), i32_dev(ref.dst_row))
    assert np.array_equal(bf16_host(packed), oracle.dispatch_bf16(x, ref.dst_row))


@pytest.mark.parametrize("T,H,K", [(1, 128, 1), (9, 384, 3), (17, 1152, 6),
                                   (33, 7168, 9), (2, 128, 32), (100, 384, 8),
                                   (513, 640, 4)])
def test_dispatch_fp8_shapes(oracle, T, H, K):
    rng = np.random.default_rng(H * K + 1)
    x = wl.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)
                        * np.exp2(rng.integers(-30, 30, (T, 1))).astype(np.float32))
    ids = wl.routing_uniform(T, max(K, 40), K, rng)
    ref = oracle.layout(ids, max(K, 40), 1)
    codes, scales = gpu_dispatch_fp8(bf16_dev(x), i32_dev(ref.dst_row))
    ec, es = oracle.dispatch_fp8(x, ref.dst_row)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), es.view(np.uint32))
    assert np.array_equal(codes.view(torch.uint8).cpu().numpy(), ec)


# ----------------------------------------------------------------- combine --

def _expert_outputs(w, inp, ref, packed_bits):
    """The workload's stand-in experts on the oracle's packed rows (CPU)."""
    if w.experts in ("identity", "dequant"):
        return packed_bits
    if w.experts == "scale":
        y = ex.scale_rows(torch.from_numpy(packed_bits.view(np.int16)).view(torch.bfloat16),
                          torch.from_numpy(ref.expert_offsets), torch.from_numpy(inp.expert_scale))
        return y.view(torch.int16).numpy().view(np.uint16)
    return wl.random_rows(packed_bits.shape[0], w.H, inp.expert_rows_seed)


@pytest.mark.parametrize("name", ALL)
def test_combine_full_size(oracle, name):
    w, inp, ref = _setup(oracle, name)
    packed = oracle.dispatch_bf16(inp.tokens, ref.dst_row)
    y = _expert_outputs(w, inp, ref, packed)
    out = gpu_combine(bf16_dev(y), f32_dev(inp.topk_weights), i32_dev(ref.dst_row))
    exp = oracle.combine(y, inp.topk_weights, ref.dst_row)
    assert np.array_equal(bf16_host(out), exp)


@pytest.mark.parametrize("T,H,K", [(1, 8, 1), (7, 24, 3), (5, 128, 5),
                                   (130, 1032, 7), (65, 4096, 16), (3, 2048, 32),
                                   (300, 24, 3), (1000, 1032, 8),
                                   # grids of >= 2^20 pieces walk flat pieces: blocks
                                   # spanning 2-3 and 16-17 tokens, ragged last block
                                   (8200, 1032, 3), (70001, 128, 2)])
def test_combine_shapes(oracle, T, H, K):
    rng = np.random.default_rng(T + H + K)
    y = wl.to_bf16_bits((rng.standard_normal((T * K, H)) *
                         np.exp2(rng.integers(-12, 12, (T * K, H)))).astype(np.float32))
    wts = (rng.standard_normal((T, K)) * 3).astype(np.float32)
    dst = rng.permutation(T * K).astype(np.int32).reshape(T, K)
    out = gpu_combine(bf16_dev(y), f32_dev(wts), i32_dev(dst))
    assert np.array_equal(bf16_host(out), oracle.combine(y, wts, dst))


def test_combine_fma_and_order_sensitive(oracle):
    """Inputs on which a separate multiply/add, another k order or a -0 start
    give different bits than the defined chain."""
    w0 = np.float32(1 + 2.0 ** -23)
    y0 = np.float32(1 - 2.0 ** -8)
    rows = np.array([[y0] * 8, [-y0] * 8, [2.0 ** 30] * 8, [1.0] * 8,
                     [-(2.0 ** 30)] * 8, [-0.0] * 8, [-0.0] * 8, [5.0] * 8,
                     [7.0] * 8], np.float32)
    y = wl.to_bf16_bits(rows)
    wts = np.array([[w0, w0, 1], [1, 1, 1], [1, 1, 0.5]], np.float32)
    dst = np.array([[0, 1, 5], [2, 4, 3], [5, 6, 6]], np.int32)
    out = gpu_combine(bf16_dev(y), f32_dev(wts), i32_dev(dst))
    exp = oracle.combine(y, wts, dst)
    assert np.array_equal(bf16_host(out), exp)
    assert np.all(exp[2] == 0)                       # +0, not -0


@pytest.mark.parametrize("K", [3, 8, 9])
def test_combine_skips_invalid_slots(oracle, K):
    """Entries whose slot is -1 or past the last row add nothing, on the
    compile-time-K path (8) and the runtime-K paths (3, and 9 in batches)."""
    T, H = 40, 264
    rng = np.random.default_rng(K + 100)
    y = wl.to_bf16_bits(rng.standard_normal((T * K, H)).astype(np.float32))
    wts = rng.standard_normal((T, K)).astype(np.float32)
    dst = rng.permutation(T * K).astype(np.int32).reshape(T, K)
    dst[rng.random((T, K)) < 0.2] = -1
    dst[5, :] = -1                                      # a token with no valid entry
    dst[6, K - 1] = T * K                               # one past the last row
    out = gpu_combine(bf16_dev(y), f32_dev(wts), i32_dev(dst))
    exp = oracle.combine(y, wts, dst)
    assert np.array_equal(bf16_host(out), exp)
    assert np.all(exp[5] == 0)


@pytest.mark.parametrize("K,fp8", [(3, False), (8, False), (8, True), (9, True)])
def test_dispatch_skips_invalid_slots(oracle, K, fp8):
    """A -1 or out-of-range slot is not written; every valid slot is."""
    T, H = 30, 384
    rng = np.random.default_rng(K * 3 + fp8)
    x = wl.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    perm = rng.permutation(T * K).astype(np.int32).reshape(T, K)
    drop = rng.random((T, K)) < 0.25
    drop[0, 0] = True
    dst = perm.copy()
    dst[drop] = -1
    dst[0, 0] = T * K + 7                               # past the last row instead
    dropped_rows, valid = perm[drop], perm[~drop]       # rows nobody / somebody writes
    if fp8:
        codes, scales = gpu_dispatch_fp8(bf16_dev(x), i32_dev(dst))
        ec, es = oracle.dispatch_fp8(x, dst)
        got = codes.view(torch.uint8).cpu().numpy()
        assert np.array_equal(got[valid], ec[valid])
        assert np.array_equal(scales.cpu().numpy()[valid].view(np.uint32), es[valid].view(np.uint32))
        assert np.all(got[dropped_rows] == 0x7F)         # untouched poison
    else:
        got = bf16_host(gpu_dispatch_bf16(bf16_dev(x), i32_dev(dst)))
        assert np.array_equal(got[valid], oracle.dispatch_bf16(x, dst)[valid])
        assert np.all(got[dropped_rows] == 0xFFFF)


# ------------------------------------------------------ the path end to end --

@pytest.mark.parametrize("name", [n for n in ALL if "bf16" in wl.get(n).dispatch])
def test_end_to_end_bf16(oracle, name):
    """layout -> bf16 dispatch -> stand-in experts -> combine, all on the GPU,
    against the same chain on the CPU oracle."""
    w, inp, ref = _setup(oracle, name)
    buf = moe.LayoutBuffers(w.T, w.K, w.E, w.R).run(i32_dev(inp.topk_ids))
    packed = gpu_dispatch_bf16(bf16_dev(inp.tokens), buf.dst_row)
    if w.experts == "scale":
        y_d = ex.scale_rows(packed, buf.expert_offsets, torch.from_numpy(inp.expert_scale))
    elif w.experts == "random":
        y_d = bf16_dev(wl.random_rows(w.T * w.K, w.H, inp.expert_rows_seed))
    else:
        y_d = packed
    out = gpu_combine(y_d, f32_dev(inp.topk_weights), buf.dst_row)
    y_h = _expert_outputs(w, inp, ref, oracle.dispatch_bf16(inp.tokens, ref.dst_row))
    exp = oracle.combine(y_h, inp.topk_weights, ref.dst_row)
    assert np.array_equal(bf16_host(out), exp)
    if w.experts == "identity":
        # combine(dispatch(x)) == x as numbers (a -0 input comes back +0)
        o = wl.bf16_bits_to_f32(bf16_host(out))
        assert np.array_equal(o, wl.bf16_bits_to_f32(inp.tokens))


@pytest.mark.parametrize("name", [n for n in ALL if "fp8" in wl.get(n).dispatch])
def test_end_to_end_fp8(oracle, name):
    """layout -> FP8 dispatch -> dequantising (or random) experts -> combine
    on the GPU, against the same chain on the CPU oracle."""
    w, inp, ref = _setup(oracle, name)
    buf = moe.LayoutBuffers(w.T, w.K, w.E, w.R).run(i32_dev(inp.topk_ids))
    codes, scales = gpu_dispatch_fp8(bf16_dev(inp.tokens), buf.dst_row)
    if w.experts == "random":
        y_h = wl.random_rows(w.T * w.K, w.H, inp.expert_rows_seed)
        y_d = bf16_dev(y_h)
    else:
        ec, es = oracle.dispatch_fp8(inp.tokens, ref.dst_row)
        y_d = ex.dequant_rows(codes, scales)
        y_h = ex.dequant_rows(torch.from_numpy(ec).view(torch.float8_e4m3fn),
                              torch.from_numpy(es)).view(torch.int16).numpy().view(np.uint16)
    out = gpu_combine(y_d, f32_dev(inp.topk_weights), buf.dst_row)
    exp = oracle.combine(y_h, inp.topk_weights, ref.dst_row)
    assert np.array_equal(bf16_host(out), exp)
    if w.experts != "random":
        # FP8 round trip: within the block-scale bound of x (amax/28 per block)
        x = wl.bf16_bits_to_f32(inp.tokens).astype(np.float64).reshape(w.T, -1, 128)
        o = wl.bf16_bits_to_f32(bf16_host(out)).astype(np.float64).reshape(w.T, -1, 128)
        amax = np.abs(x).max(axis=2, keepdims=True)
        assert np.all(np.abs(o - x) <= amax / 28 * 1.01 + np.abs(x) * 2.0 ** -7)


# ------------------------------------------- layout + dispatch in one call --

FUSED_SHAPES = [  # T, H, K, E, R, fp8: single-kernel sizes, then fallbacks
    (1, 8, 1, 1, 1, 0), (3, 24, 3, 7, 7, 0), (128, 7168, 8, 256, 32, 0),
    (256, 7168, 8, 256, 32, 1), (128, 7168, 8, 256, 32, 1), (100, 1032, 6, 64, 8, 0),
    (64, 256, 2, 8, 2, 1), (37, 4096, 32, 1024, 16, 0), (250, 384, 9, 1024, 4, 1),
    (1024, 7168, 8, 256, 32, 0), (4096, 7168, 8, 384, 48, 1), (0, 128, 4, 16, 4, 0),
    # multi-launch layout (T*K > 4096): odd K, runtime K, E = 1024, and chunks
    # capped by the scan (15000 ids per chunk)
    (5000, 264, 3, 40, 8, 0), (700, 1024, 9, 64, 4, 1), (600, 512, 32, 1024, 16, 0),
    (30000, 128, 8, 1024, 32, 0),
]


@pytest.mark.parametrize("T,H,K,E,R,fp8", FUSED_SHAPES)
def test_layout_dispatch_matches_oracle(oracle, T, H, K, E, R, fp8):
    rng = np.random.default_rng(T * 7 + H + K)
    x = wl.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)
                        * np.exp2(rng.integers(-8, 8, (T, 1))).astype(np.float32))
    ids = wl.routing_zipf(T, E, K, 1.2, rng) if T else np.zeros((0, K), np.int32)
    ref = oracle.layout(ids, E, R)
    buf = moe.LayoutBuffers(T, K, E, R)
    for t in (buf.expert_counts, buf.expert_offsets, buf.rank_offsets, buf.src_token,
              buf.dst_row, buf.dev_error):
        t.fill_(-7)
    if fp8:
        packed = torch.empty((T * K, H), dtype=torch.float8_e4m3fn, device="cuda")
        packed.view(torch.uint8).fill_(0x7F)
        scales = torch.full((T * K, H // 128), float("nan"), device="cuda")
    else:
        packed = torch.empty((T * K, H), dtype=torch.bfloat16, device="cuda")
        packed.view(torch.int16).fill_(-1)
        scales = None
    buf.run_dispatch(i32_dev(ids), bf16_dev(x), packed, scales, fp8=bool(fp8))
    torch.cuda.synchronize()
    assert_layout_equal(buf, ref, T, K, E, R)
    if T == 0:
        return
    if fp8:
        ec, es = oracle.dispatch_fp8(x, ref.dst_row)
        assert np.array_equal(packed.view(torch.uint8).cpu().numpy(), ec)
        assert np.array_equal(scales.cpu().numpy().view(np.uint32), es.view(np.uint32))
    else:
        assert np.array_equal(bf16_host(packed), oracle.dispatch_bf16(x, ref.dst_row))


@pytest.mark.parametrize("name", ALL)
def test_layout_dispatch_full_size(oracle, name):
    """The call the benchmark makes, at each workload's full size."""
    w, inp, ref = _setup(oracle, name)
    for fp8 in (False, True):
        buf = moe.LayoutBuffers(w.T, w.K, w.E, w.R)
        if fp8:
            packed = torch.empty((w.T * w.K, w.H), dtype=torch.float8_e4m3fn, device="cuda")
            scales = torch.empty((w.T * w.K, w.H // 128), device="cuda")
        else:
            packed = torch.empty((w.T * w.K, w.H), dtype=torch.bfloat16, device="cuda")
            scales = None
        buf.run_dispatch(i32_dev(inp.topk_ids), bf16_dev(inp.tokens), packed, scales, fp8=fp8)
        torch.cuda.synchronize()
        assert_layout_equal(buf, ref, w.T, w.K, w.E, w.R)
        if fp8:
            ec, es = oracle.dispatch_fp8(inp.tokens, ref.dst_row)
            assert np.array_equal(packed.view(torch.uint8).cpu().numpy(), ec)
            assert np.array_equal(scales.cpu().numpy().view(np.uint32), es.view(np.uint32))
        else:
            assert np.array_equal(bf16_host(packed), oracle.dispatch_bf16(inp.tokens, ref.dst_row))


@pytest.mark.parametrize("T,K,E,R", [(50, 4, 16, 4), (300, 8, 64, 8), (261, 8, 1024, 32),
                                     (1500, 4, 16, 4)])
def test_layout_dispatch_bad_ids(oracle, T, K, E, R):
    """Errors and -1 slots match the oracle's: single kernel with integer and
    with fp16 counters (T*K >= 2048), and the multi-launch form (T*K > 4096)."""
    rng = np.random.default_rng(T)
    H = 256
    ids = wl.routing_uniform(T, E, K, rng)
    ids[0, 0] = E + 3
    ids[9, 3] = ids[9, 1]
    ids[T - 1, K - 1] = -1
    ids[T // 2, 0] = E
    x = wl.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    ref = oracle.layout(ids, E, R)
    buf = moe.LayoutBuffers(T, K, E, R)
    packed = torch.zeros((T * K, H), dtype=torch.bfloat16, device="cuda")
    buf.run_dispatch(i32_dev(ids), bf16_dev(x), packed)
    torch.cuda.synchronize()
    assert_layout_equal(buf, ref, T, K, E, R)
    exp = oracle.dispatch_bf16(x, ref.dst_row)
    n = int(ref.expert_offsets[E])
    assert np.array_equal(bf16_host(packed)[:n], exp[:n])
