"""GPU parity of moe_combine_fp8 (combine reading e4m3 codes and block
scales directly) against the oracle's combine_fp8, bit for bit: the same
exact code widening, the same fp32 products with the scale and the same fp32
fused multiply-add chain in k order, rounded once to bf16."""
import numpy as np
import pytest
import torch

import combine_moe_layout_05_gb300 as moe
from combine_moe_layout_05_gb300 import workload as wl

from gpu_util import bf16_dev, bf16_host, f32_dev, i32_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_layout_05_gb300 import build
    build.build()
    moe.load()


def e4m3_dev(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).cuda().view(torch.float8_e4m3fn)


def gpu_combine_fp8(codes, scales, wts, dst):
    T, K = dst.shape
    H = codes.shape[1]
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    moe.moe_combine_fp8(e4m3_dev(codes), f32_dev(scales), f32_dev(wts), i32_dev(dst), out)
    torch.cuda.synchronize()
    return bf16_host(out)


@pytest.mark.parametrize("name", ["decode_dsv3_fp8", "prefill_kimi_k2", "prefill_qwen3"])
def test_combine_fp8_full_size(oracle, name):
    w = wl.get(name)
    inp = wl.make_inputs(w)
    lay = oracle.layout(inp.topk_ids, w.E, w.R)
    codes, scales = oracle.dispatch_fp8(inp.tokens, lay.dst_row)
    got = gpu_combine_fp8(codes, scales, inp.topk_weights, lay.dst_row)
    assert np.array_equal(got, oracle.combine_fp8(codes, scales, inp.topk_weights, lay.dst_row))


@pytest.mark.parametrize("T,H,K", [(1, 128, 1), (5, 384, 3), (33, 7168, 8),
                                   (17, 1152, 9), (4, 256, 32), (70, 4096, 6)])
def test_combine_fp8_shapes(oracle, T, H, K):
    rng = np.random.default_rng(T * 31 + H + K)
    codes = rng.integers(0, 256, (T * K, H)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x01                       # no NaN codes
    scales = (rng.random((T * K, H // 128)) *
              np.exp2(rng.integers(-30, 30, (T * K, H // 128)))).astype(np.float32)
    scales[0, 0] = 0.0
    wts = (rng.standard_normal((T, K)) * 2).astype(np.float32)
    dst = rng.permutation(T * K).astype(np.int32).reshape(T, K)
    if T > 2:
        dst[1, 0] = -1                                         # skipped term
    got = gpu_combine_fp8(codes, scales, wts, dst)
    assert np.array_equal(got, oracle.combine_fp8(codes, scales, wts, dst))


def test_combine_fp8_rounding_sensitive(oracle):
    """w*(q*s) - q with w, s = 1 + small multiples of 2^-23: the output is the
    low fp32 bits of the sum, so any other rounding order shows."""
    dec = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).float().numpy()
    cases = [(c, np.float32(1 + a * 2.0 ** -23), np.float32(1 + b * 2.0 ** -23))
             for c in list(range(0x38, 0x40)) + list(range(0xB8, 0xC0))
             for a in range(-5, 6) for b in range(-5, 6)]
    T, H, K = len(cases), 128, 2
    codes = np.zeros((T * K, H), np.uint8)
    scales = np.ones((T * K, 1), np.float32)
    wts = np.zeros((T, K), np.float32)
    for i, (c, w, s) in enumerate(cases):
        codes[2 * i] = codes[2 * i + 1] = c
        scales[2 * i] = s
        wts[i] = (w, -1.0)
    dst = np.arange(T * K, dtype=np.int32).reshape(T, K)
    got = gpu_combine_fp8(codes, scales, wts, dst)
    exp = oracle.combine_fp8(codes, scales, wts, dst)
    assert np.array_equal(got, exp)
    assert np.count_nonzero(exp[:, 0]) > T // 2


@pytest.mark.parametrize("name", ["decode_dsv3_fp8", "prefill_qwen3"])
def test_fp8_round_trip_end_to_end(oracle, name):
    """layout + FP8 dispatch, then combine straight from the codes and scales,
    all on the GPU, against the same chain on the oracle."""
    w = wl.get(name)
    inp = wl.make_inputs(w)
    buf = moe.LayoutBuffers(w.T, w.K, w.E, w.R)
    codes = torch.empty((w.T * w.K, w.H), dtype=torch.float8_e4m3fn, device="cuda")
    scales = torch.empty((w.T * w.K, w.H // 128), device="cuda")
    buf.run_dispatch(i32_dev(inp.topk_ids), bf16_dev(inp.tokens), codes, scales, fp8=True)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine_fp8(codes, scales, f32_dev(inp.topk_weights), buf.dst_row, out)
    torch.cuda.synchronize()
    ref = oracle.layout(inp.topk_ids, w.E, w.R)
    ec, es = oracle.dispatch_fp8(inp.tokens, ref.dst_row)
    assert np.array_equal(bf16_host(out), oracle.combine_fp8(ec, es, inp.topk_weights, ref.dst_row))
