"""A seeded sweep of random small shapes through every entry point, each
compared bit for bit with the oracle: layout, layout + dispatch (bf16 and
FP8), combine, FP8-input combine, per-rank partial combine, and the
send/receive regions.  The shapes are drawn so that every kernel path is hit
(single-kernel and multi-kernel layout, compile-time and runtime K, partial
row slices), with a few bad ids mixed in."""
import numpy as np
import pytest
import torch

import combine_moe_layout_05_gb300 as moe
from combine_moe_layout_05_gb300 import workload as wl

from gpu_util import bf16_dev, bf16_host, f32_dev, i32_dev

pytestmark = pytest.mark.gpu
CASES = 60


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_layout_05_gb300 import build
    build.build()
    moe.load()


def _shape(rng):
    R = int(rng.choice([1, 2, 4, 8, 16, 32]))
    E = R * int(rng.integers(1, max(2, 512 // R)))
    K = int(rng.integers(1, min(E, 32) + 1))
    T = int(rng.integers(0, 1200 if K <= 8 else 300))
    H = 128 * int(rng.integers(1, 24))        # FP8 needs H % 128 == 0
    return T, H, K, E, R


def _ids(rng, T, E, K, bad):
    ids = wl.routing_zipf(T, E, K, float(rng.uniform(0.5, 1.5)), rng) if T else \
        np.zeros((0, K), np.int32)
    if bad and T:
        ids[rng.integers(0, T), rng.integers(0, K)] = E + int(rng.integers(0, 5))
        ids[rng.integers(0, T), rng.integers(0, K)] = -1
    return ids


def _layout_equal(buf, ref, E):
    assert int(buf.dev_error.item()) == ref.error
    assert np.array_equal(buf.expert_counts.cpu().numpy(), ref.expert_counts)
    assert np.array_equal(buf.expert_offsets.cpu().numpy(), ref.expert_offsets)
    assert np.array_equal(buf.rank_offsets.cpu().numpy(), ref.rank_offsets)
    assert np.array_equal(buf.dst_row.cpu().numpy(), ref.dst_row)
    n = int(ref.expert_offsets[E])
    assert np.array_equal(buf.src_token.cpu().numpy()[:n], ref.src_token[:n])


@pytest.mark.parametrize("case", range(CASES))
def test_random_shape(oracle, case):
    rng = np.random.default_rng(1000 + case)
    T, H, K, E, R = _shape(rng)
    bad = case % 4 == 3
    ids = _ids(rng, T, E, K, bad)
    x = wl.to_bf16_bits((rng.standard_normal((T, H)) *
                         np.exp2(rng.integers(-20, 20, (T, 1)))).astype(np.float32))
    wts = rng.standard_normal((T, K)).astype(np.float32)
    ref = oracle.layout(ids, E, R)

    # layout, and layout + dispatch in one call (both dispatch formats)
    for fp8 in (False, True):
        buf = moe.LayoutBuffers(T, K, E, R)
        for t in (buf.dst_row, buf.src_token, buf.expert_counts):
            t.fill_(-7)
        if fp8:
            packed = torch.empty((T * K, H), dtype=torch.float8_e4m3fn, device="cuda")
            scales = torch.empty((T * K, H // 128), device="cuda")
        else:
            packed = torch.empty((T * K, H), dtype=torch.bfloat16, device="cuda")
            scales = None
        buf.run_dispatch(i32_dev(ids), bf16_dev(x), packed, scales, fp8=fp8)
        torch.cuda.synchronize()
        _layout_equal(buf, ref, E)
        n = int(ref.expert_offsets[E])
        if fp8:
            ec, es = oracle.dispatch_fp8(x, ref.dst_row)
            assert np.array_equal(packed.view(torch.uint8).cpu().numpy()[:n], ec[:n])
            assert np.array_equal(scales.cpu().numpy()[:n].view(np.uint32), es[:n].view(np.uint32))
            codes, sc = ec, es
        else:
            assert np.array_equal(bf16_host(packed)[:n], oracle.dispatch_bf16(x, ref.dst_row)[:n])
    buf = moe.LayoutBuffers(T, K, E, R).run(i32_dev(ids))
    torch.cuda.synchronize()
    _layout_equal(buf, ref, E)
    if T == 0:
        return

    # combine, FP8-input combine, per-rank partial combine on the oracle's slots
    y = wl.to_bf16_bits(rng.standard_normal((T * K, H)).astype(np.float32))
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(bf16_dev(y), f32_dev(wts), i32_dev(ref.dst_row), out)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(out), oracle.combine(y, wts, ref.dst_row))
    moe.moe_combine_fp8(torch.from_numpy(np.ascontiguousarray(codes)).cuda().view(torch.float8_e4m3fn),
                        f32_dev(sc), f32_dev(wts), i32_dev(ref.dst_row), out)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(out), oracle.combine_fp8(codes, sc, wts, ref.dst_row))
    moe.moe_combine_rank_partial(bf16_dev(y), f32_dev(wts), i32_dev(ids), i32_dev(ref.dst_row),
                                 E, R, out)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(out),
                          oracle.combine_rank_partial(y, wts, ids, ref.dst_row, E, R))

    # send / receive regions (bf16), bulk sized to the fullest rank
    P = int(rng.integers(0, 4))
    C = max(0, int(np.diff(ref.rank_offsets).max()) - P)
    priv = torch.zeros((R, P, H), dtype=torch.bfloat16, device="cuda")
    bulk = torch.zeros((R, C, H), dtype=torch.bfloat16, device="cuda")
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ro = i32_dev(ref.rank_offsets)
    moe.moe_dispatch_send(bf16_dev(x), i32_dev(ids), i32_dev(ref.dst_row), ro, E, R, priv, bulk,
                          dev_error=err)
    back = torch.zeros((T * K, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch_recv(priv, bulk, ro, T, K, back)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    n = int(ref.expert_offsets[E])
    assert np.array_equal(bf16_host(back)[:n], oracle.dispatch_bf16(x, ref.dst_row)[:n])
