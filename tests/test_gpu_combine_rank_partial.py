"""GPU parity of moe_combine_rank_partial (sender-side per-rank partial sums)
against the oracle's combine_rank_partial, bit for bit, and its distance from
the receiver-side combine on the same data."""
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


def gpu_rank_partial(y, wts, ids, dst, E, R):
    T, K = dst.shape
    H = y.shape[1]
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    moe.moe_combine_rank_partial(bf16_dev(y), f32_dev(wts), i32_dev(ids), i32_dev(dst), E, R, out)
    torch.cuda.synchronize()
    return bf16_host(out)


@pytest.mark.parametrize("name", ["decode_dsv3", "prefill_kimi_k2", "prefill_qwen3"])
def test_rank_partial_full_size(oracle, name):
    w = wl.get(name)
    inp = wl.make_inputs(w)
    lay = oracle.layout(inp.topk_ids, w.E, w.R)
    y = wl.random_rows(w.T * w.K, w.H, inp.expert_rows_seed)
    got = gpu_rank_partial(y, inp.topk_weights, inp.topk_ids, lay.dst_row, w.E, w.R)
    exp = oracle.combine_rank_partial(y, inp.topk_weights, inp.topk_ids, lay.dst_row, w.E, w.R)
    assert np.array_equal(got, exp)
    recv = oracle.combine(y, inp.topk_weights, lay.dst_row)
    assert np.count_nonzero(exp != recv) > 0            # the schemes do differ


@pytest.mark.parametrize("T,H,K,E,R", [(1, 8, 1, 4, 2), (7, 24, 3, 9, 3), (33, 1032, 5, 40, 8),
                                       (20, 256, 9, 64, 1), (9, 128, 32, 64, 16), (50, 7168, 6, 60, 60)])
def test_rank_partial_shapes(oracle, T, H, K, E, R):
    rng = np.random.default_rng(T * 13 + K + E)
    ids = wl.routing_uniform(T, E, K, rng)
    lay = oracle.layout(ids, E, R)
    y = wl.to_bf16_bits((rng.standard_normal((T * K, H)) *
                         np.exp2(rng.integers(-10, 10, (T * K, H)))).astype(np.float32))
    wts = (rng.standard_normal((T, K)) * 2).astype(np.float32)
    got = gpu_rank_partial(y, wts, ids, lay.dst_row, E, R)
    assert np.array_equal(got, oracle.combine_rank_partial(y, wts, ids, lay.dst_row, E, R))


def test_rank_partial_order_sensitive(oracle):
    """2^30, -2^30, 1 in the defined orders sum to exactly 1."""
    big = 2.0 ** 30
    ids = np.array([[4, 2, 0], [0, 1, 2]], np.int32)
    for R in (3, 2):
        lay = oracle.layout(ids[:1] if R == 3 else ids[1:], 6, R)
        y = np.zeros((3, 8), np.float32)
        vals = ((1.0, -big, big) if R == 3 else (big, -big, 1.0))
        for k, v in enumerate(vals):
            y[lay.dst_row[0, k]] = v
        yb = wl.to_bf16_bits(y)
        w = np.ones((1, 3), np.float32)
        got = gpu_rank_partial(yb, w, ids[:1] if R == 3 else ids[1:], lay.dst_row, 6, R)
        assert np.all(wl.bf16_bits_to_f32(got) == 1.0)


@pytest.mark.parametrize("K", [3, 8, 32])
def test_rank_partial_invalid_entries(oracle, K):
    """Entries with a bad expert id or an out-of-range slot are skipped, wherever
    they fall in the (rank, k) order; a token with no valid entry gives +0."""
    T, H, E, R = 40, 264, 64, 8
    rng = np.random.default_rng(K)
    ids = wl.routing_uniform(T, E, K, rng)
    ids[rng.random((T, K)) < 0.2] = -1
    ids[3, :] = E + 5                                   # no valid entry at all
    ids[5, 0] = E
    lay = oracle.layout(ids, E, R)
    dst = lay.dst_row.copy()
    ok = np.argwhere(dst >= 0)
    for t, k in ok[rng.choice(len(ok), 6, replace=False)]:
        dst[t, k] = T * K + int(rng.integers(0, 3))     # valid id, slot past the rows
    y = wl.to_bf16_bits(rng.standard_normal((T * K, H)).astype(np.float32))
    wts = rng.standard_normal((T, K)).astype(np.float32)
    got = gpu_rank_partial(y, wts, ids, dst, E, R)
    exp = oracle.combine_rank_partial(y, wts, ids, dst, E, R)
    assert np.array_equal(got, exp)
    assert np.all(got[3] == 0)
