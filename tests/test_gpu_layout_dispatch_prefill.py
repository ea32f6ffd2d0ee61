"""GPU parity of moe_layout_dispatch's large-batch path (the counting kernel,
then one grid whose first blocks rank the chunks while the others pack the
rows of ranked chunks) against the oracle, bit for bit, and the bounded wait
of the packing blocks: made to expire on purpose through a test hook (a
chunk that is never published), it reports MOE_DEV_ERR_TIMEOUT and returns."""
import ctypes
import time

import numpy as np
import pytest
import torch

import combine_moe_layout_05_gb300 as moe
from combine_moe_layout_05_gb300 import workload as wl

from gpu_util import bf16_dev, bf16_host, i32_dev

pytestmark = pytest.mark.gpu

MOE_DEV_ERR_TIMEOUT = moe.MOE_DEV_ERR_TIMEOUT


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_layout_05_gb300 import build
    build.build()
    moe.load()


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _inputs(T, H, K, E, seed, routing="zipf"):
    rng = np.random.default_rng(seed)
    x = wl.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)
                        * np.exp2(rng.integers(-6, 6, (T, 1))).astype(np.float32))
    if routing == "zipf":
        ids = wl.routing_zipf(T, E, K, 1.1, rng)
    else:
        ids = wl.routing_uniform(T, E, K, rng)
    return x, ids


def _outputs(T, H, K, fp8):
    if fp8:
        packed = torch.empty((T * K, H), dtype=torch.float8_e4m3fn, device="cuda")
        packed.view(torch.uint8).fill_(0x7F)
        scales = torch.full((T * K, H // 128), float("nan"), device="cuda")
    else:
        packed = torch.empty((T * K, H), dtype=torch.bfloat16, device="cuda")
        packed.view(torch.int16).fill_(-1)
        scales = None
    return packed, scales


def _poisoned_layout(T, K, E, R):
    buf = moe.LayoutBuffers(T, K, E, R)
    for t in (buf.expert_counts, buf.expert_offsets, buf.rank_offsets, buf.src_token,
              buf.dst_row, buf.dev_error):
        t.fill_(-7)
    if buf.workspace is not None:
        buf.workspace.fill_(0xAB)
    return buf


def _check(oracle, buf, ref, x, packed, scales, T, K, E, R, fp8, rows=None, err=None):
    assert int(buf.dev_error.item()) == (ref.error if err is None else err)
    assert np.array_equal(buf.expert_counts.cpu().numpy(), ref.expert_counts)
    assert np.array_equal(buf.expert_offsets.cpu().numpy(), ref.expert_offsets)
    assert np.array_equal(buf.rank_offsets.cpu().numpy(), ref.rank_offsets)
    assert np.array_equal(buf.dst_row.cpu().numpy(), ref.dst_row)
    n = int(ref.expert_offsets[E])
    assert np.array_equal(buf.src_token.cpu().numpy()[:n], ref.src_token[:n])
    sel = slice(0, n) if rows is None else rows
    if fp8:
        ec, es = oracle.dispatch_fp8(x, ref.dst_row)
        assert np.array_equal(packed.view(torch.uint8).cpu().numpy()[sel], ec[sel])
        assert np.array_equal(scales.cpu().numpy().view(np.uint32)[sel],
                              es.view(np.uint32)[sel])
    else:
        exp = oracle.dispatch_bf16(x, ref.dst_row)
        assert np.array_equal(bf16_host(packed)[sel], exp[sel])


PREFILL_SHAPES = [  # T, H, K, E, R, fp8: every one takes the two-launch path
    (4096, 7168, 8, 384, 48, 0),      # Kimi-K2 prefill shape
    (4096, 7168, 8, 384, 48, 1),
    (16384, 4096, 8, 128, 16, 1),     # Qwen3 prefill shape
    (16384, 4096, 8, 128, 16, 0),
    (3001, 1032, 5, 40, 8, 0),        # runtime K, rows of 129 pieces
    (3001, 1032, 5, 42, 7, 0),        # E % 4 != 0: scalar column sums
    (9001, 512, 1, 16, 4, 0),         # K = 1
    (300, 1024, 32, 64, 4, 1),        # K = 32
    (700, 1024, 9, 64, 4, 1),         # runtime K
    (5000, 512, 8, 128, 16, 0),       # four tokens per packing block
    (3000, 128, 8, 64, 8, 0),         # 16 or 17 tokens per packing block
    (6000, 384, 8, 64, 8, 0),         # rows of 48 pieces: warps span two tokens
    (2500, 2056, 3, 24, 4, 0),        # rows of 257 pieces, K = 3
    (4000, 1024, 8, 64, 8, 1),
    (40000, 1024, 6, 96, 12, 1),
    (100000, 1024, 4, 128, 16, 0),    # chunk count capped by the histogram budget
    (1100, 1024, 8, 64, 8, 0),        # 9 chunks: the second cluster one chunk + 7 empty
    (16384, 1024, 8, 256, 32, 1),     # fewer, larger chunks for the shared-memory budget
    (5000, 256, 2, 3, 3, 0),          # E = 3: most counting blocks own no expert
]


@pytest.mark.parametrize("T,H,K,E,R,fp8", PREFILL_SHAPES)
def test_prefill_path_matches_oracle(oracle, T, H, K, E, R, fp8):
    assert moe.moe_layout_dispatch_kernels(T, H, K, E, fp8) == 2
    x, ids = _inputs(T, H, K, E, seed=T + 31 * K + E)
    ref = oracle.layout(ids, E, R)
    buf = _poisoned_layout(T, K, E, R)
    packed, scales = _outputs(T, H, K, fp8)
    buf.run_dispatch(i32_dev(ids), bf16_dev(x), packed, scales, fp8=bool(fp8))
    torch.cuda.synchronize()
    _check(oracle, buf, ref, x, packed, scales, T, K, E, R, fp8)


@pytest.mark.parametrize("fp8", [0, 1])
def test_prefill_path_bad_ids(oracle, fp8):
    T, H, K, E, R = 3000, 1024, 4, 16, 4
    x, ids = _inputs(T, H, K, E, seed=5, routing="uniform")
    assert moe.moe_layout_dispatch_kernels(T, H, K, E, fp8) == 2
    ids[0, 0] = E + 3
    ids[9, 3] = ids[9, 1]
    ids[T - 1, K - 1] = -1
    ids[T // 2, 0] = E
    ref = oracle.layout(ids, E, R)
    assert ref.error == moe.MOE_DEV_ERR_EXPERT_RANGE | moe.MOE_DEV_ERR_DUPLICATE
    buf = _poisoned_layout(T, K, E, R)
    packed, scales = _outputs(T, H, K, fp8)
    buf.run_dispatch(i32_dev(ids), bf16_dev(x), packed, scales, fp8=bool(fp8))
    torch.cuda.synchronize()
    _check(oracle, buf, ref, x, packed, scales, T, K, E, R, fp8)


def test_prefill_path_graph_replay(oracle):
    """Captured once, replayed twice on new inputs: nothing carries over
    between calls (the workspace is rewritten, the error word re-zeroed)."""
    T, H, K, E, R = 5000, 512, 8, 128, 16
    assert moe.moe_layout_dispatch_kernels(T, H, K, E, 0) == 2
    buf = moe.LayoutBuffers(T, K, E, R)
    ids_d = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    x_d = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    packed, _ = _outputs(T, H, K, 0)
    s = torch.cuda.Stream()
    x0, ids0 = _inputs(T, H, K, E, seed=1)
    ids_d.copy_(i32_dev(ids0))
    x_d.copy_(bf16_dev(x0))
    buf.run_dispatch(ids_d, x_d, packed)          # first call outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        buf.run_dispatch(ids_d, x_d, packed)
    for seed in (2, 3):
        x, ids = _inputs(T, H, K, E, seed=seed)
        if seed == 3:
            ids[7, 2] = -1
        ids_d.copy_(i32_dev(ids))
        x_d.copy_(bf16_dev(x))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.layout(ids, E, R)
        _check(oracle, buf, ref, x, packed, None, T, K, E, R, 0)


def _hook(lib):
    f = lib.moe_testing_layout_dispatch_prefill
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [P, P, i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P,
                  ctypes.c_uint64, i32, P]
    f.restype = i32
    return f


SLOT_PENDING = -2**31      # a dst_row entry not yet written by its chunk's ranking block


@pytest.mark.parametrize("fp8", [0, 1])
def test_bounded_wait_expires_and_reports(oracle, fp8):
    """Chunk 1 is never ranked (its slots stay pending) and each wait is
    bounded at 2 ms: the call completes, the error word is exactly the
    timeout bit, the counts, offsets and every other chunk's slots are right,
    every row of a token outside chunk 1 is packed, chunk 1's rows are left
    alone, and the next normal call on the same context is bit-exact."""
    T, H, K, E, R = 4000, 1024, 8, 64, 8
    assert moe.moe_layout_dispatch_kernels(T, H, K, E, fp8) == 2
    tpc = 1024 // K                      # tokens per chunk at this size
    x, ids = _inputs(T, H, K, E, seed=9)
    ref = oracle.layout(ids, E, R)
    buf = _poisoned_layout(T, K, E, R)
    packed, scales = _outputs(T, H, K, fp8)
    ids_d, x_d = i32_dev(ids), bf16_dev(x)
    f = _hook(moe.load())
    t0 = time.time()
    st = f(ids_d.data_ptr(), x_d.data_ptr(), T, H, K, E, R, fp8, buf.expert_counts.data_ptr(),
           buf.expert_offsets.data_ptr(), buf.rank_offsets.data_ptr(), buf.src_token.data_ptr(),
           buf.dst_row.data_ptr(), buf.dev_error.data_ptr(), packed.data_ptr(),
           scales.data_ptr() if fp8 else None, buf.workspace.data_ptr(), 2_000_000, 1,
           torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert time.time() - t0 < 30
    assert int(buf.dev_error.item()) == MOE_DEV_ERR_TIMEOUT
    assert np.array_equal(buf.expert_counts.cpu().numpy(), ref.expert_counts)
    assert np.array_equal(buf.expert_offsets.cpu().numpy(), ref.expert_offsets)
    assert np.array_equal(buf.rank_offsets.cpu().numpy(), ref.rank_offsets)
    dr = buf.dst_row.cpu().numpy()
    assert np.all(dr[tpc:2 * tpc] == SLOT_PENDING)
    assert np.array_equal(dr[:tpc], ref.dst_row[:tpc])
    assert np.array_equal(dr[2 * tpc:], ref.dst_row[2 * tpc:])
    others = np.unique(np.concatenate([ref.dst_row[:tpc].ravel(), ref.dst_row[2 * tpc:].ravel()]))
    stalled = np.unique(ref.dst_row[tpc:2 * tpc].ravel())
    st_tok = buf.src_token.cpu().numpy()
    assert np.array_equal(st_tok[others], ref.src_token[others])
    if fp8:
        ec, es = oracle.dispatch_fp8(x, ref.dst_row)
        assert np.array_equal(packed.view(torch.uint8).cpu().numpy()[others], ec[others])
        assert np.array_equal(scales.cpu().numpy().view(np.uint32)[others],
                              es.view(np.uint32)[others])
        assert np.all(packed.view(torch.uint8).cpu().numpy()[stalled] == 0x7F)
    else:
        exp = oracle.dispatch_bf16(x, ref.dst_row)
        assert np.array_equal(bf16_host(packed)[others], exp[others])
        assert np.all(bf16_host(packed)[stalled] == 0xFFFF)
    # the context is still usable
    buf2 = _poisoned_layout(T, K, E, R)
    packed2, scales2 = _outputs(T, H, K, fp8)
    buf2.run_dispatch(ids_d, x_d, packed2, scales2, fp8=bool(fp8))
    torch.cuda.synchronize()
    _check(oracle, buf2, ref, x, packed2, scales2, T, K, E, R, fp8)


def _random_prefill_shape(rng):
    """A shape that takes the two-launch path: T*K above the single-kernel
    sizes, E and H small enough for the ranking blocks' shared memory."""
    for _ in range(1000):
        R = int(rng.choice([1, 2, 4, 8, 16]))
        E = R * int(rng.integers(1, max(2, 320 // R)))
        K = int(rng.integers(1, min(E, 16) + 1))
        T = int(rng.integers(8192 // K + 1, 160_000 // K))
        H = 128 * int(rng.integers(1, 5))
        fp8 = int(rng.integers(0, 2))
        if moe.moe_layout_dispatch_kernels(T, H, K, E, fp8) == 2:
            return T, H, K, E, R, fp8
    raise AssertionError("no two-launch shape drawn")


@pytest.mark.parametrize("case", range(16))
def test_prefill_path_random_shapes(oracle, case):
    """Seeded random shapes on the two-launch path (chunk counts up to 128,
    so 1 to 16 clusters of counting blocks, the last one often partly
    empty), Zipf routing with a few bad ids: every output bit for bit
    against the oracle."""
    rng = np.random.default_rng(5000 + case)
    T, H, K, E, R, fp8 = _random_prefill_shape(rng)
    x, ids = _inputs(T, H, K, E, seed=6000 + case)
    if case % 4 == 3:
        ids[int(rng.integers(0, T)), int(rng.integers(0, K))] = E + 1
    ref = oracle.layout(ids, E, R)
    buf = _poisoned_layout(T, K, E, R)
    packed, scales = _outputs(T, H, K, fp8)
    buf.run_dispatch(i32_dev(ids), bf16_dev(x), packed, scales, fp8=bool(fp8))
    torch.cuda.synchronize()
    _check(oracle, buf, ref, x, packed, scales, T, K, E, R, fp8)
