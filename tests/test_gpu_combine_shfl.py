"""GPU parity, bit for bit against the oracle, of the combine form kept behind
a test hook for comparison: lanes 0..7 of each warp load the token's 8 slots
and weights and shuffle them to the warp."""
import ctypes

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


@pytest.mark.parametrize("T,H", [(128, 7168), (300, 4096), (7, 136), (1000, 1032)])
def test_shuffle_combine_matches_oracle(oracle, T, H):
    K, E, R = 8, 64, 8
    rng = np.random.default_rng(T + H)
    ids = wl.routing_uniform(T, E, K, rng)
    ids[0, 3] = -1                                  # one skipped term
    ref = oracle.layout(ids, E, R)
    y = wl.to_bf16_bits(rng.standard_normal((T * K, H)).astype(np.float32))
    w = wl.routing_weights(T, K, rng)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    y_d, w_d, d_d = bf16_dev(y), f32_dev(w), i32_dev(ref.dst_row)
    f = moe.load().moe_testing_combine_shfl
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [P, P, P, i32, i32, i32, P, P]
    f.restype = i32
    assert f(y_d.data_ptr(), w_d.data_ptr(), d_d.data_ptr(), T, H, K, out.data_ptr(),
             torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(out), oracle.combine(y, w, ref.dst_row))
