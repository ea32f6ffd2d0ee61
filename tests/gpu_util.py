"""Helpers shared by the GPU tests: numpy <-> device tensors and one call of
the whole CUDA path through the C ABI."""
import numpy as np
import torch

import combine_moe_layout_05_gb300 as moe


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16))
    return t.cuda().view(torch.bfloat16)


def bf16_host(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def i32_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def f32_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def gpu_layout(ids: np.ndarray, E: int, R: int, poison: bool = True):
    T, K = ids.shape
    buf = moe.LayoutBuffers(T, K, E, R)
    if poison:
        for t in (buf.expert_counts, buf.expert_offsets, buf.rank_offsets,
                  buf.src_token, buf.dst_row, buf.dev_error):
            t.fill_(-7)
        if buf.workspace is not None:
            buf.workspace.fill_(0xAB)
    buf.run(i32_dev(ids))
    torch.cuda.synchronize()
    return buf


def gpu_dispatch_bf16(tokens_dev, dst_row_dev):
    T, H = tokens_dev.shape
    K = dst_row_dev.shape[1]
    packed = torch.empty((T * K, H), dtype=torch.bfloat16, device="cuda")
    packed.view(torch.int16).fill_(-1)          # poison: catches unwritten rows
    moe.moe_dispatch(tokens_dev, dst_row_dev, packed)
    return packed


def gpu_dispatch_fp8(tokens_dev, dst_row_dev):
    T, H = tokens_dev.shape
    K = dst_row_dev.shape[1]
    codes = torch.empty((T * K, H), dtype=torch.float8_e4m3fn, device="cuda")
    codes.view(torch.uint8).fill_(0x7F)
    scales = torch.full((T * K, H // 128), float("nan"), device="cuda")
    moe.moe_dispatch(tokens_dev, dst_row_dev, codes, scales, fp8=True)
    return codes, scales


def gpu_combine(y_dev, weights_dev, dst_row_dev):
    T, K = weights_dev.shape
    H = y_dev.shape[1]
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    moe.moe_combine(y_dev, weights_dev, dst_row_dev, out)
    return out
