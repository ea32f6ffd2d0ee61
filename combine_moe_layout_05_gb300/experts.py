"""Stand-in experts run between dispatch and combine by tests and benchmarks.

In a model the grouped GEMM multiplies the packed rows with the expert
weights between dispatch and combine (Perplexity, "Enabling trillion-parameter
models on AWS EFA", section "MoE all-to-all over EFA").  No weights exist
here, so the stand-ins below produce bf16 expert outputs from the packed rows
with plain PyTorch ops (fp32 arithmetic, one round-to-nearest-even to bf16),
identically on CPU and GPU.  They are outside the library's path.
"""
from __future__ import annotations

import torch


def expert_of_row(expert_offsets: torch.Tensor, rows: int) -> torch.Tensor:
    """Expert that owns each packed row, from the layout's offsets."""
    r = torch.arange(rows, device=expert_offsets.device, dtype=torch.int32)
    return torch.searchsorted(expert_offsets[1:].contiguous(), r, right=True)


def scale_rows(packed_bf16: torch.Tensor, expert_offsets: torch.Tensor,
               expert_scale: torch.Tensor) -> torch.Tensor:
    """y[r] = bf16(f32(packed[r]) * s[e(r)]): the per-expert-scalar expert."""
    e = expert_of_row(expert_offsets, packed_bf16.shape[0])
    s = expert_scale.to(packed_bf16.device, torch.float32)[e]
    return (packed_bf16.float() * s[:, None]).to(torch.bfloat16)


def dequant_rows(codes_e4m3: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """y[r, j] = bf16(f32(code[r, j]) * scale[r, j // 128]): the identity
    expert of an FP8 round trip."""
    rows, H = codes_e4m3.shape
    q = codes_e4m3.float().view(rows, H // 128, 128)
    return (q * scales.view(rows, H // 128, 1)).view(rows, H).to(torch.bfloat16)
