"""Thin ctypes binding over libmoe_layout.so (argument marshalling only).

Every function has the name of its C entry point and forwards raw device
pointers, sizes and the current CUDA stream; all computation happens in the
library's CUDA kernels.  There is no CPU fallback: if the library is missing
or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import build as _build

MOE_OK = 0
MOE_DEV_ERR_EXPERT_RANGE = 1
MOE_DEV_ERR_DUPLICATE = 2
MOE_DEV_ERR_REGION_OVERFLOW = 4
MOE_DEV_ERR_TIMEOUT = 8

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {moe_status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load the CUDA library (built beforehand by build.build())."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"{p} is missing: build it with "
                    "combine_moe_layout_05_gb300.build.build()")
            lib = ctypes.CDLL(p)
            P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            lib.moe_status_string.argtypes = [ctypes.c_int]
            lib.moe_status_string.restype = ctypes.c_char_p
            lib.moe_layout_workspace_bytes.argtypes = [i32, i32, i32]
            lib.moe_layout_workspace_bytes.restype = sz
            lib.moe_layout.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P,
                                       P, sz, P]
            lib.moe_layout.restype = ctypes.c_int
            lib.moe_dispatch.argtypes = [P, i32, i32, i32, P, i32, P, P, P]
            lib.moe_dispatch.restype = ctypes.c_int
            lib.moe_combine.argtypes = [P, P, P, i32, i32, i32, P, P]
            lib.moe_combine.restype = ctypes.c_int
            lib.moe_layout_dispatch.argtypes = [P, P, i32, i32, i32, i32, i32, i32,
                                                P, P, P, P, P, P, P, P, P, sz, P]
            lib.moe_layout_dispatch.restype = ctypes.c_int
            lib.moe_layout_dispatch_kernels.argtypes = [i32, i32, i32, i32, i32]
            lib.moe_layout_dispatch_kernels.restype = i32
            lib.moe_layout_kernels.argtypes = [i32, i32, i32]
            lib.moe_layout_kernels.restype = i32
            lib.moe_combine_fp8.argtypes = [P, P, P, P, i32, i32, i32, P, P]
            lib.moe_combine_fp8.restype = ctypes.c_int
            lib.moe_combine_rank_partial.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, P]
            lib.moe_combine_rank_partial.restype = ctypes.c_int
            lib.moe_dispatch_send.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, i32, i32,
                                              P, P, i32, P, P, P, P]
            lib.moe_dispatch_send.restype = ctypes.c_int
            lib.moe_dispatch_recv.argtypes = [P, P, i32, P, P, i32, P, i32, i32, i32, i32,
                                              i32, P, P, P]
            lib.moe_dispatch_recv.restype = ctypes.c_int
            lib.moe_layout_static.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P, P]
            lib.moe_layout_static.restype = ctypes.c_int
            _lib = lib
    return _lib


def declared_functions(header: str | None = None) -> list[str]:
    """Names of the functions the public header declares."""
    header = header or os.path.join(_build.INCLUDE, "moe_layout.h")
    text = open(header).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", text)))


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(name: str, t, dtype, device=None):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _raise(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status)


def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def moe_layout_workspace_bytes(T: int, K: int, E: int) -> int:
    return int(load().moe_layout_workspace_bytes(T, K, E))


def moe_layout_dispatch_kernels(T: int, H: int, K: int, E: int, fp8: bool) -> int:
    return int(load().moe_layout_dispatch_kernels(T, H, K, E, int(bool(fp8))))


def moe_layout_kernels(T: int, K: int, E: int) -> int:
    return int(load().moe_layout_kernels(T, K, E))


def moe_layout(topk_ids, E: int, R: int, expert_counts, expert_offsets,
               rank_offsets, src_token, dst_row, dev_error=None,
               workspace=None, stream=None) -> None:
    """Routing histogram, scan and stable slot map (see include/moe_layout.h)."""
    T, K = topk_ids.shape
    _check("topk_ids", topk_ids, torch.int32)
    for n, t in (("expert_counts", expert_counts), ("expert_offsets", expert_offsets),
                 ("rank_offsets", rank_offsets), ("src_token", src_token),
                 ("dst_row", dst_row)):
        _check(n, t, torch.int32)
    if expert_counts.numel() < E or expert_offsets.numel() < E + 1 or rank_offsets.numel() < R + 1:
        raise ValueError("moe_layout: output arrays too small")
    if src_token.numel() < T * K or dst_row.numel() < T * K:
        raise ValueError("moe_layout: src_token/dst_row too small")
    if dev_error is not None:
        _check("dev_error", dev_error, torch.int32)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().moe_layout(_ptr(topk_ids), T, K, E, R, _ptr(expert_counts),
                           _ptr(expert_offsets), _ptr(rank_offsets),
                           _ptr(src_token), _ptr(dst_row), _ptr(dev_error),
                           _ptr(workspace), ws_bytes, _stream(stream))
    _raise("moe_layout", st)


def moe_dispatch(tokens, dst_row, packed, scales=None, fp8: bool = False,
                 stream=None) -> None:
    """Pack token rows into their K slots, bf16 or block-scaled e4m3."""
    T, H = tokens.shape
    K = dst_row.shape[1] if dst_row.dim() == 2 else 1
    _check("tokens", tokens, torch.bfloat16)
    _check("dst_row", dst_row, torch.int32)
    if fp8:
        _check("packed", packed, torch.float8_e4m3fn)
        _check("scales", scales, torch.float32)
        if scales is None or scales.numel() < T * K * (H // 128):
            raise ValueError("moe_dispatch: scales missing or too small")
    else:
        _check("packed", packed, torch.bfloat16)
    if dst_row.numel() != T * K or packed.numel() < T * K * H:
        raise ValueError("moe_dispatch: dst_row/packed have the wrong size")
    st = load().moe_dispatch(_ptr(tokens), T, H, K, _ptr(dst_row), int(bool(fp8)),
                             _ptr(packed), _ptr(scales) if fp8 else None,
                             _stream(stream))
    _raise("moe_dispatch", st)


def moe_layout_dispatch(topk_ids, tokens, E: int, R: int, expert_counts,
                        expert_offsets, rank_offsets, src_token, dst_row, packed,
                        scales=None, fp8: bool = False, dev_error=None,
                        workspace=None, stream=None) -> None:
    """moe_layout then moe_dispatch in one call (one kernel for small batches)."""
    T, K = topk_ids.shape
    H = tokens.shape[1]
    if tokens.shape[0] != T:
        raise ValueError("moe_layout_dispatch: tokens and topk_ids disagree on T")
    _check("topk_ids", topk_ids, torch.int32)
    _check("tokens", tokens, torch.bfloat16)
    for n, t in (("expert_counts", expert_counts), ("expert_offsets", expert_offsets),
                 ("rank_offsets", rank_offsets), ("src_token", src_token),
                 ("dst_row", dst_row)):
        _check(n, t, torch.int32)
    if expert_counts.numel() < E or expert_offsets.numel() < E + 1 or rank_offsets.numel() < R + 1:
        raise ValueError("moe_layout_dispatch: output arrays too small")
    if src_token.numel() < T * K or dst_row.numel() < T * K or packed.numel() < T * K * H:
        raise ValueError("moe_layout_dispatch: src_token/dst_row/packed too small")
    if fp8:
        _check("packed", packed, torch.float8_e4m3fn)
        _check("scales", scales, torch.float32)
        if scales is None or scales.numel() < T * K * (H // 128):
            raise ValueError("moe_layout_dispatch: scales missing or too small")
    else:
        _check("packed", packed, torch.bfloat16)
    if dev_error is not None:
        _check("dev_error", dev_error, torch.int32)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().moe_layout_dispatch(
        _ptr(topk_ids), _ptr(tokens), T, H, K, E, R, int(bool(fp8)), _ptr(expert_counts),
        _ptr(expert_offsets), _ptr(rank_offsets), _ptr(src_token), _ptr(dst_row),
        _ptr(dev_error), _ptr(packed), _ptr(scales) if fp8 else None,
        _ptr(workspace), ws_bytes, _stream(stream))
    _raise("moe_layout_dispatch", st)


def moe_combine(expert_out, topk_weights, dst_row, out, stream=None) -> None:
    """Routing-weighted fp32 sum of each token's K expert rows, rounded to bf16."""
    T, K = topk_weights.shape
    H = out.shape[1]
    _check("expert_out", expert_out, torch.bfloat16)
    _check("topk_weights", topk_weights, torch.float32)
    _check("dst_row", dst_row, torch.int32)
    _check("out", out, torch.bfloat16)
    if dst_row.numel() != T * K or out.shape[0] != T or expert_out.numel() < T * K * H:
        raise ValueError("moe_combine: argument sizes disagree")
    st = load().moe_combine(_ptr(expert_out), _ptr(topk_weights), _ptr(dst_row),
                            T, H, K, _ptr(out), _stream(stream))
    _raise("moe_combine", st)


def moe_combine_rank_partial(expert_out, topk_weights, topk_ids, dst_row, E: int,
                             R: int, out, stream=None) -> None:
    """Combine with sender-side per-rank partial sums (bf16 partials)."""
    T, K = topk_weights.shape
    H = out.shape[1]
    _check("expert_out", expert_out, torch.bfloat16)
    _check("topk_weights", topk_weights, torch.float32)
    _check("topk_ids", topk_ids, torch.int32)
    _check("dst_row", dst_row, torch.int32)
    _check("out", out, torch.bfloat16)
    if dst_row.numel() != T * K or topk_ids.numel() != T * K or out.shape[0] != T \
            or expert_out.numel() < T * K * H:
        raise ValueError("moe_combine_rank_partial: argument sizes disagree")
    st = load().moe_combine_rank_partial(_ptr(expert_out), _ptr(topk_weights), _ptr(topk_ids),
                                         _ptr(dst_row), T, H, K, E, R, _ptr(out),
                                         _stream(stream))
    _raise("moe_combine_rank_partial", st)


def moe_dispatch_send(tokens, topk_ids, dst_row, rank_offsets, E: int, R: int,
                      priv, bulk, priv_scales=None, bulk_scales=None, fp8: bool = False,
                      dev_error=None, stream=None) -> None:
    """Dispatch into per-rank regions: priv [R,P,H] for each rank's first P
    rows, bulk [R,C,H] for the rest (bf16, or e4m3 codes + block scales)."""
    T, H = tokens.shape
    K = topk_ids.shape[1]
    R_, P = priv.shape[0], priv.shape[1]
    C = bulk.shape[1]
    if R_ != R or bulk.shape[0] != R:
        raise ValueError("moe_dispatch_send: region buffers must have R rows of regions")
    _check("tokens", tokens, torch.bfloat16)
    for n, t in (("topk_ids", topk_ids), ("dst_row", dst_row), ("rank_offsets", rank_offsets)):
        _check(n, t, torch.int32)
    dt = torch.float8_e4m3fn if fp8 else torch.bfloat16
    _check("priv", priv, dt)
    _check("bulk", bulk, dt)
    if fp8:
        _check("priv_scales", priv_scales, torch.float32)
        _check("bulk_scales", bulk_scales, torch.float32)
    st = load().moe_dispatch_send(_ptr(tokens), T, H, K, E, R, _ptr(topk_ids), _ptr(dst_row),
                                  _ptr(rank_offsets), int(bool(fp8)), P, _ptr(priv),
                                  _ptr(priv_scales) if fp8 else None, C, _ptr(bulk),
                                  _ptr(bulk_scales) if fp8 else None, _ptr(dev_error),
                                  _stream(stream))
    _raise("moe_dispatch_send", st)


def moe_dispatch_recv(priv, bulk, rank_offsets, T: int, K: int, packed,
                      priv_scales=None, bulk_scales=None, scales=None, fp8: bool = False,
                      stream=None) -> None:
    """Region rows back to slot order (the grouped-GEMM input)."""
    R, P = priv.shape[0], priv.shape[1]
    C = bulk.shape[1]
    H = packed.shape[1]
    _check("rank_offsets", rank_offsets, torch.int32)
    dt = torch.float8_e4m3fn if fp8 else torch.bfloat16
    for n, t in (("priv", priv), ("bulk", bulk), ("packed", packed)):
        _check(n, t, dt)
    st = load().moe_dispatch_recv(_ptr(priv), _ptr(priv_scales) if fp8 else None, P,
                                  _ptr(bulk), _ptr(bulk_scales) if fp8 else None, C,
                                  _ptr(rank_offsets), R, T, H, K, int(bool(fp8)), _ptr(packed),
                                  _ptr(scales) if fp8 else None, _stream(stream))
    _raise("moe_dispatch_recv", st)


def moe_layout_static(topk_ids, E: int, R: int, expert_counts, expert_offsets,
                      rank_offsets, src_token, dst_row, dev_error=None,
                      stream=None) -> None:
    """moe_layout for callers that cannot allocate: the large-batch scratch is
    a fixed array inside the library (see include/moe_layout.h)."""
    T, K = topk_ids.shape
    _check("topk_ids", topk_ids, torch.int32)
    for n, t in (("expert_counts", expert_counts), ("expert_offsets", expert_offsets),
                 ("rank_offsets", rank_offsets), ("src_token", src_token),
                 ("dst_row", dst_row)):
        _check(n, t, torch.int32)
    if expert_counts.numel() < E or expert_offsets.numel() < E + 1 or rank_offsets.numel() < R + 1:
        raise ValueError("moe_layout_static: output arrays too small")
    if src_token.numel() < T * K or dst_row.numel() < T * K:
        raise ValueError("moe_layout_static: src_token/dst_row too small")
    if dev_error is not None:
        _check("dev_error", dev_error, torch.int32)
    st = load().moe_layout_static(_ptr(topk_ids), T, K, E, R, _ptr(expert_counts),
                                  _ptr(expert_offsets), _ptr(rank_offsets),
                                  _ptr(src_token), _ptr(dst_row), _ptr(dev_error),
                                  _stream(stream))
    _raise("moe_layout_static", st)


def moe_combine_fp8(expert_out, expert_scales, topk_weights, dst_row, out,
                    stream=None) -> None:
    """Routing-weighted sum of e4m3 expert rows (value = code * block scale)."""
    T, K = topk_weights.shape
    H = out.shape[1]
    _check("expert_out", expert_out, torch.float8_e4m3fn)
    _check("expert_scales", expert_scales, torch.float32)
    _check("topk_weights", topk_weights, torch.float32)
    _check("dst_row", dst_row, torch.int32)
    _check("out", out, torch.bfloat16)
    if dst_row.numel() != T * K or out.shape[0] != T or expert_out.numel() < T * K * H \
            or expert_scales.numel() < T * K * (H // 128):
        raise ValueError("moe_combine_fp8: argument sizes disagree")
    st = load().moe_combine_fp8(_ptr(expert_out), _ptr(expert_scales), _ptr(topk_weights),
                                _ptr(dst_row), T, H, K, _ptr(out), _stream(stream))
    _raise("moe_combine_fp8", st)


class LayoutBuffers:
    """Device buffers for one layout of T x K entries (allocated by torch)."""

    def __init__(self, T: int, K: int, E: int, R: int, device="cuda"):
        i32 = dict(dtype=torch.int32, device=device)
        self.T, self.K, self.E, self.R = T, K, E, R
        self.expert_counts = torch.empty(E, **i32)
        self.expert_offsets = torch.empty(E + 1, **i32)
        self.rank_offsets = torch.empty(R + 1, **i32)
        self.src_token = torch.empty(T * K, **i32)
        self.dst_row = torch.empty((T, K), **i32)
        self.dev_error = torch.empty(1, **i32)
        ws = moe_layout_workspace_bytes(T, K, E)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=device) if ws else None

    def run(self, topk_ids, stream=None) -> "LayoutBuffers":
        moe_layout(topk_ids, self.E, self.R, self.expert_counts,
                   self.expert_offsets, self.rank_offsets, self.src_token,
                   self.dst_row, self.dev_error, self.workspace, stream)
        return self

    def run_dispatch(self, topk_ids, tokens, packed, scales=None, fp8=False,
                     stream=None) -> "LayoutBuffers":
        """Layout and dispatch together (moe_layout_dispatch)."""
        moe_layout_dispatch(topk_ids, tokens, self.E, self.R, self.expert_counts,
                            self.expert_offsets, self.rank_offsets, self.src_token,
                            self.dst_row, packed, scales, fp8, self.dev_error,
                            self.workspace, stream)
        return self
