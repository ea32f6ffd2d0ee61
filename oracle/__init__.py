"""CPU oracle for MoE layout, dispatch and combine (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  This package is the parity reference for the CUDA
library.  Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline / reference leg may import it.  The library package never does,
and it shares no code with the CUDA sources.

The arithmetic lives in ``moe_oracle.c`` (plain single-threaded C, built with
``-ffp-contract=off``); this module only compiles it, loads it and marshals
numpy arrays.  Method source: Perplexity, "Enabling trillion-parameter models
on AWS EFA", sections "Send/receive buffers", "Dispatch and Combine" and
"Evaluation".

Parity pins (all CPU tests): the bf16 and e4m3 codecs against PyTorch's own
conversions (exhaustive decode, constructed ties for encode); the layout
against numpy's stable argsort and brute force over all tiny routings; bf16
dispatch by bit identity; FP8 dispatch by the closed-form error bound of the
block scale; combine against exact rational arithmetic of the fused
multiply-add chain and against the identity round trip; the FP8-input combine
against exact rational arithmetic and against the bf16 combine wherever the
dequantised values are exact in bf16.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-Wall",
          "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/_build/liboracle.so (host compiler)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cc = os.environ.get("CC", "cc")
        subprocess.run([cc, *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32 = ctypes.c_int32
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f32.restype = ctypes.c_float
            lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_f32.restype = ctypes.c_float
            lib.oracle_f32_to_e4m3_satfinite.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_e4m3_satfinite.restype = ctypes.c_uint8
            lib.oracle_f32_to_bf16_n.argtypes = [P, ctypes.c_int64, P]
            lib.oracle_f32_to_bf16_n.restype = None
            lib.oracle_f32_to_e4m3_n.argtypes = [P, ctypes.c_int64, P]
            lib.oracle_f32_to_e4m3_n.restype = None
            lib.oracle_layout.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P]
            lib.oracle_layout.restype = ctypes.c_uint32
            lib.oracle_dispatch_bf16.argtypes = [P, i32, i32, i32, P, P]
            lib.oracle_dispatch_bf16.restype = None
            lib.oracle_dispatch_fp8.argtypes = [P, i32, i32, i32, P, P, P]
            lib.oracle_dispatch_fp8.restype = None
            lib.oracle_combine.argtypes = [P, P, P, i32, i32, i32, P]
            lib.oracle_combine.restype = None
            lib.oracle_combine_fp8.argtypes = [P, P, P, P, i32, i32, i32, P]
            lib.oracle_combine_fp8.restype = None
            lib.oracle_combine_rank_partial.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P]
            lib.oracle_combine_rank_partial.restype = None
            lib.oracle_dispatch_send.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, P, P]
            lib.oracle_dispatch_send.restype = ctypes.c_uint32
            lib.oracle_dispatch_recv.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, P, P]
            lib.oracle_dispatch_recv.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# --- codecs (scalar; vectorised by numpy.vectorize for the tests) ----------

def bf16_to_f32(h: int) -> float:
    return float(_load().oracle_bf16_to_f32(int(h)))


def e4m3_to_f32(c: int) -> float:
    return float(_load().oracle_e4m3_to_f32(int(c)))


def f32_to_e4m3(f: float) -> int:
    return int(_load().oracle_f32_to_e4m3_satfinite(float(np.float32(f))))


def f32_to_bf16_array(a: np.ndarray) -> np.ndarray:
    a = _c(a, np.float32).ravel()
    out = np.empty(a.size, np.uint16)
    _load().oracle_f32_to_bf16_n(_ptr(a), a.size, _ptr(out))
    return out


def f32_to_e4m3_array(a: np.ndarray) -> np.ndarray:
    a = _c(a, np.float32).ravel()
    out = np.empty(a.size, np.uint8)
    _load().oracle_f32_to_e4m3_n(_ptr(a), a.size, _ptr(out))
    return out


# --- the path ---------------------------------------------------------------

class Layout:
    """Outputs of the layout step (all int32 numpy arrays) plus error bits."""

    def __init__(self, counts, offsets, rank_offsets, src_token, dst_row, error):
        self.expert_counts = counts
        self.expert_offsets = offsets
        self.rank_offsets = rank_offsets
        self.src_token = src_token
        self.dst_row = dst_row
        self.error = int(error)


def layout(topk_ids: np.ndarray, E: int, R: int) -> Layout:
    """Per-expert counts, offsets, rank offsets and the stable slot map.

    ``topk_ids`` is [T, K] int32.  ``src_token`` rows at or beyond
    ``expert_offsets[E]`` are -1 here (the C code leaves them untouched)."""
    ids = _c(topk_ids, np.int32)
    T, K = ids.shape
    if R <= 0 or E % R != 0:
        raise ValueError("E must be a positive multiple of R")
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    rank_offsets = np.zeros(R + 1, np.int32)
    src_token = np.full(max(T * K, 1), -1, np.int32)[: T * K].copy()
    dst_row = np.zeros((T, K), np.int32)
    err = _load().oracle_layout(_ptr(ids), T, K, E, R, _ptr(counts),
                                _ptr(offsets), _ptr(rank_offsets),
                                _ptr(src_token), _ptr(dst_row))
    return Layout(counts, offsets, rank_offsets, src_token, dst_row, err)


def dispatch_bf16(tokens_bits: np.ndarray, dst_row: np.ndarray) -> np.ndarray:
    """packed[dst_row[t,k]] = tokens[t]; bf16 carried as uint16 bit patterns."""
    x = _c(tokens_bits, np.uint16)
    T, H = x.shape
    d = _c(dst_row, np.int32)
    K = d.shape[1]
    packed = np.zeros((T * K, H), np.uint16)
    _load().oracle_dispatch_bf16(_ptr(x), T, H, K, _ptr(d), _ptr(packed))
    return packed


def dispatch_fp8(tokens_bits: np.ndarray, dst_row: np.ndarray):
    """Block-scaled e4m3 dispatch; returns (codes uint8 [T*K,H], scales f32 [T*K,H/128])."""
    x = _c(tokens_bits, np.uint16)
    T, H = x.shape
    if H % 128:
        raise ValueError("H must be a multiple of 128 for FP8 dispatch")
    d = _c(dst_row, np.int32)
    K = d.shape[1]
    codes = np.zeros((T * K, H), np.uint8)
    scales = np.zeros((T * K, H // 128), np.float32)
    _load().oracle_dispatch_fp8(_ptr(x), T, H, K, _ptr(d), _ptr(codes),
                                _ptr(scales))
    return codes, scales


def combine(y_bits: np.ndarray, topk_weights: np.ndarray,
            dst_row: np.ndarray) -> np.ndarray:
    """out[t] = bf16(sum_k w[t,k] * y[dst_row[t,k]]) as an fp32 FMA chain in k order."""
    y = _c(y_bits, np.uint16)
    w = _c(topk_weights, np.float32)
    d = _c(dst_row, np.int32)
    T, K = d.shape
    H = y.shape[1]
    out = np.zeros((T, H), np.uint16)
    _load().oracle_combine(_ptr(y), _ptr(w), _ptr(d), T, H, K, _ptr(out))
    return out


def combine_fp8(codes: np.ndarray, scales: np.ndarray, topk_weights: np.ndarray,
                dst_row: np.ndarray) -> np.ndarray:
    """Weighted sum of e4m3 expert outputs: value = f32(code) * block scale,
    then the same fp32 FMA chain in k order and one bf16 rounding."""
    q = _c(codes, np.uint8)
    s = _c(scales, np.float32)
    w = _c(topk_weights, np.float32)
    d = _c(dst_row, np.int32)
    T, K = d.shape
    H = q.shape[1]
    if H % 128 or s.shape != (q.shape[0], H // 128):
        raise ValueError("codes/scales shapes disagree (H must be a multiple of 128)")
    out = np.zeros((T, H), np.uint16)
    _load().oracle_combine_fp8(_ptr(q), _ptr(s), _ptr(w), _ptr(d), T, H, K, _ptr(out))
    return out


def combine_rank_partial(y_bits: np.ndarray, topk_weights: np.ndarray,
                         topk_ids: np.ndarray, dst_row: np.ndarray, E: int,
                         R: int) -> np.ndarray:
    """Sender-side partial sums: per destination rank an fp32 FMA chain in k
    order rounded to bf16, then the receiver's fp32 sum in rank order."""
    y = _c(y_bits, np.uint16)
    w = _c(topk_weights, np.float32)
    ids = _c(topk_ids, np.int32)
    d = _c(dst_row, np.int32)
    T, K = d.shape
    H = y.shape[1]
    if R <= 0 or E % R:
        raise ValueError("E must be a positive multiple of R")
    out = np.zeros((T, H), np.uint16)
    _load().oracle_combine_rank_partial(_ptr(y), _ptr(w), _ptr(ids), _ptr(d), T, H, K,
                                        E, R, _ptr(out))
    return out


def dispatch_send(packed: np.ndarray, scales, rank_offsets: np.ndarray, P: int, C: int):
    """Split the dispatched rows into per-rank private [R,P,row_bytes] and bulk
    [R,C,row_bytes] regions (plus scale regions for FP8); returns
    (priv, priv_scales, bulk, bulk_scales, err)."""
    rows = np.ascontiguousarray(packed)
    rb = rows.shape[1] * rows.itemsize
    u8 = rows.view(np.uint8).reshape(rows.shape[0], rb)
    sc = None if scales is None else np.ascontiguousarray(scales, np.float32)
    nb = 0 if sc is None else sc.shape[1]
    R = rank_offsets.size - 1
    priv = np.zeros((R, P, rb), np.uint8)
    bulk = np.zeros((R, C, rb), np.uint8)
    ps = None if sc is None else np.zeros((R, P, nb), np.float32)
    bs = None if sc is None else np.zeros((R, C, nb), np.float32)
    ro = _c(rank_offsets, np.int32)
    err = _load().oracle_dispatch_send(
        _ptr(u8), _ptr(sc) if sc is not None else None, _ptr(ro), R, rb, nb, P, C,
        _ptr(priv), _ptr(ps) if ps is not None else None, _ptr(bulk),
        _ptr(bs) if bs is not None else None)
    return priv, ps, bulk, bs, int(err)


def dispatch_recv(priv, priv_scales, bulk, bulk_scales, rank_offsets: np.ndarray,
                  rows: int):
    """Regions back to slot order: returns (packed_bytes [rows, row_bytes], scales)."""
    R, P, rb = priv.shape
    C = bulk.shape[1]
    nb = 0 if priv_scales is None else priv_scales.shape[2]
    packed = np.zeros((rows, rb), np.uint8)
    scales = None if priv_scales is None else np.zeros((rows, nb), np.float32)
    ro = _c(rank_offsets, np.int32)
    _load().oracle_dispatch_recv(
        _ptr(_c(priv, np.uint8)), _ptr(_c(priv_scales, np.float32)) if priv_scales is not None else None,
        _ptr(_c(bulk, np.uint8)), _ptr(_c(bulk_scales, np.float32)) if bulk_scales is not None else None,
        _ptr(ro), R, rb, nb, P, C, _ptr(packed), _ptr(scales) if scales is not None else None)
    return packed, scales
