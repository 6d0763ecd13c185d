"""CPU oracle for MoE expert-parallel layout / dispatch / combine (virtual ranks).

TEST INFRASTRUCTURE ONLY. This package may be imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``; the product
(``combine_layout_02_gb300``) never imports it, and the two share no code.

The arithmetic lives in ``ep_oracle.c`` (plain single-threaded C, explicit loops);
this module only marshals numpy arrays through ctypes and allocates outputs.
bf16 arrays are ``uint16`` bit patterns, e4m3 arrays ``uint8`` bit patterns.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        I64 = ctypes.c_int64
        L.oracle_bf16_from_double.argtypes = [P, I64, P]
        L.oracle_e4m3_encode.argtypes = [P, I64, P]
        L.oracle_e4m3_decode.argtypes = [P, I64, P]
        F = ctypes.c_float
        L.oracle_quantize_row.argtypes = [P, I, P, P]
        L.oracle_quantize_row_mode.argtypes = [P, I, I, F, P, P, P]
        L.oracle_layout.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, P, P]
        L.oracle_layout.restype = I64
        L.oracle_dispatch.argtypes = [I, I, I, I, I, I, I, F, P, P, P, P, P, P, P, P, P, P, P]
        L.oracle_dispatch.restype = I64
        L.oracle_combine.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, P]
        L.oracle_combine.restype = I64
        L.oracle_ll_dispatch.argtypes = [I, I, I, I, I, I, I, I, I, F, P, P, P, P, P, P, P, P]
        L.oracle_ll_dispatch.restype = I64
        L.oracle_ll_combine.argtypes = [I, I, I, I, I, I, P, P, P, P, P]
        L.oracle_ll_combine.restype = None
        L.oracle_expert_layout.argtypes = [I, I, I, I, P, P, P]
        L.oracle_expert_layout.restype = I64
        L.oracle_dispatch_expert_major.argtypes = [I, I, I, I, I, I, I, F, P, P, P, P, P, P, P, P, P]
        L.oracle_dispatch_expert_major.restype = I64
        L.oracle_combine_expert_major.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P]
        L.oracle_combine_expert_major.restype = None
        _lib = L
    return _lib


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats

def bf16_from_double(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_bf16_from_double(_p(v), v.size, _p(out))
    return out


def e4m3_encode(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode(_p(v), v.size, _p(out))
    return out


def e4m3_decode(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    lib().oracle_e4m3_decode(_p(b), b.size, _p(out))
    return out


SCALE_FP32, SCALE_POW2, SCALE_UE8M0, SCALE_TENSOR = 0, 1, 2, 3


def quantize_rows(x: np.ndarray, scale_mode: int = SCALE_FP32, tensor_scale: float = 0.0):
    """x: [..., H] bf16 bits -> (q [..., H] uint8, scales [..., H/128]); scales are fp32,
    or uint8 biased exponents in the UE8M0 mode."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    H = x.shape[-1]
    rows = x.reshape(-1, H)
    q = np.empty(rows.shape, dtype=np.uint8)
    ue = scale_mode == SCALE_UE8M0
    sc = np.empty((rows.shape[0], H // 128), dtype=np.uint8 if ue else np.float32)
    L = lib()
    for i in range(rows.shape[0]):
        L.oracle_quantize_row_mode(_p(rows[i]), H, scale_mode, tensor_scale, _p(q[i]),
                                   None if ue else _p(sc[i]), _p(sc[i]) if ue else None)
    return q.reshape(x.shape), sc.reshape(x.shape[:-1] + (H // 128,))


# ---------------------------------------------------------------- layout

def layout(topk_idx: np.ndarray, E: int, C: int = 12) -> dict:
    """topk_idx [R, T, k] int64 -> layout / handle tensors (see ep_oracle.c)."""
    topk_idx = _c(topk_idx, np.int64)
    R, T, k = topk_idx.shape
    assert E % R == 0 and C >= 1
    out = {
        "num_tokens_per_rank": np.empty((R, R), np.int32),
        "num_tokens_per_expert": np.empty((R, E), np.int32),
        "is_token_in_rank": np.empty((R, T, R), np.uint8),
        "rank_prefix_matrix": np.empty((R, R), np.int32),
        "channel_prefix_matrix": np.empty((R, R, C), np.int32),
        "recv_channel_prefix_matrix": np.empty((R, R, C), np.int32),
        "send_head": np.empty((R, T, R), np.int32),
        "num_recv_tokens_per_expert": np.empty((R, E // R), np.int32),
    }
    bad = lib().oracle_layout(
        R, T, E, k, C, _p(topk_idx), _p(out["num_tokens_per_rank"]),
        _p(out["num_tokens_per_expert"]), _p(out["is_token_in_rank"]),
        _p(out["rank_prefix_matrix"]), _p(out["channel_prefix_matrix"]),
        _p(out["recv_channel_prefix_matrix"]), _p(out["send_head"]),
        _p(out["num_recv_tokens_per_expert"]))
    out["bad_entries"] = int(bad)
    return out


# ---------------------------------------------------------------- dispatch / combine

X_BF16, X_QUANTIZE, X_FP8 = 0, 1, 2


def dispatch(x: np.ndarray, send_head: np.ndarray, row_offset: np.ndarray, E: int,
             topk_idx: Optional[np.ndarray] = None, topk_weights: Optional[np.ndarray] = None,
             x_kind: int = X_BF16, x_scales: Optional[np.ndarray] = None,
             fill_x: int = 0, fill_idx: int = 0, fill_w: float = 0.0, fill_src: int = 0,
             scale_mode: int = SCALE_FP32, tensor_scale: float = 0.0) -> dict:
    """Normal dispatch. x [R, T, H] (uint16 bf16 bits, or uint8 e4m3 when x_kind=2).

    Output arrays are created with the given fill values, so rows that no token maps
    to keep them (tests use them as canaries). Returns dict of outputs + "bad_rows".
    """
    send_head = _c(send_head, np.int32)
    row_offset = _c(row_offset, np.int64)
    R, T, H = x.shape
    k = 0 if topk_idx is None else topk_idx.shape[-1]
    rows = int(row_offset[-1])
    out_dtype = np.uint16 if x_kind == X_BF16 else np.uint8
    res = {"recv_x": np.full((rows, H), fill_x, out_dtype),
           "recv_src_idx": np.full((rows,), fill_src, np.int32)}
    if x_kind == X_BF16:
        res["recv_x_scales"] = None
    elif x_kind == X_QUANTIZE and scale_mode == SCALE_UE8M0:
        res["recv_x_scales"] = np.full((rows, H // 128), 0xEE, np.uint8)
    else:
        res["recv_x_scales"] = np.full((rows, H // 128), np.nan, np.float32)
    if topk_idx is not None:
        res["recv_topk_idx"] = np.full((rows, k), fill_idx, np.int64)
        res["recv_topk_weights"] = (np.full((rows, k), fill_w, np.float32)
                                    if topk_weights is not None else None)
    else:
        res["recv_topk_idx"] = res["recv_topk_weights"] = None
    x = np.ascontiguousarray(x)
    bad = lib().oracle_dispatch(
        R, T, H, E, k, x_kind, scale_mode, tensor_scale, _p(x), _p(_c(x_scales, np.float32)),
        _p(_c(topk_idx, np.int64)), _p(_c(topk_weights, np.float32)),
        _p(send_head), _p(row_offset), _p(res["recv_x"]), _p(res["recv_x_scales"]),
        _p(res["recv_topk_idx"]), _p(res["recv_topk_weights"]), _p(res["recv_src_idx"]))
    res["bad_rows"] = int(bad)
    return res


COMBINE_SUM, COMBINE_WEIGHTED = 0, 1


def combine(y: np.ndarray, send_head: np.ndarray, row_offset: np.ndarray, E: int, k: int,
            mode: int = COMBINE_SUM, topk_idx: Optional[np.ndarray] = None,
            topk_weights: Optional[np.ndarray] = None,
            recv_topk_weights: Optional[np.ndarray] = None) -> dict:
    """Normal combine. y [rows, H] bf16 bits in dispatch row order -> out [R, T, H]."""
    send_head = _c(send_head, np.int32)
    row_offset = _c(row_offset, np.int64)
    R, T, _ = send_head.shape
    H = y.shape[-1]
    y = _c(y, np.uint16)
    if mode == COMBINE_WEIGHTED:
        assert topk_idx is not None and topk_weights is not None
    out = np.empty((R, T, H), np.uint16)
    cw = np.empty((R, T, k), np.float32) if recv_topk_weights is not None else None
    bad = lib().oracle_combine(
        R, T, H, E, k, mode, _p(y), _p(row_offset), _p(send_head),
        _p(_c(topk_idx, np.int64)), _p(_c(topk_weights, np.float32)),
        _p(_c(recv_topk_weights, np.float32)), _p(out), _p(cw))
    return {"out": out, "combined_topk_weights": cw, "bad_rows": int(bad)}


# ---------------------------------------------------------------- low latency

def ll_dispatch(x: np.ndarray, topk_idx: np.ndarray, E: int, nmax: int, use_fp8: bool,
                fill_x: int = 0, fill_src: int = -7, scale_mode: int = SCALE_FP32,
                tensor_scale: float = 0.0, packed: bool = False) -> dict:
    """Low-latency dispatch into fixed per-(expert, source) slots, or (packed) into
    per-expert rows without gaps between the sources."""
    x = _c(x, np.uint16)
    topk_idx = _c(topk_idx, np.int64)
    R, T, H = x.shape
    k = topk_idx.shape[-1]
    E_loc = E // R
    slots = R * nmax
    res = {
        "recv_x": np.full((R, E_loc, slots, H), fill_x, np.uint8 if use_fp8 else np.uint16),
        "recv_x_scales": (None if not use_fp8 else
                          np.full((R, E_loc, slots, H // 128), 0xEE, np.uint8)
                          if scale_mode == SCALE_UE8M0 else
                          np.full((R, E_loc, slots, H // 128), np.nan, np.float32)),
        "src_info": np.full((R, E_loc, slots), fill_src, np.int32),
        "slot": np.empty((R, T, k), np.int32),
        "recv_expert_count": np.empty((R, E_loc), np.int32),
        "layout_range": np.empty((R, E_loc, R, 2), np.int32),
    }
    bad = lib().oracle_ll_dispatch(
        R, T, H, E, k, nmax, int(bool(use_fp8)), int(bool(packed)), scale_mode, tensor_scale,
        _p(x), _p(topk_idx),
        _p(res["recv_x"]),
        _p(res["recv_x_scales"]), _p(res["src_info"]), _p(res["slot"]),
        _p(res["recv_expert_count"]), _p(res["layout_range"]))
    res["bad_entries"] = int(bad)
    return res


def ll_combine(y: np.ndarray, topk_idx: np.ndarray, topk_weights: np.ndarray,
               slot: np.ndarray, E: int, nmax: int) -> np.ndarray:
    """Low-latency weighted combine. y [R, E_loc, R*nmax, H] bf16 bits -> [R, T, H]."""
    y = _c(y, np.uint16)
    topk_idx = _c(topk_idx, np.int64)
    R, T, k = topk_idx.shape
    H = y.shape[-1]
    out = np.empty((R, T, H), np.uint16)
    lib().oracle_ll_combine(R, T, H, E, k, nmax, _p(y), _p(topk_idx),
                            _p(_c(topk_weights, np.float32)), _p(_c(slot, np.int32)), _p(out))
    return out


# ---------------------------------------------------------------- expert-major layout

def expert_layout(topk_idx: np.ndarray, E: int) -> dict:
    """Expert-major placement: expert_rows [R, T, k] (row in the destination's region or
    -1) and expert_prefix [R, E_loc + 1] (exclusive per-expert prefix; last = total)."""
    topk_idx = _c(topk_idx, np.int64)
    R, T, k = topk_idx.shape
    rows = np.empty((R, T, k), np.int32)
    pre = np.empty((R, E // R + 1), np.int32)
    bad = lib().oracle_expert_layout(R, T, E, k, _p(topk_idx), _p(rows), _p(pre))
    return {"expert_rows": rows, "expert_prefix": pre, "bad_entries": int(bad)}


def dispatch_expert_major(x, topk_idx, topk_weights, expert_rows, row_offset, E,
                          quantize=False, scale_mode=SCALE_FP32, tensor_scale=0.0,
                          fill_x=0, fill_src=-3, fill_w=-5.0) -> dict:
    x = _c(x, np.uint16)
    topk_idx = _c(topk_idx, np.int64)
    R, T, H = x.shape
    k = topk_idx.shape[-1]
    row_offset = _c(row_offset, np.int64)
    rows = int(row_offset[-1])
    res = {"recv_x": np.full((rows, H), fill_x, np.uint8 if quantize else np.uint16),
           "recv_src_idx": np.full((rows,), fill_src, np.int32),
           "recv_weights": np.full((rows,), fill_w, np.float32)}
    if quantize:
        res["recv_x_scales"] = (np.full((rows, H // 128), 0xEE, np.uint8) if scale_mode == SCALE_UE8M0
                                else np.full((rows, H // 128), np.nan, np.float32))
    else:
        res["recv_x_scales"] = None
    bad = lib().oracle_dispatch_expert_major(
        R, T, H, E, k, int(bool(quantize)), scale_mode, tensor_scale, _p(x), _p(topk_idx),
        _p(_c(topk_weights, np.float32)), _p(_c(expert_rows, np.int32)), _p(row_offset),
        _p(res["recv_x"]), _p(res["recv_x_scales"]), _p(res["recv_src_idx"]), _p(res["recv_weights"]))
    res["bad_rows"] = int(bad)
    return res


def combine_expert_major(y, topk_idx, topk_weights, expert_rows, row_offset, E,
                         weighted=True) -> np.ndarray:
    topk_idx = _c(topk_idx, np.int64)
    R, T, k = topk_idx.shape
    y = _c(y, np.uint16)
    H = y.shape[-1]
    out = np.empty((R, T, H), np.uint16)
    lib().oracle_combine_expert_major(R, T, H, E, k, int(bool(weighted)), _p(y),
                                      _p(_c(row_offset, np.int64)), _p(topk_idx),
                                      _p(_c(topk_weights, np.float32)), _p(_c(expert_rows, np.int32)),
                                      _p(out))
    return out
