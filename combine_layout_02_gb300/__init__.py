"""combine_layout_02_gb300 -- MoE expert-parallel layout / dispatch / combine on one
GB300, with the expert-parallel ranks made virtual partitions of the device memory.

This module is a thin ctypes binding over the C ABI in ``include/ep.h`` (``libep.so``,
built in-tree by ``build.py``). Functions keep the C names; they only marshal
arguments (tensor -> device pointer, stream -> cudaStream_t) and raise on a non-OK
status. Every step of the computation runs in the library's CUDA kernels. There is no
CPU fallback: if the library is missing or fails to load, every call raises.

Tensors are PyTorch CUDA tensors used as plain device memory; bf16 data may be
``torch.bfloat16`` or ``torch.int16``/``uint16`` views, e4m3 data ``torch.uint8`` or
``torch.float8_e4m3fn``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

__all__ = [
    "EP_OK", "EP_ERR_INVALID_ARG", "EP_ERR_CUDA", "EP_ERR_UNSUPPORTED",
    "EP_DEVERR_BAD_EXPERT", "EP_DEVERR_RECV_OVERFLOW", "EP_DEVERR_SLOT_OVERFLOW",
    "EP_DEVERR_TIMEOUT",
    "EP_BF16", "EP_FP8_E4M3", "EP_COMBINE_SUM", "EP_COMBINE_WEIGHTED",
    "EP_PHASE_SEND", "EP_PHASE_RECV", "EP_PHASE_BOTH", "EP_MAX_RANKS",
    "EP_FP8_SCALE_FP32", "EP_FP8_SCALE_POW2", "EP_FP8_SCALE_UE8M0", "EP_FP8_SCALE_TENSOR",
    "ep_fp8_options",
    "EpError", "ep_shape", "ep_launch", "ep_layout", "ep_handle", "ep_recv", "ep_ll_buffer",
    "lib", "library_path", "make_shape", "make_launch",
    "ep_layout_workspace_size", "ep_get_layout", "ep_get_layout_static_scratch",
    "ep_buffer_size_hint", "ep_size_hint",
    "ep_dispatch", "ep_combine", "ep_dispatch_expert_major", "ep_combine_expert_major",
    "ep_ll_dispatch", "ep_ll_combine", "ep_clean_ll_buffer", "ep_read_recv_counts_sync",
    "ep_read_error_flags_sync", "ep_selftest_wait_timeout", "ep_kernel_launch_count",
    "ep_abi_version", "EXPORTED_SYMBOLS",
]

EP_OK, EP_ERR_INVALID_ARG, EP_ERR_CUDA, EP_ERR_UNSUPPORTED = 0, 1, 2, 3
EP_DEVERR_BAD_EXPERT, EP_DEVERR_RECV_OVERFLOW, EP_DEVERR_SLOT_OVERFLOW, EP_DEVERR_TIMEOUT = 1, 2, 4, 8
EP_BF16, EP_FP8_E4M3 = 0, 1
EP_COMBINE_SUM, EP_COMBINE_WEIGHTED = 0, 1
EP_PHASE_SEND, EP_PHASE_RECV, EP_PHASE_BOTH = 1, 2, 3
EP_FP8_SCALE_FP32, EP_FP8_SCALE_POW2, EP_FP8_SCALE_UE8M0, EP_FP8_SCALE_TENSOR = 0, 1, 2, 3
EP_LL_LAYOUT_SLOTS, EP_LL_LAYOUT_PACKED = 0, 1
EP_MAX_RANKS = 64
EP_MAX_TOPK = 32
EP_EXPERT_MAJOR_MAX_EXPERTS = 4096

# Every function include/ep.h declares (checked by the ABI test).
EXPORTED_SYMBOLS = (
    "ep_layout_workspace_size", "ep_get_layout", "ep_get_layout_static_scratch",
    "ep_buffer_size_hint",
    "ep_dispatch", "ep_combine", "ep_dispatch_expert_major", "ep_combine_expert_major",
    "ep_ll_dispatch", "ep_ll_combine", "ep_clean_ll_buffer", "ep_read_recv_counts_sync",
    "ep_read_error_flags_sync", "ep_selftest_wait_timeout", "ep_status_string",
    "ep_last_cuda_error", "ep_kernel_launch_count", "ep_abi_version",
)

_HERE = os.path.dirname(os.path.abspath(__file__))
_P = ctypes.c_void_p
_I32 = ctypes.c_int32


def library_path() -> str:
    return os.path.join(_HERE, "_build", "libep.so")


class EpError(RuntimeError):
    def __init__(self, func: str, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{func} failed with status {status}: {detail}")


class ep_shape(ctypes.Structure):
    _fields_ = [("num_ranks", _I32), ("num_tokens", _I32), ("hidden", _I32),
                ("num_experts", _I32), ("num_topk", _I32), ("num_channels", _I32),
                ("num_max_dispatch_tokens_per_rank", _I32), ("num_sms", _I32)]


class ep_fp8_options(ctypes.Structure):
    _fields_ = [("scale_format", _I32), ("tensor_scale", ctypes.c_float)]


class ep_launch(ctypes.Structure):
    _fields_ = [("stream", _P), ("wait_event", _P), ("record_event", _P), ("error_flags", _P)]


class ep_layout(ctypes.Structure):
    _fields_ = [("num_tokens_per_rank", _P), ("num_tokens_per_rdma_rank", _P),
                ("num_tokens_per_expert", _P), ("is_token_in_rank", _P)]


class ep_handle(ctypes.Structure):
    _fields_ = [("rank_prefix_matrix", _P), ("channel_prefix_matrix", _P),
                ("recv_channel_prefix_matrix", _P), ("recv_src_idx", _P),
                ("is_token_in_rank", _P), ("send_head", _P),
                ("num_recv_tokens_per_expert", _P), ("expert_rows", _P), ("expert_prefix", _P)]


class ep_recv(ctypes.Structure):
    _fields_ = [("recv_x", _P), ("recv_x_scales", _P), ("recv_topk_idx", _P),
                ("recv_topk_weights", _P), ("recv_src_idx", _P), ("row_offset", _P),
                ("fp8", ep_fp8_options)]


class ep_ll_buffer(ctypes.Structure):
    _fields_ = [("recv_x", _P), ("recv_x_scales", _P), ("src_info", _P), ("slot", _P),
                ("send_count", _P), ("recv_expert_count", _P), ("layout_range", _P),
                ("fp8", ep_fp8_options), ("layout", _I32)]


class ep_size_hint(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64 if n.endswith("_rows") else ctypes.c_uint64) for n in (
        "recv_rows", "recv_x_bytes", "recv_x_scales_bytes", "recv_topk_idx_bytes",
        "recv_topk_weights_bytes", "recv_src_idx_bytes", "expert_major_rows",
        "expert_major_x_bytes", "ll_slots", "ll_recv_x_bytes", "ll_recv_x_scales_bytes",
        "ll_src_info_bytes", "ll_slot_bytes", "ll_send_count_bytes", "ll_recv_expert_count_bytes",
        "ll_layout_range_bytes", "layout_workspace_bytes")]


_lib = None


def lib():
    """Load libep.so (built by build.py / __graft_entry__.build()). Raises if absent."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"libep.so not found at {path}: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (no CPU fallback exists)")
        L = ctypes.CDLL(path)
        S = ctypes.POINTER
        L.ep_layout_workspace_size.argtypes = [S(ep_shape)]
        L.ep_layout_workspace_size.restype = ctypes.c_size_t
        L.ep_buffer_size_hint.argtypes = [S(ep_shape), ctypes.c_int, _I32, S(ep_size_hint)]
        L.ep_buffer_size_hint.restype = ctypes.c_int
        L.ep_get_layout.argtypes = [S(ep_shape), _P, S(ep_layout), S(ep_handle), _P,
                                    ctypes.c_size_t, S(ep_launch)]
        L.ep_get_layout_static_scratch.argtypes = [S(ep_shape), _P, S(ep_layout), S(ep_handle),
                                                   S(ep_launch)]
        L.ep_dispatch.argtypes = [S(ep_shape), _P, ctypes.c_int, _P, ctypes.c_int, _P, _P,
                                  S(ep_handle), S(ep_recv), S(ep_launch)]
        L.ep_combine.argtypes = [S(ep_shape), _P, _P, S(ep_handle), ctypes.c_int, _P, _P, _P,
                                 _P, _P, S(ep_launch)]
        L.ep_dispatch_expert_major.argtypes = [S(ep_shape), _P, ctypes.c_int, _P, _P, S(ep_handle),
                                                S(ep_recv), S(ep_launch)]
        L.ep_combine_expert_major.argtypes = [S(ep_shape), _P, _P, S(ep_handle), ctypes.c_int, _P, _P,
                                               _P, S(ep_launch)]
        L.ep_ll_dispatch.argtypes = [S(ep_shape), _P, _P, ctypes.c_int, ctypes.c_int,
                                     S(ep_ll_buffer), S(ep_launch)]
        L.ep_ll_combine.argtypes = [S(ep_shape), _P, _P, _P, S(ep_ll_buffer), ctypes.c_int, _P,
                                    S(ep_launch)]
        L.ep_clean_ll_buffer.argtypes = [S(ep_shape), S(ep_ll_buffer), S(ep_launch)]
        L.ep_read_recv_counts_sync.argtypes = [S(ep_shape), S(ep_handle), _P, _P]
        L.ep_read_error_flags_sync.argtypes = [_P, _P, _P]
        L.ep_selftest_wait_timeout.argtypes = [_P, _I32, _P, S(ep_launch)]
        L.ep_status_string.argtypes = [_I32]
        L.ep_status_string.restype = ctypes.c_char_p
        L.ep_last_cuda_error.argtypes = []
        L.ep_last_cuda_error.restype = ctypes.c_char_p
        L.ep_kernel_launch_count.argtypes = []
        L.ep_kernel_launch_count.restype = ctypes.c_uint64
        L.ep_abi_version.argtypes = []
        L.ep_abi_version.restype = _I32
        for name in ("ep_get_layout", "ep_get_layout_static_scratch", "ep_dispatch", "ep_combine",
                     "ep_dispatch_expert_major", "ep_combine_expert_major", "ep_ll_dispatch",
                     "ep_ll_combine", "ep_clean_ll_buffer", "ep_read_recv_counts_sync",
                     "ep_read_error_flags_sync", "ep_selftest_wait_timeout"):
            getattr(L, name).restype = _I32
        _lib = L
    return _lib


# ---------------------------------------------------------------- marshalling helpers

def _ptr(t) -> Optional[int]:
    """Device pointer of a tensor (None -> NULL). Requires a contiguous CUDA tensor."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libep takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libep takes contiguous tensors")
    return t.data_ptr() or None


def _check(func: str, status: int):
    if status != EP_OK:
        L = lib()
        detail = L.ep_status_string(status).decode()
        if status == EP_ERR_CUDA:
            detail += f" ({L.ep_last_cuda_error().decode()})"
        raise EpError(func, status, detail)


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


def _event_handle(ev) -> Optional[int]:
    if ev is None:
        return None
    return ev.cuda_event or None


def make_shape(R: int, T: int, H: int, E: int, k: int, C: int = 12, nmax: int = 0,
               num_sms: int = 0) -> ep_shape:
    return ep_shape(R, T, H, E, k, C, nmax, num_sms)


def make_launch(stream=None, wait_event=None, record_event=None, error_flags=None) -> ep_launch:
    """stream: torch.cuda.Stream (None = current); events: torch.cuda.Event (a record
    event must already exist on the device, i.e. have been created with a record);
    error_flags: int32/uint32 device tensor of one element or None."""
    return ep_launch(_stream_handle(stream), _event_handle(wait_event),
                     _event_handle(record_event), _ptr(error_flags))


def _launch(launch) -> ep_launch:
    return launch if isinstance(launch, ep_launch) else make_launch()


# ---------------------------------------------------------------- C-ABI functions

def ep_layout_workspace_size(shape: ep_shape) -> int:
    return int(lib().ep_layout_workspace_size(ctypes.byref(shape)))


def ep_buffer_size_hint(shape: ep_shape, recv_dtype: int = EP_BF16,
                        fp8_scale: int = EP_FP8_SCALE_FP32) -> dict:
    """Worst-case buffer sizes for `shape` (see ep_size_hint in ep.h) as a dict."""
    h = ep_size_hint()
    _check("ep_buffer_size_hint",
           lib().ep_buffer_size_hint(ctypes.byref(shape), recv_dtype, fp8_scale, ctypes.byref(h)))
    return {name: int(getattr(h, name)) for name, _ in ep_size_hint._fields_}


def ep_get_layout(shape: ep_shape, topk_idx, layout: Optional[ep_layout], handle: ep_handle,
                  workspace, launch: Optional[ep_launch] = None) -> None:
    L = lib()
    st = L.ep_get_layout(ctypes.byref(shape), _ptr(topk_idx),
                         ctypes.byref(layout) if layout is not None else None,
                         ctypes.byref(handle), _ptr(workspace),
                         workspace.numel() * workspace.element_size(),
                         ctypes.byref(_launch(launch)))
    _check("ep_get_layout", st)


def ep_get_layout_static_scratch(shape: ep_shape, topk_idx, layout: Optional[ep_layout],
                                 handle: ep_handle, launch: Optional[ep_launch] = None) -> None:
    """ep_get_layout for callers that cannot allocate device memory: the workspace is a
    fixed array inside libep.so (EP_LAYOUT_STATIC_SCRATCH_BYTES). Calls on one device
    share it, so calls that may run at the same time on the GPU must be ordered."""
    st = lib().ep_get_layout_static_scratch(ctypes.byref(shape), _ptr(topk_idx),
                                            ctypes.byref(layout) if layout is not None else None,
                                            ctypes.byref(handle), ctypes.byref(_launch(launch)))
    _check("ep_get_layout_static_scratch", st)


def _offsets(row_offset: Sequence[int]):
    arr = (ctypes.c_int64 * len(row_offset))(*[int(v) for v in row_offset])
    return arr


def ep_dispatch(shape: ep_shape, x, x_dtype: int, x_scales, recv_dtype: int, topk_idx,
                topk_weights, handle: ep_handle, recv_x, recv_x_scales, recv_topk_idx,
                recv_topk_weights, recv_src_idx, row_offset: Sequence[int],
                launch: Optional[ep_launch] = None, fp8_scale: int = EP_FP8_SCALE_FP32,
                tensor_scale: float = 0.0) -> None:
    off = _offsets(row_offset)
    out = ep_recv(_ptr(recv_x), _ptr(recv_x_scales), _ptr(recv_topk_idx),
                  _ptr(recv_topk_weights), _ptr(recv_src_idx),
                  ctypes.cast(off, ctypes.c_void_p), ep_fp8_options(fp8_scale, tensor_scale))
    st = lib().ep_dispatch(ctypes.byref(shape), _ptr(x), x_dtype, _ptr(x_scales), recv_dtype,
                           _ptr(topk_idx), _ptr(topk_weights), ctypes.byref(handle),
                           ctypes.byref(out), ctypes.byref(_launch(launch)))
    _check("ep_dispatch", st)


def ep_combine(shape: ep_shape, y, row_offset: Sequence[int], handle: ep_handle, mode: int,
               topk_idx, topk_weights, recv_topk_weights, out, combined_topk_weights,
               launch: Optional[ep_launch] = None) -> None:
    off = _offsets(row_offset)
    st = lib().ep_combine(ctypes.byref(shape), _ptr(y), ctypes.cast(off, ctypes.c_void_p),
                          ctypes.byref(handle), mode, _ptr(topk_idx), _ptr(topk_weights),
                          _ptr(recv_topk_weights), _ptr(out), _ptr(combined_topk_weights),
                          ctypes.byref(_launch(launch)))
    _check("ep_combine", st)


def ep_dispatch_expert_major(shape: ep_shape, x, recv_dtype: int, topk_idx, topk_weights,
                             handle: ep_handle, recv_x, recv_x_scales, recv_weights, recv_src_idx,
                             row_offset: Sequence[int], launch: Optional[ep_launch] = None,
                             fp8_scale: int = EP_FP8_SCALE_FP32, tensor_scale: float = 0.0) -> None:
    off = _offsets(row_offset)
    out = ep_recv(_ptr(recv_x), _ptr(recv_x_scales), None, _ptr(recv_weights), _ptr(recv_src_idx),
                  ctypes.cast(off, ctypes.c_void_p), ep_fp8_options(fp8_scale, tensor_scale))
    st = lib().ep_dispatch_expert_major(ctypes.byref(shape), _ptr(x), recv_dtype, _ptr(topk_idx),
                                        _ptr(topk_weights), ctypes.byref(handle), ctypes.byref(out),
                                        ctypes.byref(_launch(launch)))
    _check("ep_dispatch_expert_major", st)


def ep_combine_expert_major(shape: ep_shape, y, row_offset: Sequence[int], handle: ep_handle,
                            mode: int, topk_idx, topk_weights, out,
                            launch: Optional[ep_launch] = None) -> None:
    off = _offsets(row_offset)
    st = lib().ep_combine_expert_major(ctypes.byref(shape), _ptr(y), ctypes.cast(off, ctypes.c_void_p),
                                       ctypes.byref(handle), mode, _ptr(topk_idx), _ptr(topk_weights),
                                       _ptr(out), ctypes.byref(_launch(launch)))
    _check("ep_combine_expert_major", st)


def ep_ll_dispatch(shape: ep_shape, x, topk_idx, use_fp8: bool, phase: int, buf: ep_ll_buffer,
                   launch: Optional[ep_launch] = None) -> None:
    st = lib().ep_ll_dispatch(ctypes.byref(shape), _ptr(x), _ptr(topk_idx), int(bool(use_fp8)),
                              phase, ctypes.byref(buf), ctypes.byref(_launch(launch)))
    _check("ep_ll_dispatch", st)


def ep_ll_combine(shape: ep_shape, y, topk_idx, topk_weights, handle: ep_ll_buffer, phase: int,
                  out, launch: Optional[ep_launch] = None) -> None:
    st = lib().ep_ll_combine(ctypes.byref(shape), _ptr(y), _ptr(topk_idx), _ptr(topk_weights),
                             ctypes.byref(handle), phase, _ptr(out), ctypes.byref(_launch(launch)))
    _check("ep_ll_combine", st)


def ep_clean_ll_buffer(shape: ep_shape, buf: ep_ll_buffer, launch: Optional[ep_launch] = None) -> None:
    _check("ep_clean_ll_buffer", lib().ep_clean_ll_buffer(ctypes.byref(shape), ctypes.byref(buf),
                                                          ctypes.byref(_launch(launch))))


def ep_read_recv_counts_sync(shape: ep_shape, handle: ep_handle, stream=None) -> list:
    host = (ctypes.c_int32 * shape.num_ranks)()
    st = lib().ep_read_recv_counts_sync(ctypes.byref(shape), ctypes.byref(handle),
                                        ctypes.cast(host, ctypes.c_void_p), _stream_handle(stream))
    _check("ep_read_recv_counts_sync", st)
    return list(host)


def ep_selftest_wait_timeout(src16, timeout_ms: int, elapsed_us=None,
                             launch: Optional[ep_launch] = None) -> None:
    _check("ep_selftest_wait_timeout",
           lib().ep_selftest_wait_timeout(_ptr(src16), timeout_ms, _ptr(elapsed_us),
                                          ctypes.byref(launch or make_launch())))


def ep_read_error_flags_sync(error_flags, stream=None) -> int:
    host = ctypes.c_uint32(0)
    st = lib().ep_read_error_flags_sync(_ptr(error_flags), ctypes.byref(host),
                                        _stream_handle(stream))
    _check("ep_read_error_flags_sync", st)
    return int(host.value)


def ep_kernel_launch_count() -> int:
    return int(lib().ep_kernel_launch_count())


def ep_abi_version() -> int:
    return int(lib().ep_abi_version())
