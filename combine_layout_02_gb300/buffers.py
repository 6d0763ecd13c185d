"""Caller-side device buffers for the C ABI (PyTorch is used as the allocator only).

The library never allocates; these classes size and own the tensors each call needs
and build the plain-pointer structs (``ep_layout``, ``ep_handle``, ``ep_ll_buffer``).
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import (EP_BF16, EP_FP8_SCALE_FP32, EP_FP8_SCALE_UE8M0, EP_LL_LAYOUT_PACKED,
               EP_LL_LAYOUT_SLOTS, ep_fp8_options,
               ep_handle, ep_layout, ep_layout_workspace_size, ep_ll_buffer, ep_shape, _ptr)


def new_event(stream=None) -> torch.cuda.Event:
    """A CUDA event that already exists on the device (recorded once), usable as the
    record_event of a call."""
    ev = torch.cuda.Event()
    ev.record(stream if stream is not None else torch.cuda.current_stream())
    return ev


class EventOverlap:
    """The pages' event handle for overlap ("How DeepEP Achieves Communication-Computation
    Overlapping with EventOverlap", sections "CUDA Event Capture in Buffer" and "Explicit
    Stream Waiting"): a CUDA event plus tensors to keep alive until the work before it is
    done. Pass `.event` as a call's wait_event (previous_event) or record_event
    (async_finish) through make_launch; current_stream_wait() makes the current stream wait
    for it, and a `with` block waits on exit. Python sugar only: the C ABI takes the event."""

    def __init__(self, event: Optional[torch.cuda.Event] = None, extra_tensors: Sequence = ()):
        self.event = event
        self.extra_tensors = tuple(extra_tensors)

    def current_stream_wait(self) -> None:
        if self.event is not None:
            torch.cuda.current_stream().wait_event(self.event)

    def __enter__(self) -> "EventOverlap":
        return self

    def __exit__(self, *exc) -> None:
        self.current_stream_wait()


def capture(stream=None) -> EventOverlap:
    """Buffer.capture(): an EventOverlap recorded now on `stream` (default: current)."""
    return EventOverlap(new_event(stream))


def completion_event(stream=None) -> EventOverlap:
    """An EventOverlap to hand to a call as its record_event (async_finish): the call
    records it after its last kernel."""
    return EventOverlap(new_event(stream))


class LayoutBuffers:
    """Outputs of ep_get_layout plus the handle tensors and the layout workspace."""

    def __init__(self, shape: ep_shape, device="cuda", expert_major: bool = False):
        R, T, E, C = shape.num_ranks, shape.num_tokens, shape.num_experts, shape.num_channels
        i32 = dict(dtype=torch.int32, device=device)
        self.shape = shape
        self.num_tokens_per_rank = torch.empty((R, R), **i32)
        self.num_tokens_per_expert = torch.empty((R, E), **i32)
        self.is_token_in_rank = torch.empty((R, T, R), dtype=torch.uint8, device=device)
        self.rank_prefix_matrix = torch.empty((R, R), **i32)
        self.channel_prefix_matrix = torch.empty((R, R, C), **i32)
        self.recv_channel_prefix_matrix = torch.empty((R, R, C), **i32)
        self.send_head = torch.empty((R, T, R), **i32)
        self.num_recv_tokens_per_expert = torch.empty((R, E // R), **i32)
        ws = ep_layout_workspace_size(shape)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
        self.recv_src_idx: Optional[torch.Tensor] = None
        k = shape.num_topk
        self.expert_rows = torch.empty((R, T, k), **i32) if expert_major else None
        self.expert_prefix = torch.empty((R, E // R + 1), **i32) if expert_major else None

    def layout(self) -> ep_layout:
        return ep_layout(_ptr(self.num_tokens_per_rank), None, _ptr(self.num_tokens_per_expert),
                         _ptr(self.is_token_in_rank))

    def handle(self, recv_src_idx: Optional[torch.Tensor] = None) -> ep_handle:
        if recv_src_idx is not None:
            self.recv_src_idx = recv_src_idx
        return ep_handle(_ptr(self.rank_prefix_matrix), _ptr(self.channel_prefix_matrix),
                         _ptr(self.recv_channel_prefix_matrix), _ptr(self.recv_src_idx),
                         _ptr(self.is_token_in_rank), _ptr(self.send_head),
                         _ptr(self.num_recv_tokens_per_expert), _ptr(self.expert_rows),
                         _ptr(self.expert_prefix))

    def tensors(self) -> list:
        """Every device tensor this object owns."""
        return [v for v in vars(self).values() if isinstance(v, torch.Tensor)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k in (
            "num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank",
            "rank_prefix_matrix", "channel_prefix_matrix", "recv_channel_prefix_matrix",
            "send_head", "num_recv_tokens_per_expert")}


class RecvBuffers:
    """Receive buffers of a normal dispatch over `rows` rows (all destinations)."""

    def __init__(self, rows: int, H: int, k: int, recv_dtype: int = EP_BF16, with_topk=True,
                 device="cuda", fill: Optional[int] = None, fp8_scale: int = EP_FP8_SCALE_FP32):
        self.rows = rows
        if recv_dtype == EP_BF16:
            self.recv_x = torch.empty((rows, H), dtype=torch.bfloat16, device=device)
            self.recv_x_scales = None
        else:
            self.recv_x = torch.empty((rows, H), dtype=torch.uint8, device=device)
            sdt = torch.uint8 if fp8_scale == EP_FP8_SCALE_UE8M0 else torch.float32
            self.recv_x_scales = torch.empty((rows, H // 128), dtype=sdt, device=device)
        self.recv_topk_idx = torch.empty((rows, k), dtype=torch.int64, device=device) if with_topk else None
        self.recv_topk_weights = torch.empty((rows, k), dtype=torch.float32, device=device) if with_topk else None
        self.recv_src_idx = torch.empty((rows,), dtype=torch.int32, device=device)
        if fill is not None:
            self.recv_x.view(torch.uint8).fill_(fill)
            if self.recv_x_scales is not None:
                self.recv_x_scales.fill_(0xEE if self.recv_x_scales.dtype == torch.uint8 else float("nan"))
            if with_topk:
                self.recv_topk_idx.fill_(-99)
                self.recv_topk_weights.fill_(-5.0)
            self.recv_src_idx.fill_(-3)


class LLBuffers:
    """Low-latency receive buffers and handle for one shape."""

    def __init__(self, shape: ep_shape, use_fp8: bool, device="cuda", fill: Optional[int] = None,
                 fp8_scale: int = EP_FP8_SCALE_FP32, tensor_scale: float = 0.0,
                 packed: bool = False):
        R, T, H, E, k = (shape.num_ranks, shape.num_tokens, shape.hidden, shape.num_experts,
                         shape.num_topk)
        nmax = shape.num_max_dispatch_tokens_per_rank
        E_loc = E // R
        slots = R * nmax
        i32 = dict(dtype=torch.int32, device=device)
        self.fp8 = ep_fp8_options(fp8_scale, tensor_scale)
        self.layout = EP_LL_LAYOUT_PACKED if packed else EP_LL_LAYOUT_SLOTS
        if use_fp8:
            self.recv_x = torch.empty((R, E_loc, slots, H), dtype=torch.uint8, device=device)
            sdt = torch.uint8 if fp8_scale == EP_FP8_SCALE_UE8M0 else torch.float32
            self.recv_x_scales = torch.empty((R, E_loc, slots, H // 128), dtype=sdt, device=device)
        else:
            self.recv_x = torch.empty((R, E_loc, slots, H), dtype=torch.bfloat16, device=device)
            self.recv_x_scales = None
        self.src_info = torch.empty((R, E_loc, slots), **i32)
        self.slot = torch.empty((R, T, k), **i32)
        self.send_count = torch.empty((R, E_loc, R), **i32)
        self.recv_expert_count = torch.empty((R, E_loc), **i32)
        self.layout_range = torch.empty((R, E_loc, R, 2), **i32)
        if fill is not None:
            self.recv_x.view(torch.uint8).fill_(fill)
            self.src_info.fill_(-7)

    def tensors(self) -> list:
        """Every device tensor this object owns."""
        return [v for v in vars(self).values() if isinstance(v, torch.Tensor)]

    def struct(self) -> ep_ll_buffer:
        return ep_ll_buffer(_ptr(self.recv_x), _ptr(self.recv_x_scales), _ptr(self.src_info),
                            _ptr(self.slot), _ptr(self.send_count), _ptr(self.recv_expert_count),
                            _ptr(self.layout_range), self.fp8, self.layout)


def compact_row_offsets(counts: Sequence[int]) -> list:
    """Row offsets [R+1] for exactly sized receive regions (counts = N_d)."""
    off = [0]
    for c in counts:
        off.append(off[-1] + int(c))
    return off


def worst_case_row_offsets(R: int, T: int) -> list:
    """Row offsets [R+1] sized for every token of every source: no host sync needed."""
    return [d * R * T for d in range(R + 1)]
