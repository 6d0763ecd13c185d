"""A front end shaped like the pages' Python API, over the C ABI.

"DeepEP" README (EnflameTechnology/DeepEP), normal-kernel and low-latency examples: a
``Buffer`` object offers ``get_dispatch_layout``, ``dispatch``, ``combine`` (also used for
``dispatch_backward``; ``dispatch`` with a handle is ``combine_backward``),
``low_latency_dispatch`` and ``low_latency_combine``, each taking ``previous_event`` /
``async_finish`` and returning an event ("How DeepEP Achieves Communication-Computation
Overlapping with EventOverlap"); the low-latency calls can return a receive hook ("How
DeepEP Enables Hook-Based Overlapping Without SM Occupation").

Here the R expert-parallel ranks are virtual partitions of one GPU, so every tensor
carries a leading rank axis ([R][T][...] for tokens) and "received" tensors are lists of R
views into one allocation, one per destination rank. This module only allocates tensors
with PyTorch and calls the library; every step runs in the library's kernels.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch

from . import (EP_BF16, EP_COMBINE_SUM, EP_COMBINE_WEIGHTED, EP_FP8_E4M3, EP_FP8_SCALE_FP32,
               EP_FP8_SCALE_UE8M0, EP_PHASE_BOTH, EP_PHASE_RECV, EP_PHASE_SEND, ep_buffer_size_hint,
               ep_clean_ll_buffer, ep_combine, ep_combine_expert_major, ep_dispatch,
               ep_dispatch_expert_major, ep_get_layout, ep_ll_combine, ep_ll_dispatch,
               ep_read_error_flags_sync, ep_read_recv_counts_sync, make_launch, make_shape)
from .buffers import EventOverlap, LayoutBuffers, LLBuffers, new_event, worst_case_row_offsets

__all__ = ["Buffer", "DispatchHandle", "ExpertMajorHandle", "LowLatencyHandle"]


class DispatchHandle:
    """The normal-mode handle ("How DeepEP Optimizes Handle Reuse for Repeated
    Dispatches", "What the Handle Contains"): the layout tensors, the receive regions and
    recv_src_idx of the dispatch that produced it."""

    def __init__(self, layout: LayoutBuffers, row_offset: List[int], recv_src_idx: torch.Tensor,
                 num_tokens: int):
        self.layout = layout
        self.row_offset = row_offset
        self.recv_src_idx = recv_src_idx
        self.num_tokens = num_tokens

    @property
    def rank_prefix_matrix(self) -> torch.Tensor:
        return self.layout.rank_prefix_matrix

    @property
    def channel_prefix_matrix(self) -> torch.Tensor:
        return self.layout.channel_prefix_matrix

    @property
    def recv_channel_prefix_matrix(self) -> torch.Tensor:
        return self.layout.recv_channel_prefix_matrix

    @property
    def is_token_in_rank(self) -> torch.Tensor:
        return self.layout.is_token_in_rank

    @property
    def send_head(self) -> torch.Tensor:
        return self.layout.send_head


class ExpertMajorHandle:
    """Layout with the expert-major placement, and the region of every destination."""

    def __init__(self, layout: LayoutBuffers, row_offset: List[int], expert_prefix: List[List[int]],
                 num_tokens: int):
        self.layout = layout
        self.row_offset = row_offset
        self.expert_prefix = expert_prefix
        self.num_tokens = num_tokens


class LowLatencyHandle:
    """The low-latency handle: the slot buffers of one low_latency_dispatch."""

    def __init__(self, buf: LLBuffers, topk_idx: torch.Tensor):
        self.buf = buf
        self.topk_idx = topk_idx


def _split(t: torch.Tensor, row_offset: Sequence[int]) -> List[torch.Tensor]:
    return [t[row_offset[d]:row_offset[d + 1]] for d in range(len(row_offset) - 1)]


class _Call:
    """Where one Buffer call runs: the stream, the event it waits on first, the event it
    records last (async_finish), and the tensors it touches on that stream."""

    def __init__(self, compute, stream, wait, done, on_comm_alloc: bool):
        self.compute, self.stream, self.wait, self.done = compute, stream, wait, done
        self.on_comm_alloc = on_comm_alloc
        self.tensors: List[torch.Tensor] = []

    def launch(self, err: torch.Tensor):
        return make_launch(self.stream, wait_event=self.wait, record_event=self.done, error_flags=err)

    def alloc(self):
        """Context for allocating the call's outputs: the comm stream's pool with
        allocate_on_comm_stream, else the compute stream's."""
        return torch.cuda.stream(self.stream if self.on_comm_alloc else self.compute)

    def use(self, *tensors) -> None:
        for t in tensors:
            if isinstance(t, torch.Tensor) and t.is_cuda:
                self.tensors.append(t)


class Buffer:
    """One virtual expert-parallel group of `num_ranks` ranks on the current GPU.

    Mirrors the pages' Buffer: get_dispatch_layout -> dispatch -> combine (normal kernels)
    and low_latency_dispatch -> low_latency_combine (low-latency kernels). As "How DeepEP
    Achieves Communication-Computation Overlapping with EventOverlap" describes, the calls
    run on the Buffer's own communication stream (get_comm_stream()): it first waits for
    `previous_event` (an EventOverlap), or else for all work issued so far on the current
    (compute) stream. With `async_finish=True` the call returns an EventOverlap that
    completes with its kernels, and the compute stream does not wait until
    current_stream_wait() (or the end of a `with` block); with `async_finish=False` the
    compute stream waits for the call's kernels before its next work (the host is never
    blocked, except by the counts read of an exact-size dispatch). A low-latency call with
    `return_recv_hook=True` runs on the compute stream instead ("How DeepEP Enables
    Hook-Based Overlapping Without SM Occupation": launch_stream = compute_stream). The
    expert-major calls run on the compute stream. Device problems the kernels detect (bad
    expert ids, undersized regions) accumulate in an error word that check_errors() reads.
    """

    def __init__(self, num_ranks: int, num_experts: int, hidden: int, num_topk: int,
                 num_channels: int = 12, device="cuda"):
        self.R, self.E, self.H, self.k, self.C = num_ranks, num_experts, hidden, num_topk, num_channels
        self.device = torch.device(device)
        self.num_sms = 0
        self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.comm_stream = torch.cuda.Stream(device=self.device)
        self._layout = None           # (id(num_tokens_per_rank), LayoutBuffers, topk_idx)

    # ----------------------------------------------------------------- common
    def set_num_sms(self, num_sms: int) -> None:
        """Caps the grid of the copy kernels (0 = every SM), as Buffer.set_num_sms."""
        self.num_sms = int(num_sms)

    def get_comm_stream(self) -> torch.cuda.Stream:
        """The stream the normal and (without a receive hook) low-latency calls run on."""
        return self.comm_stream

    @staticmethod
    def capture() -> EventOverlap:
        """An EventOverlap recorded now on the current stream (Buffer.capture()), to pass
        as a call's previous_event."""
        return EventOverlap(new_event(torch.cuda.current_stream()))

    def get_buffer_size_hint(self, num_tokens: int, fp8: bool = False,
                             num_max_dispatch_tokens_per_rank: int = 0,
                             fp8_scale: int = EP_FP8_SCALE_FP32) -> dict:
        """Worst-case byte sizes of the receive and low-latency buffers for num_tokens per
        rank (the pages' size-hint calls; the caller, not the library, allocates)."""
        sh = self._shape(num_tokens, num_max_dispatch_tokens_per_rank)
        return ep_buffer_size_hint(sh, EP_FP8_E4M3 if fp8 else EP_BF16, fp8_scale)

    def check_errors(self) -> int:
        """Waits for the comm stream and the current stream, then returns the
        EP_DEVERR_* bits seen so far."""
        self.comm_stream.synchronize()
        return ep_read_error_flags_sync(self.err)

    def _shape(self, T: int, nmax: int = 0):
        return make_shape(self.R, T, self.H, self.E, self.k, self.C, nmax=nmax, num_sms=self.num_sms)

    def _begin(self, previous_event: Optional[EventOverlap], async_finish: bool,
               allocate_on_comm_stream: bool = False, on_compute: bool = False) -> _Call:
        compute = torch.cuda.current_stream(self.device)
        stream = compute if on_compute else self.comm_stream
        if previous_event is not None:
            wait = previous_event.event
        elif stream is not compute:
            wait = new_event(compute)          # the comm stream follows the compute stream
        else:
            wait = None
        done = new_event(stream) if async_finish else None   # re-recorded after the kernels
        return _Call(compute, stream, wait, done, allocate_on_comm_stream and not on_compute)

    def _end(self, call: _Call, keep=()) -> EventOverlap:
        """Marks the tensors the call touched as in use on its stream (so the caching
        allocator does not hand them out again before its kernels are done) and, without
        async_finish, makes the compute stream wait for the call. Outputs allocated from
        the comm stream's pool are read on the compute stream, so they are also marked as
        in use there: freeing them then waits for the compute stream's work issued so far
        before the block can serve another comm-stream call (one that passes an older
        previous_event does not wait for the compute stream itself)."""
        if call.stream is not call.compute:
            for t in call.tensors:
                t.record_stream(call.stream)
                if call.on_comm_alloc:
                    t.record_stream(call.compute)
            if call.done is None:
                call.compute.wait_stream(call.stream)
        return EventOverlap(call.done, tuple(keep))

    # ----------------------------------------------------------------- normal kernels
    def get_dispatch_layout(self, topk_idx: torch.Tensor, previous_event: Optional[EventOverlap] = None,
                            async_finish: bool = False, allocate_on_comm_stream: bool = False):
        """topk_idx [R][T][k] int64 (-1 masked) -> (num_tokens_per_rank [R][R],
        None (no RDMA domain), num_tokens_per_expert [R][E], is_token_in_rank [R][T][R] uint8,
        event)."""
        T = topk_idx.shape[1]
        sh = self._shape(T)
        call = self._begin(previous_event, async_finish, allocate_on_comm_stream)
        with call.alloc():
            lb = LayoutBuffers(sh, self.device)
        call.use(topk_idx, *lb.tensors())
        ep_get_layout(sh, topk_idx, lb.layout(), lb.handle(), lb.workspace, call.launch(self.err))
        self._layout = (id(lb.num_tokens_per_rank), lb, topk_idx)
        return (lb.num_tokens_per_rank, None, lb.num_tokens_per_expert, lb.is_token_in_rank,
                self._end(call, (lb.workspace,)))

    def dispatch(self, x, handle: Optional[DispatchHandle] = None,
                 num_tokens_per_rank: Optional[torch.Tensor] = None,
                 topk_idx: Optional[torch.Tensor] = None, topk_weights: Optional[torch.Tensor] = None,
                 fp8: bool = False, fp8_scale: int = EP_FP8_SCALE_FP32, tensor_scale: float = 0.0,
                 num_worst_tokens: bool = False, previous_event: Optional[EventOverlap] = None,
                 async_finish: bool = False, allocate_on_comm_stream: bool = False):
        """x: bf16 [R][T][H], or the pre-quantised tuple (e4m3 [R][T][H] uint8, scales
        [R][T][H/128] fp32). A first dispatch passes topk_idx (and topk_weights) with the
        layout from get_dispatch_layout (its num_tokens_per_rank tensor) or none (the
        layout is then computed here); a repeated dispatch passes only `handle`.
        fp8=True quantises bf16 x to e4m3 on the way (per-128-channel scales).
        Receive regions are exact (the host reads the counts first, the pages' CPU wait)
        unless num_worst_tokens=True (worst-case regions of R*T rows, no host wait).

        Returns (recv_x, recv_topk_idx, recv_topk_weights, num_recv_tokens_per_expert_list,
        handle, event); recv_x is a list of R row tensors (or of (e4m3, scales) pairs), the
        topk lists are None for a repeated dispatch."""
        pre_quantised = isinstance(x, (tuple, list))
        xq, xs = (x[0], x[1]) if pre_quantised else (x, None)
        R, T, H = xq.shape[0], xq.shape[1], xq.shape[2]
        sh = self._shape(T)
        if handle is None and topk_idx is None:
            raise ValueError("dispatch needs topk_idx or a handle")
        if handle is not None and (topk_idx is not None or topk_weights is not None):
            raise ValueError("a reused handle takes no topk_idx / topk_weights")
        call = self._begin(previous_event, async_finish, allocate_on_comm_stream)
        launch = call.launch(self.err)
        call.use(xq, xs, topk_idx, topk_weights)
        if handle is None:
            lb = None
            if self._layout is not None and num_tokens_per_rank is not None and \
                    self._layout[0] == id(num_tokens_per_rank) and self._layout[2] is topk_idx:
                lb = self._layout[1]
            if lb is None:
                with call.alloc():
                    lb = LayoutBuffers(sh, self.device)
                call.use(*lb.tensors())
                ep_get_layout(sh, topk_idx, lb.layout(), lb.handle(), lb.workspace, launch)
                launch.wait_event = None          # waited once already
            if num_worst_tokens:
                off = list(worst_case_row_offsets(R, T))
            else:
                counts = ep_read_recv_counts_sync(sh, lb.handle(), call.stream)   # the CPU wait
                off = [0]
                for n in counts:
                    off.append(off[-1] + int(n))
            with call.alloc():
                recv_src_idx = torch.empty((max(off[-1], 1),), dtype=torch.int32, device=self.device)
            handle = DispatchHandle(lb, off, recv_src_idx, T)
            reuse = False
        else:
            reuse = True
        off = handle.row_offset
        rows = max(off[-1], 1)
        quant = fp8 or pre_quantised
        with call.alloc():
            if quant:
                rx = torch.empty((rows, H), dtype=torch.uint8, device=self.device)
                ue8m0 = fp8 and not pre_quantised and fp8_scale == EP_FP8_SCALE_UE8M0
                sdt = torch.uint8 if ue8m0 else torch.float32
                rs = torch.empty((rows, H // 128), dtype=sdt, device=self.device)
            else:
                rx = torch.empty((rows, H), dtype=torch.bfloat16, device=self.device)
                rs = None
            rti = None if reuse else torch.empty((rows, self.k), dtype=torch.int64, device=self.device)
            rtw = None if (reuse or topk_weights is None) else \
                torch.empty((rows, self.k), dtype=torch.float32, device=self.device)
        call.use(rx, rs, rti, rtw, handle.recv_src_idx, *handle.layout.tensors())
        ep_dispatch(sh, xq, EP_FP8_E4M3 if pre_quantised else EP_BF16, xs,
                    EP_FP8_E4M3 if quant else EP_BF16, None if reuse else topk_idx,
                    None if reuse else topk_weights, handle.layout.handle(handle.recv_src_idx),
                    rx, rs, rti, rtw, handle.recv_src_idx, off, launch,
                    fp8_scale=fp8_scale if (fp8 and not pre_quantised) else EP_FP8_SCALE_FP32,
                    tensor_scale=tensor_scale if (fp8 and not pre_quantised) else 0.0)
        recv_x = list(zip(_split(rx, off), _split(rs, off))) if quant else _split(rx, off)
        per_expert = handle.layout.num_recv_tokens_per_expert
        return (recv_x, None if rti is None else _split(rti, off),
                None if rtw is None else _split(rtw, off), per_expert, handle,
                self._end(call, (rx,)))

    def combine(self, x, handle: DispatchHandle, topk_weights=None,
                weight_by: Optional[Tuple[torch.Tensor, torch.Tensor]] = None,
                previous_event: Optional[EventOverlap] = None, async_finish: bool = False,
                allocate_on_comm_stream: bool = False):
        """x: the expert outputs in the dispatch's row order -- one bf16 tensor of all rows,
        or the list of R per-destination views of one allocation that dispatch returned.
        Plain sum over the ranks a token was sent to (the pages' combine); with
        weight_by=(topk_idx, topk_weights), each rank's row is scaled by the token's
        weights of the experts on that rank (the weighted top-k reduce). topk_weights (a
        list of R [rows_d][k] tensors, or one tensor) are reduced alongside
        (dispatch_backward). Returns (combined_x [R][T][H], combined_topk_weights, event)."""
        y = self._rows_tensor(x, handle.row_offset)
        T = handle.num_tokens
        sh = self._shape(T)
        call = self._begin(previous_event, async_finish, allocate_on_comm_stream)
        rtw = None if topk_weights is None else self._rows_tensor(topk_weights, handle.row_offset)
        with call.alloc():
            out = torch.empty((self.R, T, self.H), dtype=torch.bfloat16, device=self.device)
            cw = None if rtw is None else torch.empty((self.R, T, self.k), dtype=torch.float32,
                                                      device=self.device)
        mode = EP_COMBINE_WEIGHTED if weight_by is not None else EP_COMBINE_SUM
        tk, tw = weight_by if weight_by is not None else (None, None)
        call.use(y, rtw, out, cw, tk, tw, handle.recv_src_idx, *handle.layout.tensors())
        ep_combine(sh, y, handle.row_offset, handle.layout.handle(handle.recv_src_idx), mode, tk, tw,
                   rtw, out, cw, call.launch(self.err))
        return out, cw, self._end(call, (y,))

    @staticmethod
    def _rows_tensor(x, row_offset: Sequence[int]) -> torch.Tensor:
        """One tensor over all rows: x itself, or the allocation the R views share."""
        if isinstance(x, torch.Tensor):
            return x
        base = x[0]
        row = base.shape[1] * base.element_size() if base.dim() > 1 else base.element_size()
        for d, t in enumerate(x):
            if t.data_ptr() != base.data_ptr() + (row_offset[d] - row_offset[0]) * row:
                raise ValueError("combine takes the rows as one allocation in region order "
                                 "(the views dispatch returned); got separate tensors")
        n = row_offset[-1] - row_offset[0]
        return base.as_strided((max(n, 1),) + tuple(base.shape[1:]), base.stride())

    # ----------------------------------------------------------------- expert-major
    def dispatch_expert_major(self, x: torch.Tensor, topk_idx: torch.Tensor,
                              topk_weights: Optional[torch.Tensor] = None, fp8: bool = False,
                              fp8_scale: int = EP_FP8_SCALE_FP32, tensor_scale: float = 0.0):
        """One row per valid (token, expert) entry, each destination's rows grouped by local
        expert (contiguous blocks a grouped GEMM can take as they are; the README's
        "specific format" for the received rows). The host reads the per-expert counts
        (a CPU wait) to size exact regions. Returns (recv_x: R lists of E_loc row tensors,
        or of (e4m3, scales) pairs; recv_src_idx and recv_weights: R lists of E_loc
        tensors (the token index and the entry's weight of each row); handle)."""
        R, T, H = x.shape[0], x.shape[1], x.shape[2]
        E_loc = self.E // self.R
        sh = self._shape(T)
        lb = LayoutBuffers(sh, self.device, expert_major=True)
        launch = self._begin(None, False, on_compute=True).launch(self.err)
        ep_get_layout(sh, topk_idx, lb.layout(), lb.handle(), lb.workspace, launch)
        prefix = lb.expert_prefix.cpu().tolist()                 # the CPU wait
        off = [0]
        for d in range(R):
            off.append(off[-1] + int(prefix[d][-1]))
        rows = max(off[-1], 1)
        if fp8:
            rx = torch.empty((rows, H), dtype=torch.uint8, device=self.device)
            sdt = torch.uint8 if fp8_scale == EP_FP8_SCALE_UE8M0 else torch.float32
            rs = torch.empty((rows, H // 128), dtype=sdt, device=self.device)
        else:
            rx = torch.empty((rows, H), dtype=torch.bfloat16, device=self.device)
            rs = None
        ri = torch.empty((rows,), dtype=torch.int32, device=self.device)
        rw = None if topk_weights is None else torch.empty((rows,), dtype=torch.float32, device=self.device)
        ep_dispatch_expert_major(sh, x, EP_FP8_E4M3 if fp8 else EP_BF16, topk_idx, topk_weights,
                                 lb.handle(), rx, rs, rw, ri, off, launch,
                                 fp8_scale=fp8_scale if fp8 else EP_FP8_SCALE_FP32,
                                 tensor_scale=tensor_scale if fp8 else 0.0)

        def blocks(t):
            if t is None:
                return None
            return [[t[off[d] + prefix[d][e]: off[d] + prefix[d][e + 1]] for e in range(E_loc)]
                    for d in range(R)]
        recv_x = [list(zip(a, b)) for a, b in zip(blocks(rx), blocks(rs))] if fp8 else blocks(rx)
        return recv_x, blocks(ri), blocks(rw), ExpertMajorHandle(lb, off, prefix, T)

    def combine_expert_major(self, y: torch.Tensor, handle: ExpertMajorHandle, topk_idx: torch.Tensor,
                             topk_weights: Optional[torch.Tensor] = None):
        """y: the grouped GEMM's output, one tensor of all rows in the dispatch's order.
        Sums each token's entry rows, weighted by topk_weights when given. Returns
        combined_x [R][T][H]."""
        sh = self._shape(handle.num_tokens)
        out = torch.empty((self.R, handle.num_tokens, self.H), dtype=torch.bfloat16, device=self.device)
        launch = self._begin(None, False, on_compute=True).launch(self.err)
        mode = EP_COMBINE_WEIGHTED if topk_weights is not None else EP_COMBINE_SUM
        ep_combine_expert_major(sh, y, handle.row_offset, handle.layout.handle(), mode, topk_idx,
                                topk_weights, out, launch)
        return out

    # ----------------------------------------------------------------- low latency
    def low_latency_dispatch(self, x: torch.Tensor, topk_idx: torch.Tensor,
                             num_max_dispatch_tokens_per_rank: int, use_fp8: bool = True,
                             packed: bool = False, fp8_scale: int = EP_FP8_SCALE_FP32,
                             tensor_scale: float = 0.0, previous_event: Optional[EventOverlap] = None,
                             async_finish: bool = False, return_recv_hook: bool = False,
                             allocate_on_comm_stream: bool = False):
        """x bf16 [R][T][H], topk_idx [R][T][k] -> (recv_x [R][E_loc][R*Nmax][H] (or
        (e4m3, scales)), recv_count [R][E_loc] int32, handle, event, hook). With
        return_recv_hook the send phase runs now and hook() runs the receive phase."""
        T = x.shape[1]
        nmax = num_max_dispatch_tokens_per_rank
        sh = self._shape(T, nmax)
        call = self._begin(previous_event, async_finish, allocate_on_comm_stream,
                           on_compute=return_recv_hook)
        with call.alloc():
            buf = LLBuffers(sh, use_fp8, device=self.device, fp8_scale=fp8_scale,
                            tensor_scale=tensor_scale, packed=packed)
        call.use(x, topk_idx, *buf.tensors())
        phase = EP_PHASE_SEND if return_recv_hook else EP_PHASE_BOTH
        ep_ll_dispatch(sh, x, topk_idx, use_fp8, phase, buf.struct(), call.launch(self.err))
        hook: Optional[Callable[[], None]] = None
        if return_recv_hook:
            def hook() -> None:
                ep_ll_dispatch(sh, x, topk_idx, use_fp8, EP_PHASE_RECV, buf.struct(),
                               make_launch(torch.cuda.current_stream(), error_flags=self.err))
        recv_x = (buf.recv_x, buf.recv_x_scales) if use_fp8 else buf.recv_x
        return recv_x, buf.recv_expert_count, LowLatencyHandle(buf, topk_idx), \
            self._end(call, (buf.recv_x,)), hook

    def low_latency_combine(self, x: torch.Tensor, topk_idx: torch.Tensor, topk_weights: torch.Tensor,
                            handle: LowLatencyHandle, previous_event: Optional[EventOverlap] = None,
                            async_finish: bool = False, return_recv_hook: bool = False,
                            allocate_on_comm_stream: bool = False):
        """x bf16 [R][E_loc][R*Nmax][H] (expert outputs in the dispatch's slots) ->
        (combined_x [R][T][H], event, hook): the weighted top-k sum per token. With
        return_recv_hook the reduction runs when hook() is called."""
        buf = handle.buf
        R, T = topk_idx.shape[0], topk_idx.shape[1]
        nmax = buf.recv_x.shape[2] // R
        sh = self._shape(T, nmax)
        call = self._begin(previous_event, async_finish, allocate_on_comm_stream,
                           on_compute=return_recv_hook)
        with call.alloc():
            out = torch.empty((R, T, self.H), dtype=torch.bfloat16, device=self.device)
        call.use(x, topk_idx, topk_weights, out, *buf.tensors())
        launch = call.launch(self.err)
        hook: Optional[Callable[[], None]] = None
        if return_recv_hook:
            ep_ll_combine(sh, x, topk_idx, topk_weights, buf.struct(), EP_PHASE_SEND, out, launch)

            def hook() -> None:
                ep_ll_combine(sh, x, topk_idx, topk_weights, buf.struct(), EP_PHASE_RECV, out,
                              make_launch(torch.cuda.current_stream(), error_flags=self.err))
        else:
            ep_ll_combine(sh, x, topk_idx, topk_weights, buf.struct(), EP_PHASE_BOTH, out, launch)
        return out, self._end(call, (x,)), hook

    def clean_low_latency_buffer(self, handle: LowLatencyHandle) -> None:
        """Zeroes the count signals, receive counts and layout ranges of a low-latency
        handle's buffers (clean_low_latency_buffer; optional here, since every send phase
        rewrites them), on the current stream."""
        buf = handle.buf
        R, T = handle.topk_idx.shape[0], handle.topk_idx.shape[1]
        sh = self._shape(T, buf.recv_x.shape[2] // R)
        ep_clean_ll_buffer(sh, buf.struct(), self._begin(None, False, on_compute=True).launch(self.err))
