"""Benchmark: MoE expert-parallel layout + dispatch + combine on one GB300.

One step = ep_get_layout -> ep_dispatch (bf16) -> ep_combine (weighted, identity
experts: y = recv_x) over the DeepSeek-V3-shaped workload: R=8 virtual ranks x 4096
tokens, hidden 7168 bf16, 256 experts (32 per rank), top-8 distinct uniform, fp32
softmax weights, 12 channels, receive regions sized for the worst case (no host sync).

Prints one JSON line. `value` is the effective HBM bandwidth of the whole step
(algorithmic bytes of layout + dispatch + combine / device time per step, inputs
resident in HBM, inputs larger than L2), timed with CUDA events only around each region
of K steps, so the kernels chain through programmatic dependent launch as in use. Every
timed pass repeats its K steps until half a second of wall time has passed, so the
nvidia-smi clock sampler sees the whole window under load; figures are means over all
repeats (`repeats`, `timed_steps`). `dispatch_gbs`, `combine_gbs`, `layout_dispatch_us`
and `roofline` come from a second timed pass of the same steps with CUDA events on the
launching stream around every phase; `layout_dispatch_region_us` from a third pass with
one event before the layout and one after the dispatch (the dispatch chained to the layout
kernels as in use). `layout_dispatch_synced_us` is the exact-size
variant: layout, a host wait for the received counts, then the dispatch into regions of
exactly those sizes. `e2e` is the same metric through the same C-ABI calls with host
buffers: pinned host -> device copy of x / topk_idx / topk_weights and a device -> host
copy of the combined output inside every timed step.

The same line carries, under `workloads`, the other workloads of the benchmark, each
timed the same way with its own roofline and clock record: group_limited (fused e4m3
dispatch + combine), zipf_reuse (dispatch and combine with a cached handle) and
ll_decode (low-latency send, receive hook and combine, L2 flushed before every step).
--workload picks another step as the headline instead (group_limited, zipf_reuse,
ll_decode, ll_decode_packed, dsv3_expert_major, dsv3_backward; see WORKLOAD_TEXT);
--fp8-scale picks the scale format of the e4m3 sends. The roofline's traffic comes from
the committed ncu counters only when they were taken on the same workload and kernel
sources.

--impl reference times the CPU oracle (test infrastructure; single-threaded C) on a
bounded token sample of the same workload and prints the same metric with the same
config.

Multi-GPU: the path does not shard (virtual ranks live in one GPU's memory), so
`--gpus N` under torchrun runs N independent replicas; the barrier and max-over-ranks
timing keep the contract and `value` sums all replicas' bytes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "dispatch/combine effective HBM GB/s (% of GB300 peak); µs per layout+dispatch"
WORKLOAD = workloads.CONFIGS["dsv3"]
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


# ----------------------------------------------------------------------------- bytes model

def algorithmic_bytes(R, T, H, k, N, weighted=True):
    """Bytes that must be read + written once (bf16 payload, int64 topk_idx, fp32
    weights, int32 send_head / src_idx, uint8 is_token_in_rank). N = received rows."""
    Tt = R * T
    layout = Tt * k * 8 + Tt * R * (1 + 4)
    dispatch = Tt * H * 2 + N * H * 2 + Tt * (k * 12 + R * 4) + N * (k * 12 + 4)
    combine = N * H * 2 + Tt * H * 2 + Tt * R * 4 + (Tt * k * 12 if weighted else 0)
    return {"layout": layout, "dispatch": dispatch, "combine": combine}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = {
    "dispatch_tma_kernel": ("dispatch.cu", "rowops.cuh", "ep_internal.cuh"),
    "dispatch_kernel<quant>": ("dispatch.cu", "rowops.cuh", "ep_internal.cuh"),
    "combine_kernel": ("combine.cu", "rowops.cuh", "ep_internal.cuh"),
    "ll_send_kernel": ("ll.cu", "rowops.cuh", "ep_internal.cuh"),
    "ll_combine_kernel": ("ll.cu", "rowops.cuh", "ep_internal.cuh"),
    "dispatch_em_tma_kernel": ("expert_major.cu", "rowops.cuh", "ep_internal.cuh"),
    "combine_em_kernel": ("expert_major.cu", "rowops.cuh", "ep_internal.cuh"),
}


def strip_comments(text: str) -> str:
    """C/C++ source without its comments (string and character literals kept), so that
    edits to comments do not read as a changed kernel."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "".join(out)


def source_digest(files):
    """sha256 over the named kernel source files, comments removed."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "combine_layout_02_gb300", "csrc")
    for name in sorted(files):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + strip_comments(f.read()).encode())
    return h.hexdigest()


def traffic_from_profiles(kernel: str, workload: str = "dsv3"):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu counters,
    if they were taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path) or kernel not in KERNEL_SOURCES:
        return None
    with open(path) as f:
        entries = json.load(f).get("entries", [])
    digest = source_digest(KERNEL_SOURCES[kernel])
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload and e.get("source_sha256") == digest:
            return e.get("dram_bytes_per_launch")
    return None


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            return
        self.first = threading.Event()
        self.active = False
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        self.first.wait(timeout=10)

    def _read(self):
        for line in self.proc.stdout:
            self.first.set()
            if self.active:
                self.lines.append(line.strip())

    def start(self):
        self.active = True

    def stop(self) -> dict:
        self.active = False
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- our path

def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(v: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_e2e(world, dev, plan, ep, err, total_bytes, e2e_steps, copy_streams=1):
    """The dsv3 step through the same C-ABI calls with host buffers: every step copies its
    inputs (x, topk_idx, topk_weights) from pinned host memory to the device and its result
    (the combined output) back to pinned host memory.

    Measured two ways: serial (copy in, compute, copy out on one stream) and pipelined as a
    user would run consecutive steps -- input copies, kernels and output copies on three
    streams with double-buffered device inputs and outputs, so step i+1's input copy and
    step i-1's output copy overlap step i's kernels (the two copy directions are
    independent). `value` is the pipelined figure: the median of three timed regions of
    `e2e_steps` steps each."""
    import torch
    w = plan["w"]
    R, T, H, E, k, C = w.R, w.T, w.H, w.E, w.k, w.C
    sh = ep.make_shape(R, T, H, E, k, C)
    lb, rb = plan["keep"][0], plan["keep"][1]
    from combine_layout_02_gb300.buffers import worst_case_row_offsets
    off = worst_case_row_offsets(R, T)
    x0, topk0, wts0, out0 = plan["x"], plan["topk"], plan["wts"], plan["out"]
    x_h = torch.empty(x0.shape, dtype=x0.dtype, pin_memory=True)
    x_h.copy_(x0)
    topk_h = torch.empty(topk0.shape, dtype=topk0.dtype, pin_memory=True)
    topk_h.copy_(topk0)
    wts_h = torch.empty(wts0.shape, dtype=wts0.dtype, pin_memory=True)
    wts_h.copy_(wts0)
    out_h = [torch.empty(out0.shape, dtype=out0.dtype, pin_memory=True) for _ in range(2)]
    x_d = [x0, torch.empty_like(x0)]
    topk_d = [topk0, torch.empty_like(topk0)]
    wts_d = [wts0, torch.empty_like(wts0)]
    out_d = [out0, torch.empty_like(out0)]
    layout_s, handle = lb.layout(), lb.handle(rb.recv_src_idx)

    def kernels(b, stream):
        launch = ep.make_launch(stream, error_flags=err)
        ep.ep_get_layout(sh, topk_d[b], layout_s, handle, lb.workspace, launch)
        ep.ep_dispatch(sh, x_d[b], ep.EP_BF16, None, ep.EP_BF16, topk_d[b], wts_d[b], handle,
                       rb.recv_x, None, rb.recv_topk_idx, rb.recv_topk_weights, rb.recv_src_idx,
                       off, launch)
        ep.ep_combine(sh, rb.recv_x, off, handle, ep.EP_COMBINE_WEIGHTED, topk_d[b], wts_d[b],
                      None, out_d[b], None, launch)

    # serial: one stream, copy in -> kernels -> copy out
    cur = torch.cuda.current_stream()

    def serial_step():
        x_d[0].copy_(x_h, non_blocking=True)
        topk_d[0].copy_(topk_h, non_blocking=True)
        wts_d[0].copy_(wts_h, non_blocking=True)
        kernels(0, cur)
        out_h[0].copy_(out_d[0], non_blocking=True)

    serial_step()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(e2e_steps):
        serial_step()
    e1.record(cur)
    torch.cuda.synchronize()
    serial_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, world, dev)

    # pipelined: input copies, kernels and output copies on their own streams,
    # double-buffered device inputs / outputs
    nc = max(1, copy_streams)
    s_in = [torch.cuda.Stream() for _ in range(nc)]
    s_out = [torch.cuda.Stream() for _ in range(nc)]
    s_comp = torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in range(nc)] for _ in range(2)]
    ev_comp = [torch.cuda.Event(), torch.cuda.Event()]
    ev_out = [[torch.cuda.Event() for _ in range(nc)] for _ in range(2)]
    xh_parts = list(torch.chunk(x_h.view(-1, H), nc))
    oh_parts = [list(torch.chunk(o.view(-1, H), nc)) for o in out_h]
    xd_parts = [list(torch.chunk(xd.view(-1, H), nc)) for xd in x_d]
    od_parts = [list(torch.chunk(od.view(-1, H), nc)) for od in out_d]

    def issue(i):
        b = i & 1
        for c in range(nc):
            with torch.cuda.stream(s_in[c]):
                if i >= 2:
                    s_in[c].wait_event(ev_comp[b])   # step i-2 has finished reading inputs b
                xd_parts[b][c].copy_(xh_parts[c], non_blocking=True)
                if c == 0:
                    topk_d[b].copy_(topk_h, non_blocking=True)
                    wts_d[b].copy_(wts_h, non_blocking=True)
                ev_in[b][c].record(s_in[c])
            s_comp.wait_event(ev_in[b][c])
            if i >= 2:
                s_comp.wait_event(ev_out[b][c])      # step i-2's output b has left the device
        kernels(b, s_comp)
        ev_comp[b].record(s_comp)
        for c in range(nc):
            with torch.cuda.stream(s_out[c]):
                s_out[c].wait_event(ev_comp[b])
                oh_parts[b][c].copy_(od_parts[b][c], non_blocking=True)
                ev_out[b][c].record(s_out[c])

    for i in range(4):
        issue(i)
    torch.cuda.synchronize()

    def pipelined_region():
        barrier(world)
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record(s_in[0])
        for i in range(e2e_steps):
            issue(i)
        for bb in range(2):
            for c in range(nc):
                s_in[0].wait_event(ev_out[bb][c])
        p1.record(s_in[0])
        torch.cuda.synchronize()
        return reduce_max(p0.elapsed_time(p1) / e2e_steps, world, dev)

    # The host link is shared with the machine's other work, and the overlap of the two
    # copy directions varies between runs: three regions, the median is reported.
    pipe_runs = [pipelined_region() for _ in range(3)]
    pipe_ms = statistics.median(pipe_runs)

    h2d = x_h.numel() * x_h.element_size() + topk_h.numel() * 8 + wts_h.numel() * 4
    d2h = out_h[0].numel() * out_h[0].element_size()

    # raw pinned-copy bandwidth of the link, each direction alone (context for the above)
    def copy_gbs(dst, src, nbytes):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dst.copy_(src, non_blocking=True)
        a.record(cur)
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        b.record(cur)
        torch.cuda.synchronize()
        return round(3 * nbytes / (a.elapsed_time(b) * 1e6), 1)

    link = {"h2d_gbs": copy_gbs(x_d[0], x_h, x_h.numel() * 2),
            "d2h_gbs": copy_gbs(out_h[0], out_d[0], d2h)}
    return {"value": round(world * total_bytes / (pipe_ms * 1e6), 1), "unit": "GB/s",
            "ms_per_step": round(pipe_ms, 4), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "mode": f"pipelined: input copies and output copies ({nc} streams each) and "
                    "kernels on their own streams, double-buffered device inputs/outputs",
            "pipelined_ms_per_step_runs": [round(v, 4) for v in pipe_runs],
            "serial_ms_per_step": round(serial_ms, 4),
            "serial_value": round(world * total_bytes / (serial_ms * 1e6), 1),
            "link": link}


PHASE_KERNEL = {"dispatch": "dispatch_tma_kernel", "dispatch_fp8": "dispatch_kernel<quant>",
                "combine_backward": "dispatch_tma_kernel", "dispatch_backward": "combine_kernel",
                "dispatch_em": "dispatch_em_tma_kernel", "combine_em": "combine_em_kernel",
                "combine": "combine_kernel", "layout": "layout_count+layout_prefix",
                "ll_send": "ll_send_kernel", "ll_recv": "ll_recv_kernel",
                "ll_combine": "ll_combine_kernel"}

WORKLOAD_TEXT = {
    "dsv3": "R=8 virtual ranks x {T} tokens, hidden 7168 bf16, 256 experts (32/rank), top-8 "
            "distinct uniform, fp32 softmax weights, 12 channels; layout + bf16 dispatch + "
            "weighted bf16 combine (identity experts), worst-case receive capacity",
    "group_limited": "dsv3 shape, 4-of-8 expert groups then top-8 inside them; layout + fused "
                     "e4m3 dispatch (per-128-channel fp32 scales) + weighted bf16 combine",
    "ll_decode": "R=8 x {T} tokens, hidden 7168, 256 experts, top-8 with 5% masked; low-latency "
                 "e4m3 dispatch send phase, receive phase, weighted bf16 combine; Nmax={nmax}",
    "zipf_reuse": "R=16 x {T} tokens, hidden 4096, 128 experts, top-6 Zipf(1.2); layout once, "
                  "then dispatch(handle) of fresh x + weighted combine(handle)",
    "dsv3_expert_major": "dsv3 shape; layout with the expert-major placement + expert-major bf16 "
                         "dispatch (one row per token-expert entry, grouped per local expert) + "
                         "weighted combine; worst-case regions R*T*min(k, E_loc) rows per rank",
    "ll_decode_packed": "ll_decode with the packed receive layout (no gaps between the sources' "
                        "rows of an expert; send phase = per-source rank kernel + send kernel)",
    "dsv3_backward": "dsv3 shape; layout and forward dispatch once, then per step the backward "
                     "pair with the cached handle: combine_backward = dispatch of a fresh output "
                     "gradient, dispatch_backward = sum combine of the received gradient rows "
                     "with the received weights' gradient reduced per token",
}
BASE_WORKLOAD = {"dsv3_expert_major": "dsv3", "ll_decode_packed": "ll_decode", "dsv3_backward": "dsv3"}
FP8_SCALE = {"fp32": 0, "pow2": 1, "ue8m0": 2, "tensor": 3}
DSV3_L2 = "inputs larger than L2; no flush"


def workload_config(name: str):
    """The synthetic workload behind a bench workload name (the expert-major and packed
    low-latency measurements run on the dsv3 / ll_decode workloads)."""
    return workloads.CONFIGS[BASE_WORKLOAD.get(name, name)]


def make_plan(args, ep, dev, stream, launch):
    """Device buffers and the step of one workload: a list of (phase, call) pairs, plus a
    function giving each phase's algorithmic bytes once the layout is known."""
    import dataclasses
    import torch
    from combine_layout_02_gb300.buffers import (LayoutBuffers, LLBuffers, RecvBuffers,
                                                 worst_case_row_offsets)
    w = workload_config(args.workload)
    if args.tokens:
        w = dataclasses.replace(w, T=args.tokens)
    if args.nmax:
        w = dataclasses.replace(w, nmax=args.nmax)
    R, T, H, E, k, C = w.R, w.T, w.H, w.E, w.k, w.C
    inp = workloads.make_workload(w)
    x = torch.from_numpy(inp["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    topk = torch.from_numpy(inp["topk_idx"]).to(dev)
    wts = torch.from_numpy(inp["topk_weights"]).to(dev)
    Tt = R * T
    plan = {"w": w, "inp": inp, "x": x, "topk": topk, "wts": wts, "flush": False}
    fmt = FP8_SCALE[args.fp8_scale]
    if fmt != FP8_SCALE["fp32"] and args.workload not in ("group_limited", "ll_decode", "ll_decode_packed"):
        raise SystemExit(f"--fp8-scale applies to the e4m3 workloads, not {args.workload}")
    tscale = 0.0
    if fmt == FP8_SCALE["tensor"]:
        # Per-tensor scale: one value for the whole input (its amax over the e4m3 maximum).
        xf = (inp["x"].view(np.uint16).astype(np.uint32) << 16).view(np.float32)
        tscale = float(np.abs(xf).max()) / 448.0
    sbytes = 1 if fmt == FP8_SCALE["ue8m0"] else 4

    if args.workload in ("dsv3", "group_limited", "zipf_reuse"):
        sh = ep.make_shape(R, T, H, E, k, C)
        off = worst_case_row_offsets(R, T)
        lb = LayoutBuffers(sh, dev)
        fp8 = args.workload == "group_limited"
        reuse = args.workload == "zipf_reuse"
        rb = RecvBuffers(off[-1], H, k, recv_dtype=ep.EP_FP8_E4M3 if fp8 else ep.EP_BF16,
                         with_topk=not reuse, device=dev, fp8_scale=fmt)
        out = torch.empty((R, T, H), dtype=torch.bfloat16, device=dev)
        layout_s, handle = lb.layout(), lb.handle(rb.recv_src_idx)

        def layout():
            ep.ep_get_layout(sh, topk, layout_s, handle, lb.workspace, launch)

        if fp8:
            # bf16 expert outputs for the combine: the bf16 rows of the same routing
            y = RecvBuffers(off[-1], H, k, with_topk=False, device=dev).recv_x
            layout()
            ep.ep_dispatch(sh, x, ep.EP_BF16, None, ep.EP_BF16, None, None, handle, y, None,
                           None, None, None, off, launch)
        else:
            y = rb.recv_x
        xs = [x]
        if reuse:
            layout()      # once, outside the timed steps
            rng = np.random.default_rng(w.seed + 77)
            xs.append(torch.from_numpy(workloads.make_hidden(rng, R, T, H).view(np.int16))
                      .to(dev).view(torch.bfloat16))
        it = [0]

        def dispatch():
            xi = xs[it[0] % len(xs)]
            it[0] += 1
            if reuse:
                ep.ep_dispatch(sh, xi, ep.EP_BF16, None, ep.EP_BF16, None, None, handle, rb.recv_x,
                               None, None, None, rb.recv_src_idx, off, launch)
            else:
                ep.ep_dispatch(sh, xi, ep.EP_BF16, None, ep.EP_FP8_E4M3 if fp8 else ep.EP_BF16,
                               topk, wts, handle, rb.recv_x, rb.recv_x_scales, rb.recv_topk_idx,
                               rb.recv_topk_weights, rb.recv_src_idx, off, launch,
                               fp8_scale=fmt, tensor_scale=tscale)

        def combine():
            ep.ep_combine(sh, y, off, handle, ep.EP_COMBINE_WEIGHTED, topk, wts, None, out, None,
                          launch)

        def layout_dispatch_synced():
            # The pages' exact-size path: layout, the CPU waits for the received counts,
            # then the dispatch writes into regions of exactly those sizes.
            layout()
            counts = ep.ep_read_recv_counts_sync(sh, handle, stream)
            exact = [0]
            for n in counts:
                exact.append(exact[-1] + int(n))
            ep.ep_dispatch(sh, x, ep.EP_BF16, None, ep.EP_FP8_E4M3 if fp8 else ep.EP_BF16, topk, wts,
                           handle, rb.recv_x, rb.recv_x_scales, rb.recv_topk_idx,
                           rb.recv_topk_weights, rb.recv_src_idx, exact, launch,
                           fp8_scale=fmt, tensor_scale=tscale)

        if not reuse:
            plan["layout_dispatch_synced"] = layout_dispatch_synced
            plan["layout_kernels"] = "layout_count+layout_prefix"
        dname = "dispatch_fp8" if fp8 else "dispatch"
        # The plan owns every buffer whose raw pointers the calls use.
        plan["keep"] = (lb, rb, y, out, xs)
        plan["phases"] = ([] if reuse else [("layout", layout)]) + [(dname, dispatch), ("combine", combine)]
        plan["out"] = out

        def nbytes():
            N = int(lb.rank_prefix_matrix[-1].sum().item())
            lay = Tt * k * 8 + Tt * R * (1 + 4)
            meta_in = Tt * R * 4 + (0 if reuse else Tt * k * 12)
            meta_out = N * 4 + (0 if reuse else N * k * 12)
            payload = N * H * (1 if fp8 else 2) + (N * (H // 128) * sbytes if fp8 else 0)
            b = {dname: Tt * H * 2 + payload + meta_in + meta_out,
                 "combine": N * H * 2 + Tt * H * 2 + Tt * R * 4 + Tt * k * 12}
            if not reuse:
                b["layout"] = lay
            return b, N
        plan["nbytes"] = nbytes
        plan["l2"] = "inputs larger than L2; no flush"
    elif args.workload == "dsv3_backward":
        # [README] normal-kernel example: the backward of combine is a dispatch with the
        # handle, the backward of dispatch a combine that also reduces the received weights'
        # gradient. Layout and one forward dispatch (for recv_topk_weights, the stand-in for
        # their gradient) run once, outside the timed steps.
        sh = ep.make_shape(R, T, H, E, k, C)
        off = worst_case_row_offsets(R, T)
        lb = LayoutBuffers(sh, dev)
        rb = RecvBuffers(off[-1], H, k, device=dev)
        layout_s, handle = lb.layout(), lb.handle(rb.recv_src_idx)
        ep.ep_get_layout(sh, topk, layout_s, handle, lb.workspace, launch)
        ep.ep_dispatch(sh, x, ep.EP_BF16, None, ep.EP_BF16, topk, wts, handle, rb.recv_x, None,
                       rb.recv_topk_idx, rb.recv_topk_weights, rb.recv_src_idx, off, launch)
        rng = np.random.default_rng(w.seed + 78)
        grad_out = (torch.from_numpy(workloads.make_hidden(rng, R, T, H).view(np.int16))
                    .to(dev).view(torch.bfloat16))
        grad_recv = torch.empty((off[-1], H), dtype=torch.bfloat16, device=dev)
        grad_x = torch.empty((R, T, H), dtype=torch.bfloat16, device=dev)
        grad_w = torch.empty((R, T, k), dtype=torch.float32, device=dev)
        plan["keep"] = (lb, rb, grad_out, grad_recv, grad_x, grad_w)
        plan["out"] = grad_x
        plan["phases"] = [
            ("combine_backward", lambda: ep.ep_dispatch(sh, grad_out, ep.EP_BF16, None, ep.EP_BF16, None,
                                                        None, handle, grad_recv, None, None, None,
                                                        rb.recv_src_idx, off, launch)),
            ("dispatch_backward", lambda: ep.ep_combine(sh, grad_recv, off, handle, ep.EP_COMBINE_SUM,
                                                        None, None, rb.recv_topk_weights, grad_x, grad_w,
                                                        launch)),
        ]
        plan["l2"] = "inputs larger than L2; no flush"

        def nbytes():
            N = int(lb.rank_prefix_matrix[-1].sum().item())
            return {"combine_backward": Tt * H * 2 + N * H * 2 + Tt * R * 4 + N * 4,
                    "dispatch_backward": N * H * 2 + Tt * H * 2 + Tt * R * 4 + N * k * 4 + Tt * k * 4}, N
        plan["nbytes"] = nbytes
    elif args.workload == "dsv3_expert_major":
        sh = ep.make_shape(R, T, H, E, k, C)
        lb = LayoutBuffers(sh, dev, expert_major=True)
        cap = R * T * min(k, E // R)
        off = [d * cap for d in range(R + 1)]
        recv_x = torch.empty((off[-1], H), dtype=torch.bfloat16, device=dev)
        recv_w = torch.empty((off[-1],), dtype=torch.float32, device=dev)
        recv_src = torch.empty((off[-1],), dtype=torch.int32, device=dev)
        out = torch.empty((R, T, H), dtype=torch.bfloat16, device=dev)
        layout_s, handle = lb.layout(), lb.handle()
        plan["keep"] = (lb, recv_x, recv_w, recv_src, out)
        plan["out"] = out
        plan["layout_kernels"] = "layout_count+layout_prefix+layout_expert_rows"
        plan["phases"] = [
            ("layout", lambda: ep.ep_get_layout(sh, topk, layout_s, handle, lb.workspace, launch)),
            ("dispatch_em", lambda: ep.ep_dispatch_expert_major(sh, x, ep.EP_BF16, topk, wts, handle,
                                                                recv_x, None, recv_w, recv_src, off,
                                                                launch)),
            ("combine_em", lambda: ep.ep_combine_expert_major(sh, recv_x, off, handle,
                                                              ep.EP_COMBINE_WEIGHTED, topk, wts, out,
                                                              launch)),
        ]
        plan["l2"] = "inputs larger than L2; no flush"

        def nbytes():
            M = int(lb.expert_prefix[:, -1].sum().item())
            lay = Tt * k * 8 + Tt * R * (1 + 4) + Tt * k * (8 + 4)
            return {"layout": lay,
                    "dispatch_em": Tt * H * 2 + M * H * 2 + Tt * k * (8 + 4 + 4) + M * (4 + 4),
                    "combine_em": M * H * 2 + Tt * H * 2 + Tt * k * (8 + 4 + 4)}, M
        plan["nbytes"] = nbytes
    elif args.workload in ("ll_decode", "ll_decode_packed"):
        sh = ep.make_shape(R, T, H, E, k, C, nmax=w.nmax)
        packed = args.workload == "ll_decode_packed"
        buf = LLBuffers(sh, True, device=dev, packed=packed, fp8_scale=fmt, tensor_scale=tscale)
        ybuf = LLBuffers(sh, False, device=dev, packed=packed)
        ep.ep_ll_dispatch(sh, x, topk, False, ep.EP_PHASE_BOTH, ybuf.struct(), launch)
        out = torch.empty((R, T, H), dtype=torch.bfloat16, device=dev)
        s_buf, s_y = buf.struct(), ybuf.struct()
        # The plan owns every buffer whose raw pointers the calls use (s_buf / s_y hold
        # only addresses; without this, buf's memory would be freed after this function).
        plan["keep"] = (buf, ybuf, out)
        plan["phases"] = [
            ("ll_send", lambda: ep.ep_ll_dispatch(sh, x, topk, True, ep.EP_PHASE_SEND, s_buf, launch)),
            ("ll_recv", lambda: ep.ep_ll_dispatch(sh, x, topk, True, ep.EP_PHASE_RECV, s_buf, launch)),
            ("ll_combine", lambda: ep.ep_ll_combine(sh, ybuf.recv_x, topk, wts, s_y,
                                                    ep.EP_PHASE_RECV, out, launch)),
        ]
        plan["flush"] = True
        plan["l2"] = "L2 flushed before every step (a 512 MB buffer is zeroed outside the timed kernels)"

        def nbytes():
            M = int((inp["topk_idx"] >= 0).sum())
            G = H // 128
            return {"ll_send": Tt * H * 2 + M * (H + G * sbytes) + Tt * k * (8 + 4) + M * 4 + E * R * 4,
                    "ll_recv": E * R * 4 + E * R * 8 + E * 4,
                    "ll_combine": M * H * 2 + Tt * H * 2 + Tt * k * (8 + 4 + 4)}, M
        plan["nbytes"] = nbytes
    else:
        raise ValueError(args.workload)
    return plan


def run_synced(args, world, dev, stream, call, reps=50):
    """µs per layout + host wait for the received counts + dispatch into exact regions,
    between CUDA events on the launching stream (the GPU idles while the host reads the
    counts; that gap is part of the figure)."""
    import torch
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    barrier(world)
    times = []
    for _ in range(min(reps, max(args.steps, 3))):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    return round(reduce_max(statistics.mean(times), world, dev) * 1e3, 2)


def run_graph(args, world, dev, launch, step, flush_buf, total_bytes):
    """The same step captured once as a CUDA graph and replayed K times (whole-step time;
    with a flush, each replay is timed alone after the flush)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    saved = launch.stream
    try:
        with torch.cuda.graph(g, stream=s):
            launch.stream = torch.cuda.current_stream().cuda_stream
            step()
    finally:
        launch.stream = saved
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    n = args.steps
    if flush_buf is None:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            flush_buf.zero_()
            a.record()
            g.replay()
            b.record()
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in evs) / n
    ms = reduce_max(ms, world, dev)
    return {"ms_per_step": round(ms, 4), "value": round(world * total_bytes / (ms * 1e6), 1),
            "unit": "GB/s"}


MIN_WINDOW_S = 0.5       # each timed pass repeats its K steps until this much wall time passed
MAX_REPEATS = 2000


def config_dict(name, w, units, world, l2):
    """The `config` object of a bench line (shared by the GPU and the reference arm)."""
    key = "valid_entries" if name in ("ll_decode", "ll_decode_packed", "dsv3_expert_major") else "recv_rows"
    return {"workload": f"{name}: " + WORKLOAD_TEXT[name].format(T=w.T, nmax=w.nmax),
            "R": w.R, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "C": w.C, key: units,
            "parallelism": f"replicas x{world} (virtual EP{w.R} inside each GPU)", "l2": l2}


def measure_workload(args, world, dev, ep, err, stream, launch, gpu_id):
    """Times one workload's step (args.workload) and returns (result dict, inputs, plan
    extras). Every timed pass repeats its K steps until MIN_WINDOW_S of wall time have
    passed, so the clock sampler sees the GPU under load for the whole window; the
    figures are means over all repeats."""
    import torch
    plan = make_plan(args, ep, dev, stream, launch)
    phases = plan["phases"]
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if plan["flush"] else None

    def step(ev=None, bounds=None):
        """One step; with events, ev[j] is recorded before phase bounds[j] (every phase
        when bounds is None) and the last event after the step."""
        j = 0
        for i, (_, call) in enumerate(phases):
            if ev is not None and (bounds is None or i in bounds):
                ev[j].record(stream)
                j += 1
            call()
        if ev is not None:
            ev[j].record(stream)

    for _ in range(max(args.warmup, 3)):
        if flush_buf is not None:
            flush_buf.zero_()
        step()
    torch.cuda.synchronize()
    nbytes, units = plan["nbytes"]()
    total_bytes = sum(nbytes.values())

    def timed_window(sampler, per_phase, flush=True, bounds=None):
        """Repeats of K steps between a barrier and a synchronisation on each side, until
        MIN_WINDOW_S have passed. per_phase=False (the headline pass): events only around
        each K-step region (around each step when L2 is flushed between steps, so the flush
        stays outside), so consecutive kernels overlap through programmatic dependent
        launch as they do in use. per_phase=True (the breakdown pass): an event before
        every phase (or before the phases listed in `bounds` only, timing the runs of
        phases between them as one segment) and after the step. Returns (ms per step,
        per-segment ms lists keyed by the segment's phase names joined with "+", launches,
        clocks, repeats)."""
        n = args.steps
        fbuf = flush_buf if flush else None
        cuts = list(range(len(phases))) if bounds is None else sorted(bounds)
        seg_names = segment_names(phases_names(phases), cuts)
        barrier(world)
        torch.cuda.synchronize()
        n0 = ep.ep_kernel_launch_count()
        if sampler:
            sampler.start()
        t0 = time.perf_counter()
        total_ms, reps = 0.0, 0
        per = {name: [] for name in seg_names} if per_phase else None
        while True:
            if per_phase:
                evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(cuts) + 1)] for _ in range(n)]
            elif fbuf is not None:
                evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
            else:
                evs = None
            t_start = torch.cuda.Event(enable_timing=True)
            t_end = torch.cuda.Event(enable_timing=True)
            t_start.record(stream)
            for i in range(n):
                if fbuf is not None:
                    fbuf.zero_()
                if per_phase:
                    step(evs[i], bounds)
                elif evs is not None:
                    evs[i][0].record(stream)
                    step()
                    evs[i][1].record(stream)
                else:
                    step()
            t_end.record(stream)
            torch.cuda.synchronize()
            reps += 1
            if per_phase:
                for j, name in enumerate(seg_names):
                    per[name].extend(e[j].elapsed_time(e[j + 1]) for e in evs)
            if evs is not None:
                total_ms += sum(e[0].elapsed_time(e[-1]) for e in evs)
            else:
                total_ms += t_start.elapsed_time(t_end)
            if time.perf_counter() - t0 >= args.min_window_s or reps >= MAX_REPEATS:
                break
        clocks = sampler.stop() if sampler else None
        barrier(world)
        launches = ep.ep_kernel_launch_count() - n0
        return total_ms / (n * reps), per, launches, clocks, reps

    remeasured = False
    ms_step, _, launches, clocks, reps = timed_window(ClockSampler(gpu_id), per_phase=False)
    if clocks and any(r in clocks["reasons"] for r in BAD_REASONS):
        remeasured = True
        ms_step, _, launches, clocks, reps = timed_window(ClockSampler(gpu_id), per_phase=False)
    # Per-phase breakdown (and the roofline's per-kernel durations): a second timed pass of
    # the same steps with an event around every phase.
    phase_ms, per, _, phase_clocks, phase_reps = timed_window(ClockSampler(gpu_id), per_phase=True)
    # Layout and dispatch as one region (the dispatch chained to the layout kernels by
    # programmatic dependent launch, as in use): events before the layout, before the phase
    # after the dispatch, and after the step.
    region_us = None
    names = phases_names(phases)
    if len(names) >= 2 and names[0] == "layout" and names[1].startswith("dispatch"):
        _, seg, _, _, _ = timed_window(None, per_phase=True, bounds=(0, 2) if len(names) > 2 else (0,))
        region_us = round(reduce_max(statistics.mean(seg[f"layout+{names[1]}"]), world, dev) * 1e3, 2)
    warm = None
    if flush_buf is not None:
        # Small working sets may stay in L2 between steps in use: the same steps unflushed.
        warm_ms, _, _, _, _ = timed_window(None, per_phase=False, flush=False)
        warm = {"ms_per_step": round(reduce_max(warm_ms, world, dev), 4), "note": "no L2 flush between steps"}

    ms_step = reduce_max(ms_step, world, dev)
    flags = int(err.item())
    if flags != 0:
        raise RuntimeError(f"device error flags set: {flags}")

    graph = None if args.no_graph else run_graph(args, world, dev, launch, step, flush_buf, total_bytes)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flags set: {int(err.item())}")

    synced = None
    if "layout_dispatch_synced" in plan:
        synced = run_synced(args, world, dev, stream, plan["layout_dispatch_synced"])
        if int(err.item()) != 0:
            raise RuntimeError(f"device error flags set: {int(err.item())}")

    peak, peak_kind = measured_peaks()
    w = plan["w"]
    mean_ms = {name: reduce_max(statistics.mean(v), world, dev) for name, v in per.items()}
    gbs = {name: nbytes[name] / (mean_ms[name] * 1e6) for name in mean_ms}
    dom = max(mean_ms, key=lambda n: mean_ms[n])
    kernels = dict(PHASE_KERNEL)
    if "layout" in phases_names(phases):
        kernels["layout"] = plan.get("layout_kernels", kernels["layout"])
    result = {
        "value": round(world * total_bytes / (ms_step * 1e6), 1),
        "unit": "GB/s",
        "ms_per_step": round(ms_step, 4),
        "config": config_dict(args.workload, w, units, world, plan["l2"]),
    }
    if args.workload in ("group_limited", "ll_decode", "ll_decode_packed"):
        result["config"]["fp8_scale"] = args.fp8_scale
    for name in mean_ms:
        short = name.replace("_fp8", "")
        result[f"{short}_us"] = round(mean_ms[name] * 1e3, 2)
        if name != "layout" and name != "ll_recv":
            result[f"{short}_gbs"] = round(gbs[name], 1)
            result[f"{short}_frac_of_peak"] = round(gbs[name] / peak, 4)
    if "layout" in mean_ms:
        dname = next(n for n in mean_ms if n.startswith("dispatch"))
        result["layout_dispatch_us"] = round((mean_ms["layout"] + mean_ms[dname]) * 1e3, 2)
    if region_us is not None:
        result["layout_dispatch_region_us"] = region_us
    result["bytes_per_step"] = nbytes
    result["roofline"] = {"bound": "hbm", "kernel": kernels[dom], "achieved": round(gbs[dom], 1),
                          "peak": peak, "unit": "GB/s", "frac": round(gbs[dom] / peak, 4),
                          "peak_source": f"{peak_kind} hbm_gbs (copy), of {peak_kind}",
                          "traffic": traffic_from_profiles(kernels[dom], args.workload),
                          "algorithmic_bytes_per_launch": nbytes[dom]}
    result["layout_dispatch_synced_us"] = synced
    if warm is not None:
        warm["value"] = round(world * total_bytes / (warm["ms_per_step"] * 1e6), 1)
        result["warm"] = warm
    result["graph"] = graph
    result["timing"] = (f"value / ms_per_step: {args.steps} steps with events only around the region "
                        "(around each step when L2 is flushed), repeated until "
                        f"{args.min_window_s} s of wall time had passed ({reps} repeats, "
                        f"{reps * args.steps} steps; the mean over all of them); *_us, *_gbs and "
                        "roofline: a second pass with an event around every phase "
                        f"({phase_reps} repeats; its step: {phase_ms:.4f} ms); "
                        "layout_dispatch_us: the sum of the layout and dispatch phases of that pass; "
                        "layout_dispatch_region_us: a third pass with one event before the layout "
                        "and one after the dispatch")
    result["repeats"] = reps
    result["timed_steps"] = reps * args.steps
    result["gpu_launches"] = launches
    result["gpu_launches_per_step"] = round(launches / (reps * args.steps), 3)
    result["clocks"] = clocks
    result["phase_pass_clocks"] = phase_clocks
    result["clocks_remeasured"] = remeasured
    return result, plan["inp"], {"plan": plan, "total_bytes": total_bytes}


def phases_names(phases):
    return [name for name, _ in phases]


def segment_names(names, cuts):
    """Names of the timed segments when events are recorded before the phases at the
    sorted indices `cuts` and after the last phase: each segment runs from one cut to the
    next and is named by its phases joined with "+"."""
    ends = list(cuts[1:]) + [len(names)]
    return ["+".join(names[c:e]) for c, e in zip(cuts, ends)]


# The extra workloads the default (dsv3) line also measures, each in its own object.
EXTRA_WORKLOADS = ("group_limited", "zipf_reuse", "ll_decode")
EXTRA_KEYS = ("value", "unit", "ms_per_step", "config", "layout_us", "dispatch_us", "dispatch_gbs",
              "dispatch_frac_of_peak", "combine_us", "combine_gbs", "combine_frac_of_peak",
              "layout_dispatch_us", "layout_dispatch_region_us", "ll_send_us", "ll_send_gbs", "ll_send_frac_of_peak", "ll_recv_us",
              "ll_combine_us", "ll_combine_gbs", "ll_combine_frac_of_peak", "bytes_per_step",
              "roofline", "warm", "graph", "repeats", "timed_steps", "gpu_launches", "clocks",
              "phase_pass_clocks", "clocks_remeasured", "layout_dispatch_synced_us")


def run_ours(args, rank, world):
    import copy
    import torch
    import combine_layout_02_gb300 as ep

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    ep.lib()                                              # fails loudly without libep.so
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    launch = ep.make_launch(stream, error_flags=err)
    gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
    gpu_id = gpu_uuid if gpu_uuid.startswith("GPU-") else "GPU-" + gpu_uuid

    res, inp, extra = measure_workload(args, world, dev, ep, err, stream, launch, gpu_id)
    e2e = None
    if args.workload == "dsv3" and not args.no_e2e:
        e2e = run_e2e(world, dev, extra["plan"], ep, err, extra["total_bytes"],
                      max(4, min(args.steps, 20)), args.e2e_copy_streams)
    del extra
    torch.cuda.empty_cache()
    result = {
        "metric": METRIC,
        "value": res.pop("value"),
        "unit": res.pop("unit"),
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": res.pop("ms_per_step"),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": res.pop("config"),
    }
    result.update(res)
    result["e2e"] = e2e
    if args.workload == "dsv3" and not args.no_extra:
        # The other workloads of the same benchmark, each with its own roofline and clocks.
        result["workloads"] = {}
        for name in EXTRA_WORKLOADS:
            sub_args = copy.copy(args)
            sub_args.workload, sub_args.fp8_scale, sub_args.tokens, sub_args.nmax = name, "fp32", 0, 0
            sub, _, extra = measure_workload(sub_args, world, dev, ep, err, stream, launch, gpu_id)
            del extra
            torch.cuda.empty_cache()
            result["workloads"][name] = {k: sub[k] for k in EXTRA_KEYS if k in sub}
    return result, inp


# ----------------------------------------------------------------------------- oracle

def oracle_sample(inp, steps: int, budget_s: float):
    """Times the CPU oracle (layout + dispatch + weighted combine) on the first T_s tokens
    of every source rank, T_s chosen by a short calibration so that `steps` steps take
    about budget_s seconds. Returns (GB/s, description, seconds per step)."""
    import oracle
    w = WORKLOAD

    def one(Ts):
        topk = np.ascontiguousarray(inp["topk_idx"][:, :Ts])
        wts = np.ascontiguousarray(inp["topk_weights"][:, :Ts])
        x = np.ascontiguousarray(inp["x"][:, :Ts])
        t0 = time.perf_counter()
        lay = oracle.layout(topk, w.E, w.C)
        n = lay["rank_prefix_matrix"][-1]
        off = np.concatenate([[0], np.cumsum(n)]).astype(np.int64)
        d = oracle.dispatch(x, lay["send_head"], off, w.E, topk, wts)
        oracle.combine(d["recv_x"], lay["send_head"], off, w.E, w.k, oracle.COMBINE_WEIGHTED, topk, wts)
        dt = time.perf_counter() - t0
        return dt, int(off[-1])

    cal_T = 32
    dt, _ = one(cal_T)
    per_tok = dt / cal_T
    Ts = int(max(8, min(w.T, budget_s / max(steps, 1) / per_tok)))
    times, N = [], 0
    for _ in range(max(steps, 1)):
        dt, N = one(Ts)
        times.append(dt)
    sec = statistics.mean(times)
    b = algorithmic_bytes(w.R, Ts, w.H, w.k, N)
    gbs = sum(b.values()) / (sec * 1e9)
    desc = (f"first {Ts} of {w.T} tokens of each of the {w.R} source ranks of the same seeded "
            f"workload ({N} received rows), {len(times)} step(s), single-threaded C oracle")
    return gbs, desc, sec


def run_reference(args, rank, world):
    if rank != 0:
        return None
    inp = workloads.make_workload(WORKLOAD)
    gbs, desc, sec = oracle_sample(inp, args.steps, budget_s=float(os.environ.get("EP_ORACLE_BUDGET_S", 90)))
    import oracle
    N = int(oracle.layout(inp["topk_idx"], WORKLOAD.E, WORKLOAD.C)["rank_prefix_matrix"][-1].sum())
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        # the GPU arm's config of the same workload (the timed sample is in cpu_baseline)
        "config": config_dict("dsv3", WORKLOAD, N, world, DSV3_L2),
        "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay measurement")
    ap.add_argument("--min-window-s", type=float, default=MIN_WINDOW_S,
                    help="each timed pass repeats its K steps until this much wall time has "
                         "passed (0: one pass of K steps, for profiler captures)")
    ap.add_argument("--no-extra", action="store_true",
                    help="dsv3 only: skip the group_limited / zipf_reuse / ll_decode objects")
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="streams per copy direction in the pipelined end-to-end measurement")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_TEXT), default="dsv3",
                    help="dsv3 is the benchmark line; the others are extra measurements")
    ap.add_argument("--fp8-scale", choices=sorted(FP8_SCALE), default="fp32",
                    help="scale format of the e4m3 sends (group_limited, ll_decode*)")
    ap.add_argument("--nmax", type=int, default=0,
                    help="low-latency slot capacity override (profiler captures only)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="tokens per source rank (default 4096); smaller cases are for "
                         "profiler captures, not bench lines")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        # The oracle runs on rank 0's host cores only; other ranks exit without work.
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group(backend)

    res, inp = run_ours(args, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == "dsv3":
        gbs, desc, _ = oracle_sample(inp, 2, budget_s=20.0)
        res["cpu_baseline"] = {"value": round(gbs, 3), "unit": "GB/s", "cores": 1,
                               "kind": "oracle", "sample": desc}
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
