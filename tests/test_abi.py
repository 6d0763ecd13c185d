"""The C-ABI library builds, loads and exports every symbol include/ep.h declares;
host-side argument validation rejects bad calls before any CUDA work (no GPU needed:
no call here reaches a kernel launch or a CUDA API)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ep():
    from combine_layout_02_gb300 import build
    build.build()
    import combine_layout_02_gb300 as ep
    ep.lib()
    return ep


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ep.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set()
    for m in re.finditer(r"^[A-Za-z_][\w \t\*]*?\b(ep_\w+)\s*\(", text, flags=re.M):
        if not m.group(0).lstrip().startswith(("typedef", "#")):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(ep):
    declared = declared_functions()
    assert declared, "no declarations parsed"
    assert declared == set(ep.EXPORTED_SYMBOLS)
    L = ctypes.CDLL(ep.library_path())
    for name in declared:
        assert hasattr(L, name), name


def test_host_only_helpers(ep):
    assert ep.ep_abi_version() == 103
    assert ep.ep_kernel_launch_count() >= 0
    assert ep.lib().ep_status_string(1).startswith(b"EP_ERR_INVALID_ARG")
    assert ep.lib().ep_last_cuda_error() == b""


def test_workspace_size_formula_and_limits(ep):
    sh = ep.make_shape(8, 4096, 7168, 256, 8, C=12)
    ws = ep.ep_layout_workspace_size(sh)
    cnt = (8 * 8 * 12 * 4 + 255) // 256 * 256
    assert ws == cnt + 8 * 12 * 256 * 4 + 256 * 4
    assert ep.ep_layout_workspace_size(ep.make_shape(65, 16, 128, 65, 1)) == 0     # R > 64
    assert ep.ep_layout_workspace_size(ep.make_shape(8, 16, 100, 64, 2)) == 0      # H % 128
    assert ep.ep_layout_workspace_size(ep.make_shape(3, 16, 128, 8, 2)) == 0       # E % R


def test_invalid_arguments_rejected_on_host(ep):
    L = ep.lib()
    sh = ep.make_shape(2, 4, 128, 4, 2, C=2)
    launch = ep.ep_launch(None, None, None, None)
    h = ep.ep_handle()
    # NULL handle fields
    st = L.ep_get_layout(ctypes.byref(sh), None, None, ctypes.byref(h), None, 0, ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG
    # dispatch with topk weights but no topk_idx (the handle-reuse assertion)
    h.send_head = 0x1000
    out = ep.ep_recv(0x2000, None, None, None, None, None)
    st = L.ep_dispatch(ctypes.byref(sh), 0x3000, ep.EP_BF16, None, ep.EP_BF16, None, 0x4000,
                       ctypes.byref(h), ctypes.byref(out), ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG
    # fp8 input cannot be dispatched as bf16
    st = L.ep_dispatch(ctypes.byref(sh), 0x3000, ep.EP_FP8_E4M3, 0x5000, ep.EP_BF16, None, None,
                       ctypes.byref(h), ctypes.byref(out), ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG
    # decreasing row offsets
    off = (ctypes.c_int64 * 3)(0, 10, 5)
    out.row_offset = ctypes.cast(off, ctypes.c_void_p)
    st = L.ep_dispatch(ctypes.byref(sh), 0x3000, ep.EP_BF16, None, ep.EP_BF16, None, None,
                       ctypes.byref(h), ctypes.byref(out), ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG
    # weighted combine without weights
    off2 = (ctypes.c_int64 * 3)(0, 8, 16)
    st = L.ep_combine(ctypes.byref(sh), 0x3000, ctypes.cast(off2, ctypes.c_void_p), ctypes.byref(h),
                      ep.EP_COMBINE_WEIGHTED, None, None, None, 0x6000, None, ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG
    # low-latency: T > Nmax
    sh_ll = ep.make_shape(2, 8, 128, 4, 2, nmax=4)
    buf = ep.ep_ll_buffer(0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000)
    st = L.ep_ll_dispatch(ctypes.byref(sh_ll), 0x7000, 0x8000, 0, ep.EP_PHASE_BOTH, ctypes.byref(buf),
                          ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG
    # bad phase value
    sh_ll2 = ep.make_shape(2, 4, 128, 4, 2, nmax=4)
    st = L.ep_ll_dispatch(ctypes.byref(sh_ll2), 0x7000, 0x8000, 0, 4, ctypes.byref(buf),
                          ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG
    # FP8 scale options: unknown format, non-positive per-tensor scale, or a scale format
    # without a fused quantisation
    off3 = (ctypes.c_int64 * 3)(0, 8, 16)
    for fmt, ts, rdt in ((7, 0.0, ep.EP_FP8_E4M3), (ep.EP_FP8_SCALE_TENSOR, 0.0, ep.EP_FP8_E4M3),
                         (ep.EP_FP8_SCALE_TENSOR, float("nan"), ep.EP_FP8_E4M3),
                         (ep.EP_FP8_SCALE_POW2, 0.0, ep.EP_BF16)):
        o = ep.ep_recv(0x2000, 0x2800, None, None, None, ctypes.cast(off3, ctypes.c_void_p),
                       ep.ep_fp8_options(fmt, ts))
        st = L.ep_dispatch(ctypes.byref(sh), 0x3000, ep.EP_BF16, None, rdt, None, None,
                           ctypes.byref(h), ctypes.byref(o), ctypes.byref(launch))
        assert st == ep.EP_ERR_INVALID_ARG, (fmt, ts, rdt)
    buf_b = ep.ep_ll_buffer(0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000,
                            ep.ep_fp8_options(ep.EP_FP8_SCALE_UE8M0, 0.0))
    st = L.ep_ll_dispatch(ctypes.byref(sh_ll2), 0x7000, 0x8000, 0, ep.EP_PHASE_SEND,
                          ctypes.byref(buf_b), ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG        # a scale format needs use_fp8
    buf_l = ep.ep_ll_buffer(0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000,
                            ep.ep_fp8_options(0, 0.0), 2)
    st = L.ep_ll_dispatch(ctypes.byref(sh_ll2), 0x7000, 0x8000, 0, ep.EP_PHASE_SEND,
                          ctypes.byref(buf_l), ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG        # unknown receive layout
    # expert-major: no expert_rows in the handle, recv_topk_idx given (one entry per row),
    # a scale format without e4m3, too many experts
    off4 = (ctypes.c_int64 * 3)(0, 8, 16)
    oe = ep.ep_recv(0x2000, None, None, None, None, ctypes.cast(off4, ctypes.c_void_p))
    st = L.ep_dispatch_expert_major(ctypes.byref(sh), 0x3000, ep.EP_BF16, 0x4000, None,
                                    ctypes.byref(ep.ep_handle()), ctypes.byref(oe), ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG
    he = ep.ep_handle()
    he.expert_rows = 0x1000
    he.expert_prefix = 0x1800
    oe_bad = ep.ep_recv(0x2000, None, 0x2400, None, None, ctypes.cast(off4, ctypes.c_void_p))
    st = L.ep_dispatch_expert_major(ctypes.byref(sh), 0x3000, ep.EP_BF16, 0x4000, None,
                                    ctypes.byref(he), ctypes.byref(oe_bad), ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG
    oe_fmt = ep.ep_recv(0x2000, None, None, None, None, ctypes.cast(off4, ctypes.c_void_p),
                        ep.ep_fp8_options(ep.EP_FP8_SCALE_UE8M0, 0.0))
    st = L.ep_dispatch_expert_major(ctypes.byref(sh), 0x3000, ep.EP_BF16, 0x4000, None,
                                    ctypes.byref(he), ctypes.byref(oe_fmt), ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG
    many = ep.make_shape(2, 4, 128, ep.EP_EXPERT_MAJOR_MAX_EXPERTS * 2, 2)
    st = L.ep_dispatch_expert_major(ctypes.byref(many), 0x3000, ep.EP_BF16, 0x4000, None,
                                    ctypes.byref(he), ctypes.byref(oe), ctypes.byref(launch))
    assert st == ep.EP_ERR_UNSUPPORTED
    # expert-major combine: weighted without weights, unknown mode
    for mode, w in ((ep.EP_COMBINE_WEIGHTED, None), (5, 0x5000)):
        st = L.ep_combine_expert_major(ctypes.byref(sh), 0x3000, ctypes.cast(off4, ctypes.c_void_p),
                                       ctypes.byref(he), mode, 0x4000, w, 0x6000, ctypes.byref(launch))
        assert st == ep.EP_ERR_INVALID_ARG, mode
    # low-latency combine: misaligned output, bad phase
    st = L.ep_ll_combine(ctypes.byref(sh_ll2), 0x3000, 0x4000, 0x5000, ctypes.byref(buf),
                         ep.EP_PHASE_BOTH, 0x6008, ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG
    st = L.ep_ll_combine(ctypes.byref(sh_ll2), 0x3000, 0x4000, 0x5000, ctypes.byref(buf),
                         8, 0x6000, ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG
    # low-latency: a source's entry count T*k beyond int32 (R*T and R*Nmax within limits)
    huge = ep.make_shape(1, 1 << 28, 128, 8, 8, nmax=1 << 28)
    for phase in (ep.EP_PHASE_SEND, ep.EP_PHASE_RECV, ep.EP_PHASE_BOTH):
        st = L.ep_ll_dispatch(ctypes.byref(huge), 0x7000, 0x8000, 0, phase, ctypes.byref(buf),
                              ctypes.byref(launch))
        assert st == ep.EP_ERR_UNSUPPORTED, phase
    st = L.ep_ll_combine(ctypes.byref(huge), 0x3000, 0x4000, 0x5000, ctypes.byref(buf),
                         ep.EP_PHASE_RECV, 0x6000, ctypes.byref(launch))
    assert st == ep.EP_ERR_UNSUPPORTED
    # unsupported shape
    big = ep.make_shape(65, 4, 128, 65, 1)
    st = L.ep_dispatch(ctypes.byref(big), 0x3000, ep.EP_BF16, None, ep.EP_BF16, None, None,
                       ctypes.byref(h), ctypes.byref(out), ctypes.byref(launch))
    assert st == ep.EP_ERR_UNSUPPORTED


@pytest.mark.parametrize("recv_dtype,fmt", [(0, 0), (1, 0), (1, 2)])
def test_buffer_size_hint_matches_the_python_buffers(ep, recv_dtype, fmt):
    """ep_buffer_size_hint (host only) against the sizes the binding's buffer classes
    allocate for the same shape (CPU tensors; nothing runs on a GPU)."""
    import torch
    from combine_layout_02_gb300.buffers import LLBuffers, RecvBuffers, worst_case_row_offsets
    sh = ep.make_shape(4, 37, 256, 16, 6, 5, nmax=40)
    h = ep.ep_buffer_size_hint(sh, recv_dtype, fmt)
    rows = worst_case_row_offsets(4, 37)[-1]
    assert h["recv_rows"] == rows == 4 * 4 * 37
    rb = RecvBuffers(rows, 256, 6, recv_dtype=recv_dtype, device="cpu", fp8_scale=fmt)
    nbytes = lambda t: 0 if t is None else t.numel() * t.element_size()   # noqa: E731
    assert h["recv_x_bytes"] == nbytes(rb.recv_x)
    assert h["recv_x_scales_bytes"] == nbytes(rb.recv_x_scales)
    assert h["recv_topk_idx_bytes"] == nbytes(rb.recv_topk_idx)
    assert h["recv_topk_weights_bytes"] == nbytes(rb.recv_topk_weights)
    assert h["recv_src_idx_bytes"] == nbytes(rb.recv_src_idx)
    assert h["expert_major_rows"] == rows * min(6, 16 // 4)
    ll = LLBuffers(sh, bool(recv_dtype), device="cpu", fp8_scale=fmt)
    assert h["ll_slots"] == ll.src_info.numel()
    for key in ("recv_x", "recv_x_scales", "src_info", "slot", "send_count", "recv_expert_count",
                "layout_range"):
        assert h[f"ll_{key}_bytes"] == nbytes(getattr(ll, key)), key
    assert h["layout_workspace_bytes"] == ep.ep_layout_workspace_size(sh)
    del torch


def test_buffer_size_hint_rejects_bad_arguments_and_overflow(ep):
    L = ep.lib()
    h = ep.ep_size_hint()
    sh = ep.make_shape(4, 37, 256, 16, 6, 5, nmax=40)
    assert L.ep_buffer_size_hint(ctypes.byref(sh), 7, 0, ctypes.byref(h)) == ep.EP_ERR_INVALID_ARG
    assert L.ep_buffer_size_hint(ctypes.byref(sh), 1, 9, ctypes.byref(h)) == ep.EP_ERR_INVALID_ARG
    assert L.ep_buffer_size_hint(ctypes.byref(sh), 0, 0, None) == ep.EP_ERR_INVALID_ARG
    huge = ep.make_shape(64, 1 << 24, 1 << 30, 64, 8, 1, nmax=1 << 24)
    assert L.ep_buffer_size_hint(ctypes.byref(huge), 0, 0, ctypes.byref(h)) == ep.EP_ERR_UNSUPPORTED
