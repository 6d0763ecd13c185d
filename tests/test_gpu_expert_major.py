"""GPU parity of the expert-major packed layout (rows of each destination grouped by
local expert, then source rank, then token) against the oracle: the handle's
expert_rows / expert_prefix bit-exact on shapes that exercise every bitmask width
(E from 4 to 4096), dispatch rows / scales / metadata bit-exact (bf16, e4m3 with every
scale format), combine within 1e-3 absolute + 1e-2 relative on every combine form (rows of
at most 256 channels, up to 1024, at most two rows per token, the rest), and the dsv3 shape
at full size with exact receive regions."""
import ctypes

import numpy as np
import pytest
import torch

import combine_layout_02_gb300 as ep
from combine_layout_02_gb300.buffers import LayoutBuffers
import oracle
import workloads
from gpu_util import assert_close_bf16, bf16_to_f64, dev_bf16, host_bits

pytestmark = pytest.mark.gpu

W = workloads.Workload
CASES = {
    "tiny": workloads.CONFIGS["tiny"],
    "ragged": W("emr", R=4, T=1000, H=384, E=32, k=5, C=7, mask_p=0.1, seed=301),
    "r3_odd": W("em3", R=3, T=257, H=128, E=9, k=3, C=12, seed=302),
    "zipf16": W("emz", R=16, T=300, H=512, E=128, k=6, C=5, routing="zipf", zipf_s=1.2, seed=303),
    "group8": W("emg", R=8, T=513, H=1024, E=256, k=8, C=12, routing="group", groups=8,
                topk_groups=4, seed=304),
    "r64": W("em64", R=64, T=40, H=128, E=64, k=4, C=2, seed=305),
    "k32": W("emk", R=8, T=64, H=128, E=64, k=32, C=3, seed=306),
    "e1024": W("em1k", R=8, T=200, H=128, E=1024, k=8, C=4, seed=307),
    "e4096": W("em4k", R=16, T=100, H=128, E=4096, k=8, C=3, seed=308),
    "top2_h2048": W("em2", R=8, T=200, H=2048, E=64, k=2, C=4, seed=309),     # <= 2 rows per token
    "h4096": W("em4", R=4, T=100, H=4096, E=16, k=4, C=3, seed=310),           # wide rows, k > 2
}


class EmRun:
    def __init__(self, w, inp):
        self.w, self.inp = w, inp
        self.sh = ep.make_shape(w.R, w.T, w.H, w.E, w.k, w.C)
        self.topk = torch.from_numpy(inp["topk_idx"]).cuda()
        self.wts = torch.from_numpy(inp["topk_weights"]).cuda()
        self.x = dev_bf16(inp["x"])
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.launch = ep.make_launch(error_flags=self.err)
        self.lb = LayoutBuffers(self.sh, expert_major=True)
        ep.ep_get_layout(self.sh, self.topk, self.lb.layout(), self.lb.handle(), self.lb.workspace,
                         self.launch)

    def flags(self):
        torch.cuda.synchronize()
        return int(self.err.item())

    def dispatch(self, off, recv_dtype=ep.EP_BF16, fp8_scale=0, tensor_scale=0.0, x=None):
        rows, H = off[-1], self.w.H
        if recv_dtype == ep.EP_BF16:
            rx = torch.full((rows, H), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
            rs = None
        else:
            rx = torch.full((rows, H), 0x5A, dtype=torch.uint8, device="cuda")
            rs = (torch.full((rows, H // 128), 0xEE, dtype=torch.uint8, device="cuda")
                  if fp8_scale == ep.EP_FP8_SCALE_UE8M0 else
                  torch.full((rows, H // 128), float("nan"), device="cuda"))
        rw = torch.full((rows,), -5.0, device="cuda")
        ri = torch.full((rows,), -3, dtype=torch.int32, device="cuda")
        ep.ep_dispatch_expert_major(self.sh, self.x if x is None else x, recv_dtype, self.topk,
                                    self.wts, self.lb.handle(), rx, rs, rw, ri, off, self.launch,
                                    fp8_scale=fp8_scale, tensor_scale=tensor_scale)
        return rx, rs, rw, ri

    def combine(self, y, off, mode):
        out = torch.empty((self.w.R, self.w.T, self.w.H), dtype=torch.bfloat16, device="cuda")
        ep.ep_combine_expert_major(self.sh, y, off, self.lb.handle(), mode, self.topk, self.wts,
                                   out, self.launch)
        return out


def _setup(name):
    w = CASES[name]
    inp = workloads.make_workload(w)
    run = EmRun(w, inp)
    ref = oracle.expert_layout(inp["topk_idx"], w.E)
    off = np.concatenate([[0], np.cumsum(ref["expert_prefix"][:, -1])]).astype(np.int64)
    return w, inp, run, ref, [int(v) for v in off]


@pytest.mark.parametrize("name", list(CASES))
def test_expert_layout_bit_exact(name):
    w, inp, run, ref, off = _setup(name)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bits(run.lb.expert_rows), ref["expert_rows"])
    np.testing.assert_array_equal(host_bits(run.lb.expert_prefix), ref["expert_prefix"])
    # the rank-major outputs of the same call are unchanged by the extra placement
    lay = oracle.layout(inp["topk_idx"], w.E, w.C)
    for key, t in run.lb.as_dict().items():
        np.testing.assert_array_equal(t.cpu().numpy(), lay[key], err_msg=key)
    assert run.flags() == 0


@pytest.mark.parametrize("name", ["tiny", "ragged", "zipf16", "group8", "k32", "e4096", "top2_h2048",
                                  "h4096"])
def test_dispatch_expert_major_bf16_bit_exact(name):
    w, inp, run, ref, off = _setup(name)
    rx, _, rw, ri = run.dispatch(off)
    exp = oracle.dispatch_expert_major(inp["x"], inp["topk_idx"], inp["topk_weights"],
                                       ref["expert_rows"], np.array(off), w.E, fill_x=0xFFFF)
    np.testing.assert_array_equal(host_bits(rx), exp["recv_x"])
    np.testing.assert_array_equal(host_bits(ri), exp["recv_src_idx"])
    np.testing.assert_array_equal(host_bits(rw).view(np.uint32), exp["recv_weights"].view(np.uint32))
    assert run.flags() == 0


@pytest.mark.parametrize("name", ["tiny", "group8", "h4096"])
@pytest.mark.parametrize("mode,ts", [(0, 0.0), (1, 0.0), (2, 0.0), (3, 0.0173)])
def test_dispatch_expert_major_fp8_bit_exact(name, mode, ts):
    w, inp, run, ref, off = _setup(name)
    rx, rs, _, _ = run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3, fp8_scale=mode, tensor_scale=ts)
    exp = oracle.dispatch_expert_major(inp["x"], inp["topk_idx"], inp["topk_weights"],
                                       ref["expert_rows"], np.array(off), w.E, quantize=True,
                                       scale_mode=mode, tensor_scale=ts, fill_x=0x5A)
    np.testing.assert_array_equal(host_bits(rx), exp["recv_x"])
    if mode == 2:
        np.testing.assert_array_equal(host_bits(rs), exp["recv_x_scales"])
    else:
        np.testing.assert_array_equal(host_bits(rs).view(np.uint32), exp["recv_x_scales"].view(np.uint32))


@pytest.mark.parametrize("name", ["tiny", "ragged", "zipf16", "group8", "k32", "top2_h2048", "h4096"])
@pytest.mark.parametrize("mode", [ep.EP_COMBINE_SUM, ep.EP_COMBINE_WEIGHTED])
def test_combine_expert_major_within_tolerance(name, mode):
    w, inp, run, ref, off = _setup(name)
    rng = np.random.default_rng(w.seed + 9)
    y32 = rng.standard_normal((max(off[-1], 1), w.H)).astype(np.float32)
    yb = torch.from_numpy(y32).to(torch.bfloat16)
    out = run.combine(yb.cuda(), off, mode)
    exp = oracle.combine_expert_major(yb.view(torch.int16).numpy().view(np.uint16)[: off[-1]],
                                      inp["topk_idx"], inp["topk_weights"], ref["expert_rows"],
                                      np.array(off), w.E, weighted=mode == ep.EP_COMBINE_WEIGHTED)
    assert_close_bf16(host_bits(out), exp)
    assert run.flags() == 0


def test_expert_major_identity_round_trip_full_size_dsv3():
    """dsv3 shape at full size with exact regions (the prefix totals): layout bit-exact,
    every row equal to its token's row, weighted combine of identity experts returns x
    within bf16 rounding."""
    w = workloads.CONFIGS["dsv3"]
    inp = workloads.make_workload(w)
    run = EmRun(w, inp)
    ref = oracle.expert_layout(inp["topk_idx"], w.E)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bits(run.lb.expert_rows), ref["expert_rows"])
    np.testing.assert_array_equal(host_bits(run.lb.expert_prefix), ref["expert_prefix"])
    off = [0]
    for n in ref["expert_prefix"][:, -1]:
        off.append(off[-1] + int(n))
    rx, _, _, _ = run.dispatch(off)
    s_i, t_i, j_i = np.nonzero(inp["topk_idx"] >= 0)
    d_i = inp["topk_idx"][s_i, t_i, j_i] // (w.E // w.R)
    rows = torch.from_numpy(np.asarray(off)[d_i] + ref["expert_rows"][s_i, t_i, j_i]).cuda()
    toks = torch.from_numpy(s_i.astype(np.int64) * w.T + t_i).cuda()
    xf = run.x.view(-1, w.H)
    for i in range(0, len(rows), 32768):
        assert torch.equal(rx[rows[i:i + 32768]].view(torch.int16), xf[toks[i:i + 32768]].view(torch.int16))
    out = run.combine(rx, off, ep.EP_COMBINE_WEIGHTED)
    xs = bf16_to_f64(inp["x"][:, :64])
    ws = inp["topk_weights"][:, :64].astype(np.float64).sum(-1)[..., None]
    got = bf16_to_f64(host_bits(out[:, :64]))
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(xs), 2.0 ** -126))) - 7)
    assert np.all(np.abs(got - xs * ws) <= 2 * ulp)
    assert run.flags() == 0


def test_expert_major_argument_checks():
    L = ep.lib()
    sh = ep.make_shape(8, 16, 128, 8192, 8)
    h = ep.ep_handle(0x1000, 0x1000, 0x1000, None, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000)
    launch = ep.make_launch()
    ws = torch.empty(ep.ep_layout_workspace_size(sh), dtype=torch.uint8, device="cuda")
    st = L.ep_get_layout(ctypes.byref(sh), ctypes.c_void_p(0x2000), None, ctypes.byref(h),
                         ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.byref(launch))
    assert st == ep.EP_ERR_UNSUPPORTED                     # E beyond the expert-major limit
    sh2 = ep.make_shape(8, 16, 128, 64, 8)
    h2 = ep.ep_handle(0x1000, 0x1000, 0x1000, None, 0x1000, 0x1000, 0x1000, 0x1000, None)
    st = L.ep_get_layout(ctypes.byref(sh2), ctypes.c_void_p(0x2000), None, ctypes.byref(h2),
                         ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.byref(launch))
    assert st == ep.EP_ERR_INVALID_ARG                     # expert_rows without expert_prefix
