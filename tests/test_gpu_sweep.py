"""Seeded sweep of random small shapes through every entry point, against the oracle
(three sets: small shapes, wide rows with capped grids, many experts per rank).

Each case draws R (1 to 64, including primes), experts per rank, k (1 to 32), T
(including 0, 1 and non-multiples of the channel and tile sizes), H, C, masking and
routing, then checks in one pass: layout and handle (with the expert-major placement)
bit-exact; bf16 dispatch rows and metadata bit-exact into exact regions; fused e4m3
dispatch with a scale format chosen per case bit-exact; combine (sum and weighted, with
the weight reduction) within 1e-3 absolute + 1e-2 relative; expert-major dispatch
bit-exact and its combine within tolerance; low-latency dispatch in both receive layouts
bit-exact and its combine within tolerance (where the slot buffers stay small).
"""
import numpy as np
import pytest
import torch

import combine_layout_02_gb300 as ep
from combine_layout_02_gb300.buffers import LayoutBuffers
import oracle
import workloads
from gpu_util import GpuRun, assert_close_bf16, compact_offsets, host_bits, assert_weight_sums_close

pytestmark = pytest.mark.gpu

LL_MAX_ELEMS = 1 << 25          # slot-buffer elements (R * E * Nmax * H) the sweep allows


def _draw_cases(n=24, seed=2024, name="sweep", wide=False):
    """wide=True also draws rows too wide for the bulk-copy buffers (H = 26624, on small
    R*T) and a capped grid (num_sms), so warps walk many tokens."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        R = int(rng.choice([1, 2, 3, 4, 5, 8, 13, 16, 32, 64]))
        E_loc = int(rng.choice([1, 2, 3, 4, 8]))
        E = R * E_loc
        k = int(rng.integers(1, min(E, 32) + 1))
        T = int(rng.choice([0, 1, 2, 17, 64, 129, 300]))
        H = int(rng.choice([128, 256, 384, 1024] + ([2048, 26624] if wide else [])))
        if H > 2048 and R * T > 512:
            H = 2048
        C = int(rng.integers(1, 13))
        mask_p = float(rng.choice([0.0, 0.15]))
        routing = "zipf" if rng.random() < 0.3 else "uniform"
        sms = int(rng.choice([0, 1, 5])) if wide else 0
        cases.append((workloads.Workload(f"{name}{i}", R=R, T=T, H=H, E=E, k=k, C=C, mask_p=mask_p,
                                         routing=routing, zipf_s=1.1 if routing == "zipf" else 0.0,
                                         nmax=max(T, 1) + int(rng.integers(0, 5)), seed=5000 + i
                                         + (1000 if wide else 0)), sms))
    return cases


def _draw_cases_many_experts(n=12, seed=2026, name="manyexp"):
    """Many experts per rank (16 to 256, E up to 8192), rows up to 7168 wide, 1 to 24
    channels, masking up to one entry in two, and uniform, Zipf or group-limited routing."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        R = int(rng.choice([2, 3, 4, 6, 8, 12, 16]))
        E_loc = min(int(rng.choice([16, 32, 64, 128, 256])), 8192 // R)
        E = R * E_loc
        k = int(rng.integers(1, min(E, 32) + 1))
        T = int(rng.choice([1, 3, 31, 64, 200, 513]))
        H = int(rng.choice([128, 512, 1536, 4096, 7168]))
        if R * T * H > (1 << 24):
            H = 512
        C = int(rng.integers(1, 25))
        mask_p = float(rng.choice([0.0, 0.05, 0.5]))
        routing = str(rng.choice(["uniform", "zipf", "group"]))
        kw = {}
        if routing == "group":
            kw = dict(groups=R, topk_groups=int(rng.integers(1, R + 1)))
            k = min(k, kw["topk_groups"] * E_loc)
        sms = int(rng.choice([0, 0, 3, 40]))
        cases.append((workloads.Workload(f"{name}{i}", R=R, T=T, H=H, E=E, k=k, C=C, mask_p=mask_p,
                                         routing=routing, zipf_s=1.2 if routing == "zipf" else 0.0,
                                         nmax=T + int(rng.integers(0, 3)), seed=7000 + i, **kw), sms))
    return cases


CASES = (_draw_cases() + _draw_cases(16, seed=2025, name="wide", wide=True)
         + _draw_cases_many_experts())


def _ids(case):
    w, sms = case
    return f"{w.name}-R{w.R}-T{w.T}-H{w.H}-E{w.E}-k{w.k}-C{w.C}" + (f"-sms{sms}" if sms else "")


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_sweep_all_entry_points(case):
    w, sms = case
    inp = workloads.make_workload(w)
    run = GpuRun(w.R, w.T, w.H, w.E, w.k, w.C, inp, nmax=w.nmax)
    run.sh = ep.make_shape(w.R, w.T, w.H, w.E, w.k, w.C, nmax=w.nmax, num_sms=sms)
    expert_major = w.E <= ep.EP_EXPERT_MAJOR_MAX_EXPERTS
    # ---- layout + handle (+ expert-major placement)
    run.lb = LayoutBuffers(run.sh, expert_major=expert_major)
    ep.ep_get_layout(run.sh, run.topk, run.lb.layout(), run.lb.handle(), run.lb.workspace, run.launch)
    ref = oracle.layout(inp["topk_idx"], w.E, w.C)
    for key, t in run.lb.as_dict().items():
        np.testing.assert_array_equal(t.cpu().numpy(), ref[key], err_msg=key)
    em = oracle.expert_layout(inp["topk_idx"], w.E)
    if expert_major:
        np.testing.assert_array_equal(host_bits(run.lb.expert_rows), em["expert_rows"])
        np.testing.assert_array_equal(host_bits(run.lb.expert_prefix), em["expert_prefix"])

    # ---- bf16 dispatch into exact regions
    off = compact_offsets(ref["rank_prefix_matrix"])
    rb = run.dispatch(off)
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, inp["topk_idx"],
                          inp["topk_weights"], fill_x=0xA5A5, fill_idx=-99, fill_w=-5.0, fill_src=-3)
    np.testing.assert_array_equal(host_bits(rb.recv_x), exp["recv_x"])
    np.testing.assert_array_equal(host_bits(rb.recv_src_idx), exp["recv_src_idx"])
    np.testing.assert_array_equal(host_bits(rb.recv_topk_idx), exp["recv_topk_idx"])
    np.testing.assert_array_equal(host_bits(rb.recv_topk_weights).view(np.uint32),
                                  exp["recv_topk_weights"].view(np.uint32))

    # ---- fused e4m3 dispatch, one scale format per case
    mode = int(w.seed % 4)
    ts = 0.0213 if mode == ep.EP_FP8_SCALE_TENSOR else 0.0
    rq = run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3, with_topk=False, fp8_scale=mode, tensor_scale=ts)
    eq = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, x_kind=oracle.X_QUANTIZE,
                         scale_mode=mode, tensor_scale=ts)
    np.testing.assert_array_equal(host_bits(rq.recv_x), eq["recv_x"])
    gs, es = host_bits(rq.recv_x_scales), eq["recv_x_scales"]
    if mode == ep.EP_FP8_SCALE_UE8M0:
        np.testing.assert_array_equal(gs, es)
    else:
        np.testing.assert_array_equal(gs.view(np.uint32), es.view(np.uint32))

    # ---- combine, both modes, with the weight reduction
    rng = np.random.default_rng(w.seed + 1)
    rows = max(off[-1], 1)
    yb = torch.from_numpy(rng.standard_normal((rows, w.H)).astype(np.float32)).to(torch.bfloat16)
    ybits = yb.view(torch.int16).numpy().view(np.uint16)[: off[-1]]
    rtw = rng.standard_normal((rows, w.k)).astype(np.float32)
    for mode_c in (ep.EP_COMBINE_SUM, ep.EP_COMBINE_WEIGHTED):
        out, cw = run.combine(yb.cuda(), off, mode_c, recv_topk_weights=torch.from_numpy(rtw).cuda())
        ec = oracle.combine(ybits, ref["send_head"], np.array(off), w.E, w.k, mode_c,
                            inp["topk_idx"], inp["topk_weights"], recv_topk_weights=rtw[: off[-1]])
        assert_close_bf16(host_bits(out), ec["out"])
        assert_weight_sums_close(cw.cpu().numpy(), ec["combined_topk_weights"], rtw[: off[-1]],
                                 ref["send_head"], off)

    # ---- expert-major dispatch + combine
    if expert_major:
        eoff = [0]
        for n in em["expert_prefix"][:, -1]:
            eoff.append(eoff[-1] + int(n))
        erows = max(eoff[-1], 1)
        rx = torch.full((erows, w.H), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        rw = torch.full((erows,), -5.0, device="cuda")
        ri = torch.full((erows,), -3, dtype=torch.int32, device="cuda")
        ep.ep_dispatch_expert_major(run.sh, run.x, ep.EP_BF16, run.topk, run.wts, run.lb.handle(),
                                    rx, None, rw, ri, eoff, run.launch)
        ee = oracle.dispatch_expert_major(inp["x"], inp["topk_idx"], inp["topk_weights"],
                                          em["expert_rows"], np.array(eoff), w.E, fill_x=0xFFFF)
        np.testing.assert_array_equal(host_bits(rx)[: eoff[-1]], ee["recv_x"])
        np.testing.assert_array_equal(host_bits(ri)[: eoff[-1]], ee["recv_src_idx"])
        np.testing.assert_array_equal(host_bits(rw)[: eoff[-1]].view(np.uint32),
                                      ee["recv_weights"].view(np.uint32))
        ye = torch.from_numpy(rng.standard_normal((erows, w.H)).astype(np.float32)).to(torch.bfloat16)
        oute = torch.empty((w.R, w.T, w.H), dtype=torch.bfloat16, device="cuda")
        ep.ep_combine_expert_major(run.sh, ye.cuda(), eoff, run.lb.handle(), ep.EP_COMBINE_WEIGHTED,
                                   run.topk, run.wts, oute, run.launch)
        eec = oracle.combine_expert_major(ye.view(torch.int16).numpy().view(np.uint16)[: eoff[-1]],
                                          inp["topk_idx"], inp["topk_weights"], em["expert_rows"],
                                          np.array(eoff), w.E, weighted=True)
        assert_close_bf16(host_bits(oute), eec)

    # ---- low latency, both receive layouts
    if w.R * w.E * w.nmax * w.H <= LL_MAX_ELEMS:
        use_fp8 = bool(w.seed % 2)
        for packed in (False, True):
            buf = run.ll_dispatch(use_fp8, packed=packed)
            el = oracle.ll_dispatch(inp["x"], inp["topk_idx"], w.E, w.nmax, use_fp8, packed=packed,
                                    fill_x=0x5A if use_fp8 else 0x5A5A)
            for key in ("slot", "recv_expert_count", "layout_range", "src_info", "recv_x"):
                np.testing.assert_array_equal(host_bits(getattr(buf, key)), el[key], err_msg=key)
            if use_fp8:
                filled = el["src_info"] != -7
                np.testing.assert_array_equal(host_bits(buf.recv_x_scales)[filled].view(np.uint32),
                                              el["recv_x_scales"][filled].view(np.uint32))
            else:
                out_ll = run.ll_combine(buf.recv_x, buf)
                ref_ll = oracle.ll_combine(el["recv_x"], inp["topk_idx"], inp["topk_weights"],
                                           el["slot"], w.E, w.nmax)
                assert_close_bf16(host_bits(out_ll), ref_ll)
    assert run.flags() == 0
