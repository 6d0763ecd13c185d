"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by
element, on seeded inputs spanning several tiles and ragged tails: the tiny workload,
ragged shapes, R not a multiple of 8, R > 32, R = 1, R = 64, k = 32, every expert chosen,
8192 experts, 16384-wide rows, top-2 and two-rank shapes (at most two rows per token),
empty inputs, masked entries, skewed and group-limited routing.

Bit-exact: every layout / handle tensor, receive rows (bf16 and e4m3), FP8 scales,
recv_topk_idx / recv_topk_weights / recv_src_idx, low-latency slots and counts, and
the canaries of rows nothing maps to. Combine: within 1e-3 absolute + 1e-2 relative.
"""
import numpy as np
import pytest
import torch

import combine_layout_02_gb300 as ep
import oracle
import workloads
from gpu_util import GpuRun, assert_close_bf16, bf16_to_f64, compact_offsets, dev_bf16, host_bits, assert_weight_sums_close

pytestmark = pytest.mark.gpu

W = workloads.Workload
CASES = {
    "tiny": workloads.CONFIGS["tiny"],
    "ragged": W("ragged", R=4, T=1000, H=384, E=32, k=5, C=7, mask_p=0.1, seed=101),
    "r3_odd": W("r3", R=3, T=257, H=128, E=9, k=3, C=12, seed=102),
    "zipf16": W("z16", R=16, T=300, H=512, E=128, k=6, C=5, routing="zipf", zipf_s=1.2, seed=103),
    "group8": W("g8", R=8, T=513, H=1024, E=256, k=8, C=12, routing="group", groups=8,
                topk_groups=4, seed=104),
    "r1": W("r1", R=1, T=70, H=128, E=4, k=2, C=3, seed=105),
    "r64": W("r64", R=64, T=40, H=128, E=64, k=4, C=2, seed=106),
    "r33": W("r33", R=33, T=50, H=256, E=66, k=3, C=4, seed=107),
    "k32": W("k32", R=8, T=64, H=128, E=64, k=32, C=3, seed=108),
    "many_channels": W("mc", R=2, T=9, H=128, E=8, k=2, C=12, seed=109),
    "e8192": W("e8k", R=16, T=50, H=128, E=8192, k=8, C=3, seed=115),       # most experts
    "h16k": W("h16k", R=4, T=33, H=16384, E=16, k=4, C=2, seed=116),       # 32 KB rows
    "k_all": W("kall", R=4, T=40, H=256, E=32, k=32, C=5, seed=117),       # every expert
    "top2_h4096": W("t2", R=8, T=300, H=4096, E=64, k=2, C=5, seed=119),   # <= 2 rows per token
    "r2_h2048": W("r2w", R=2, T=200, H=2048, E=8, k=4, C=3, seed=120),    # <= 2 rows per token
}


def _setup(name):
    w = CASES[name]
    inp = workloads.make_workload(w)
    run = GpuRun(w.R, w.T, w.H, w.E, w.k, w.C, inp)
    ref = oracle.layout(inp["topk_idx"], w.E, w.C)
    return w, inp, run, ref


@pytest.mark.parametrize("name", list(CASES))
def test_layout_bit_exact(name):
    w, inp, run, ref = _setup(name)
    got = run.layout()
    for key, arr in got.items():
        np.testing.assert_array_equal(arr, ref[key], err_msg=key)
    assert run.flags() == 0


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("offsets", ["compact", "worst"])
def test_dispatch_bf16_bit_exact(name, offsets):
    w, inp, run, ref = _setup(name)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"]) if offsets == "compact" else \
        [int(v) for v in workloads.worst_case_row_offsets(w.R, w.T)]
    rb = run.dispatch(off)
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, inp["topk_idx"],
                          inp["topk_weights"], fill_x=0xA5A5, fill_idx=-99, fill_w=-5.0, fill_src=-3)
    np.testing.assert_array_equal(host_bits(rb.recv_x), exp["recv_x"])
    np.testing.assert_array_equal(host_bits(rb.recv_src_idx), exp["recv_src_idx"])
    np.testing.assert_array_equal(host_bits(rb.recv_topk_idx), exp["recv_topk_idx"])
    np.testing.assert_array_equal(host_bits(rb.recv_topk_weights).view(np.uint32),
                                  exp["recv_topk_weights"].view(np.uint32))
    assert run.flags() == 0


@pytest.mark.parametrize("name", ["tiny", "ragged", "r3_odd", "group8", "r33", "k32", "h16k",
                                  "top2_h4096", "r2_h2048"])
def test_dispatch_fp8_fused_bit_exact(name):
    """Every form of the fused quantisation: rows up to 1024 channels, at most two
    destinations per token, and the rest."""
    w, inp, run, ref = _setup(name)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rb = run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3)
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, inp["topk_idx"],
                          inp["topk_weights"], x_kind=oracle.X_QUANTIZE)
    np.testing.assert_array_equal(host_bits(rb.recv_x), exp["recv_x"])
    np.testing.assert_array_equal(host_bits(rb.recv_x_scales).view(np.uint32),
                                  exp["recv_x_scales"].view(np.uint32))
    np.testing.assert_array_equal(host_bits(rb.recv_topk_idx), exp["recv_topk_idx"])
    # pre-quantised (fp8, scales) input tuple is copied byte for byte
    q, sc = oracle.quantize_rows(inp["x"])
    rb2 = run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3, with_topk=False,
                       x=torch.from_numpy(q).cuda(), x_dtype=ep.EP_FP8_E4M3,
                       x_scales=torch.from_numpy(sc).cuda())
    np.testing.assert_array_equal(host_bits(rb2.recv_x), exp["recv_x"])
    np.testing.assert_array_equal(host_bits(rb2.recv_x_scales).view(np.uint32),
                                  exp["recv_x_scales"].view(np.uint32))
    assert run.flags() == 0


def test_fp8_extreme_values():
    """Groups with zeros, values below the amax floor, huge magnitudes, ties."""
    R, T, H, E, k = 2, 8, 256, 4, 2
    rng = np.random.default_rng(110)
    x32 = rng.standard_normal((R, T, H)).astype(np.float32)
    x32[0, 0] = 0.0
    x32[0, 1, :128] = 3e-5
    x32[0, 2] *= 1e30
    x32[0, 3, 128:] = -1e-38
    x32[1, 0, :] = np.tile(np.array([2.0, -3 / 1024, 1.0, 0.01], np.float32), H // 4)
    xb = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    topk = np.tile(np.array([0, 3], np.int64), (R, T, 1))
    inp = {"x": xb, "topk_idx": topk, "topk_weights": np.full((R, T, k), 0.5, np.float32)}
    run = GpuRun(R, T, H, E, k, 1, inp)
    ref = oracle.layout(topk, E, 1)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rb = run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3)
    exp = oracle.dispatch(xb, ref["send_head"], np.array(off), E, x_kind=oracle.X_QUANTIZE)
    np.testing.assert_array_equal(host_bits(rb.recv_x), exp["recv_x"])
    np.testing.assert_array_equal(host_bits(rb.recv_x_scales).view(np.uint32),
                                  exp["recv_x_scales"].view(np.uint32))


@pytest.mark.parametrize("name", list(CASES))
def test_handle_reuse_bit_identical(name):
    w, inp, run, ref = _setup(name)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    first = run.dispatch(off)
    again = run.dispatch(off, with_topk=False)
    assert torch.equal(first.recv_x.view(torch.int16), again.recv_x.view(torch.int16))
    assert torch.equal(first.recv_src_idx, again.recv_src_idx)
    # fresh x through the cached handle equals the oracle on that x
    rng = np.random.default_rng(w.seed + 1000)
    x2 = workloads.make_hidden(rng, w.R, w.T, w.H)
    rb = run.dispatch(off, with_topk=False, x=dev_bf16(x2))
    exp = oracle.dispatch(x2, ref["send_head"], np.array(off), w.E)
    np.testing.assert_array_equal(host_bits(rb.recv_x), exp["recv_x"])


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("mode", [ep.EP_COMBINE_SUM, ep.EP_COMBINE_WEIGHTED])
def test_combine_within_tolerance(name, mode):
    w, inp, run, ref = _setup(name)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rng = np.random.default_rng(w.seed + 2000)
    y32 = rng.standard_normal((max(off[-1], 1), w.H)).astype(np.float32)
    yb = torch.from_numpy(y32).to(torch.bfloat16)
    ybits = yb.view(torch.int16).numpy().view(np.uint16)[: off[-1]]
    rtw = rng.standard_normal((max(off[-1], 1), w.k)).astype(np.float32)
    out, cw = run.combine(yb.cuda(), off, mode, recv_topk_weights=torch.from_numpy(rtw).cuda())
    exp = oracle.combine(ybits, ref["send_head"], np.array(off), w.E, w.k, mode,
                         inp["topk_idx"], inp["topk_weights"], recv_topk_weights=rtw[: off[-1]])
    assert_close_bf16(host_bits(out), exp["out"])
    assert_weight_sums_close(cw.cpu().numpy(), exp["combined_topk_weights"], rtw[: off[-1]],
                             ref["send_head"], off)
    assert run.flags() == 0


@pytest.mark.parametrize("name", ["tiny", "zipf16", "group8", "k32"])
def test_identity_round_trip(name):
    """dispatch -> identity experts -> weighted combine returns x within bf16 rounding."""
    w, inp, run, ref = _setup(name)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rb = run.dispatch(off)
    out, _ = run.combine(rb.recv_x, off, ep.EP_COMBINE_WEIGHTED)
    xf, of = bf16_to_f64(inp["x"]), bf16_to_f64(host_bits(out))
    sent = ref["is_token_in_rank"].sum(-1) > 0
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(xf), 2.0 ** -126))) - 7)
    assert np.all(np.abs(of - xf)[sent] <= 2 * ulp[sent])


def test_empty_tokens():
    R, T, H, E, k, C = 4, 0, 128, 8, 2, 3
    inp = {"x": np.zeros((R, T, H), np.uint16), "topk_idx": np.zeros((R, T, k), np.int64),
           "topk_weights": np.zeros((R, T, k), np.float32)}
    run = GpuRun(R, T, H, E, k, C, inp)
    got = run.layout()
    ref = oracle.layout(inp["topk_idx"], E, C)
    for key, arr in got.items():
        np.testing.assert_array_equal(arr, ref[key], err_msg=key)


def test_device_error_flags():
    """Bad expert ids are skipped (as masked) and flagged; undersized receive regions
    flag an overflow and skip the rows -- no fault, no trap."""
    w = CASES["ragged"]
    inp = workloads.make_workload(w)
    bad = inp["topk_idx"].copy()
    bad[0, 3, 1] = w.E
    bad[2, 10, 0] = -5
    inp2 = dict(inp, topk_idx=bad)
    run = GpuRun(w.R, w.T, w.H, w.E, w.k, w.C, inp2)
    got = run.layout()
    assert run.flags() & ep.EP_DEVERR_BAD_EXPERT
    ref = oracle.layout(bad, w.E, w.C)
    assert ref["bad_entries"] == 2
    for key, arr in got.items():
        np.testing.assert_array_equal(arr, ref[key], err_msg=key)
    # overflow: every region one row short
    run.err.zero_()
    off = compact_offsets(ref["rank_prefix_matrix"])
    short = [0] + [off[d + 1] - (d + 1) for d in range(w.R)]
    rb = run.dispatch(short)
    assert run.flags() & ep.EP_DEVERR_RECV_OVERFLOW
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(short), w.E, bad, inp["topk_weights"],
                          fill_x=0xA5A5, fill_idx=-99, fill_w=-5.0, fill_src=-3)
    assert exp["bad_rows"] > 0
    np.testing.assert_array_equal(host_bits(rb.recv_x), exp["recv_x"])
    np.testing.assert_array_equal(host_bits(rb.recv_topk_idx), exp["recv_topk_idx"])


# ----------------------------------------------------------------------------- low latency

LL_CASES = {
    "tiny": W("lt", R=2, T=128, H=256, E=8, k=2, nmax=128, seed=0),
    "masked": W("lm", R=4, T=40, H=512, E=32, k=6, nmax=48, mask_p=0.05, seed=111),
    "r8": W("l8", R=8, T=100, H=1024, E=64, k=8, nmax=128, mask_p=0.05, seed=112),
    # more earlier entries than a send block loads up front (t*k > 1024)
    "long": W("ll", R=2, T=300, H=256, E=16, k=8, nmax=300, mask_p=0.05, seed=118),
    # rows longer than a send block loads up front (bf16 > 16 KB, e4m3 source > 16 KB)
    "wide": W("lw", R=2, T=20, H=16384, E=8, k=4, nmax=24, seed=119),
    # the rank kernel's running counts across chunks: 8192 entries per source (8 chunks)
    "chunks": W("lc", R=2, T=1024, H=128, E=64, k=8, nmax=1024, mask_p=0.05, seed=120),
    # many experts: fewer warps per rank-kernel chunk (5 at E = 4096), 4 chunks per source
    "experts4096": W("le", R=4, T=64, H=128, E=4096, k=8, nmax=64, mask_p=0.05, seed=121),
}


def _ll_setup(name):
    w = LL_CASES[name]
    inp = workloads.make_workload(w)
    return w, inp, GpuRun(w.R, w.T, w.H, w.E, w.k, 1, inp, nmax=w.nmax)


@pytest.mark.parametrize("name", list(LL_CASES))
@pytest.mark.parametrize("use_fp8", [False, True])
@pytest.mark.parametrize("packed", [False, True])
def test_ll_dispatch_bit_exact(name, use_fp8, packed):
    w, inp, run = _ll_setup(name)
    buf = run.ll_dispatch(use_fp8, packed=packed)
    exp = oracle.ll_dispatch(inp["x"], inp["topk_idx"], w.E, w.nmax, use_fp8, packed=packed,
                             fill_x=0x5A5A if not use_fp8 else 0x5A)
    for key in ("slot", "recv_expert_count", "layout_range", "src_info"):
        np.testing.assert_array_equal(host_bits(getattr(buf, key)), exp[key], err_msg=key)
    np.testing.assert_array_equal(host_bits(buf.recv_x), exp["recv_x"])
    if use_fp8:
        filled = exp["src_info"] != -7
        np.testing.assert_array_equal(host_bits(buf.recv_x_scales)[filled].view(np.uint32),
                                      exp["recv_x_scales"][filled].view(np.uint32))
    assert run.flags() == 0


@pytest.mark.parametrize("name", list(LL_CASES))
@pytest.mark.parametrize("packed", [False, True])
def test_ll_phase_split_equals_single_call(name, packed):
    w, inp, run = _ll_setup(name)
    both = run.ll_dispatch(True, packed=packed)
    split = run.ll_dispatch(True, phase=ep.EP_PHASE_SEND, packed=packed)
    torch.cuda.synchronize()
    run.ll_dispatch(True, phase=ep.EP_PHASE_RECV, buf=split)
    for key in ("recv_x", "recv_x_scales", "src_info", "slot", "send_count", "recv_expert_count",
                "layout_range"):
        a, b = getattr(both, key), getattr(split, key)
        if key == "recv_x_scales":
            filled = (both.src_info != -7)
            a, b = a[filled], b[filled]
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.int32 else a,
                           b.view(torch.uint8) if b.dtype != torch.int32 else b), key


@pytest.mark.parametrize("name", list(LL_CASES))
@pytest.mark.parametrize("packed", [False, True])
def test_ll_combine_within_tolerance(name, packed):
    w, inp, run = _ll_setup(name)
    buf = run.ll_dispatch(False, packed=packed)
    rng = np.random.default_rng(w.seed + 3000)
    y32 = rng.standard_normal(tuple(buf.recv_x.shape)).astype(np.float32)
    yb = torch.from_numpy(y32).to(torch.bfloat16)
    out_send = run.ll_combine(yb.cuda(), buf, phase=ep.EP_PHASE_SEND)   # event-only phase
    out = run.ll_combine(yb.cuda(), buf, phase=ep.EP_PHASE_RECV)
    exp = oracle.ll_combine(yb.view(torch.int16).numpy().view(np.uint16), inp["topk_idx"],
                            inp["topk_weights"], host_bits(buf.slot), w.E, w.nmax)
    assert_close_bf16(host_bits(out), exp)
    # identity experts: returns x * sum of valid weights (= x) within rounding
    out2 = run.ll_combine(buf.recv_x, buf)
    xf = bf16_to_f64(inp["x"]) * inp["topk_weights"].astype(np.float64).sum(-1)[..., None]
    assert np.all(np.abs(bf16_to_f64(host_bits(out2)) - xf) <= 1e-3 + 1e-2 * np.abs(xf))
    del out_send


@pytest.mark.parametrize("packed", [False, True])
def test_ll_slot_overflow_flag(packed):
    """Duplicate experts in a token push a (source, expert) count past Nmax: flagged and
    skipped exactly like the oracle, no fault."""
    R, T, H, E, k, nmax = 2, 4, 128, 4, 2, 4
    topk = np.zeros((R, T, k), np.int64)
    rng = np.random.default_rng(113)
    inp = {"x": workloads.make_hidden(rng, R, T, H), "topk_idx": topk,
           "topk_weights": np.full((R, T, k), 0.5, np.float32)}
    run = GpuRun(R, T, H, E, k, 1, inp, nmax=nmax)
    buf = run.ll_dispatch(False, packed=packed)
    assert run.flags() & ep.EP_DEVERR_SLOT_OVERFLOW
    exp = oracle.ll_dispatch(inp["x"], topk, E, nmax, False, packed=packed)
    assert exp["bad_entries"] == 2 * 4
    np.testing.assert_array_equal(host_bits(buf.slot), exp["slot"])
    np.testing.assert_array_equal(host_bits(buf.recv_expert_count), exp["recv_expert_count"])
    np.testing.assert_array_equal(host_bits(buf.layout_range), exp["layout_range"])


# ----------------------------------------------------------------------------- FP8 scale modes

MODES = [(ep.EP_FP8_SCALE_POW2, 0.0), (ep.EP_FP8_SCALE_UE8M0, 0.0), (ep.EP_FP8_SCALE_TENSOR, 0.0173)]


def _cmp_scales(got, exp, mode):
    if mode == ep.EP_FP8_SCALE_UE8M0:
        np.testing.assert_array_equal(got, exp)
    else:
        np.testing.assert_array_equal(got.view(np.uint32), exp.view(np.uint32))


@pytest.mark.parametrize("name", ["tiny", "ragged", "group8", "k32", "h16k", "top2_h4096"])
@pytest.mark.parametrize("mode,ts", MODES)
def test_dispatch_fp8_scale_modes_bit_exact(name, mode, ts):
    """round_scale / UE8M0 / per-tensor scale ("DeepEP" README feature notes)."""
    w, inp, run, ref = _setup(name)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rb = run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3, fp8_scale=mode, tensor_scale=ts)
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, inp["topk_idx"],
                          inp["topk_weights"], x_kind=oracle.X_QUANTIZE, scale_mode=mode,
                          tensor_scale=ts)
    np.testing.assert_array_equal(host_bits(rb.recv_x), exp["recv_x"])
    _cmp_scales(host_bits(rb.recv_x_scales), exp["recv_x_scales"], mode)
    assert run.flags() == 0


@pytest.mark.parametrize("mode,ts", MODES + [(ep.EP_FP8_SCALE_TENSOR, 1e-30)])
def test_fp8_scale_modes_extreme_values(mode, ts):
    R, T, H, E, k = 2, 8, 256, 4, 2
    rng = np.random.default_rng(114)
    x32 = rng.standard_normal((R, T, H)).astype(np.float32)
    x32[0, 0] = 0.0
    x32[0, 1, :128] = 3e-5
    x32[0, 2] *= 1e30
    x32[0, 3, 128:] = -1e-38
    x32[1, 0, :] = np.tile(np.array([2.0, -3 / 1024, 1.0, 0.01], np.float32), H // 4)
    xb = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    topk = np.tile(np.array([0, 3], np.int64), (R, T, 1))
    inp = {"x": xb, "topk_idx": topk, "topk_weights": np.full((R, T, k), 0.5, np.float32)}
    run = GpuRun(R, T, H, E, k, 1, inp)
    ref = oracle.layout(topk, E, 1)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rb = run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3, with_topk=False, fp8_scale=mode, tensor_scale=ts)
    exp = oracle.dispatch(xb, ref["send_head"], np.array(off), E, x_kind=oracle.X_QUANTIZE,
                          scale_mode=mode, tensor_scale=ts)
    np.testing.assert_array_equal(host_bits(rb.recv_x), exp["recv_x"])
    _cmp_scales(host_bits(rb.recv_x_scales), exp["recv_x_scales"], mode)


@pytest.mark.parametrize("mode,ts", MODES)
@pytest.mark.parametrize("packed", [False, True])
def test_ll_dispatch_scale_modes_bit_exact(mode, ts, packed):
    w, inp, run = _ll_setup("masked")
    buf = run.ll_dispatch(True, fp8_scale=mode, tensor_scale=ts, packed=packed)
    exp = oracle.ll_dispatch(inp["x"], inp["topk_idx"], w.E, w.nmax, True, fill_x=0x5A,
                             scale_mode=mode, tensor_scale=ts, packed=packed)
    np.testing.assert_array_equal(host_bits(buf.recv_x), exp["recv_x"])
    filled = exp["src_info"] != -7
    _cmp_scales(host_bits(buf.recv_x_scales)[filled], exp["recv_x_scales"][filled], mode)
    np.testing.assert_array_equal(host_bits(buf.slot), exp["slot"])


def test_all_entries_masked_empty_regions():
    """Every entry masked: exact regions hold no row, so the receive arrays are empty
    (NULL pointers) and the calls must still succeed; combine gives +0 everywhere."""
    R, T, H, E, k, C = 4, 33, 256, 8, 3, 5
    rng = np.random.default_rng(114)
    inp = {"x": workloads.make_hidden(rng, R, T, H), "topk_idx": np.full((R, T, k), -1, np.int64),
           "topk_weights": np.zeros((R, T, k), np.float32)}
    run = GpuRun(R, T, H, E, k, C, inp)
    ref = oracle.layout(inp["topk_idx"], E, C)
    got = run.layout()
    for key, arr in got.items():
        np.testing.assert_array_equal(arr, ref[key], err_msg=key)
    off = compact_offsets(ref["rank_prefix_matrix"])
    assert off[-1] == 0
    run.dispatch(off)
    run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3, with_topk=False)
    y = torch.empty((0, H), dtype=torch.bfloat16, device="cuda")
    out, cw = run.combine(y, off, ep.EP_COMBINE_WEIGHTED,
                          recv_topk_weights=torch.empty((0, k), device="cuda"))
    assert torch.count_nonzero(out.view(torch.int16)) == 0
    assert torch.count_nonzero(cw) == 0
    assert run.flags() == 0


@pytest.mark.parametrize("name", ["zipf16", "group8", "r64"])
def test_run_twice_bit_identical(name):
    """No atomics decide any value: layout, dispatch (bf16 and e4m3), combine and the
    low-latency path give the same bits on a second run over fresh buffers."""
    w, inp, run, ref = _setup(name)
    outs = []
    for _ in range(2):
        lay = run.layout()
        off = compact_offsets(ref["rank_prefix_matrix"])
        rb = run.dispatch(off)
        rq = run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3, with_topk=False)
        out, _ = run.combine(rb.recv_x, off, ep.EP_COMBINE_WEIGHTED)
        outs.append([*lay.values(), host_bits(rb.recv_x), host_bits(rb.recv_topk_weights),
                     host_bits(rq.recv_x), host_bits(rq.recv_x_scales), host_bits(out)])
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)
    run_ll = GpuRun(w.R, min(w.T, 64), w.H, w.E, w.k, 1,
                    {key: np.ascontiguousarray(v[:, :64]) for key, v in inp.items()}, nmax=64)
    lls = []
    for _ in range(2):
        buf = run_ll.ll_dispatch(False, packed=True)
        lls.append((host_bits(buf.recv_x), host_bits(buf.slot), host_bits(run_ll.ll_combine(buf.recv_x, buf))))
    for a, b in zip(*lls):
        np.testing.assert_array_equal(a, b)
    assert run.flags() == 0 and run_ll.flags() == 0



def test_dispatch_16_byte_aligned_buffers():
    """x and the receive rows need only 16-byte alignment: buffers that start 16 bytes past
    a 32-byte boundary give the oracle's bytes too."""
    w, inp, run, ref = _setup("ragged")
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    n_x = w.R * w.T * w.H
    xbuf = torch.empty(n_x + 8, dtype=torch.bfloat16, device="cuda")
    x16 = xbuf[8:].view(w.R, w.T, w.H)
    x16.copy_(run.x)
    assert x16.data_ptr() % 32 == 16
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, fill_x=0xA5A5)
    from combine_layout_02_gb300.buffers import LayoutBuffers, RecvBuffers
    rb = RecvBuffers(off[-1] + 1, w.H, w.k, with_topk=False, fill=0xA5)
    recv16 = rb.recv_x.view(-1)[8: 8 + off[-1] * w.H].view(off[-1], w.H)
    assert recv16.data_ptr() % 32 == 16
    ep.ep_dispatch(run.sh, x16, ep.EP_BF16, None, ep.EP_BF16, None, None, run.lb.handle(rb.recv_src_idx),
                   recv16, None, None, None, rb.recv_src_idx, off, run.launch)
    np.testing.assert_array_equal(host_bits(recv16), exp["recv_x"])
    # fused e4m3 from a 16-byte-aligned x (two 16-byte loads per unit instead of one 32-byte)
    eq = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, x_kind=oracle.X_QUANTIZE)
    for x_in in (run.x, x16):
        rq = run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3, with_topk=False, x=x_in)
        np.testing.assert_array_equal(host_bits(rq.recv_x), eq["recv_x"])
        np.testing.assert_array_equal(host_bits(rq.recv_x_scales).view(np.uint32),
                                      eq["recv_x_scales"].view(np.uint32))
    lb = LayoutBuffers(run.sh, expert_major=True)
    ep.ep_get_layout(run.sh, run.topk, lb.layout(), lb.handle(), lb.workspace, run.launch)
    em = oracle.expert_layout(inp["topk_idx"], w.E)
    eoff = [0]
    for n in em["expert_prefix"][:, -1]:
        eoff.append(eoff[-1] + int(n))
    ee = oracle.dispatch_expert_major(inp["x"], inp["topk_idx"], inp["topk_weights"], em["expert_rows"],
                                      np.array(eoff), w.E, quantize=True)
    for x_in in (run.x, x16):
        rx = torch.zeros((eoff[-1], w.H), dtype=torch.uint8, device="cuda")
        rs = torch.zeros((eoff[-1], w.H // 128), dtype=torch.float32, device="cuda")
        ep.ep_dispatch_expert_major(run.sh, x_in, ep.EP_FP8_E4M3, run.topk, run.wts, lb.handle(), rx, rs,
                                    None, None, eoff, run.launch)
        np.testing.assert_array_equal(host_bits(rx), ee["recv_x"])
        np.testing.assert_array_equal(host_bits(rs).view(np.uint32), ee["recv_x_scales"].view(np.uint32))
    assert run.flags() == 0


@pytest.mark.parametrize("num_sms", [1, 3])
def test_num_sms_cap_persistent_grid(num_sms):
    """ep_shape.num_sms caps the grid (Buffer.set_num_sms): each warp then walks many
    tokens, reusing its row buffer and barrier phases. Results stay bit-exact."""
    w, inp, run, ref = _setup("group8")
    run.sh = ep.make_shape(w.R, w.T, w.H, w.E, w.k, w.C, num_sms=num_sms)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rb = run.dispatch(off)
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, inp["topk_idx"],
                          inp["topk_weights"], fill_x=0xA5A5, fill_idx=-99, fill_w=-5.0, fill_src=-3)
    np.testing.assert_array_equal(host_bits(rb.recv_x), exp["recv_x"])
    np.testing.assert_array_equal(host_bits(rb.recv_topk_idx), exp["recv_topk_idx"])
    np.testing.assert_array_equal(host_bits(rb.recv_src_idx), exp["recv_src_idx"])
    rq = run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3, with_topk=False)
    eq = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, x_kind=oracle.X_QUANTIZE)
    np.testing.assert_array_equal(host_bits(rq.recv_x), eq["recv_x"])
    np.testing.assert_array_equal(host_bits(rq.recv_x_scales).view(np.uint32),
                                  eq["recv_x_scales"].view(np.uint32))
    q, sc = oracle.quantize_rows(inp["x"])
    rp = run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3, with_topk=False,
                      x=torch.from_numpy(q).cuda(), x_dtype=ep.EP_FP8_E4M3,
                      x_scales=torch.from_numpy(sc).cuda())
    np.testing.assert_array_equal(host_bits(rp.recv_x), eq["recv_x"])
    out, _ = run.combine(rb.recv_x, off, ep.EP_COMBINE_WEIGHTED)
    ec = oracle.combine(exp["recv_x"], ref["send_head"], np.array(off), w.E, w.k,
                        ep.EP_COMBINE_WEIGHTED, inp["topk_idx"], inp["topk_weights"])
    assert_close_bf16(host_bits(out), ec["out"])
    assert run.flags() == 0


def test_rows_too_wide_for_bulk_copies_use_the_register_copy():
    """bf16 rows above 50 KB (H > 25600) do not fit four shared-memory row buffers and take
    the 16-byte register copy, rank-major and expert-major: still bit-exact."""
    w = W("wide", R=2, T=21, H=26624, E=4, k=2, C=3, seed=118)
    inp = workloads.make_workload(w)
    run = GpuRun(w.R, w.T, w.H, w.E, w.k, w.C, inp)
    ref = oracle.layout(inp["topk_idx"], w.E, w.C)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rb = run.dispatch(off)
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, inp["topk_idx"],
                          inp["topk_weights"], fill_x=0xA5A5, fill_idx=-99, fill_w=-5.0, fill_src=-3)
    np.testing.assert_array_equal(host_bits(rb.recv_x), exp["recv_x"])
    np.testing.assert_array_equal(host_bits(rb.recv_topk_idx), exp["recv_topk_idx"])
    from combine_layout_02_gb300.buffers import LayoutBuffers
    lb = LayoutBuffers(run.sh, expert_major=True)
    ep.ep_get_layout(run.sh, run.topk, lb.layout(), lb.handle(), lb.workspace, run.launch)
    em = oracle.expert_layout(inp["topk_idx"], w.E)
    eoff = [0]
    for n in em["expert_prefix"][:, -1]:
        eoff.append(eoff[-1] + int(n))
    rx = torch.full((eoff[-1], w.H), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    ep.ep_dispatch_expert_major(run.sh, run.x, ep.EP_BF16, run.topk, run.wts, lb.handle(), rx, None,
                                None, None, eoff, run.launch)
    ee = oracle.dispatch_expert_major(inp["x"], inp["topk_idx"], inp["topk_weights"],
                                      em["expert_rows"], np.array(eoff), w.E, fill_x=0xFFFF)
    np.testing.assert_array_equal(host_bits(rx), ee["recv_x"])
    assert run.flags() == 0


@pytest.mark.parametrize("name", ["zipf16", "tiny", "h16k", "top2_h4096"])
def test_combine_16_byte_aligned_y_takes_the_16_byte_gather(name):
    """y that is 16- but not 32-byte aligned uses a 16-byte-load gather (aligned y uses
    32-byte loads): both match the oracle, rank-major and expert-major, for each form of the
    combine (rows of at most 256 channels, rows up to 1024, at most two rows per token, the
    rest)."""
    w, inp, run, ref = _setup(name)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rng = np.random.default_rng(w.seed + 4000)
    y32 = rng.standard_normal((off[-1], w.H)).astype(np.float32)
    yb = torch.from_numpy(y32).to(torch.bfloat16)
    ybits = yb.view(torch.int16).numpy().view(np.uint16)
    ybuf = torch.empty(off[-1] * w.H + 8, dtype=torch.bfloat16, device="cuda")
    y16 = ybuf[8:].view(off[-1], w.H)
    y16.copy_(yb.cuda())
    assert y16.data_ptr() % 32 == 16
    exp = oracle.combine(ybits, ref["send_head"], np.array(off), w.E, w.k, ep.EP_COMBINE_WEIGHTED,
                         inp["topk_idx"], inp["topk_weights"])
    for y in (yb.cuda(), y16):
        out, _ = run.combine(y, off, ep.EP_COMBINE_WEIGHTED)
        assert_close_bf16(host_bits(out), exp["out"])
    from combine_layout_02_gb300.buffers import LayoutBuffers
    lb = LayoutBuffers(run.sh, expert_major=True)
    ep.ep_get_layout(run.sh, run.topk, lb.layout(), lb.handle(), lb.workspace, run.launch)
    em = oracle.expert_layout(inp["topk_idx"], w.E)
    eoff = [0]
    for n in em["expert_prefix"][:, -1]:
        eoff.append(eoff[-1] + int(n))
    ye = rng.standard_normal((eoff[-1], w.H)).astype(np.float32)
    yeb = torch.from_numpy(ye).to(torch.bfloat16)
    ebuf = torch.empty(eoff[-1] * w.H + 8, dtype=torch.bfloat16, device="cuda")
    ye16 = ebuf[8:].view(eoff[-1], w.H)
    ye16.copy_(yeb.cuda())
    eexp = oracle.combine_expert_major(yeb.view(torch.int16).numpy().view(np.uint16), inp["topk_idx"],
                                       inp["topk_weights"], em["expert_rows"], np.array(eoff), w.E)
    for y in (yeb.cuda(), ye16):
        oute = torch.empty((w.R, w.T, w.H), dtype=torch.bfloat16, device="cuda")
        ep.ep_combine_expert_major(run.sh, y, eoff, lb.handle(), ep.EP_COMBINE_WEIGHTED, run.topk,
                                   run.wts, oute, run.launch)
        assert_close_bf16(host_bits(oute), eexp)
    assert run.flags() == 0


def test_clean_ll_buffer_zeroes_the_signals_and_counts():
    """clean_low_latency_buffer: the count signals, receive counts and layout ranges are
    zero afterwards, and the next dispatch into the same buffer is exact again."""
    w, inp, run = _ll_setup("masked")
    buf = run.ll_dispatch(True)
    assert int(buf.recv_expert_count.sum().item()) > 0
    ep.ep_clean_ll_buffer(run.sh, buf.struct(), run.launch)
    torch.cuda.synchronize()
    for key in ("send_count", "recv_expert_count", "layout_range"):
        assert int(torch.count_nonzero(getattr(buf, key)).item()) == 0, key
    run.ll_dispatch(True, buf=buf)
    exp = oracle.ll_dispatch(inp["x"], inp["topk_idx"], w.E, w.nmax, True)
    for key in ("slot", "recv_expert_count", "layout_range"):
        np.testing.assert_array_equal(host_bits(getattr(buf, key)), exp[key], err_msg=key)
    # ep_read_recv_counts_sync returns each destination's received row count
    ref = oracle.layout(inp["topk_idx"], w.E, 3)
    run3 = GpuRun(w.R, w.T, w.H, w.E, w.k, 3, inp)
    run3.layout()
    counts = ep.ep_read_recv_counts_sync(run3.sh, run3.lb.handle())
    np.testing.assert_array_equal(counts, ref["rank_prefix_matrix"][-1])
    assert run.flags() == 0


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("use_fp8", [False, True])
def test_ll_repeated_experts_bit_exact(packed, use_fp8):
    """Tokens that name an expert more than once (no overflow): every entry gets its own
    slot in entry order, exactly as the oracle places it."""
    rng = np.random.default_rng(121)
    R, T, H, E, k, nmax = 2, 30, 256, 4, 3, 128
    topk = rng.integers(-1, E, size=(R, T, k)).astype(np.int64)
    inp = {"x": workloads.make_hidden(rng, R, T, H), "topk_idx": topk,
           "topk_weights": np.full((R, T, k), 1.0 / k, np.float32)}
    run = GpuRun(R, T, H, E, k, 1, inp, nmax=nmax)
    buf = run.ll_dispatch(use_fp8, packed=packed)
    exp = oracle.ll_dispatch(inp["x"], topk, E, nmax, use_fp8, packed=packed,
                             fill_x=0x5A5A if not use_fp8 else 0x5A)
    assert exp["bad_entries"] == 0
    for key in ("slot", "recv_expert_count", "layout_range", "src_info"):
        np.testing.assert_array_equal(host_bits(getattr(buf, key)), exp[key], err_msg=key)
    np.testing.assert_array_equal(host_bits(buf.recv_x), exp["recv_x"])
    assert run.flags() == 0


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("E", [4, 2048])
def test_ll_repeated_experts_across_rank_chunks(packed, E):
    """Repeated experts over many rank-kernel chunks: k = 5 entries per token from few
    experts (E = 4), or from a large expert set where a chunk holds only a few warps
    (E = 2048), T*k = 4000 entries per source, so equal experts meet across lanes, warps
    and chunks. Every slot, count and range equals the oracle's."""
    rng = np.random.default_rng(122 + E)
    R, T, H, k = 2, 800, 128, 5
    nmax = 4096 if E == 4 else 800
    pool = np.array([0, 1, 2, 3]) if E == 4 else rng.choice(E, 12, replace=False)
    topk = pool[rng.integers(0, len(pool), size=(R, T, k))].astype(np.int64)
    topk[rng.random((R, T, k)) < 0.05] = -1
    inp = {"x": workloads.make_hidden(rng, R, T, H), "topk_idx": topk,
           "topk_weights": np.full((R, T, k), 1.0 / k, np.float32)}
    run = GpuRun(R, T, H, E, k, 1, inp, nmax=nmax)
    buf = run.ll_dispatch(True, packed=packed)
    exp = oracle.ll_dispatch(inp["x"], topk, E, nmax, True, packed=packed, fill_x=0x5A)
    assert exp["bad_entries"] == 0
    for key in ("slot", "recv_expert_count", "layout_range", "src_info"):
        np.testing.assert_array_equal(host_bits(getattr(buf, key)), exp[key], err_msg=key)
    filled = exp["src_info"] != -7
    np.testing.assert_array_equal(host_bits(buf.recv_x)[filled], exp["recv_x"][filled])
    assert run.flags() == 0


@pytest.mark.parametrize("name", ["h16k", "group8"])
def test_fp8_receive_rows_16_byte_aligned(name):
    """Fused e4m3 into receive rows that are 16- but not 32-byte aligned (the 32-byte-store
    pair form then falls back to 16-byte stores), rank-major and expert-major, against the
    oracle; and into aligned rows (the pair form where it applies)."""
    w, inp, run, ref = _setup(name)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    G = w.H // 128
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, x_kind=oracle.X_QUANTIZE)
    for shift in (0, 16):
        qbuf = torch.zeros(off[-1] * w.H + 32, dtype=torch.uint8, device="cuda")
        rq = qbuf[shift: shift + off[-1] * w.H].view(off[-1], w.H)
        assert rq.data_ptr() % 32 == shift
        rs = torch.zeros((off[-1], G), dtype=torch.float32, device="cuda")
        ep.ep_dispatch(run.sh, run.x, ep.EP_BF16, None, ep.EP_FP8_E4M3, None, None,
                       run.lb.handle(), rq, rs, None, None, None, off, run.launch)
        np.testing.assert_array_equal(host_bits(rq), exp["recv_x"], err_msg=f"shift {shift}")
        np.testing.assert_array_equal(host_bits(rs).view(np.uint32), exp["recv_x_scales"].view(np.uint32))
    from combine_layout_02_gb300.buffers import LayoutBuffers
    lb = LayoutBuffers(run.sh, expert_major=True)
    ep.ep_get_layout(run.sh, run.topk, lb.layout(), lb.handle(), lb.workspace, run.launch)
    em = oracle.expert_layout(inp["topk_idx"], w.E)
    eoff = [0]
    for n in em["expert_prefix"][:, -1]:
        eoff.append(eoff[-1] + int(n))
    ee = oracle.dispatch_expert_major(inp["x"], inp["topk_idx"], inp["topk_weights"], em["expert_rows"],
                                      np.array(eoff), w.E, quantize=True)
    for shift in (0, 16):
        ebuf = torch.zeros(eoff[-1] * w.H + 32, dtype=torch.uint8, device="cuda")
        rx = ebuf[shift: shift + eoff[-1] * w.H].view(eoff[-1], w.H)
        rs = torch.zeros((eoff[-1], G), dtype=torch.float32, device="cuda")
        ep.ep_dispatch_expert_major(run.sh, run.x, ep.EP_FP8_E4M3, run.topk, run.wts, lb.handle(), rx, rs,
                                    None, None, eoff, run.launch)
        np.testing.assert_array_equal(host_bits(rx), ee["recv_x"], err_msg=f"expert-major shift {shift}")
        np.testing.assert_array_equal(host_bits(rs).view(np.uint32), ee["recv_x_scales"].view(np.uint32))
    assert run.flags() == 0
