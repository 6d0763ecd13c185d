"""GPU parity at the workloads' full sizes, in the launch configuration the benchmark
uses (worst-case receive capacity, no host sync):

  dsv3           R8 x T4096, H7168, E256, k8     bf16 dispatch, weighted combine
  group_limited  same shape, 4-of-8 group gating FP8 (e4m3, per-128 scales) dispatch
  ll_decode      R8 x T128, H7168, E256, k8, 5% masked, Nmax 128, FP8 LL dispatch
  zipf_reuse     R16 x T2048, H4096, E128, k6 Zipf(1.2); layout once, then 10 x
                 (fresh x -> dispatch(handle) -> combine(handle))

Checks: every layout / handle tensor bit-exact against the oracle at full size; every
received row equal to its source row at the oracle's mapping (a device-side gather over
all rows) and every unmapped row still holding its canary; receive metadata bit-exact
against the oracle run at full size with a narrow hidden size (metadata does not depend
on H); FP8 bytes and scales of every received row bit-exact against the oracle's
quantisation of every source token; every combined token against the oracle's own
layout -> dispatch -> combine pipeline over the whole workload (compared on the device,
within the combine tolerance).
"""
import numpy as np
import pytest
import torch

import combine_layout_02_gb300 as ep
import oracle
import workloads
from gpu_util import GpuRun, assert_close_bf16, assert_close_bf16_dev, dev_bf16, host_bits

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _run(name):
    w = workloads.CONFIGS[name]
    inp = workloads.make_workload(w)
    run = GpuRun(w.R, w.T, w.H, w.E, w.k, w.C, inp, nmax=w.nmax)
    return w, inp, run


def _mapping(send_head, off):
    """(row, token) index pairs of every in-rank (s, t, d) from the oracle's send_head."""
    R, T, _ = send_head.shape
    s, t, d = np.nonzero(send_head >= 0)
    rows = np.asarray(off, np.int64)[d] + send_head[s, t, d]
    return rows, s.astype(np.int64) * T + t


def _check_rows_gather(recv_x, x_flat, rows, toks, total_rows, canary_byte):
    rows_t = torch.from_numpy(rows).cuda()
    toks_t = torch.from_numpy(toks).cuda()
    for i in range(0, len(rows), 16384):
        a = recv_x[rows_t[i:i + 16384]].view(torch.uint8)
        b = x_flat[toks_t[i:i + 16384]].view(torch.uint8)
        assert torch.equal(a, b), f"row mismatch in chunk {i}"
    mapped = torch.zeros(total_rows, dtype=torch.bool, device="cuda")
    mapped[rows_t] = True
    free = recv_x.view(torch.uint8)[~mapped]
    assert bool((free == canary_byte).all()), "an unmapped row was written"


def _layout_and_compare(run, w, inp):
    got = run.layout()
    ref = oracle.layout(inp["topk_idx"], w.E, w.C)
    for key, arr in got.items():
        np.testing.assert_array_equal(arr, ref[key], err_msg=key)
    return ref


def _oracle_pipeline(w, inp, weighted=True):
    """The oracle's layout -> dispatch (exact regions) -> combine over every token of the
    workload: the expected combine output of identity experts."""
    lay = oracle.layout(inp["topk_idx"], w.E, w.C)
    off = np.concatenate([[0], np.cumsum(lay["rank_prefix_matrix"][-1])]).astype(np.int64)
    d = oracle.dispatch(inp["x"], lay["send_head"], off, w.E)
    mode = oracle.COMBINE_WEIGHTED if weighted else oracle.COMBINE_SUM
    out = oracle.combine(d["recv_x"], lay["send_head"], off, w.E, w.k, mode, inp["topk_idx"],
                         inp["topk_weights"])["out"]
    del d
    return out


def _check_fp8_rows(recv_x, recv_x_scales, exp_q, exp_s, rows, rows_exp, total_rows, canary_byte,
                    chunk=16384):
    """Every received e4m3 row and scale row (rows, in the GPU's regions) equals the
    oracle dispatch's row (rows_exp, in the oracle's regions); unmapped rows keep the
    canary byte and NaN scales."""
    q_d = torch.from_numpy(np.ascontiguousarray(exp_q)).cuda()
    s_d = torch.from_numpy(np.ascontiguousarray(exp_s).view(np.int32)).cuda()
    rows_t = torch.from_numpy(rows).cuda()
    exp_t = torch.from_numpy(rows_exp).cuda()
    for i in range(0, len(rows), chunk):
        r, e = rows_t[i:i + chunk], exp_t[i:i + chunk]
        assert torch.equal(recv_x[r], q_d[e]), f"e4m3 bytes differ in chunk {i}"
        assert torch.equal(recv_x_scales[r].view(torch.int32), s_d[e]), f"scales differ in chunk {i}"
    mapped = torch.zeros(total_rows, dtype=torch.bool, device="cuda")
    mapped[rows_t] = True
    assert bool((recv_x[~mapped] == canary_byte).all()), "an unmapped row was written"
    assert bool(torch.isnan(recv_x_scales[~mapped]).all()), "an unmapped scale row was written"


def _metadata_reference(w, inp, ref, off):
    """Oracle dispatch at full size with a 128-wide dummy hidden state: the metadata
    (recv_topk_idx, recv_topk_weights, recv_src_idx) does not depend on H."""
    x_small = np.zeros((w.R, w.T, 128), np.uint16)
    return oracle.dispatch(x_small, ref["send_head"], np.asarray(off, np.int64), w.E,
                           inp["topk_idx"], inp["topk_weights"], fill_idx=-99, fill_w=-5.0,
                           fill_src=-3)


def test_dsv3_full_size():
    w, inp, run = _run("dsv3")
    ref = _layout_and_compare(run, w, inp)
    off = [int(v) for v in workloads.worst_case_row_offsets(w.R, w.T)]
    rb = run.dispatch(off)
    rows, toks = _mapping(ref["send_head"], off)
    _check_rows_gather(rb.recv_x, run.x.view(-1, w.H), rows, toks, off[-1], 0xA5)
    meta = _metadata_reference(w, inp, ref, off)
    np.testing.assert_array_equal(host_bits(rb.recv_src_idx), meta["recv_src_idx"])
    np.testing.assert_array_equal(host_bits(rb.recv_topk_idx), meta["recv_topk_idx"])
    np.testing.assert_array_equal(host_bits(rb.recv_topk_weights).view(np.uint32),
                                  meta["recv_topk_weights"].view(np.uint32))
    out, _ = run.combine(rb.recv_x, off, ep.EP_COMBINE_WEIGHTED)
    assert_close_bf16_dev(out, _oracle_pipeline(w, inp))
    assert run.flags() == 0


def test_group_limited_fp8_full_size():
    w, inp, run = _run("group_limited")
    ref = _layout_and_compare(run, w, inp)
    assert (ref["is_token_in_rank"].sum(-1) <= 4).all()        # group-limited: <= 4 ranks
    off = [int(v) for v in workloads.worst_case_row_offsets(w.R, w.T)]
    rb = run.dispatch(off, recv_dtype=ep.EP_FP8_E4M3)
    rows, _ = _mapping(ref["send_head"], off)
    # every received row: bytes and scales equal the oracle's FP8 dispatch of the same
    # routing (into exact regions; rows_c are the same entries' rows there)
    off_c = np.concatenate([[0], np.cumsum(ref["rank_prefix_matrix"][-1])]).astype(np.int64)
    rows_c, _ = _mapping(ref["send_head"], off_c)
    exp = oracle.dispatch(inp["x"], ref["send_head"], off_c, w.E, x_kind=oracle.X_QUANTIZE)
    _check_fp8_rows(rb.recv_x, rb.recv_x_scales, exp["recv_x"], exp["recv_x_scales"], rows, rows_c,
                    off[-1], 0xA5)
    del exp
    # bf16 combine of the bf16 rows, every token
    rb16 = run.dispatch(off)
    out, _ = run.combine(rb16.recv_x, off, ep.EP_COMBINE_WEIGHTED)
    assert_close_bf16_dev(out, _oracle_pipeline(w, inp))
    assert run.flags() == 0


@pytest.mark.parametrize("packed", [False, True])
def test_ll_decode_full_size(packed):
    w, inp, run = _run("ll_decode")
    buf = run.ll_dispatch(True, phase=ep.EP_PHASE_SEND, packed=packed)
    run.ll_dispatch(True, phase=ep.EP_PHASE_RECV, buf=buf)
    exp = oracle.ll_dispatch(inp["x"], inp["topk_idx"], w.E, w.nmax, True, fill_x=0x5A,
                             packed=packed)
    for key in ("slot", "recv_expert_count", "layout_range", "src_info"):
        np.testing.assert_array_equal(host_bits(getattr(buf, key)), exp[key], err_msg=key)
    filled = exp["src_info"] != -7
    idx = torch.from_numpy(np.argwhere(filled)).cuda()
    got_q = buf.recv_x[idx[:, 0], idx[:, 1], idx[:, 2]].cpu().numpy()
    got_s = buf.recv_x_scales[idx[:, 0], idx[:, 1], idx[:, 2]].cpu().numpy()
    np.testing.assert_array_equal(got_q, exp["recv_x"][filled])
    np.testing.assert_array_equal(got_s.view(np.uint32), exp["recv_x_scales"][filled].view(np.uint32))
    # bf16 slots + weighted LL combine of identity experts, against the oracle pipeline
    b16 = run.ll_dispatch(False, packed=packed)
    out = run.ll_combine(b16.recv_x, b16)
    e16 = oracle.ll_dispatch(inp["x"], inp["topk_idx"], w.E, w.nmax, False, packed=packed)
    ref = oracle.ll_combine(e16["recv_x"], inp["topk_idx"], inp["topk_weights"], e16["slot"],
                            w.E, w.nmax)
    assert_close_bf16(host_bits(out), ref)
    assert run.flags() == 0


def test_zipf_handle_reuse_full_size():
    w, inp, run = _run("zipf_reuse")
    ref = _layout_and_compare(run, w, inp)
    off = [int(v) for v in workloads.worst_case_row_offsets(w.R, w.T)]
    rows, toks = _mapping(ref["send_head"], off)
    rng = np.random.default_rng(99)
    for it in range(10):
        x_it = workloads.make_hidden(rng, w.R, w.T, w.H)
        xd = dev_bf16(x_it)
        rb = run.dispatch(off, with_topk=False, x=xd)
        out, _ = run.combine(rb.recv_x, off, ep.EP_COMBINE_WEIGHTED)
        if it in (0, 9):
            _check_rows_gather(rb.recv_x, xd.view(-1, w.H), rows, toks, off[-1], 0xA5)
            assert_close_bf16_dev(out, _oracle_pipeline(w, dict(inp, x=x_it)))
    assert run.flags() == 0


def test_tiny_all_modes_full_compare():
    """The tiny workload end to end in every mode against the full oracle."""
    w, inp, run = _run("tiny")
    ref = _layout_and_compare(run, w, inp)
    off = [int(v) for v in workloads.worst_case_row_offsets(w.R, w.T)]
    rb = run.dispatch(off)
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, inp["topk_idx"],
                          inp["topk_weights"], fill_x=0xA5A5, fill_idx=-99, fill_w=-5.0, fill_src=-3)
    np.testing.assert_array_equal(host_bits(rb.recv_x), exp["recv_x"])
    for mode in (ep.EP_COMBINE_SUM, ep.EP_COMBINE_WEIGHTED):
        out, _ = run.combine(rb.recv_x, off, mode)
        cexp = oracle.combine(exp["recv_x"], ref["send_head"], np.array(off), w.E, w.k, mode,
                              inp["topk_idx"], inp["topk_weights"])["out"]
        assert_close_bf16(host_bits(out), cexp)
