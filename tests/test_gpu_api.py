"""The Buffer front end (combine_layout_02_gb300.api), shaped like the pages' Python API,
against the oracle: layout, exact-region and worst-case dispatch, FP8 and pre-quantised
dispatch, handle reuse, weighted combine and the weight reduction, and the low-latency
calls with and without the receive hook, and the expert-major blocks."""
import numpy as np
import pytest
import torch

import combine_layout_02_gb300 as ep
from combine_layout_02_gb300.api import Buffer
import oracle
import workloads
from gpu_util import assert_close_bf16, dev_bf16, host_bits, assert_weight_sums_close

pytestmark = pytest.mark.gpu

W = workloads.Workload("api", R=4, T=300, H=512, E=32, k=6, C=5, mask_p=0.05, seed=501)


def _inputs(w=W):
    inp = workloads.make_workload(w)
    return inp, dev_bf16(inp["x"]), torch.from_numpy(inp["topk_idx"]).cuda(), \
        torch.from_numpy(inp["topk_weights"]).cuda()


def test_buffer_normal_path_matches_the_oracle():
    inp, x, topk, wts = _inputs()
    buf = Buffer(W.R, W.E, W.H, W.k, W.C)
    ntpr, rdma, ntpe, in_rank, ev = buf.get_dispatch_layout(topk, async_finish=True)
    ev.current_stream_wait()
    ref = oracle.layout(inp["topk_idx"], W.E, W.C)
    assert rdma is None
    np.testing.assert_array_equal(ntpr.cpu().numpy(), ref["num_tokens_per_rank"])
    np.testing.assert_array_equal(ntpe.cpu().numpy(), ref["num_tokens_per_expert"])
    np.testing.assert_array_equal(in_rank.cpu().numpy(), ref["is_token_in_rank"])

    recv_x, recv_ti, recv_tw, per_expert, handle, ev = buf.dispatch(
        x, num_tokens_per_rank=ntpr, topk_idx=topk, topk_weights=wts, previous_event=ev,
        async_finish=True)
    with ev:
        pass
    off = handle.row_offset
    assert off[-1] == int(ref["rank_prefix_matrix"][-1].sum())
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), W.E, inp["topk_idx"],
                          inp["topk_weights"])
    for d in range(W.R):
        np.testing.assert_array_equal(host_bits(recv_x[d]), exp["recv_x"][off[d]:off[d + 1]])
        np.testing.assert_array_equal(host_bits(recv_ti[d]), exp["recv_topk_idx"][off[d]:off[d + 1]])
        np.testing.assert_array_equal(host_bits(recv_tw[d]).view(np.uint32),
                                      exp["recv_topk_weights"][off[d]:off[d + 1]].view(np.uint32))
    np.testing.assert_array_equal(per_expert.cpu().numpy(), ref["num_recv_tokens_per_expert"])

    # weighted combine of the received rows (identity experts) and the weight reduction
    out, cw, _ = buf.combine(recv_x, handle, topk_weights=recv_tw, weight_by=(topk, wts))
    ec = oracle.combine(exp["recv_x"], ref["send_head"], np.array(off), W.E, W.k,
                        oracle.COMBINE_WEIGHTED, inp["topk_idx"], inp["topk_weights"],
                        recv_topk_weights=exp["recv_topk_weights"])
    assert_close_bf16(host_bits(out), ec["out"])
    assert_weight_sums_close(cw.cpu().numpy(), ec["combined_topk_weights"], exp["recv_topk_weights"],
                             ref["send_head"], off)

    # handle reuse with fresh x, then a plain-sum combine of one tensor of rows
    rng = np.random.default_rng(502)
    x2 = workloads.make_hidden(rng, W.R, W.T, W.H)
    recv2, ti2, tw2, _, h2, _ = buf.dispatch(dev_bf16(x2), handle=handle)
    assert ti2 is None and tw2 is None and h2 is handle
    exp2 = oracle.dispatch(x2, ref["send_head"], np.array(off), W.E)
    for d in range(W.R):
        np.testing.assert_array_equal(host_bits(recv2[d]), exp2["recv_x"][off[d]:off[d + 1]])
    out2, cw2, _ = buf.combine(recv2, handle)
    es = oracle.combine(exp2["recv_x"], ref["send_head"], np.array(off), W.E, W.k, oracle.COMBINE_SUM)
    assert_close_bf16(host_bits(out2), es["out"])
    assert cw2 is None
    assert buf.check_errors() == 0


def test_buffer_worst_case_regions_fp8_and_pre_quantised():
    inp, x, topk, wts = _inputs()
    buf = Buffer(W.R, W.E, W.H, W.k, W.C)
    ref = oracle.layout(inp["topk_idx"], W.E, W.C)
    recv_x, _, _, _, handle, _ = buf.dispatch(x, topk_idx=topk, topk_weights=wts, fp8=True,
                                              num_worst_tokens=True)
    off = handle.row_offset
    assert off == [d * W.R * W.T for d in range(W.R + 1)]
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), W.E, x_kind=oracle.X_QUANTIZE)
    counts = ref["rank_prefix_matrix"][-1]
    for d in range(W.R):
        q, sc = recv_x[d]
        n = int(counts[d])
        np.testing.assert_array_equal(host_bits(q)[:n], exp["recv_x"][off[d]:off[d] + n])
        np.testing.assert_array_equal(host_bits(sc)[:n].view(np.uint32),
                                      exp["recv_x_scales"][off[d]:off[d] + n].view(np.uint32))
    # the pages' pre-quantised (fp8, scales) tuple, through the cached handle
    qx, sx = oracle.quantize_rows(inp["x"])
    recv_p, _, _, _, _, _ = buf.dispatch((torch.from_numpy(qx).cuda(), torch.from_numpy(sx).cuda()),
                                         handle=handle)
    for d in range(W.R):
        n = int(counts[d])
        np.testing.assert_array_equal(host_bits(recv_p[d][0])[:n], exp["recv_x"][off[d]:off[d] + n])
    assert buf.check_errors() == 0


@pytest.mark.parametrize("hook", [False, True])
def test_buffer_low_latency_calls(hook):
    w = workloads.Workload("apill", R=4, T=48, H=512, E=32, k=6, mask_p=0.05, nmax=64, seed=503)
    inp, x, topk, wts = _inputs(w)
    buf = Buffer(w.R, w.E, w.H, w.k)
    recv_x, count, handle, ev, recv_hook = buf.low_latency_dispatch(
        x, topk, w.nmax, use_fp8=False, async_finish=True, return_recv_hook=hook)
    if hook:
        assert recv_hook is not None
        recv_hook()
    ev.current_stream_wait()
    exp = oracle.ll_dispatch(inp["x"], inp["topk_idx"], w.E, w.nmax, False)
    np.testing.assert_array_equal(count.cpu().numpy(), exp["recv_expert_count"])
    np.testing.assert_array_equal(host_bits(handle.buf.slot), exp["slot"])
    out, _, comb_hook = buf.low_latency_combine(recv_x, topk, wts, handle, return_recv_hook=hook)
    if hook:
        comb_hook()
    ref = oracle.ll_combine(exp["recv_x"], inp["topk_idx"], inp["topk_weights"], exp["slot"], w.E, w.nmax)
    assert_close_bf16(host_bits(out), ref)
    assert buf.check_errors() == 0


def test_buffer_rejects_rows_in_separate_allocations():
    inp, x, topk, wts = _inputs()
    buf = Buffer(W.R, W.E, W.H, W.k, W.C)
    recv_x, _, _, _, handle, _ = buf.dispatch(x, topk_idx=topk, topk_weights=wts)
    copies = [t.clone() for t in recv_x]
    with pytest.raises(ValueError):
        buf.combine(copies, handle)
    with pytest.raises(ValueError):
        buf.dispatch(x, handle=handle, topk_idx=topk)
    assert ep.EP_OK == 0


def test_buffer_expert_major_blocks():
    inp, x, topk, wts = _inputs()
    buf = Buffer(W.R, W.E, W.H, W.k, W.C)
    recv_x, recv_src, recv_w, handle = buf.dispatch_expert_major(x, topk, wts)
    em = oracle.expert_layout(inp["topk_idx"], W.E)
    off = handle.row_offset
    exp = oracle.dispatch_expert_major(inp["x"], inp["topk_idx"], inp["topk_weights"], em["expert_rows"],
                                       np.array(off), W.E)
    E_loc = W.E // W.R
    for d in range(W.R):
        for e in range(E_loc):
            a, b = off[d] + int(em["expert_prefix"][d][e]), off[d] + int(em["expert_prefix"][d][e + 1])
            np.testing.assert_array_equal(host_bits(recv_x[d][e]), exp["recv_x"][a:b])
            np.testing.assert_array_equal(host_bits(recv_src[d][e]), exp["recv_src_idx"][a:b])
            np.testing.assert_array_equal(host_bits(recv_w[d][e]).view(np.uint32),
                                          exp["recv_weights"][a:b].view(np.uint32))
    y = recv_x[0][0]                                   # all rows start at the first block
    rows = torch.as_strided(y, (off[-1], W.H), y.stride())
    out = buf.combine_expert_major(rows, handle, topk, wts)
    ref = oracle.combine_expert_major(exp["recv_x"], inp["topk_idx"], inp["topk_weights"],
                                      em["expert_rows"], np.array(off), W.E, weighted=True)
    assert_close_bf16(host_bits(out), ref)
    assert buf.check_errors() == 0


def test_buffer_comm_stream_events_and_helpers():
    """The calls run on the Buffer's comm stream after a captured event; with
    async_finish the compute stream waits only through the returned event. Also the
    size hint and clean_low_latency_buffer helpers."""
    inp, x, topk, wts = _inputs()
    buf = Buffer(W.R, W.E, W.H, W.k, W.C)
    assert buf.get_comm_stream() != torch.cuda.current_stream()
    prev = Buffer.capture()
    recv_x, _, _, _, handle, ev = buf.dispatch(x, topk_idx=topk, topk_weights=wts, num_worst_tokens=True,
                                               previous_event=prev, async_finish=True,
                                               allocate_on_comm_stream=True)
    ev.current_stream_wait()
    ref = oracle.layout(inp["topk_idx"], W.E, W.C)
    off = handle.row_offset
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), W.E)
    counts = ref["rank_prefix_matrix"][-1]
    for d in range(W.R):
        n = int(counts[d])
        np.testing.assert_array_equal(host_bits(recv_x[d])[:n], exp["recv_x"][off[d]:off[d] + n])
    # a combine chained on the dispatch's event, without async_finish: the compute stream
    # waits for it before the copy to the host
    out, _, _ = buf.combine(recv_x, handle, previous_event=ev, weight_by=(topk, wts))
    ec = oracle.combine(exp["recv_x"], ref["send_head"], np.array(off), W.E, W.k,
                        oracle.COMBINE_WEIGHTED, inp["topk_idx"], inp["topk_weights"])
    assert_close_bf16(host_bits(out), ec["out"])

    hint = buf.get_buffer_size_hint(W.T, fp8=True, num_max_dispatch_tokens_per_rank=W.T)
    assert hint["recv_rows"] == W.R * W.R * W.T
    w = workloads.Workload("apic", R=4, T=16, H=256, E=16, k=4, mask_p=0.0, nmax=16, seed=504)
    _, xl, tl, _ = _inputs(w)
    bl = Buffer(w.R, w.E, w.H, w.k)
    _, count, lh, _, _ = bl.low_latency_dispatch(xl, tl, w.nmax, use_fp8=True)
    assert int(count.sum().item()) == w.R * w.T * w.k
    bl.clean_low_latency_buffer(lh)
    assert int(lh.buf.recv_expert_count.abs().sum().item()) == 0
    assert int(lh.buf.send_count.abs().sum().item()) == 0
    assert buf.check_errors() == 0 and bl.check_errors() == 0


def test_buffer_comm_stream_follows_a_delayed_compute_stream():
    """Without previous_event the comm stream waits for the work already issued on the
    compute stream: x is written there after a bounded busy kernel, and the dispatch on
    the comm stream still sees the final x."""
    inp, x, topk, wts = _inputs()
    buf = Buffer(W.R, W.E, W.H, W.k, W.C)
    x2 = torch.zeros_like(x)
    torch.cuda.synchronize()
    torch.cuda._sleep(20_000_000)          # keep the compute stream busy (bounded)
    x2.copy_(x)
    recv_x, _, _, _, handle, ev = buf.dispatch(x2, topk_idx=topk, num_worst_tokens=True,
                                               async_finish=True)
    ev.current_stream_wait()
    ref = oracle.layout(inp["topk_idx"], W.E, W.C)
    off = handle.row_offset
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), W.E)
    counts = ref["rank_prefix_matrix"][-1]
    for d in range(W.R):
        n = int(counts[d])
        np.testing.assert_array_equal(host_bits(recv_x[d])[:n], exp["recv_x"][off[d]:off[d] + n])
    assert buf.check_errors() == 0


def test_buffer_comm_pool_outputs_stay_reserved_for_compute_stream_readers():
    """allocate_on_comm_stream: the outputs come from the comm stream's pool and are read
    on the compute stream. A compute-stream reader, delayed by a bounded busy kernel, must
    still see the first call's outputs after the host has dropped them and later calls
    (waiting only on an older previous_event, not on the compute stream) allocated from
    the same pool and ran."""
    import dataclasses
    inp, _, topk, _ = _inputs()
    inp2 = workloads.make_workload(dataclasses.replace(W, seed=502), with_hidden=False)
    topk2 = torch.from_numpy(inp2["topk_idx"]).cuda()
    buf = Buffer(W.R, W.E, W.H, W.k, W.C)
    stale = buf.capture()
    torch.cuda.synchronize()
    _, _, ntpe, in_rank, ev = buf.get_dispatch_layout(topk, previous_event=stale, async_finish=True,
                                                      allocate_on_comm_stream=True)
    ev.current_stream_wait()
    torch.cuda._sleep(20_000_000)          # the reader below runs late (bounded busy kernel)
    seen_rank, seen_expert = in_rank.clone(), ntpe.clone()
    del ntpe, in_rank, ev
    # The Buffer keeps the latest layout, so the first call's buffers are released by the
    # second call and may be handed out again to the third.
    for _ in range(2):
        out = buf.get_dispatch_layout(topk2, previous_event=stale, async_finish=True,
                                      allocate_on_comm_stream=True)
        del out
    torch.cuda.synchronize()
    ref = oracle.layout(inp["topk_idx"], W.E, W.C)
    np.testing.assert_array_equal(seen_rank.cpu().numpy(), ref["is_token_in_rank"])
    np.testing.assert_array_equal(seen_expert.cpu().numpy(), ref["num_tokens_per_expert"])
    assert buf.check_errors() == 0
