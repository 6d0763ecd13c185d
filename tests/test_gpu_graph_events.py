"""Ordering, CUDA-graph capture and backward identities through the C ABI.

- Event ordering ("How DeepEP Achieves Communication-Computation Overlapping with
  EventOverlap", "Propagation Through EP Operations"): a call given wait_event
  (previous_event) sees everything recorded before that event on another stream, and
  its record_event (async_finish) orders a consumer stream after the call.
- CUDA graphs ("DeepEP" README: the low-latency calls are compatible with CUDA graphs):
  the normal step (layout -> dispatch -> combine) and the low-latency step (send ->
  receive -> combine) captured once and replayed on fresh inputs give the eager results,
  with no buffer state to restore between replays.
- Backward identities ("DeepEP" README, dispatch_backward / combine_backward): the
  backward of dispatch is a combine (sum over ranks) and the backward of combine is a
  dispatch with the handle, i.e. <dispatch(x), y> == <x, combine_sum(y)> exactly on
  small-integer data, and the weight gradients are reduced by combine.
"""
import numpy as np
import pytest
import torch

import combine_layout_02_gb300 as ep
from combine_layout_02_gb300.buffers import LayoutBuffers, LLBuffers, RecvBuffers, new_event
import oracle
import workloads
from gpu_util import GpuRun, assert_close_bf16, bf16_to_f64, compact_offsets, dev_bf16, host_bits, assert_weight_sums_close

pytestmark = pytest.mark.gpu

W = workloads.Workload("ev", R=8, T=512, H=1024, E=64, k=6, C=12, seed=201)


def test_wait_event_orders_producer_before_dispatch():
    inp = workloads.make_workload(W)
    run = GpuRun(W.R, W.T, W.H, W.E, W.k, W.C, inp)
    ref = oracle.layout(inp["topk_idx"], W.E, W.C)
    run.layout()
    torch.cuda.synchronize()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rng = np.random.default_rng(202)
    x_new = workloads.make_hidden(rng, W.R, W.T, W.H)
    x_new_d = dev_bf16(x_new)
    x_buf = torch.zeros_like(run.x)
    producer, consumer = torch.cuda.Stream(), torch.cuda.Stream()
    rb = RecvBuffers(off[-1], W.H, W.k, with_topk=False)
    torch.cuda.synchronize()
    with torch.cuda.stream(producer):
        torch.cuda._sleep(20_000_000)                 # keep the producer busy (bounded)
        x_buf.copy_(x_new_d)
        prev = new_event(producer)                    # previous_event
    done = new_event(consumer)
    launch = ep.make_launch(consumer, wait_event=prev, record_event=done)
    ep.ep_dispatch(run.sh, x_buf, ep.EP_BF16, None, ep.EP_BF16, None, None,
                   run.lb.handle(rb.recv_src_idx), rb.recv_x, None, None, None, rb.recv_src_idx,
                   off, launch)
    torch.cuda.current_stream().wait_event(done)      # current_stream_wait on async_finish
    got = host_bits(rb.recv_x)
    exp = oracle.dispatch(x_new, ref["send_head"], np.array(off), W.E)["recv_x"]
    np.testing.assert_array_equal(got, exp)


def test_record_event_orders_consumer_after_combine():
    inp = workloads.make_workload(W)
    run = GpuRun(W.R, W.T, W.H, W.E, W.k, W.C, inp)
    ref = oracle.layout(inp["topk_idx"], W.E, W.C)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rb = run.dispatch(off)
    torch.cuda.synchronize()
    comm = torch.cuda.Stream()
    out = torch.empty((W.R, W.T, W.H), dtype=torch.bfloat16, device="cuda")
    done = new_event(comm)
    with torch.cuda.stream(comm):
        torch.cuda._sleep(20_000_000)
    ep.ep_combine(run.sh, rb.recv_x, off, run.lb.handle(), ep.EP_COMBINE_WEIGHTED, run.topk, run.wts,
                  None, out, None, ep.make_launch(comm, record_event=done))
    torch.cuda.current_stream().wait_event(done)
    copy = out.clone()                                # ordered after the combine by the event
    exp = oracle.combine(host_bits(rb.recv_x), ref["send_head"], np.array(off), W.E, W.k,
                         oracle.COMBINE_WEIGHTED, inp["topk_idx"], inp["topk_weights"])["out"]
    assert_close_bf16(host_bits(copy), exp)


def test_normal_step_cuda_graph_replay():
    inp = workloads.make_workload(W)
    R, T, H, E, k, C = W.R, W.T, W.H, W.E, W.k, W.C
    sh = ep.make_shape(R, T, H, E, k, C)
    off = [int(v) for v in workloads.worst_case_row_offsets(R, T)]
    topk = torch.from_numpy(inp["topk_idx"]).cuda()
    wts = torch.from_numpy(inp["topk_weights"]).cuda()
    x = dev_bf16(inp["x"])
    lb = LayoutBuffers(sh)
    rb = RecvBuffers(off[-1], H, k)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    handle = lb.handle(rb.recv_src_idx)

    def step(stream):
        launch = ep.make_launch(stream, error_flags=err)
        ep.ep_get_layout(sh, topk, lb.layout(), handle, lb.workspace, launch)
        ep.ep_dispatch(sh, x, ep.EP_BF16, None, ep.EP_BF16, topk, wts, handle, rb.recv_x, None,
                       rb.recv_topk_idx, rb.recv_topk_weights, rb.recv_src_idx, off, launch)
        ep.ep_combine(sh, rb.recv_x, off, handle, ep.EP_COMBINE_WEIGHTED, topk, wts, None, out,
                      None, launch)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)                                       # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    for it in range(2):
        w2 = workloads.Workload("ev2", R=R, T=T, H=H, E=E, k=k, C=C, seed=300 + it)
        inp2 = workloads.make_workload(w2)
        x.copy_(dev_bf16(inp2["x"]))
        topk.copy_(torch.from_numpy(inp2["topk_idx"]))
        wts.copy_(torch.from_numpy(inp2["topk_weights"]))
        g.replay()
        torch.cuda.synchronize()
        lay = oracle.layout(inp2["topk_idx"], E, C)
        for key, t in lb.as_dict().items():
            np.testing.assert_array_equal(t.cpu().numpy(), lay[key], err_msg=key)
        sub = {kk: np.ascontiguousarray(v[:, :64]) for kk, v in inp2.items()}
        slay = oracle.layout(sub["topk_idx"], E, C)
        soff = np.concatenate([[0], np.cumsum(slay["rank_prefix_matrix"][-1])]).astype(np.int64)
        sd = oracle.dispatch(sub["x"], slay["send_head"], soff, E)
        cexp = oracle.combine(sd["recv_x"], slay["send_head"], soff, E, k, oracle.COMBINE_WEIGHTED,
                              sub["topk_idx"], sub["topk_weights"])["out"]
        assert_close_bf16(host_bits(out[:, :64]), cexp)
    assert int(err.item()) == 0


@pytest.mark.parametrize("packed", [False, True])
def test_low_latency_step_cuda_graph_replay(packed):
    w = workloads.Workload("llg", R=8, T=96, H=1024, E=64, k=8, nmax=128, mask_p=0.05, seed=210)
    inp = workloads.make_workload(w)
    sh = ep.make_shape(w.R, w.T, w.H, w.E, w.k, 1, nmax=w.nmax)
    topk = torch.from_numpy(inp["topk_idx"]).cuda()
    wts = torch.from_numpy(inp["topk_weights"]).cuda()
    x = dev_bf16(inp["x"])
    buf = LLBuffers(sh, use_fp8=True, packed=packed)
    ybuf = LLBuffers(sh, use_fp8=False, packed=packed)
    out = torch.empty((w.R, w.T, w.H), dtype=torch.bfloat16, device="cuda")

    def step(stream):
        launch = ep.make_launch(stream)
        ep.ep_ll_dispatch(sh, x, topk, True, ep.EP_PHASE_SEND, buf.struct(), launch)
        ep.ep_ll_dispatch(sh, x, topk, True, ep.EP_PHASE_RECV, buf.struct(), launch)
        ep.ep_ll_dispatch(sh, x, topk, False, ep.EP_PHASE_BOTH, ybuf.struct(), launch)
        ep.ep_ll_combine(sh, ybuf.recv_x, topk, wts, ybuf.struct(), ep.EP_PHASE_RECV, out, launch)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    for it in range(2):
        w2 = workloads.Workload("llg2", R=w.R, T=w.T, H=w.H, E=w.E, k=w.k, nmax=w.nmax,
                                mask_p=0.05, seed=400 + it)
        inp2 = workloads.make_workload(w2)
        x.copy_(dev_bf16(inp2["x"]))
        topk.copy_(torch.from_numpy(inp2["topk_idx"]))
        wts.copy_(torch.from_numpy(inp2["topk_weights"]))
        g.replay()
        torch.cuda.synchronize()
        exp = oracle.ll_dispatch(inp2["x"], inp2["topk_idx"], w.E, w.nmax, True, packed=packed)
        for key in ("slot", "recv_expert_count", "layout_range"):
            np.testing.assert_array_equal(host_bits(getattr(buf, key)), exp[key], err_msg=key)
        filled = exp["src_info"] != -7
        np.testing.assert_array_equal(host_bits(buf.recv_x)[filled], exp["recv_x"][filled])
        e16 = oracle.ll_dispatch(inp2["x"], inp2["topk_idx"], w.E, w.nmax, False, packed=packed)
        cexp = oracle.ll_combine(e16["recv_x"], inp2["topk_idx"], inp2["topk_weights"], e16["slot"],
                                 w.E, w.nmax)
        assert_close_bf16(host_bits(out), cexp)


def test_backward_identities_exact_on_integer_data():
    """dispatch_backward = combine (sum) and combine_backward = dispatch(handle): the two
    are adjoint, exactly, when every value and partial sum is a small integer."""
    inp = workloads.make_workload(W)
    run = GpuRun(W.R, W.T, W.H, W.E, W.k, W.C, inp)
    ref = oracle.layout(inp["topk_idx"], W.E, W.C)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rng = np.random.default_rng(204)
    xi = rng.integers(-4, 5, (W.R, W.T, W.H)).astype(np.float32)
    yi = rng.integers(-4, 5, (off[-1], W.H)).astype(np.float32)
    xd = torch.from_numpy(xi).to(torch.bfloat16).cuda()
    yd = torch.from_numpy(yi).to(torch.bfloat16).cuda()
    fwd = run.dispatch(off, with_topk=False, x=xd)                     # forward dispatch
    cy, _ = run.combine(yd, off, ep.EP_COMBINE_SUM)                     # dispatch_backward
    lhs = np.sum(bf16_to_f64(host_bits(fwd.recv_x)) * yi.astype(np.float64))
    rhs = np.sum(xi.astype(np.float64) * bf16_to_f64(host_bits(cy)))
    assert lhs == rhs
    # combine_backward: gradient of the summed output wrt the received rows is the
    # dispatch of the output gradient through the same handle
    g = rng.integers(-4, 5, (W.R, W.T, W.H)).astype(np.float32)
    gd = torch.from_numpy(g).to(torch.bfloat16).cuda()
    back = run.dispatch(off, with_topk=False, x=gd)
    lhs2 = np.sum(bf16_to_f64(host_bits(cy)) * g.astype(np.float64))
    rhs2 = np.sum(yi.astype(np.float64) * bf16_to_f64(host_bits(back.recv_x)))
    assert lhs2 == rhs2
    # weight gradients: combine reduces grad_recv_topk_weights back to token order
    gw = rng.standard_normal((off[-1], W.k)).astype(np.float32)
    _, cw = run.combine(yd, off, ep.EP_COMBINE_SUM, recv_topk_weights=torch.from_numpy(gw).cuda())
    exp = oracle.combine(yd.view(torch.int16).cpu().numpy().view(np.uint16), ref["send_head"],
                         np.array(off), W.E, W.k, recv_topk_weights=gw)["combined_topk_weights"]
    assert_weight_sums_close(cw.cpu().numpy(), exp, gw, ref["send_head"], off)


def test_event_overlap_helpers_order_like_the_raw_events():
    """capture() on the producer stream as previous_event, completion_event() as
    async_finish, and EventOverlap.current_stream_wait / the `with` block on the consumer
    side give the same ordering as raw events."""
    from combine_layout_02_gb300.buffers import EventOverlap, capture, completion_event
    inp = workloads.make_workload(W)
    run = GpuRun(W.R, W.T, W.H, W.E, W.k, W.C, inp)
    ref = oracle.layout(inp["topk_idx"], W.E, W.C)
    run.layout()
    torch.cuda.synchronize()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rng = np.random.default_rng(203)
    x_new = workloads.make_hidden(rng, W.R, W.T, W.H)
    x_new_d = dev_bf16(x_new)
    x_buf = torch.zeros_like(run.x)
    producer, comm = torch.cuda.Stream(), torch.cuda.Stream()
    rb = RecvBuffers(off[-1], W.H, W.k, with_topk=False)
    torch.cuda.synchronize()
    with torch.cuda.stream(producer):
        torch.cuda._sleep(20_000_000)
        x_buf.copy_(x_new_d)
        previous = capture(producer)
    finish = completion_event(comm)
    launch = ep.make_launch(comm, wait_event=previous.event, record_event=finish.event)
    ep.ep_dispatch(run.sh, x_buf, ep.EP_BF16, None, ep.EP_BF16, None, None,
                   run.lb.handle(rb.recv_src_idx), rb.recv_x, None, None, None, rb.recv_src_idx,
                   off, launch)
    with EventOverlap(finish.event, extra_tensors=(rb.recv_x,)):
        pass                                         # the current stream waits on exit
    got = host_bits(rb.recv_x)
    exp = oracle.dispatch(x_new, ref["send_head"], np.array(off), W.E)["recv_x"]
    np.testing.assert_array_equal(got, exp)
