"""Failure detection on the GPU without a fault: the library's bounded device waits (the
bulk-copy dispatch waits for each row load on a shared-memory barrier) give up after their
time limit and report EP_DEVERR_TIMEOUT, and the context stays usable afterwards."""
import numpy as np
import pytest
import torch

import combine_layout_02_gb300 as ep
import oracle
from gpu_util import GpuRun, compact_offsets, host_bits
import workloads

pytestmark = pytest.mark.gpu


def test_wait_that_never_completes_gives_up_and_reports():
    src = torch.zeros(4, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_selftest_wait_timeout(src, 200, elapsed, ep.make_launch(error_flags=err))
    torch.cuda.synchronize()
    assert int(err.item()) == ep.EP_DEVERR_TIMEOUT
    assert 200_000 <= int(elapsed.item()) < 2_000_000           # µs: gave up after the limit
    # the context is still usable: a dispatch right after is bit-exact and flag-free
    w = workloads.CONFIGS["tiny"]
    inp = workloads.make_workload(w)
    run = GpuRun(w.R, w.T, w.H, w.E, w.k, w.C, inp)
    ref = oracle.layout(inp["topk_idx"], w.E, w.C)
    run.layout()
    off = compact_offsets(ref["rank_prefix_matrix"])
    rb = run.dispatch(off)
    exp = oracle.dispatch(inp["x"], ref["send_head"], np.array(off), w.E, fill_x=0xA5A5)
    np.testing.assert_array_equal(host_bits(rb.recv_x), exp["recv_x"])
    assert run.flags() == 0


def test_selftest_argument_checks():
    src = torch.zeros(8, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = ep.lib()
    import ctypes
    launch = ep.make_launch(error_flags=err)
    for ptr, ms in ((src.data_ptr() + 4, 10), (src.data_ptr(), 0), (src.data_ptr(), 20000)):
        assert L.ep_selftest_wait_timeout(ctypes.c_void_p(ptr), ms, None, ctypes.byref(launch)) == \
            ep.EP_ERR_INVALID_ARG
    assert int(err.item()) == 0
