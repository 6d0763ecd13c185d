"""Layout edge cases against the oracle, bit for bit: shapes past the largest benchmark
size, channel boundaries that do not divide the tokens, many small sources, channels
with no token, odd top-k (scalar id loads), rank counts that are not multiples of 4 or 8
(scalar stores), masked and bad ids, a second run over the first run's outputs, and
optional layout outputs. A ninth top-k column that is always masked must not change any
output."""
import ctypes

import numpy as np
import pytest
import torch

import combine_layout_02_gb300 as ep
from combine_layout_02_gb300.buffers import LayoutBuffers
import oracle
import workloads
from gpu_util import GpuRun

pytestmark = pytest.mark.gpu

W = workloads.Workload
CASES = {
    "r16_t4096": W("c1", R=16, T=4096, H=128, E=256, k=8, C=12, seed=601),
    "r8_t8200": W("c2", R=8, T=8200, H=128, E=256, k=8, C=12, seed=602),
    "ranges_cross_sources": W("c3", R=7, T=3001, H=128, E=28, k=6, C=5, mask_p=0.1, seed=603),
    "many_sources_per_cta": W("c4", R=64, T=3, H=128, E=128, k=4, C=2, seed=604),
    "empty_channels": W("c5", R=4, T=5, H=128, E=16, k=2, C=12, seed=605),
    "odd_k_r6": W("c6", R=6, T=777, H=128, E=36, k=7, C=4, routing="zipf", zipf_s=1.2, seed=606),
    "one_token": W("c7", R=1, T=1, H=128, E=4, k=3, C=3, seed=607),
    "r5_masked": W("c8", R=5, T=2049, H=128, E=40, k=5, C=12, mask_p=0.3, seed=608),
}


@pytest.mark.parametrize("name", list(CASES))
def test_layout_edge_cases_bit_exact(name):
    w = CASES[name]
    inp = workloads.make_workload(w, with_hidden=False)
    run = GpuRun(w.R, w.T, w.H, w.E, w.k, w.C, inp)
    ref = oracle.layout(inp["topk_idx"], w.E, w.C)
    for _ in range(2):                       # a second run over the first one's outputs
        got = run.layout()
        for key, arr in got.items():
            np.testing.assert_array_equal(arr, ref[key], err_msg=key)
    assert run.flags() == 0


def test_bad_ids_flagged_and_skipped():
    w = W("bad", R=4, T=600, H=128, E=16, k=4, C=3, seed=609)
    inp = workloads.make_workload(w, with_hidden=False)
    topk = inp["topk_idx"].copy()
    topk[1, 5, 2] = 16          # == E
    topk[3, 599, 0] = -5
    for extra in (0, 1):        # k = 4, and k = 5 with a masked fifth column
        t = np.concatenate([topk, np.full((w.R, w.T, extra), -1, np.int64)], axis=2)
        run = GpuRun(w.R, w.T, w.H, w.E, w.k + extra, w.C, dict(inp, topk_idx=t))
        got = run.layout()
        ref = oracle.layout(t, w.E, w.C)
        assert ref["bad_entries"] == 2
        for key, arr in got.items():
            np.testing.assert_array_equal(arr, ref[key], err_msg=key)
        assert run.flags() == ep.EP_DEVERR_BAD_EXPERT


def test_masked_extra_column_changes_nothing():
    w = workloads.CONFIGS["dsv3"]
    inp = workloads.make_workload(w, with_hidden=False)
    outs = []
    for extra in (0, 1):
        t = np.concatenate([inp["topk_idx"], np.full((w.R, w.T, extra), -1, np.int64)], axis=2)
        run = GpuRun(w.R, w.T, w.H, w.E, w.k + extra, w.C, dict(inp, topk_idx=t))
        outs.append(run.layout())
        assert run.flags() == 0
    for key in outs[0]:
        np.testing.assert_array_equal(outs[0][key], outs[1][key], err_msg=key)


def test_layout_outputs_optional():
    """The layout struct's fields may be NULL (and the struct itself): the handle is
    still complete."""
    w = CASES["ranges_cross_sources"]
    inp = workloads.make_workload(w, with_hidden=False)
    ref = oracle.layout(inp["topk_idx"], w.E, w.C)
    sh = ep.make_shape(w.R, w.T, w.H, w.E, w.k, w.C)
    topk = torch.from_numpy(inp["topk_idx"]).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    launch = ep.make_launch(error_flags=err)
    for with_struct in (False, True):
        lb = LayoutBuffers(sh)
        lay = ep.ep_layout(None, None, None, None) if with_struct else None
        ep.ep_get_layout(sh, topk, lay, lb.handle(), lb.workspace, launch)
        torch.cuda.synchronize()
        for key in ("rank_prefix_matrix", "channel_prefix_matrix", "recv_channel_prefix_matrix",
                    "send_head", "num_recv_tokens_per_expert", "is_token_in_rank"):
            np.testing.assert_array_equal(getattr(lb, key).cpu().numpy(), ref[key], err_msg=key)
    assert int(err.item()) == 0
