"""Pins for the oracle's expert-major packed receive layout (rows of each destination
grouped by local expert, then source rank, then token): a hand-worked example,
exhaustive tiny tables against a sorting characterisation, bincount / cumsum for the
per-expert prefix, and dispatch / combine round trips."""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint32) << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def test_hand_example():
    with open(os.path.join(GOLDEN, "layout_hand_example.json")) as f:
        g = json.load(f)
    r = oracle.expert_layout(np.array(g["topk_idx"], np.int64), g["E"])
    np.testing.assert_array_equal(r["expert_rows"], np.array(g["expert_rows"]))
    np.testing.assert_array_equal(r["expert_prefix"], np.array(g["expert_prefix"]))


def check_expert_layout(topk, E, res):
    R, T, k = topk.shape
    E_loc = E // R
    rows, pre = res["expert_rows"], res["expert_prefix"]
    valid = (topk >= 0) & (topk < E)
    counts = np.bincount(topk[valid], minlength=E).reshape(R, E_loc)
    np.testing.assert_array_equal(pre[:, 0], 0)
    np.testing.assert_array_equal(np.diff(pre, axis=1), counts)
    assert np.all(rows[~valid] == -1)
    s_i, t_i, j_i = np.nonzero(valid)
    e = topk[s_i, t_i, j_i]
    d, el = e // E_loc, e % E_loc
    r = rows[s_i, t_i, j_i]
    for dd in range(R):
        m = d == dd
        # the entries of d, sorted by (local expert, source, token, entry), are rows 0..M_d-1
        order = np.lexsort((j_i[m], t_i[m], s_i[m], el[m]))
        np.testing.assert_array_equal(r[m][order], np.arange(m.sum()))


@pytest.mark.parametrize("T,k", [(2, 1), (1, 2), (3, 1)])
def test_exhaustive_tiny_tables(T, k):
    R, E = 2, 4
    for vals in itertools.product(range(-1, E), repeat=R * T * k):
        topk = np.array(vals, np.int64).reshape(R, T, k)
        check_expert_layout(topk, E, oracle.expert_layout(topk, E))


@pytest.mark.parametrize("routing", ["uniform", "zipf", "group"])
def test_invariants_on_workload_shapes(routing):
    w = workloads.Workload("em", R=8, T=200, H=128, E=64, k=6, routing=routing, zipf_s=1.2,
                           groups=8, topk_groups=4, mask_p=0.05, seed=51)
    topk = workloads.make_workload(w, with_hidden=False)["topk_idx"]
    res = oracle.expert_layout(topk, w.E)
    assert res["bad_entries"] == 0
    check_expert_layout(topk, w.E, res)
    lay = oracle.layout(topk, w.E)
    np.testing.assert_array_equal(res["expert_prefix"][:, -1], lay["num_recv_tokens_per_expert"].sum(1))


def _case(seed=52, R=4, T=60, H=256, E=16, k=4, mask_p=0.1):
    w = workloads.Workload("emd", R=R, T=T, H=H, E=E, k=k, mask_p=mask_p, seed=seed)
    inp = workloads.make_workload(w)
    res = oracle.expert_layout(inp["topk_idx"], E)
    off = np.concatenate([[0], np.cumsum(res["expert_prefix"][:, -1])]).astype(np.int64)
    return w, inp, res, off


def test_dispatch_expert_major_rows():
    w, inp, res, off = _case()
    E_loc = w.E // w.R
    d = oracle.dispatch_expert_major(inp["x"], inp["topk_idx"], inp["topk_weights"],
                                     res["expert_rows"], off, w.E)
    assert d["bad_rows"] == 0
    written = np.zeros(int(off[-1]), bool)
    for s in range(w.R):
        for t in range(w.T):
            for j in range(w.k):
                e = inp["topk_idx"][s, t, j]
                if e < 0:
                    continue
                row = off[e // E_loc] + res["expert_rows"][s, t, j]
                written[row] = True
                np.testing.assert_array_equal(d["recv_x"][row], inp["x"][s, t])
                assert d["recv_src_idx"][row] == t
                assert d["recv_weights"][row] == inp["topk_weights"][s, t, j]
    assert written.all()                                  # the packing has no gaps
    q = oracle.dispatch_expert_major(inp["x"], inp["topk_idx"], inp["topk_weights"],
                                     res["expert_rows"], off, w.E, quantize=True)
    qr, sc = oracle.quantize_rows(inp["x"])
    s_i, t_i, j_i = np.nonzero(inp["topk_idx"] >= 0)
    rr = off[inp["topk_idx"][s_i, t_i, j_i] // E_loc] + res["expert_rows"][s_i, t_i, j_i]
    np.testing.assert_array_equal(q["recv_x"][rr], qr[s_i, t_i])
    np.testing.assert_array_equal(q["recv_x_scales"][rr], sc[s_i, t_i])


def test_combine_expert_major_round_trip_and_fp64_reference():
    w, inp, res, off = _case(seed=53, R=8, T=40, E=64, k=8, mask_p=0.05)
    E_loc = w.E // w.R
    d = oracle.dispatch_expert_major(inp["x"], inp["topk_idx"], inp["topk_weights"],
                                     res["expert_rows"], off, w.E)
    out = oracle.combine_expert_major(d["recv_x"], inp["topk_idx"], inp["topk_weights"],
                                      res["expert_rows"], off, w.E)
    xf = _bf16_to_f64(inp["x"]) * inp["topk_weights"].astype(np.float64).sum(-1)[..., None]
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(xf), 2.0 ** -126))) - 7)
    assert np.all(np.abs(_bf16_to_f64(out) - xf) <= ulp)
    rng = np.random.default_rng(54)
    y = (rng.standard_normal((int(off[-1]), w.H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    out2 = oracle.combine_expert_major(y, inp["topk_idx"], inp["topk_weights"], res["expert_rows"],
                                       off, w.E)
    topk = inp["topk_idx"]
    valid = topk >= 0
    rows = np.where(valid, off[np.where(valid, topk // E_loc, 0)] + res["expert_rows"], 0)
    ref = np.einsum("rtk,rtkh->rth", np.where(valid, inp["topk_weights"], 0).astype(np.float64),
                    _bf16_to_f64(y)[rows])
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 8)
    assert np.all(np.abs(_bf16_to_f64(out2) - ref) <= half_ulp * (1 + 1e-9))
