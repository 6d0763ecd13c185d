"""Pins for the oracle's low-latency dispatch / combine (fixed per-expert slots).

Checks: every valid (token, expert) pair lands in exactly one slot inside its source's
sub-slot, in token order; counts equal bincounts; src_info inverts slot; rows equal the
source rows (bf16) or the pinned quantiser's rows (FP8) and the normal dispatch's rows;
weighted combine of identity experts returns x within bf16 rounding; an fp64 numpy
reference; capacity overflow is reported.
"""
import numpy as np
import pytest

import oracle
import workloads


def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint32) << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def _case(R=4, T=20, H=256, E=16, k=4, nmax=24, mask_p=0.1, seed=41):
    w = workloads.Workload("ll", R=R, T=T, H=H, E=E, k=k, mask_p=mask_p, nmax=nmax, seed=seed)
    return w, workloads.make_workload(w)


@pytest.mark.parametrize("use_fp8", [False, True])
def test_ll_dispatch_slots_counts_rows(use_fp8):
    w, inp = _case()
    R, T, E, k, nmax = w.R, w.T, w.E, w.k, w.nmax
    E_loc = E // R
    topk = inp["topk_idx"]
    res = oracle.ll_dispatch(inp["x"], topk, E, nmax, use_fp8)
    assert res["bad_entries"] == 0
    q, sc = oracle.quantize_rows(inp["x"])
    seen = set()
    for s in range(R):
        cnt = np.bincount(topk[s][topk[s] >= 0], minlength=E)
        for e in range(E):
            d, el = divmod(e, E_loc)
            np.testing.assert_array_equal(res["layout_range"][d, el, s], [s * nmax, cnt[e]])
        for t in range(T):
            for j in range(k):
                e = topk[s, t, j]
                pos = res["slot"][s, t, j]
                if e < 0:
                    assert pos == -1
                    continue
                d, el = divmod(int(e), E_loc)
                # in token order inside the source's sub-slot
                earlier = int(np.any(topk[s, :t] == e, axis=-1).sum())
                assert pos == s * nmax + earlier
                key = (d, el, int(pos))
                assert key not in seen
                seen.add(key)
                assert res["src_info"][d, el, pos] == t
                if use_fp8:
                    np.testing.assert_array_equal(res["recv_x"][d, el, pos], q[s, t])
                    np.testing.assert_array_equal(res["recv_x_scales"][d, el, pos], sc[s, t])
                else:
                    np.testing.assert_array_equal(res["recv_x"][d, el, pos], inp["x"][s, t])
    assert len(seen) == (topk >= 0).sum()
    np.testing.assert_array_equal(res["recv_expert_count"].reshape(-1),
                                  np.bincount(topk[topk >= 0], minlength=E))
    # untouched slots keep the canary
    touched = np.zeros(res["src_info"].shape, bool)
    for d, el, pos in seen:
        touched[d, el, pos] = True
    assert np.all(res["src_info"][~touched] == -7)


def test_ll_rows_equal_normal_dispatch_rows():
    w, inp = _case(seed=42)
    E_loc = w.E // w.R
    ll = oracle.ll_dispatch(inp["x"], inp["topk_idx"], w.E, w.nmax, False)
    lay = oracle.layout(inp["topk_idx"], w.E, 3)
    off = np.concatenate([[0], np.cumsum(lay["rank_prefix_matrix"][-1])]).astype(np.int64)
    nd = oracle.dispatch(inp["x"], lay["send_head"], off, w.E)
    for s in range(w.R):
        for t in range(w.T):
            for j in range(w.k):
                e = inp["topk_idx"][s, t, j]
                if e < 0:
                    continue
                d, el = divmod(int(e), E_loc)
                row = off[d] + lay["send_head"][s, t, d]
                np.testing.assert_array_equal(ll["recv_x"][d, el, ll["slot"][s, t, j]],
                                              nd["recv_x"][row])


def test_ll_combine_identity_round_trip_and_fp64_reference():
    w, inp = _case(R=8, T=32, H=256, E=64, k=8, nmax=40, mask_p=0.05, seed=43)
    E_loc = w.E // w.R
    ll = oracle.ll_dispatch(inp["x"], inp["topk_idx"], w.E, w.nmax, False)
    out = oracle.ll_combine(ll["recv_x"], inp["topk_idx"], inp["topk_weights"], ll["slot"],
                            w.E, w.nmax)
    xf, of = _bf16_to_f64(inp["x"]), _bf16_to_f64(out)
    wsum = inp["topk_weights"].astype(np.float64).sum(-1)
    # weights are a softmax over the valid entries: they sum to 1 (0 if all masked)
    ref = xf * wsum[..., None]
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
    assert np.all(np.abs(of - ref) <= ulp)
    # general expert outputs vs an fp64 numpy gather
    rng = np.random.default_rng(44)
    y = ((rng.standard_normal(ll["recv_x"].shape).astype(np.float32).view(np.uint32) >> 16)
         .astype(np.uint16))                            # any bf16 bit patterns will do
    out2 = oracle.ll_combine(y, inp["topk_idx"], inp["topk_weights"], ll["slot"], w.E, w.nmax)
    yf = _bf16_to_f64(y)
    topk = inp["topk_idx"]
    valid = topk >= 0
    d = np.where(valid, topk // E_loc, 0)
    el = np.where(valid, topk % E_loc, 0)
    pos = np.where(valid, ll["slot"], 0)
    g = yf[d, el, pos]                                   # [R, T, k, H]
    ref2 = np.einsum("rtk,rtkh->rth", np.where(valid, inp["topk_weights"], 0).astype(np.float64), g)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref2), 2.0 ** -126))) - 8)
    assert np.all(np.abs(_bf16_to_f64(out2) - ref2) <= half_ulp * (1 + 1e-9))
    # fully masked token -> +0
    topk3 = topk.copy()
    topk3[0, 0, :] = -1
    ll3 = oracle.ll_dispatch(inp["x"], topk3, w.E, w.nmax, False)
    out3 = oracle.ll_combine(ll3["recv_x"], topk3, inp["topk_weights"], ll3["slot"], w.E, w.nmax)
    assert np.all(out3[0, 0] == 0)


def test_ll_capacity_overflow_is_reported():
    # 10 tokens of one source all pick expert 0, slot capacity 4
    topk = np.full((2, 10, 1), 0, np.int64)
    x = np.zeros((2, 10, 128), np.uint16)
    res = oracle.ll_dispatch(x, topk, 4, 4, False)
    assert res["bad_entries"] == 2 * 6
    assert np.all(res["slot"][:, 4:] == -1)
    np.testing.assert_array_equal(res["recv_expert_count"][0], [8, 0])


def _golden_ll():
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "ll_hand_example.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("packed", [False, True])
def test_ll_hand_example(packed):
    g = _golden_ll()
    R, T, E, k, nmax = g["R"], g["T"], g["E"], g["k"], g["nmax"]
    topk = np.array(g["topk_idx"], np.int64)
    x = (np.arange(R * T * 128, dtype=np.uint16) % 7919).reshape(R, T, 128)
    res = oracle.ll_dispatch(x, topk, E, nmax, False, packed=packed)
    pre = "packed_" if packed else ""
    assert res["bad_entries"] == 0
    np.testing.assert_array_equal(res["slot"], g[pre + "slot"])
    np.testing.assert_array_equal(res["layout_range"], g[pre + "layout_range"])
    np.testing.assert_array_equal(res["recv_expert_count"], g["recv_expert_count"])
    E_loc = E // R
    for e in range(E):
        d, el = divmod(e, E_loc)
        want = g[pre + "src_info"][f"e{e}"]
        items = enumerate(want) if packed else ((int(p), t) for p, t in want.items())
        for pos, t in items:
            assert res["src_info"][d, el, pos] == t


def test_ll_packed_is_the_gapless_compaction_of_the_slot_layout():
    """The packed layout, checked three independent ways: (1) each expert's region is
    the concatenation over sources of the slot layout's filled sub-slots; (2) a source's
    start is the running sum of the earlier sources' counts (numpy cumsum); (3) the
    position of each entry is its rank among the expert's entries sorted by (source,
    token), which is also the expert-major placement's row minus the expert's start."""
    w, inp = _case(R=4, T=24, H=256, E=16, k=4, nmax=30, mask_p=0.1, seed=45)
    R, T, E, k, nmax = w.R, w.T, w.E, w.k, w.nmax
    E_loc = E // R
    topk = inp["topk_idx"]
    for use_fp8 in (False, True):
        sl = oracle.ll_dispatch(inp["x"], topk, E, nmax, use_fp8)
        pk = oracle.ll_dispatch(inp["x"], topk, E, nmax, use_fp8, packed=True)
        assert pk["bad_entries"] == 0
        np.testing.assert_array_equal(pk["recv_expert_count"], sl["recv_expert_count"])
        cnt = sl["layout_range"][..., 1]                       # [R][E_loc][R]
        np.testing.assert_array_equal(pk["layout_range"][..., 1], cnt)
        starts = np.concatenate([np.zeros(cnt.shape[:-1] + (1,), cnt.dtype),
                                 np.cumsum(cnt, -1)[..., :-1]], -1)
        np.testing.assert_array_equal(pk["layout_range"][..., 0], starts)
        for d in range(R):
            for el in range(E_loc):
                n = int(pk["recv_expert_count"][d, el])
                keys = ["recv_x", "src_info"] + (["recv_x_scales"] if use_fp8 else [])
                for key in keys:
                    parts = [sl[key][d, el, s * nmax: s * nmax + cnt[d, el, s]] for s in range(R)]
                    np.testing.assert_array_equal(pk[key][d, el, :n], np.concatenate(parts))
    ranks = {}
    for e in range(E):
        entries = sorted((s, t) for s in range(R) for t in range(T) if e in topk[s, t])
        for i, st in enumerate(entries):
            ranks[(e,) + st] = i
    em = oracle.expert_layout(topk, E)
    for s in range(R):
        for t in range(T):
            for j in range(k):
                e = int(topk[s, t, j])
                if e < 0:
                    assert pk["slot"][s, t, j] == -1
                    continue
                d, el = divmod(e, E_loc)
                assert pk["slot"][s, t, j] == ranks[(e, s, t)]
                assert pk["slot"][s, t, j] == em["expert_rows"][s, t, j] - em["expert_prefix"][d, el]


def test_ll_packed_combine_equals_slot_layout_combine():
    w, inp = _case(R=4, T=16, H=256, E=16, k=4, nmax=16, mask_p=0.1, seed=46)
    E_loc = w.E // w.R
    sl = oracle.ll_dispatch(inp["x"], inp["topk_idx"], w.E, w.nmax, False)
    pk = oracle.ll_dispatch(inp["x"], inp["topk_idx"], w.E, w.nmax, False, packed=True)
    # the same expert outputs, placed by each layout's slots
    rng = np.random.default_rng(47)
    ys = np.zeros_like(sl["recv_x"])
    yp = np.zeros_like(pk["recv_x"])
    topk = inp["topk_idx"]
    for s, t, j in zip(*np.nonzero(topk >= 0)):
        d, el = divmod(int(topk[s, t, j]), E_loc)
        row = (rng.standard_normal(w.H).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        ys[d, el, sl["slot"][s, t, j]] = row
        yp[d, el, pk["slot"][s, t, j]] = row
    a = oracle.ll_combine(ys, topk, inp["topk_weights"], sl["slot"], w.E, w.nmax)
    b = oracle.ll_combine(yp, topk, inp["topk_weights"], pk["slot"], w.E, w.nmax)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("packed", [False, True])
def test_ll_repeated_experts_take_one_slot_per_entry_in_entry_order(packed):
    """A token may name an expert twice: each entry takes its own slot, ranked by entry
    order (token, then k) among the source's entries with that expert (brute force)."""
    rng = np.random.default_rng(57)
    R, T, k, E, nmax = 2, 6, 3, 4, 40
    topk = rng.integers(-1, E, size=(R, T, k)).astype(np.int64)
    assert any(len(set(r[r >= 0].tolist())) < int((r >= 0).sum()) for r in topk.reshape(-1, k))
    x = workloads.make_hidden(rng, R, T, 128)
    res = oracle.ll_dispatch(x, topk, E, nmax, False, packed=packed)
    assert res["bad_entries"] == 0
    E_loc = E // R
    counts = np.array([[int(np.sum(topk[s] == e)) for s in range(R)] for e in range(E)])
    for s in range(R):
        seen = {}
        for t in range(T):
            for j in range(k):
                e = int(topk[s, t, j])
                if e < 0:
                    assert res["slot"][s, t, j] == -1
                    continue
                r = seen.get(e, 0)
                seen[e] = r + 1
                start = int(counts[e, :s].sum()) if packed else s * nmax
                assert res["slot"][s, t, j] == start + r
                d, el = divmod(e, E_loc)
                assert res["src_info"][d, el, start + r] == t
                np.testing.assert_array_equal(res["recv_x"][d, el, start + r], x[s, t])
    np.testing.assert_array_equal(res["recv_expert_count"].reshape(-1), counts.sum(1))
