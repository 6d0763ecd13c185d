"""Pins for the oracle's dispatch and combine (normal mode).

Dispatch: byte equality with the source rows at the rows the (separately pinned)
layout assigns, canaries elsewhere, inverse maps, local-id / weight routing invariants,
FP8 rows equal to the pinned per-row quantiser, pre-quantised rows copied verbatim.
Combine: adjointness <dispatch(x), y> = <x, combine_sum(y)> (exact, integer data), the
identity-expert round trip returning x within bf16 rounding, an fp64 numpy reference
within half a bf16 ulp, and the weight-gradient reduction.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint32) << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def _f64_to_bf16_torch(v):
    # library cast (fp32 in between is exact for the small-integer values used with it)
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _case(R=4, T=50, H=256, E=16, k=3, C=5, mask_p=0.1, seed=21, routing="uniform"):
    w = workloads.Workload("t", R=R, T=T, H=H, E=E, k=k, C=C, mask_p=mask_p, seed=seed,
                           routing=routing, zipf_s=1.2)
    inp = workloads.make_workload(w)
    lay = oracle.layout(inp["topk_idx"], E, C)
    return w, inp, lay


def _compact_offsets(lay):
    n = lay["rank_prefix_matrix"][-1]
    return np.concatenate([[0], np.cumsum(n)]).astype(np.int64)


@pytest.mark.parametrize("offsets", ["compact", "worst"])
def test_dispatch_bf16_rows_and_metadata(offsets):
    w, inp, lay = _case()
    R, T, E, k = w.R, w.T, w.E, w.k
    E_loc = E // R
    off = (_compact_offsets(lay) if offsets == "compact"
           else workloads.worst_case_row_offsets(R, T))
    res = oracle.dispatch(inp["x"], lay["send_head"], off, E, inp["topk_idx"],
                          inp["topk_weights"], fill_x=0xDEAD, fill_idx=-99, fill_w=-5.0,
                          fill_src=-3)
    assert res["bad_rows"] == 0
    written = np.zeros(int(off[-1]), bool)
    for s in range(R):
        for t in range(T):
            for d in range(R):
                h = lay["send_head"][s, t, d]
                if h < 0:
                    continue
                row = off[d] + h
                written[row] = True
                np.testing.assert_array_equal(res["recv_x"][row], inp["x"][s, t])
                assert res["recv_src_idx"][row] == t
                ids, ws = res["recv_topk_idx"][row], res["recv_topk_weights"][row]
                # local ids map back to the original expert; non-local entries are -1/0
                orig = inp["topk_idx"][s, t]
                loc = ids >= 0
                assert loc.any()          # a row is only sent because of a local expert
                np.testing.assert_array_equal(ids[loc] + d * E_loc, orig[loc])
                assert np.all((orig[~loc] < 0) | (orig[~loc] // E_loc != d))
                np.testing.assert_array_equal(ws[loc], inp["topk_weights"][s, t][loc])
                assert np.all(ws[~loc] == 0.0) and np.all(ids[~loc] == -1)
    # rows that no token maps to keep their canaries
    assert np.all(res["recv_x"][~written] == 0xDEAD)
    assert np.all(res["recv_src_idx"][~written] == -3)
    assert np.all(res["recv_topk_idx"][~written] == -99)


def test_dispatch_is_a_row_permutation_count():
    """Every in-rank (s, t, d) triple appears once; total rows = sum of rank counts."""
    w, inp, lay = _case(R=8, T=120, E=64, k=6, C=12, seed=22)
    off = _compact_offsets(lay)
    res = oracle.dispatch(inp["x"], lay["send_head"], off, w.E, inp["topk_idx"],
                          inp["topk_weights"])
    assert off[-1] == lay["is_token_in_rank"].sum()
    # reconstruct the source of every row from recv_src_idx + region + rank_prefix
    rp = lay["rank_prefix_matrix"]
    for d in range(w.R):
        rows = np.arange(off[d], off[d + 1])
        local = rows - off[d]
        src_rank = np.searchsorted(rp[:, d], local, side="right")
        np.testing.assert_array_equal(res["recv_x"][rows],
                                      inp["x"][src_rank, res["recv_src_idx"][rows]])


def test_dispatch_fp8_rows_equal_quantised_rows():
    w, inp, lay = _case(H=512, seed=23)
    off = _compact_offsets(lay)
    res = oracle.dispatch(inp["x"], lay["send_head"], off, w.E, inp["topk_idx"],
                          inp["topk_weights"], x_kind=oracle.X_QUANTIZE)
    q, sc = oracle.quantize_rows(inp["x"])
    for s in range(w.R):
        for t in range(w.T):
            for d in range(w.R):
                h = lay["send_head"][s, t, d]
                if h >= 0:
                    np.testing.assert_array_equal(res["recv_x"][off[d] + h], q[s, t])
                    np.testing.assert_array_equal(res["recv_x_scales"][off[d] + h], sc[s, t])
    # pre-quantised input tuple: bytes and scales copied verbatim
    res2 = oracle.dispatch(q, lay["send_head"], off, w.E, x_kind=oracle.X_FP8, x_scales=sc)
    np.testing.assert_array_equal(res2["recv_x"], res["recv_x"])
    np.testing.assert_array_equal(res2["recv_x_scales"], res["recv_x_scales"])


def test_dispatch_capacity_overflow_is_reported():
    w, inp, lay = _case(seed=24)
    off = _compact_offsets(lay)
    short = off.copy()
    short[1:] -= np.arange(1, w.R + 1)            # every region one row too small
    short[0] = 0
    res = oracle.dispatch(inp["x"], lay["send_head"], short, w.E)
    assert res["bad_rows"] > 0


# ----------------------------------------------------------------------------- combine

def test_combine_sum_is_adjoint_of_dispatch():
    """<dispatch(x), y> == <x, combine_sum(y)> exactly, with small-integer data."""
    w, inp, lay = _case(R=4, T=40, H=128, E=16, k=4, seed=25)
    rng = np.random.default_rng(26)
    off = _compact_offsets(lay)
    x = _f64_to_bf16_torch(rng.integers(-4, 5, (w.R, w.T, w.H))).reshape(w.R, w.T, w.H)
    y = _f64_to_bf16_torch(rng.integers(-4, 5, (int(off[-1]), w.H))).reshape(-1, w.H)
    dx = oracle.dispatch(x, lay["send_head"], off, w.E)["recv_x"]
    cy = oracle.combine(y, lay["send_head"], off, w.E, w.k)["out"]
    lhs = np.sum(_bf16_to_f64(dx) * _bf16_to_f64(y))
    rhs = np.sum(_bf16_to_f64(x) * _bf16_to_f64(cy))
    assert lhs == rhs


def test_combine_sum_of_identity_experts_scales_by_fanout():
    w, inp, lay = _case(R=8, T=64, H=256, E=64, k=8, seed=27)
    off = _compact_offsets(lay)
    y = oracle.dispatch(inp["x"], lay["send_head"], off, w.E)["recv_x"]
    out = oracle.combine(y, lay["send_head"], off, w.E, w.k)["out"]
    fan = lay["is_token_in_rank"].sum(-1).astype(np.float64)
    ref = _f64_to_bf16_torch(_bf16_to_f64(inp["x"]) * fan[..., None]).reshape(out.shape)
    np.testing.assert_array_equal(out, ref)


@pytest.mark.parametrize("routing", ["uniform", "zipf"])
def test_weighted_combine_identity_round_trip(routing):
    """dispatch -> identity experts -> weighted combine returns x within bf16 rounding
    (weights sum to 1 per token)."""
    w, inp, lay = _case(R=8, T=64, H=256, E=64, k=6, mask_p=0.0, seed=28, routing=routing)
    off = _compact_offsets(lay)
    y = oracle.dispatch(inp["x"], lay["send_head"], off, w.E)["recv_x"]
    out = oracle.combine(y, lay["send_head"], off, w.E, w.k, oracle.COMBINE_WEIGHTED,
                         inp["topk_idx"], inp["topk_weights"])["out"]
    xf, of = _bf16_to_f64(inp["x"]), _bf16_to_f64(out)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(xf), 2.0 ** -126))) - 7)
    assert np.all(np.abs(of - xf) <= ulp)


def test_weighted_combine_matches_fp64_reference():
    w, inp, lay = _case(R=4, T=60, H=256, E=16, k=4, seed=29)
    rng = np.random.default_rng(30)
    off = _compact_offsets(lay)
    y = _f64_to_bf16_torch(rng.standard_normal((int(off[-1]), w.H))).reshape(-1, w.H)
    out = oracle.combine(y, lay["send_head"], off, w.E, w.k, oracle.COMBINE_WEIGHTED,
                         inp["topk_idx"], inp["topk_weights"])["out"]
    E_loc = w.E // w.R
    yf = _bf16_to_f64(y)
    ref = np.zeros((w.R, w.T, w.H))
    topk, wt = inp["topk_idx"], inp["topk_weights"].astype(np.float64)
    for d in range(w.R):
        c = np.where((topk >= 0) & (topk // E_loc == d), wt, 0.0).sum(-1)      # [R, T]
        h = lay["send_head"][:, :, d]
        rows = np.where(h >= 0, off[d] + h, 0)
        ref += np.where((h >= 0)[..., None], c[..., None] * yf[rows], 0.0)
    of = _bf16_to_f64(out)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 8)
    assert np.all(np.abs(of - ref) <= half_ulp * (1 + 1e-9))


def test_combine_reduces_weight_gradients():
    w, inp, lay = _case(R=4, T=50, E=16, k=3, seed=31)
    off = _compact_offsets(lay)
    d = oracle.dispatch(inp["x"], lay["send_head"], off, w.E, inp["topk_idx"], inp["topk_weights"])
    c = oracle.combine(d["recv_x"], lay["send_head"], off, w.E, w.k,
                       recv_topk_weights=d["recv_topk_weights"])
    # each weight comes back from exactly the rank that owns its expert (others send 0)
    np.testing.assert_array_equal(c["combined_topk_weights"], inp["topk_weights"])
    # general gradients: sum over the ranks the token was sent to
    rng = np.random.default_rng(32)
    g = rng.standard_normal(d["recv_topk_weights"].shape).astype(np.float32)
    c2 = oracle.combine(d["recv_x"], lay["send_head"], off, w.E, w.k, recv_topk_weights=g)
    ref = np.zeros((w.R, w.T, w.k))
    for dd in range(w.R):
        h = lay["send_head"][:, :, dd]
        ref += np.where((h >= 0)[..., None], g[np.where(h >= 0, off[dd] + h, 0)].astype(np.float64), 0)
    np.testing.assert_allclose(c2["combined_topk_weights"], ref, rtol=1e-6, atol=1e-7)


def test_handle_reuse_same_result():
    """Dispatch with the cached send_head (no topk) gives the same rows as a fresh one."""
    w, inp, lay = _case(seed=33)
    off = _compact_offsets(lay)
    a = oracle.dispatch(inp["x"], lay["send_head"], off, w.E, inp["topk_idx"], inp["topk_weights"])
    b = oracle.dispatch(inp["x"], lay["send_head"], off, w.E)
    np.testing.assert_array_equal(a["recv_x"], b["recv_x"])
    np.testing.assert_array_equal(a["recv_src_idx"], b["recv_src_idx"])
