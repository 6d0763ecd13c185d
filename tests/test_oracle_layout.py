"""Pins for the oracle's layout (get_dispatch_layout + the handle's prefix matrices).

Checks: a hand-worked example; exhaustive enumeration of every routing table of tiny
shapes against set-membership / sorting characterisations; invariants on larger random
and skewed tables (bincount, cumsum, stable-sort inverse maps); error counting.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_example():
    with open(os.path.join(GOLDEN, "layout_hand_example.json")) as f:
        g = json.load(f)
    lay = oracle.layout(np.array(g["topk_idx"], np.int64), g["E"], g["C"])
    for key in ("num_tokens_per_expert", "is_token_in_rank", "num_tokens_per_rank",
                "channel_prefix_matrix", "rank_prefix_matrix", "recv_channel_prefix_matrix",
                "send_head", "num_recv_tokens_per_expert"):
        np.testing.assert_array_equal(lay[key], np.array(g[key]), err_msg=key)
    assert lay["bad_entries"] == 0


def check_layout_invariants(topk, E, C, lay):
    """Characterise every layout tensor without the oracle's running counters."""
    R, T, k = topk.shape
    E_loc = E // R
    tpc = -(-T // C) if T else 1
    valid = (topk >= 0) & (topk < E)
    # experts: bincount of valid entries per source
    for s in range(R):
        np.testing.assert_array_equal(
            lay["num_tokens_per_expert"][s], np.bincount(topk[s][valid[s]], minlength=E))
    # rank membership: set of ranks of the token's valid experts
    in_rank = np.zeros((R, T, R), np.uint8)
    for d in range(R):
        in_rank[:, :, d] = np.any(valid & (topk // E_loc == d), axis=-1)
    np.testing.assert_array_equal(lay["is_token_in_rank"], in_rank)
    np.testing.assert_array_equal(lay["num_tokens_per_rank"], in_rank.sum(1))
    # channel prefix: cumsum of per-channel bincounts, ends at the count
    for s in range(R):
        for d in range(R):
            toks = np.nonzero(in_rank[s, :, d])[0]
            ref = np.cumsum(np.bincount(toks // tpc, minlength=C)[:C])
            np.testing.assert_array_equal(lay["channel_prefix_matrix"][s, d], ref)
    cp = lay["channel_prefix_matrix"]
    assert np.all(np.diff(cp, axis=-1) >= 0)
    np.testing.assert_array_equal(cp[:, :, -1], lay["num_tokens_per_rank"])
    rp = lay["rank_prefix_matrix"]
    np.testing.assert_array_equal(rp, np.cumsum(lay["num_tokens_per_rank"], axis=0))
    # send_head: rows of d enumerate {(s, t): in_rank} in lexicographic order; the map
    # is a bijection onto [0, N_d)
    for d in range(R):
        s_idx, t_idx = np.nonzero(in_rank[:, :, d])
        order = np.lexsort((t_idx, s_idx))            # stable sort by (s, t)
        expect = np.full((R, T), -1, np.int64)
        expect[s_idx[order], t_idx[order]] = np.arange(len(order))
        np.testing.assert_array_equal(lay["send_head"][:, :, d], expect)
        heads = lay["send_head"][:, :, d][in_rank[:, :, d] == 1]
        assert sorted(heads.tolist()) == list(range(rp[-1, d] if R else 0))
    # recv_channel_prefix_matrix[d][s][c] = #rows of d that come before the first token
    # of (s, c) in (s, t) order
    for d in range(R):
        for s in range(R):
            for c in range(C):
                before = in_rank[:s, :, d].sum() + in_rank[s, :min(c * tpc, T), d].sum()
                assert lay["recv_channel_prefix_matrix"][d, s, c] == before
    # per-expert receive counts
    allv = topk[valid]
    np.testing.assert_array_equal(lay["num_recv_tokens_per_expert"].reshape(-1),
                                  np.bincount(allv, minlength=E))


@pytest.mark.parametrize("T,k", [(1, 1), (2, 1), (1, 2), (3, 1)])
def test_exhaustive_tiny_tables(T, k):
    """Every table with entries in {-1, 0, 1, 2, 3} for R=2, E=4 (duplicates allowed)."""
    R, E, C = 2, 4, 2
    n = R * T * k
    for vals in itertools.product(range(-1, E), repeat=n):
        topk = np.array(vals, np.int64).reshape(R, T, k)
        lay = oracle.layout(topk, E, C)
        assert lay["bad_entries"] == 0
        check_layout_invariants(topk, E, C, lay)


def test_random_tiny_tables_k2():
    rng = np.random.default_rng(7)
    for _ in range(1500):
        topk = rng.integers(-1, 4, (2, 2, 2)).astype(np.int64)
        lay = oracle.layout(topk, 4, 3)
        check_layout_invariants(topk, 4, 3, lay)


@pytest.mark.parametrize("name", ["tiny", "zipf_reuse_small", "group_small", "masked"])
def test_invariants_on_workload_shapes(name):
    W = workloads.Workload
    w = {
        "tiny": workloads.CONFIGS["tiny"],
        "zipf_reuse_small": W("z", R=16, T=150, H=128, E=128, k=6, C=7, routing="zipf",
                              zipf_s=1.2, seed=11),
        "group_small": W("g", R=8, T=300, H=128, E=256, k=8, C=12, routing="group",
                         groups=8, topk_groups=4, seed=12),
        "masked": W("m", R=4, T=77, H=128, E=32, k=5, C=5, mask_p=0.3, seed=13),
    }[name]
    topk = workloads.make_workload(w, with_hidden=False)["topk_idx"]
    lay = oracle.layout(topk, w.E, w.C)
    assert lay["bad_entries"] == 0
    check_layout_invariants(topk, w.E, w.C, lay)
    # sum of expert counts = number of valid entries
    assert lay["num_tokens_per_expert"].sum() == (topk >= 0).sum()


def test_invalid_entries_are_counted_and_skipped():
    topk = np.array([[[0, 4], [-2, 1]], [[3, -1], [7, 2]]], np.int64)   # E = 4
    lay = oracle.layout(topk, 4, 1)
    assert lay["bad_entries"] == 3
    clean = np.where((topk >= 0) & (topk < 4), topk, -1)
    ref = oracle.layout(clean, 4, 1)
    for key in ("num_tokens_per_expert", "is_token_in_rank", "send_head", "rank_prefix_matrix"):
        np.testing.assert_array_equal(lay[key], ref[key])


def test_empty_and_degenerate_shapes():
    # T = 0: all counts zero
    lay = oracle.layout(np.zeros((3, 0, 2), np.int64), 6, 4)
    assert lay["num_tokens_per_rank"].sum() == 0 and lay["send_head"].size == 0
    assert np.all(lay["channel_prefix_matrix"] == 0)
    # R = 1: every valid token goes to rank 0 in token order
    topk = np.array([[[0, 1], [-1, -1], [2, 0]]], np.int64)
    lay = oracle.layout(topk, 3, 2)
    np.testing.assert_array_equal(lay["send_head"][0, :, 0], [0, -1, 1])
    # all masked
    lay = oracle.layout(np.full((2, 5, 3), -1, np.int64), 4, 2)
    assert np.all(lay["send_head"] == -1) and lay["num_recv_tokens_per_expert"].sum() == 0
