"""Seeded synthetic inputs for MoE expert-parallel layout / dispatch / combine.

This module only draws random numbers. It holds none of the method's arithmetic, so
both the CPU oracle (``oracle/``) and the CUDA path (``combine_layout_02_gb300``) can
consume the same inputs without sharing code. Random draws use numpy's PCG64
(``numpy.random.default_rng(seed)``); the fp32 -> bf16 conversion of the hidden
states is done by PyTorch's own tensor cast (a library routine), so no rounding
code of this project is involved.

Routing shapes follow the workloads the pages describe:

* uniform top-k distinct experts (the DeepSeek-V3-shaped training / prefill case),
* group-limited gating (DeepSeek-V3 style: pick groups first, then experts inside the
  chosen groups; "DeepEP" README, introduction on group-limited gating),
* masked entries (``-1``) for low-latency decode,
* Zipf-skewed expert popularity for the handle-reuse workload.

Each token's ``k`` entries are stored in the order in which they were drawn.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = ["Workload", "CONFIGS", "make_workload", "make_hidden", "make_topk",
           "make_weights", "worst_case_row_offsets"]


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and routing recipe of one synthetic workload.

    R: virtual expert-parallel ranks; T: tokens per source rank; H: hidden size;
    E: experts (E % R == 0); k: top-k; C: channels per source rank;
    nmax: ``num_max_dispatch_tokens_per_rank`` (low-latency mode only).
    """
    name: str
    R: int
    T: int
    H: int
    E: int
    k: int
    C: int = 12
    routing: str = "uniform"          # uniform | group | zipf
    groups: int = 0                    # group-limited gating: number of expert groups
    topk_groups: int = 0               # group-limited gating: groups chosen per token
    mask_p: float = 0.0                # probability that an entry is masked to -1
    zipf_s: float = 0.0                # Zipf exponent for skewed routing
    nmax: int = 0                      # low-latency slot capacity per (expert, source)
    seed: int = 0


# The five workloads: tiny parity case, DeepSeek-V3 shape, group-limited gating,
# low-latency decode, and Zipf skew with handle reuse.
CONFIGS = {
    "tiny": Workload("tiny", R=2, T=128, H=256, E=8, k=2, seed=0),
    "dsv3": Workload("dsv3", R=8, T=4096, H=7168, E=256, k=8, seed=1),
    "group_limited": Workload("group_limited", R=8, T=4096, H=7168, E=256, k=8,
                              routing="group", groups=8, topk_groups=4, seed=2),
    "ll_decode": Workload("ll_decode", R=8, T=128, H=7168, E=256, k=8,
                          mask_p=0.05, nmax=128, seed=3),
    "zipf_reuse": Workload("zipf_reuse", R=16, T=2048, H=4096, E=128, k=6,
                           routing="zipf", zipf_s=1.2, seed=4),
}


def make_hidden(rng: np.random.Generator, R: int, T: int, H: int) -> np.ndarray:
    """Hidden states x ~ N(0, 1), drawn in fp32 and cast to bf16 by PyTorch.

    Returns the bf16 bit patterns as a ``uint16`` array of shape [R, T, H].
    """
    import torch
    x32 = rng.standard_normal((R, T, H), dtype=np.float32)
    xb = torch.from_numpy(x32).to(torch.bfloat16)
    return xb.view(torch.int16).numpy().view(np.uint16)


def _distinct_uniform(rng: np.random.Generator, n: int, E: int, k: int) -> np.ndarray:
    """k distinct experts per row, uniform without replacement, in draw order."""
    keys = rng.random((n, E), dtype=np.float64)
    return np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int64)


def make_topk(rng: np.random.Generator, w: Workload) -> np.ndarray:
    """Routing table topk_idx [R, T, k] (int64, -1 = masked)."""
    n = w.R * w.T
    if w.routing == "uniform":
        idx = _distinct_uniform(rng, n, w.E, w.k)
    elif w.routing == "group":
        # Pick topk_groups groups uniformly without replacement, then k distinct
        # experts uniformly among the experts of the chosen groups.
        gsize = w.E // w.groups
        g = _distinct_uniform(rng, n, w.groups, w.topk_groups)            # [n, G']
        cand = (g[:, :, None] * gsize + np.arange(gsize)[None, None, :]).reshape(n, -1)
        pick = _distinct_uniform(rng, n, cand.shape[1], w.k)              # [n, k]
        idx = np.take_along_axis(cand, pick, axis=1).astype(np.int64)
    elif w.routing == "zipf":
        # Sequential sampling without replacement with p(rank r) ~ r^-s over a random
        # permutation of the experts, drawn by the Gumbel-top-k trick (which has the
        # same distribution as sequential draws without replacement).
        perm = rng.permutation(w.E)
        rank_of_expert = np.empty(w.E, dtype=np.int64)
        rank_of_expert[perm] = np.arange(1, w.E + 1)
        logp = -w.zipf_s * np.log(rank_of_expert.astype(np.float64))
        keys = logp[None, :] + rng.gumbel(size=(n, w.E))
        idx = np.argsort(-keys, axis=1, kind="stable")[:, :w.k].astype(np.int64)
    else:
        raise ValueError(f"unknown routing {w.routing!r}")
    if w.mask_p > 0:
        idx = np.where(rng.random(idx.shape) < w.mask_p, -1, idx)
    return np.ascontiguousarray(idx.reshape(w.R, w.T, w.k))


def make_weights(rng: np.random.Generator, topk_idx: np.ndarray) -> np.ndarray:
    """topk_weights [R, T, k] fp32: softmax of N(0, 1) logits over the token's
    unmasked entries; masked entries get weight 0."""
    logits = rng.standard_normal(topk_idx.shape).astype(np.float32)
    valid = topk_idx >= 0
    logits = np.where(valid, logits, -np.inf).astype(np.float32)
    m = np.max(logits, axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0).astype(np.float32)
    ex = np.where(valid, np.exp(logits - m), 0).astype(np.float32)
    den = np.sum(ex, axis=-1, keepdims=True, dtype=np.float32)
    den = np.where(den > 0, den, 1).astype(np.float32)
    return (ex / den).astype(np.float32)


def make_workload(w: Workload, with_hidden: bool = True, seed: Optional[int] = None):
    """Return dict(x [R,T,H] uint16 bf16 bits | None, topk_idx, topk_weights)."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    topk_idx = make_topk(rng, w)
    topk_weights = make_weights(rng, topk_idx)
    x = make_hidden(rng, w.R, w.T, w.H) if with_hidden else None
    return {"x": x, "topk_idx": topk_idx, "topk_weights": topk_weights}


def worst_case_row_offsets(R: int, T: int) -> np.ndarray:
    """Receive-region row offsets [R+1] when each destination is sized for the worst
    case (every token of every source rank): region d = rows [d*R*T, (d+1)*R*T)."""
    return (np.arange(R + 1, dtype=np.int64) * (R * T)).astype(np.int64)
