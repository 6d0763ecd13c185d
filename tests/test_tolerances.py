"""The fp32 summation bound used for the weight-gradient reduction (combined_topk_weights),
checked on the CPU: sums formed the way the kernel forms them (fp32, one destination row
after another in ascending rank order) always pass against the binary64 sum rounded once,
including cases with heavy cancellation, and a sum that lost a single term does not pass."""
import numpy as np

from gpu_util import assert_weight_sums_close


def _case(seed, R=64, T=40, k=32, p_route=0.6, scale=1.0, cancel=False):
    rng = np.random.default_rng(seed)
    in_rank = rng.random((R, T, R)) < p_route
    send_head = np.full((R, T, R), -1, np.int32)
    counts = np.zeros(R, np.int64)
    for d in range(R):                      # rows of d in (source, token) order
        idx = np.flatnonzero(in_rank[:, :, d].reshape(-1))
        flat = np.full(R * T, -1, np.int32)
        flat[idx] = np.arange(idx.size)
        send_head[:, :, d] = flat.reshape(R, T)
        counts[d] = idx.size
    off = np.concatenate([[0], np.cumsum(counts)])
    w = (rng.standard_normal((int(off[-1]), k)) * scale).astype(np.float32)
    if cancel:
        # each token's last row nearly cancels the others: large terms, a small sum
        for s in range(R):
            for t in range(T):
                ds = np.flatnonzero(send_head[s, t] >= 0)
                if ds.size < 2:
                    continue
                rows = off[ds] + send_head[s, t, ds]
                rest = w[rows[:-1]].astype(np.float64).sum(axis=0)
                w[rows[-1]] = (-rest + 1e-3 * rng.standard_normal(k)).astype(np.float32)
    got = np.zeros((R, T, k), np.float32)
    exact = np.zeros((R, T, k), np.float64)
    for d in range(R):                      # the kernel's order: ascending destination
        h = send_head[:, :, d]
        m = h >= 0
        rows = off[d] + h[m]
        got[m] = (got[m] + w[rows]).astype(np.float32)
        exact[m] += w[rows].astype(np.float64)
    return got, exact.astype(np.float32), w, send_head, off


def test_fp32_sequential_sums_pass():
    for seed in range(6):
        got, exp, w, sh, off = _case(seed, scale=10.0 ** (seed - 2))
        assert_weight_sums_close(got, exp, w, sh, off)


def test_cancellation_heavy_sums_pass():
    # large terms around a small result: the relative error of the fp32 sum is large there,
    # and the bound (relative to the sum of magnitudes) still holds
    got, exp, w, sh, off = _case(11, R=32, T=30, k=8, p_route=0.9, scale=100.0, cancel=True)
    rel = np.abs(got.astype(np.float64) - exp) / np.maximum(np.abs(exp), 1e-30)
    assert rel.max() > 1e-4          # far outside a fixed relative tolerance of 1e-5
    assert_weight_sums_close(got, exp, w, sh, off)


def test_a_dropped_term_fails():
    got, exp, w, sh, off = _case(7)
    # drop one row's contribution from one token (a destination it was sent to)
    s, t = 3, 5
    d = int(np.flatnonzero(sh[s, t] >= 0)[0])
    row = off[d] + sh[s, t, d]
    j = int(np.argmax(np.abs(w[row])))
    bad = got.copy()
    bad[s, t, j] = np.float32(bad[s, t, j] - w[row, j])
    try:
        assert_weight_sums_close(bad, exp, w, sh, off)
    except AssertionError:
        return
    raise AssertionError("a sum missing one term passed the bound")
