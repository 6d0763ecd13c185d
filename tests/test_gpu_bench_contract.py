"""bench.py's JSON line on small cases: one line with the contract's keys, a roofline
with a measured peak, a clock record, the end-to-end object with the bytes it moved, the
count of this library's kernel launches, and (for the low-latency step) the flushed
per-phase figures. Small token counts keep each run to a few seconds; the numbers are
not checked, only that the line is well formed and self-consistent."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMALL = ["--steps", "3", "--warmup", "3", "--min-window-s", "0", "--no-cpu-baseline", "--no-graph"]


def _bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *SMALL, *args],
                       capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def _common(d):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "clocks", "gpu_launches", "e2e"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert d["gpu_launches"] > 0 and d["timed_steps"] == 3 * d["repeats"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]


def test_bench_line_dsv3_small():
    d = _bench("--tokens", "256", "--no-extra")
    _common(d)
    assert d["config"]["workload"].startswith("dsv3:") and d["config"]["T"] == 256
    assert set(d["bytes_per_step"]) == {"layout", "dispatch", "combine"}
    # layout + dispatch as one event-bounded region, and as the sum of the two phases
    assert 0 < d["layout_dispatch_region_us"] and 0 < d["layout_dispatch_us"]
    # layout + dispatch + combine launches per step (the layout is two kernels)
    assert d["gpu_launches_per_step"] == 4
    e2e = d["e2e"]
    assert e2e["h2d_bytes_per_step"] == 8 * 256 * (7168 * 2 + 8 * 8 + 8 * 4)
    assert e2e["d2h_bytes_per_step"] == 8 * 256 * 7168 * 2 and e2e["value"] > 0


def test_bench_line_low_latency_small():
    d = _bench("--workload", "ll_decode", "--tokens", "32", "--nmax", "32", "--no-e2e")
    _common(d)
    assert d["config"]["workload"].startswith("ll_decode:") and "Nmax=32" in d["config"]["workload"]
    for k in ("ll_send_us", "ll_recv_us", "ll_combine_us", "warm"):
        assert k in d, k
    assert d["roofline"]["kernel"] in ("ll_combine_kernel", "ll_send_kernel")
    assert d["gpu_launches_per_step"] == 4   # rank + send, receive, combine
