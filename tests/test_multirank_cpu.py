"""The benchmark's multi-rank path on CPU (gloo, world size 2): barrier, max-over-ranks
timing and the reference arm's rank-0-only rule. The hot path itself does not shard
(the virtual ranks live in one GPU's memory), so N > 1 means independent replicas."""
import multiprocessing as mp
import os
import socket
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            init_method=f"tcp://127.0.0.1:{port}")
    import bench
    mx = bench.reduce_max(float(10 * (rank + 1)), world)
    bench.barrier(world)

    class A:
        steps, warmup = 1, 0
    ref = bench.run_reference(A, rank, world) if rank != 0 else "skipped"
    q.put((rank, mx, ref))
    dist.destroy_process_group()


def test_reduce_max_and_reference_rank_rule_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [20.0, 20.0]
    assert res[1][2] is None          # non-zero ranks of the reference arm do no work


def test_reduce_max_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5


def test_bytes_model_counts_each_byte_once():
    sys.path.insert(0, ROOT)
    import bench
    b = bench.algorithmic_bytes(R=8, T=4096, H=7168, k=8, N=173_000)
    # payload: x read once + N rows written (dispatch); N rows read + x written (combine)
    assert b["dispatch"] - (8 * 4096 * 7168 * 2 + 173_000 * 7168 * 2) == \
        8 * 4096 * (8 * 12 + 8 * 4) + 173_000 * (8 * 12 + 4)
    assert b["combine"] - (173_000 * 7168 * 2 + 8 * 4096 * 7168 * 2) == \
        8 * 4096 * 8 * 4 + 8 * 4096 * 8 * 12


def test_every_bench_workload_resolves():
    sys.path.insert(0, ROOT)
    import bench
    for name in bench.WORKLOAD_TEXT:
        w = bench.workload_config(name)
        assert w.E % w.R == 0 and w.H % 128 == 0


def test_roofline_traffic_only_for_its_own_workload_and_sources():
    """The committed DRAM counters are reported only for the (kernel, workload) pair and
    the kernel sources they were taken on; any other workload reads as null."""
    sys.path.insert(0, ROOT)
    import json
    import bench
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)["entries"]
    assert entries
    for e in entries:
        kernel, workload = e["kernel"], e["workload"]
        assert kernel in bench.KERNEL_SOURCES and workload in bench.WORKLOAD_TEXT
        got = bench.traffic_from_profiles(kernel, workload)
        current = e["source_sha256"] == bench.source_digest(bench.KERNEL_SOURCES[kernel])
        assert got == (e["dram_bytes_per_launch"] if current else None)
        others = [w for w in bench.WORKLOAD_TEXT
                  if not any(x["kernel"] == kernel and x["workload"] == w for x in entries)]
        for w in others:
            assert bench.traffic_from_profiles(kernel, w) is None
    assert bench.traffic_from_profiles("no_such_kernel") is None


def test_fp8_scale_names_match_the_abi():
    sys.path.insert(0, ROOT)
    import bench
    import combine_layout_02_gb300 as ep
    assert bench.FP8_SCALE == {"fp32": ep.EP_FP8_SCALE_FP32, "pow2": ep.EP_FP8_SCALE_POW2,
                               "ue8m0": ep.EP_FP8_SCALE_UE8M0, "tensor": ep.EP_FP8_SCALE_TENSOR}
    # every phase a workload can time names the kernel its roofline would cite
    assert {"combine_backward", "dispatch_backward", "dispatch", "dispatch_fp8", "combine",
            "dispatch_em", "combine_em", "ll_send", "ll_recv", "ll_combine"} <= set(bench.PHASE_KERNEL)


def test_source_digest_ignores_comments_only():
    sys.path.insert(0, ROOT)
    import bench
    a = 'int f() { return 1; } // one\n/* two */ const char* s = "// kept";\n'
    b = 'int f() { return 1; } // changed\n/* other\n text */ const char* s = "// kept";\n'
    c = 'int f() { return 2; } // one\n/* two */ const char* s = "// kept";\n'
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert bench.strip_comments(a) != bench.strip_comments(c)
    assert '"// kept"' in bench.strip_comments(a)


def test_reference_arm_line_has_the_gpu_arm_config(monkeypatch):
    """The reference arm (the CPU oracle on a bounded token sample) reports the same
    metric, unit and config object as the GPU arm's dsv3 line: the same workload string,
    shape keys, received-row count (from the oracle's layout of the whole workload),
    parallelism and L2 note."""
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    monkeypatch.setenv("EP_ORACLE_BUDGET_S", "0.5")

    class A:
        steps, warmup = 1, 3
    res = bench.run_reference(A, 0, 1)
    w = bench.WORKLOAD
    inp = bench.workloads.make_workload(w, with_hidden=False)
    N = int(oracle.layout(inp["topk_idx"], w.E, w.C)["rank_prefix_matrix"][-1].sum())
    assert res["impl"] == "reference" and res["metric"] == bench.METRIC and res["unit"] == "GB/s"
    assert res["config"] == bench.config_dict("dsv3", w, N, 1, bench.DSV3_L2)
    assert res["config"]["recv_rows"] == N
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["e2e"]["value"] == res["value"]
    assert res["cpu_baseline"]["kind"] == "oracle" and res["cpu_baseline"]["cores"] == 1


def test_segment_names_of_the_timed_passes():
    import bench
    names = ["layout", "dispatch", "combine"]
    assert bench.segment_names(names, [0, 1, 2]) == names
    assert bench.segment_names(names, [0, 2]) == ["layout+dispatch", "combine"]
    assert bench.segment_names(names, [0]) == ["layout+dispatch+combine"]
    assert bench.segment_names(["layout", "dispatch_fp8"], [0]) == ["layout+dispatch_fp8"]
