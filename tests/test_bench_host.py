"""Host logic of the benchmark: the replica reduction over ranks (gloo,
world size 2, CPU), argument defaults and workload bookkeeping."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), TSD_BENCH_BACKEND="gloo")
    import bench
    w, r, _ = bench.dist_setup()
    mx = bench.dist_max(10.0 + r, w)          # per-rank time -> slowest rank
    tot = bench.dist_sum(100.0 * (r + 1), w)   # per-rank units -> job total
    bench.dist_barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, mx, tot))


def test_replica_reduction_gloo_world2():
    import torch.multiprocessing as mp
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
    assert res == [(0, 11.0, 300.0), (1, 11.0, 300.0)]


def test_defaults_and_flops():
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.workload == "long" and a.warmup >= 3 and a.min_seconds >= 2.0
    assert bench.attn_flops(1, 16, 4096, 4096, 64, False) == 4 * 16 * 4096 * 4096 * 64
    assert bench.attn_flops(1, 16, 4096, 4096, 64, True) == 2 * 16 * 4096 * 4096 * 64


def test_reference_arm_reports_the_oracle(monkeypatch):
    import bench
    a = bench.parse_args(["--impl", "reference", "--workload", "long", "--n", "512", "--steps", "1",
                          "--warmup", "0"])
    line, rank = bench.run_reference_arm(a, 1, 0)
    assert rank == 0 and line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert bench.run_reference_arm(a, 2, 1) == (None, 1)   # other ranks do no work


def test_profiled_traffic_requires_matching_source(tmp_path, monkeypatch):
    import bench
    assert bench.profiled_traffic("attn_fwd_bf16", "no_such_workload") is None


def test_overridden_shape_takes_no_committed_traffic():
    """A committed ncu summary describes its workload's own launch: --n, --d,
    --B, --h or --causal that change the shape leave `traffic` null."""
    import bench
    assert not bench.config_overridden(bench.parse_args([]))
    assert not bench.config_overridden(bench.parse_args(["--n", "4096", "--causal", "0"]))
    for extra in (["--causal", "1"], ["--n", "8192"], ["--d", "128"], ["--B", "2"], ["--h", "8"]):
        assert bench.config_overridden(bench.parse_args(extra)), extra
    assert bench.config_overridden(bench.parse_args(["--workload", "big_self", "--causal", "1"]))
    assert not bench.config_overridden(bench.parse_args(["--workload", "big_self_causal"]))
