"""The multi-GPU path of bench.py on CPU: two gloo ranks (world size 2).

The attention shards by request and kv head with no exchange, so N GPUs run
N independent replicas of the workload: the host logic is the slowest rank's
time (an all-reduce MAX) and the whole-job rate (N x the per-replica work in
that time); the reference arm runs on rank 0 only."""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [3.0, 5.0][rank]                      # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, world)
        rate = bench.job_rate(world, 2e12, slowest)
        dist.barrier()
        q.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, rate in got:
        assert slowest == 5.0
        assert rate == pytest.approx(2 * 2e12 / 5e-3 / 1e12)   # 2 replicas x work / slowest time


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_rate(1, 1e12, 1.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Ranks other than 0 return at once, before touching the workload or the oracle."""
    import argparse

    import bench
    args = argparse.Namespace(workload="no_such_workload", steps=1, warmup=3)
    assert bench.run_reference(args, rank=1, world=2) is None


@pytest.mark.parametrize("workload", ["chunked_prefill", "mixed_window"])
def test_multi_rank_run_refuses_prefill_workloads(workload):
    """The prefill kernel loads K/V tiles with cluster multicast, which runs on
    one GPU only: a multi-rank bench run of a prefill workload exits with a
    clear message before touching a device or a process group."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0", MASTER_ADDR="127.0.0.1", MASTER_PORT="1")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--workload", workload, "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 2, (r.returncode, r.stderr[-2000:])
    assert "1-GPU library" in r.stderr and "multicast" in r.stderr
    assert r.stdout == ""


def test_uses_prefill_follows_the_packed_row_rule():
    import bench
    from paged_attention_relative_gb300.workloads import make_case, tiny_mixed
    assert not bench.uses_prefill(tiny_mixed(0))                      # 5 tokens x 2 heads per kv head
    c = make_case(seed=0, seqlens_q=[17], seqlens_k=[40], num_heads=8, num_kv_heads=2, head_dim=64)
    assert bench.uses_prefill(c)                                      # 17 x 4 = 68 rows > 64
    c = make_case(seed=0, seqlens_q=[16], seqlens_k=[40], num_heads=8, num_kv_heads=2, head_dim=64)
    assert not bench.uses_prefill(c)                                  # 64 rows
