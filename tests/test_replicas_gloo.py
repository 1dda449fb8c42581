"""The multi-GPU benchmark path on CPU: two gloo ranks run the host logic of
independent replicas (per-rank inputs, the slowest rank's time, the whole
job's throughput). No GPU and no kernel is involved."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from dsa_inputs import WORKLOADS, make_inputs, small_workload
        wl = small_workload(batch=1, q_len=1, total_len=300, top_k=32, seed=5)
        x = make_inputs(wl, seed=bench.replica_seed(wl, rank))["q"].float().sum().item()
        ms = bench.slowest_rank_ms(1.5 + rank, world, device="cpu")
        value = bench.whole_job_value(world, WORKLOADS["decode_128k"].query_tokens, ms)
        q.put((rank, ms, value, x))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    # both ranks see the slowest rank's time; the job counts both ranks' tokens
    assert res[0][1] == res[1][1] == 2.5
    assert res[0][2] == res[1][2] == pytest.approx(2 * 1 / 2.5e-3)
    # each rank draws its own inputs
    assert res[0][3] != res[1][3]
