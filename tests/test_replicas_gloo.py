"""The multi-process (replica) path of bench.py on CPU: world size 2 over gloo.

Output tiles are independent, so N GPUs run N replicas with no exchange; the only
cross-rank step is the timing reduction (the job takes as long as its slowest rank)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        local_ms = [100.0, 125.0][rank]
        tflops, t = bench.job_throughput(local_ms, steps=10, flops_per_step=2e12, ws=ws)
        assert bench.dist_env() == (ws, rank, rank)
        # the modes a replica times: no cluster shape that shares operands by TMA multicast
        table = bench.mode_table(1, 256, 148, 152, bench.dist_env()[0])
        assert table and not any(r["tma_multicast"] for r in table)
        assert not any(r["sel"] == "clusters" for r in table)
        q.put((rank, t, tflops))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, t, tflops in res:
        assert t == 125.0
        # 2 replicas x 10 steps x 2 TFLOP in 125 ms
        assert tflops == pytest.approx(2 * 10 * 2.0 / 0.125)


def test_mode_table_alone_keeps_the_cluster_rows():
    """A process alone on its GPU (world size 1) also times the larger cluster shapes,
    three of which share operands by TMA multicast; world size 2 drops all of them."""
    import bench
    alone = bench.mode_table(1, 256, 148, 152, 1)
    assert sum(r["tma_multicast"] for r in alone) == 3
    assert {r["key"] for r in alone if r["tma_multicast"]} == {
        "clc_cluster2_shared_b", "clc_cluster4_shared_b", "clc_cluster2x2_shared_ab"}
    two = bench.mode_table(1, 256, 148, 152, 2)
    assert [r["key"] for r in two] == [r["key"] for r in alone if r["sel"] != "clusters"]


def test_single_process_needs_no_group():
    import bench
    tflops, t = bench.job_throughput(50.0, steps=4, flops_per_step=1e12, ws=1)
    assert t == 50.0 and tflops == pytest.approx(4 * 1.0 / 0.05)
