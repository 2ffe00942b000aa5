"""Host logic of the N > 1 benchmark path, on CPU with gloo (world size 2):
max-over-ranks timing, whole-job throughput, distinct per-rank replicas, and
the reference arm doing no work on ranks other than 0."""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    from moe_grouped_block_gb300 import workloads
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 2.0 + rank  # rank 1 is the slowest
    m = bench.max_over_ranks(ms, dist, "cpu")
    wl = bench.replica_workload(workloads.WORKLOADS["tiny_fprop_mxfp8"], rank)
    x = workloads.make_inputs(wl)["x"]
    digest = float(x.float().sum())
    t = torch.tensor([digest], dtype=torch.float64)
    all_d = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(all_d, t)

    class A:
        steps, warmup = 1, 0
    ref = bench.run_reference(A, workloads.WORKLOADS["tiny_fprop_mxfp8"], world, rank) if rank else None
    q.put((rank, m, [float(v) for v in all_d], ref))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_gloo_host_logic():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, digests, ref in res:
        assert m == 3.0                      # max over ranks
        assert digests[0] != digests[1]      # independent replicas
        if rank == 1:
            assert ref is None               # reference arm: rank 0 only
    import bench
    assert np.isclose(bench.job_tflops(1e12, 2, 1.0), 2000.0)
