"""The benchmark's N > 1 path on the CPU (gloo, world size 2): one replica
per rank on its own seeded batch, no data-path collective, and the slowest
rank's time for the whole job."""
import os
import socket
import sys
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from decode_attention_paged_gb300 import workloads as W

    local_ms = 10.0 + 5.0 * rank
    got = bench.max_over_ranks(local_ms, dist)
    w = bench.replica_workload(W, "tiny", rank)
    # the replicas' inputs differ; gather a fingerprint of each rank's q
    fp = torch.tensor([float(w.q.float().sum())], dtype=torch.float64)
    fps = [torch.zeros_like(fp) for _ in range(world)]
    dist.all_gather(fps, fp)
    args = types.SimpleNamespace(workload="tiny", steps=1, warmup=0)
    ref_rc = bench.reference_arm(args, rank, world) if rank == 1 else None
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got, [float(x) for x in fps], ref_rc))


@pytest.mark.timeout(300)
def test_two_rank_replicas_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(world):
        rank, got, fps, ref_rc = q.get(timeout=240)
        out[rank] = (got, fps, ref_rc)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank reports the slowest rank's time
    assert out[0][0] == out[1][0] == 15.0
    # the two replicas decode different seeded batches
    assert out[0][1][0] != out[0][1][1]
    # the reference arm runs on rank 0 only; other ranks exit 0 without work
    assert out[1][2] == 0
