"""The N > 1 benchmark path on the CPU: two gloo ranks, each with its own batch
(weak scaling); whole-job throughput = all ranks' units over the slowest
rank's time; the only cross-rank calls are the barrier and those reductions."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import synth
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    bench.init_dist(ws, "gloo")
    bench.barrier(ws)
    units = 1000.0 * (rank + 1)
    elapsed = 0.5 + rank            # rank 1 is slower
    total, slowest, thr = bench.aggregate(units, elapsed, ws, torch.device("cpu"))
    w = synth.workload("tiny", seed=rank)
    k = synth.rows(w.seed, synth.STREAM_K, 0, 8, w.H, w.dk, torch.float32, True)
    gathered = [torch.zeros_like(k) for _ in range(world)]
    dist.all_gather(gathered, k)
    out[rank] = (total, slowest, thr, bool(torch.equal(gathered[0], gathered[1])))
    dist.destroy_process_group()


def test_two_rank_aggregation_and_independent_batches():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        total, slowest, thr, same = res[rank]
        assert total == 3000.0 and slowest == 1.5 and abs(thr - 2000.0) < 1e-9
        assert not same, "each rank must scan its own batch"
