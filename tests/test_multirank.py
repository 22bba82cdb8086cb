"""The multi-GPU path of bench.py shards by batch (one replica per GPU, no
data-path collective); its host logic -- the max-over-ranks step time and the
summed throughput -- runs here on two gloo ranks on the CPU."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    w, r, lr = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    # rank r took (r + 1) ms per step; the slowest rank sets the step time
    t_max = bench.reduce_max((rank + 1) * 1e-3, dist)
    total_roof = bench.reduce_sum(0.5e-3, dist)        # each rank's roofline time per step
    dist.barrier()
    q.put((rank, w, r, t_max, total_roof, 100.0 * total_roof / t_max))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
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
    for rank, w, r, t_max, total_roof, value in res:
        assert w == 2 and r == rank
        assert t_max == pytest.approx(2e-3)
        assert total_roof == pytest.approx(1e-3)
        assert value == pytest.approx(50.0)   # 2 GPUs at 25% of one GPU's roofline each
