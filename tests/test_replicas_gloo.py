"""The benchmark's multi-GPU mode runs independent replicas (the layer does not
shard); the only cross-rank work is a barrier and the max of the timed region.
Checked here with two gloo ranks on CPU."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_env()
    dist = bench.init_dist(w)
    dist.barrier()
    got = bench.max_over_ranks(dist, 10.0 + rank)   # each rank's timed region
    out[rank] = (w, r, got)
    dist.destroy_process_group()


def test_two_replicas_take_the_max_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == (2, 0, 11.0) and res[1] == (2, 1, 11.0)
