"""bench.py's multi-rank harness on CPU: two gloo ranks share only a barrier
and a max-reduction of their times (each rank runs an independent replica;
nothing on the data path crosses ranks), and the reference arm runs on rank
0 only."""
import argparse
import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    dist = bench.init_dist(world)
    slowest = bench.max_over_ranks(dist, 10.0 * (rank + 1))
    bench.barrier(dist)
    args = argparse.Namespace(steps=1, warmup=3, seed=0)
    ref = bench.run_reference(args, world, rank) if rank != 0 else "skipped"
    dist.destroy_process_group()
    q.put((rank, slowest, ref))


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got = {r: (v, ref) for r, v, ref in out}
    assert got[0][0] == 20.0 and got[1][0] == 20.0
    assert got[1][1] is None  # non-zero ranks print nothing on the reference arm


def test_byte_model_matches_hand_count():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    bm = bench.byte_model(32768, 256, 8, 7168)
    assert bm["combine"] == 32768 * 8 * 7168 * 2 + 32768 * 7168 * 2 + 32768 * 8 * 12
    assert bm["dispatch"] == 32768 * 7168 * 2 + 32768 * 8 * (7168 + 56 * 4) + 32768 * 8 * 8
