"""Multi-process host logic of bench.py on CPU (gloo, world size 2): each rank
gets its own requests (weak scaling) and the reported time is the slowest
rank's.  No GPU and no data-path collective is involved."""
import os
import socket


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import sys
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    import workload as wl
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = bench.rank_workload(wl.WORKLOADS["tiny"], rank, world)
    walk = wl.query_walk(w, 0, 0, 2)
    t = bench.max_over_ranks(float(10 + rank), world)
    q.put((rank, w.base_seed, walk.tobytes(), t))
    dist.destroy_process_group()


def test_two_ranks_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, w0, t0), (r1, s1, w1, t1) = got
    assert s0 != s1 and w0 != w1          # independent requests per rank
    assert t0 == t1 == 11.0               # slowest rank's time on both


def test_single_rank_is_identity():
    import bench
    import workload as wl
    w = wl.WORKLOADS["tiny"]
    assert bench.rank_workload(w, 0, 1) is w
    assert bench.max_over_ranks(3.5, 1) == 3.5
