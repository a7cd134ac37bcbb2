"""The bench's multi-rank host logic on CPU: two gloo ranks agree on the max / sum over
ranks, and the reference arm prints only on rank 0."""

import io
import os
import socket
import contextlib

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import bench
    w, r, local = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    cpu = torch.device("cpu")
    mx = bench.max_over_ranks(dist, 10.0 + r, cpu)
    sm = bench.sum_over_ranks(dist, 1.0 + r, cpu)
    bench.barrier(dist)
    args = type("A", (), dict(config="layer_256x256", steps=1, warmup=0))()
    buf = io.StringIO()
    if r == 1:
        with contextlib.redirect_stdout(buf):
            bench.run_reference(args, w, r)
    q.put((r, mx, sm, buf.getvalue()))
    dist.destroy_process_group()


def test_two_gloo_ranks():
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
    assert [r[1] for r in res] == [11.0, 11.0]
    assert [r[2] for r in res] == [3.0, 3.0]
    assert res[1][3] == ""          # rank 1 of the reference arm prints nothing
