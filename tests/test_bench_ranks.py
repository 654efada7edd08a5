"""bench.py's multi-rank path on CPU: two gloo ranks, independent problems,
the job time is the slowest rank's and the work is summed."""

import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.dist_env()
    t, f, b = bench.reduce_over_ranks(10.0 + 5 * rank, 1000 * (rank + 1), 7 * (rank + 1), dist)
    out[rank] = (w, r, lr, t, f, b)
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(world):
            w, rank, lr, t, f, b = out[r]
            assert (w, rank, lr) == (world, r, r)
            assert t == 15.0 and f == 3000.0 and b == 21.0


def test_single_rank_passthrough():
    import bench

    assert bench.reduce_over_ranks(3.5, 10, 20) == (3.5, 10.0, 20.0)


def test_failing_leg_is_reported_not_fatal(capsys):
    """An auxiliary measurement that raises becomes {"error": ...} in its
    key; a disabled one is None; a working one returns its result."""
    import bench

    def boom(x):
        raise RuntimeError(f"no device {x}")

    def ok(x, y):
        return {"ms_per_step": x + y}

    assert bench.run_leg(False, boom, 1) is None
    assert bench.run_leg(True, ok, 1, 2) == {"ms_per_step": 3}
    r = bench.run_leg(True, boom, 7)
    assert r == {"error": "RuntimeError('no device 7')"}
    assert "boom failed" in capsys.readouterr().err
