"""The N > 1 host logic of bench.py on CPU: two gloo ranks (127.0.0.1) reduce
their step times to the slowest one and report the whole job's throughput.
The operator has no exchange between ranks (replicas), so this is all the
multi-rank code there is."""
import importlib.util
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    b = _bench()
    env = b.dist_env()
    my_ms = 10.0 + 5.0 * rank          # rank 1 is the slower one
    mx = b.max_over_ranks(my_ms, dist, "cpu")
    value = b.job_throughput(1000.0, 4, ws, mx)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, env, mx, value))


def test_two_gloo_ranks_reduce_to_the_slowest():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, mx, value in got:
        assert env == (ws, rank, rank)
        assert mx == 15.0                                     # every rank sees the slowest time
        assert value == pytest.approx(1000.0 * 4 * ws / 15e-3)   # all ranks' units / slowest time


def test_single_rank_needs_no_process_group():
    b = _bench()
    assert b.max_over_ranks(3.5, None, "cpu") == 3.5
    assert b.job_throughput(10.0, 2, 1, 4.0) == pytest.approx(10.0 * 2 / 4e-3)
