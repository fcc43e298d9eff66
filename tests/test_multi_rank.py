"""Host logic of the bench's N > 1 path on CPU: two `gloo` ranks (one process
each) agree on the slowest rank's time, report the whole-job rate over all
replicas, draw different batches (weak scaling, no data-path collective), and
only rank 0 runs the reference arm."""
import importlib.util
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        r, w, local = bench.dist_env()
        local_ms = 10.0 * (rank + 1)                 # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, dist, "cpu")
        rate = bench.job_rate_gbs(1e9, 5, w, ms)

        class A:                                     # the args bench.py parses
            workload, batch, layers = "serving", 64, 36
        wl, sparse = bench.make_workload(A, r)
        q.put((r, w, ms, rate, [int(x) for x in wl.seq_lens[:8]], sparse))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_and_rate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()                              # both ranks rendezvous on it
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for r, w, ms, rate, lens, sparse in res:
        assert w == world and ms == 20.0             # both ranks see the slowest time
        assert rate == pytest.approx(1e9 * 5 * world / 0.020 / 1e9)
        assert not sparse
    assert res[0][4] != res[1][4]                    # each replica draws its own batch


def test_single_rank_is_a_no_op_and_reference_arm_runs_on_rank_0_only():
    bench = _bench()
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5
    assert bench.job_rate_gbs(2e9, 10, 1, 1000.0) == pytest.approx(20.0)

    class A:
        workload, steps, warmup, batch, layers, gpus = "serving", 1, 0, 64, 36, 2
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A, 1, 2)                 # rank 1 of 2: no work, no line
    assert buf.getvalue() == ""
