"""The replicas path of bench.py (one independent verify-pass stream per GPU, no collective
on the data path): the time reported is the slowest rank's and the rate counts every rank's
passes.  Run here as two gloo ranks on the CPU; the reference arm prints only on rank 0."""
import contextlib
import io
import multiprocessing as mp
import os
import socket
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as td

    import bench
    td.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(10.0 + 3.0 * rank)  # rank 1 is the slow replica
    out.put((rank, ms, bench.replica_rate(5, world, ms)))
    td.barrier()
    td.destroy_process_group()


def test_two_gloo_ranks_report_slowest_time_and_all_passes():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate in res:
        assert ms == 13.0                       # the max over ranks, on every rank
        assert abs(rate - 2 * 5 / 0.013) < 1e-9  # both ranks' passes over the slowest time


def test_without_a_group_the_local_time_is_used():
    import bench
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.replica_rate(3, 1, 1500.0) == 2.0


def test_percentiles():
    import bench
    p = bench.percentiles([float(x) for x in range(1, 12)])  # 1..11
    assert p == {"median": 6.0, "p10": 2.0, "p90": 10.0}
    assert bench.percentiles([4.0]) == {"median": 4.0, "p10": 4.0, "p90": 4.0}


def test_reference_arm_prints_on_rank_zero_only():
    import bench
    args = types.SimpleNamespace(steps=1, warmup=0, gpus=2)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, rank=1)
    assert buf.getvalue() == ""


def test_reference_arm_sample_sizing():
    import bench
    # 23 whole passes of 8.4 s fit in 240 s: whole passes
    assert bench.ref_sample_layers(8.4, 22, budget=240.0) == 64
    # 510 steps do not: a share of the layers so that they fit in what the first pass left
    n = bench.ref_sample_layers(8.4, 509, budget=240.0)
    assert n == int(64 * (240.0 - 8.4) / (509 * 8.4))
    assert n * 509 * 8.4 / 64 <= 240.0 - 8.4
    # never below one layer, never above all of them
    assert bench.ref_sample_layers(100.0, 1000, budget=240.0) == 1
    assert bench.ref_sample_layers(1.0, 0, budget=240.0) == 64
