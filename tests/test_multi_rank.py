"""The N > 1 path of bench.py on CPU: world size 2 with the gloo backend.
Each rank is an independent replica; timings are maximised over the ranks and
the job throughput counts every rank's tokens.  No GPU."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r "took" 10 + r ms for the device loop and 20 - r ms end to end
    ms, e2e = bench.max_over_ranks([10.0 + rank, 20.0 - rank], torch.device("cpu"), world)
    out_q.put((rank, ms, e2e, bench.job_throughput(world, 1, 128, ms / 1e3)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_is_the_max_over_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, ms, e2e, value in res:
        assert ms == 11.0 and e2e == 20.0           # every rank sees the slowest replica
        assert value == pytest.approx(2 * 128 / 0.011)  # tokens of both replicas / the max time


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(bench.parse()) == 0  # returns at once: only rank 0 times the oracle
