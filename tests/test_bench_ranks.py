"""bench.py's multi-rank host logic on CPU (gloo, world size 2): under torchrun every rank
runs its own replica of the step, the job's step time is the slowest rank's, and the
reference arm runs on rank 0 alone (the other ranks exit without work)."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out.put((rank, bench._max_over_ranks(values[rank], world, "cpu")))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_step_time_is_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    values = [0.412, 0.437]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: max(values), 1: max(values)}


def test_single_process_keeps_its_own_time():
    assert bench._max_over_ranks(0.25, 1, "cpu") == 0.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                                      "--warmup", "0"])
    a = bench._args()
    assert bench._reference_arm(a) == 0
    assert capsys.readouterr().out == ""
