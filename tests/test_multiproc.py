"""The N>1 path of bench.py on CPU: two gloo ranks. Every rank runs its own
replica of the workload (no collective on the data path); the only exchanges
are the barrier around the timed region and the max over ranks of the elapsed
time, which these tests exercise."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    class A:
        impl = "reference"          # forces the gloo backend
    r, w = bench.dist_init(A())
    assert (r, w) == (rank, world)
    bench.barrier(w)
    # each rank reports a different elapsed time; all must agree on the max
    got = bench.max_over_ranks(10.0 + rank, w)
    q.put((rank, got))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_barrier_and_max_over_ranks(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert res == [(r, 10.0 + world - 1) for r in range(world)]


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.main() is None
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank0(monkeypatch, capsys):
    import json
    import bench
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                                     "--workload", "tiny_linear"])
    bench.main()
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GOPS" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"] == "linear_64x256x512_f32"
