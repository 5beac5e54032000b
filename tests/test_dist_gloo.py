"""Multi-process host logic of the benchmark on CPU (gloo, world size 2):
the barrier, the max-over-ranks timing that makes `value` a whole-job
figure, and the rule that only rank 0 runs the reference arm. The data path
itself needs no collective (each rank runs its own batches)."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.init("gloo")
    slowest = d.max(1.5 * (rank + 1))          # per-rank elapsed ms
    d.barrier()
    # whole-job throughput: units of every rank over the slowest rank's time
    value = 1000.0 * d.world / slowest
    q.put((rank, d.world, slowest, value))
    d.close()


def test_two_ranks_share_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [2, 2]
    assert all(o[2] == 3.0 for o in out)            # max over ranks
    assert all(abs(o[3] - 2000.0 / 3.0) < 1e-9 for o in out)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.rank, d.world = 1, 2
    args = bench.argparse.Namespace(steps=1, warmup=0, gpus=2)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args, d) == 0
    assert buf.getvalue() == ""                     # non-zero ranks print nothing


def test_reference_arm_line(monkeypatch):
    sys.path.insert(0, ROOT)
    import json
    import bench
    monkeypatch.setattr(bench, "oracle_fwd_sample", lambda units, seed=1: (0.5, 4096.0, 4, "sample"))
    d = bench.Dist()
    args = bench.argparse.Namespace(steps=2, warmup=1, gpus=1)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args, d) == 0
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference" and line["unit"] == "tokens/s"
    assert line["value"] == pytest.approx(4096.0 / 0.5)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
