"""The N > 1 path of bench.py on CPU: two ranks over gloo (127.0.0.1).

The forward shards by (batch, head) with no exchange step, so N GPUs run N
independent replicas; what the ranks share is the rendezvous, the barriers
around the timed region, the max-over-ranks reduction of the step time, and
the rule that only rank 0 runs and prints the reference (oracle) arm.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)


def _reduce_worker(rank, world, port, out):
    _env(rank, world, port)
    import bench
    w, r, _ = bench.dist_setup("gloo")
    bench.barrier(w)
    m = bench.max_over_ranks(1.5 * (rank + 1), w, torch.device("cpu"))
    bench.barrier(w)
    out.put((r, w, m))
    torch.distributed.destroy_process_group()


def _reference_worker(rank, world, port, out):
    _env(rank, world, port)
    import bench
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--config", "tiny_f32", "--gpus", "2", "--steps", "1", "--warmup", "3",
                         "--cpu-budget", "0.2"])
    out.put((rank, rc, buf.getvalue()))
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


def _run(target, world=2):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = [out.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0, f"rank process exited with {p.exitcode}"
    return sorted(res)


def test_two_ranks_take_the_max_step_time():
    res = _run(_reduce_worker)
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 for r in res)
    assert all(r[2] == pytest.approx(3.0) for r in res), res


def test_reference_arm_runs_on_rank0_only():
    res = _run(_reference_worker)
    (r0, rc0, out0), (r1, rc1, out1) = res
    assert (r0, r1) == (0, 1) and rc0 == 0 and rc1 == 0
    assert out1.strip() == ""
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
