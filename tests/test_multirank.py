"""The N > 1 host logic of bench.py, run as two gloo ranks on the CPU.

Packs are independent, so bench.py has no data-path collective: under
torchrun every rank draws its own tensor values for the same pack shapes,
times its own steps, and the job's time is the slowest rank's.  These tests
check, with world_size 2 over gloo:

  - rank_workload gives each rank the same shapes and different values;
  - max_over_ranks returns the slowest rank's time on every rank;
  - job_tflops counts every rank's FLOPs over that time (weak scaling);
  - the reference arm runs on rank 0 alone (one JSON line) while the other
    rank exits 0 without output.
"""
import contextlib
import io
import json
import os
import socket
import sys
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.WORKLOADS["tiny"](0)
        t = synth.draw_tensors(bench.rank_workload(wl, rank), with_grad=True)
        mine = (tuple(t["q"].shape), float(t["q"].double().abs().sum()), float(t["do"].double().abs().sum()))
        packs = [None] * world
        dist.all_gather_object(packs, mine)
        ms = 2.0 + 3.0 * rank  # the second rank is the slower one
        ms_max = bench.max_over_ranks(ms, dist)
        args = types.SimpleNamespace(workload="tiny", seed=0, warmup=0, steps=1)
        out = io.StringIO()
        with contextlib.redirect_stdout(out):
            rc = bench.run_reference(args)
        results.put((rank, packs, ms_max, rc, out.getvalue()))
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_ranks():
    ctx = mp.get_context("spawn")
    results = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        rank, *rest = results.get()
        got[rank] = rest
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return got


def test_each_rank_draws_its_own_values_for_the_same_shapes(two_ranks):
    packs = two_ranks[0][0]
    assert packs == two_ranks[1][0]          # both ranks saw the same gathered list
    (shape0, q0, do0), (shape1, q1, do1) = packs
    assert shape0 == shape1
    assert q0 != q1 and do0 != do1


def test_job_time_is_the_slowest_rank(two_ranks):
    assert two_ranks[0][1] == two_ranks[1][1] == 5.0


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    flop = 11.34e12
    assert bench.job_tflops(1, flop, 10.0) == pytest.approx(1134.0)
    # two ranks, each with the same pack, timed by the slower one: twice the work in the same time
    assert bench.job_tflops(2, flop, 10.0) == pytest.approx(2 * 1134.0)
    assert bench.max_over_ranks(3.5) == 3.5  # no process group: the rank's own value


def test_reference_arm_runs_on_rank_zero_only(two_ranks):
    rc0, out0 = two_ranks[0][2], two_ranks[0][3]
    rc1, out1 = two_ranks[1][2], two_ranks[1][3]
    assert rc0 == 0 and rc1 == 0
    assert out1 == ""
    lines = [l for l in out0.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
