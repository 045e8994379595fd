"""The benchmark's multi-rank host logic on CPU ranks (gloo, world size 2):
rendezvous, max-over-ranks timing, the barrier, and the reference arm's
rank > 0 exit.  Replicas exchange no data; only timing is reduced."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, local = bench.dist_setup()
    elapsed = [0.25, 0.75][r]                       # rank 1 is the slow one
    m = bench.max_over_ranks(elapsed, w, "cpu")
    bench.barrier(w)
    # weak scaling: every rank ran its own T tokens, the job took the slowest rank's time
    tokens_per_s = w * 16384 * 10 / m
    q.put((r, w, local, m, tokens_per_s))
    dist.destroy_process_group()


def test_two_rank_max_timing_and_weak_scaling_value():
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
    assert [o[0] for o in out] == [0, 1]
    for r, w, local, m, tps in out:
        assert w == 2 and local == r
        assert m == 0.75                             # max over ranks, same on both
        assert tps == pytest.approx(2 * 16384 * 10 / 0.75)


def test_reference_arm_other_ranks_exit_without_work():
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    from mixture_experts_routing_router_gb300 import synth
    args = argparse.Namespace(gpus=2, steps=3, warmup=3)
    assert bench.run_reference(args, synth.WORKLOADS["large"], world=2, rank=1) == 0


def test_reference_arm_line_on_rank0(capsys):
    """Rank 0 of the reference arm times the oracle on a bounded sample and
    prints one JSON line with the contract's keys: its own value as the
    end-to-end figure (no host-device copies) and a cpu_baseline that names
    the host."""
    sys.path.insert(0, ROOT)
    import argparse
    import json

    import bench
    from mixture_experts_routing_router_gb300 import synth
    args = argparse.Namespace(gpus=1, steps=2, warmup=1)
    assert bench.run_reference(args, synth.WORKLOADS["tiny"], world=1, rank=0) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "tokens/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] == 1 and line["dtype"] == "f64"
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert "nproc" in cb and "cpu_model" in cb and cb["sample"]
