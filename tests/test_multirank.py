"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): each rank
decodes its own replica, the reported step time is the maximum over ranks, and
only rank 0 runs and prints the CPU reference leg."""
from __future__ import annotations

import io
import os
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank)  # rank 1 is the slow replica
        # the reference leg: rank 0 alone does the CPU work and prints one line
        class Args:
            workload, ref_frames, warmup, steps, gpus = "tiny_cal", 2, 0, 1, world
        buf = io.StringIO()
        with redirect_stdout(buf):
            rc = bench.run_reference(Args, rank, world)
        q.put((rank, got, rc, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rank0_reference():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, got, rc, out = q.get(timeout=300)
        res[rank] = (got, rc, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == res[1][1] == 0
    assert '"impl": "reference"' in res[0][2] and res[0][2].count("\n") == 1
    assert res[1][2] == ""


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5


def test_every_workload_has_a_sample_rate_and_config():
    """bench.py can report every workload it accepts (--workload choices)."""
    import bench
    from dac_vocoder_decode_gb300 import workloads as W
    for name in W.WORKLOADS:
        assert name in bench.SAMPLE_RATE, name
        wl = W.make_workload(name, T=2, B=1)
        cfg = bench.config_of(wl, name)
        assert cfg["sample_rate"] == bench.SAMPLE_RATE[name]
    for name in W.ENC_WORKLOADS:  # encoder workloads: audio in, latents out
        assert name in bench.SAMPLE_RATE, name
        wl = bench.load_workload(name, frames=2)
        cfg = bench.workload_config(wl, name)
        assert cfg["sample_rate"] == bench.SAMPLE_RATE[name]
        assert cfg["latent"][2] * cfg["hop"] == cfg["audio"][2]
        assert bench.metric_of(name) == bench.ENC_METRIC
