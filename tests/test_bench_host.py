"""CPU: the host-side logic of bench.py: the host-mirror placement policy, the
whole-job rate and the max-over-ranks reduction with two gloo ranks, and the
reference arm under torchrun with two ranks (rank 0 alone prints)."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_placement_mask_coldest_first_shared_last():
    w = gen.get_workload(1)  # 512 routed experts, Zipf router bias, a shared expert
    n = w.n_experts_total
    assert bench.placement_mask(w, 0.0, 0) is None
    m = bench.placement_mask(w, 0.25, 0)
    assert m.dtype == bool and m.shape == (n,) and int((~m).sum()) == round(0.25 * n)
    assert m[w.E], "the always-used shared expert keeps its HBM slot"
    bias = gen.router_bias(w)
    host = np.where(~m[:w.E])[0]
    hbm = np.where(m[:w.E])[0]
    assert bias[host].max() <= bias[hbm].min(), "the mirror holds the coldest experts"
    full = bench.placement_mask(w, 1.0, 0)
    assert not full.any(), "everything in the mirror, the shared expert last"
    no_bias = gen.get_workload(0)  # no router bias: ties by expert index
    m0 = bench.placement_mask(no_bias, 0.5, 0)
    k = int((~m0).sum())
    assert np.array_equal(np.where(~m0)[0], np.arange(k))


def test_job_rate():
    assert bench.job_rate(1, 1, 32, 2000, 1.0) == 64000
    assert bench.job_rate(2, 1, 32, 2000, 2.0) == 64000  # weak scaling, slowest rank's time


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(1.5 + rank, world)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    assert got == {0: 2.5, 1: 2.5}
    assert bench.max_over_ranks(3.0, 1) == 3.0


def test_reference_arm_two_ranks_rank0_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--workload", "0", "--steps", "3", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
