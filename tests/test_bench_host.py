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


def test_profile_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    """The roofline's `traffic` comes from a committed ncu summary only while the
    kernel's translation unit and the local headers it includes (followed
    through other headers) hash as they did when the summary was written; a
    header it does not include does not matter."""
    csrc = tmp_path / "csrc"
    csrc.mkdir()
    (csrc / "k.cu").write_text('#include "a.cuh"\n__global__ void kern() {}\n')
    (csrc / "a.cuh").write_text('#include "b.cuh"\n// a\n')
    (csrc / "b.cuh").write_text("// b\n")
    (csrc / "other.cuh").write_text("// not included\n")
    sha = bench.sources_sha256(str(csrc), "k.cu")
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "kern_wl.md").write_text(
        f"# kern\n\ndram_bytes_per_launch: 12345\nsource_unit: k.cu\nsource_sha256: {sha}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile("kern", "wl", str(csrc)) == 12345.0
    (csrc / "other.cuh").write_text("// changed, still not included\n")
    assert bench.traffic_from_profile("kern", "wl", str(csrc)) == 12345.0
    (csrc / "b.cuh").write_text("// b changed\n")  # included through a.cuh
    assert bench.traffic_from_profile("kern", "wl", str(csrc)) is None
    assert bench.traffic_from_profile("kern", "missing", str(csrc)) is None


def test_prefill_flops_count_the_routed_pairs():
    """bench.prefill_flops: 2 (T k + T) 2I H FLOPs for the gate/up GEMM (the
    routed pairs and the shared expert's tokens), and the MMA's padding of each
    work item of at most 128 tokens to a multiple of 16, on hand-counted items."""
    w = gen.get_workload(4)
    counts = np.zeros(w.E, dtype=np.int64)
    counts[:3] = [1, 130, 16]  # experts with 1, 130 (items of 128 and 2) and 16 tokens
    algo, as_run = bench.prefill_flops(w, counts)
    unit = 2.0 * 2 * w.I * w.H  # FLOPs of one token through one expert's gate/up
    assert algo == unit * (1 + 130 + 16 + w.T)
    # items padded: 1 -> 16; 130 -> 128 + 16; 16 -> 16; the shared 4096 -> 32 x 128
    assert as_run == unit * (16 + 128 + 16 + 16 + 4096)
    assert bench.prefill_flops(w, np.zeros(w.E))[0] == unit * w.T * w.shared
