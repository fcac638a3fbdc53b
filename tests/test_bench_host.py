"""Host logic of bench.py without a GPU: the N > 1 replica aggregation over gloo
ranks (slowest rank's time, bytes of all ranks), the profile-digest check and the
reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, value = bench.aggregate(1.0 + rank, 1_000_000, world, dist, "cpu")
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_aggregation_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    # both ranks see the slowest rank's 2.0 ms; value = 2 ranks x 1 MB / 2 ms
    for r in range(2):
        ms, value = out[r]
        assert ms == 2.0
        assert abs(value - 2 * 1_000_000 / 2e-3 / 1e9) < 1e-9


def test_single_rank_aggregation():
    import bench
    ms, value = bench.aggregate(0.5, 2_000_000, 1)
    assert ms == 0.5 and abs(value - 4.0) < 1e-12


def test_profile_traffic_requires_matching_digest(tmp_path, monkeypatch):
    import bench
    # the committed summary names the digest of the current kernel source or is ignored
    t = bench.read_profile_traffic()
    assert t is None or t > 1e8


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                         timeout=120, cwd=ROOT, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_reference_arm_matches_the_headline_config():
    import bench
    # both arms describe the same workload (the driver compares the two lines) and
    # the reference arm runs the warm-up it was asked for
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["config"] == bench.headline_config(2, 1)
    assert line["warmup"] == 1 and line["steps"] == 2
    assert line["cpu_baseline"]["cores"] == bench.host_threads()


def test_oracle_config_time_on_a_sample():
    import bench
    import workloads as wl
    # the per-config oracle time comes from a bounded sample scaled to the batch
    inp = wl.make_batch(512, (64, 32), 100, "q4", seed=3)
    ms, frac = bench.oracle_config_ms(inp, threads=2, budget_macs=4e5)
    assert ms > 0 and 0 < frac < 1
    ms_full, frac_full = bench.oracle_config_ms(wl.make_batch(64, (16,), 2, "bf16", seed=3), threads=2)
    assert frac_full == 1.0 and ms_full > 0
