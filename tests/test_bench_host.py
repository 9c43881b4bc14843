"""bench.py host logic without a GPU: the reference arm (the CPU oracle),
its silence on ranks other than 0, the replica aggregation over two gloo
ranks, and the byte count the headline metric divides by."""
import json
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from tests.conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _run_bench(args, env_extra=None, timeout=300):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                          env=env, timeout=timeout, cwd=ROOT)


def test_reference_arm_prints_the_contract_line():
    r = _run_bench(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] >= 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == bench.host_cores()
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("tiny")


def test_cpu_baseline_reports_all_cores_and_one():
    """The oracle timed on every host core (one spawned process each) and on
    one, over whole steps of the config's first token."""
    d = bench.cpu_baseline("tiny")
    assert d["kind"] == "oracle" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cores"] == bench.host_cores()
    one = d["single_core"]
    assert one["cores"] == 1 and one["value"] > 0 and one["kind"] == "oracle"
    assert "top-2" in d["sample"] and "spawned" in d["sample"]


def test_reference_arm_runs_on_rank_0_only():
    r = _run_bench(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "1"],
                   {"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def _replica_rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank  # rank 1 is the slower replica
    total = bench.max_over_ranks(ms, dist, "cpu")
    out[rank] = (total, bench.replica_throughput(world, 1e9, total))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_over_gloo():
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_replica_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # two replicas of 1 GB each in the slower rank's 15 ms
    assert res[0][1] == pytest.approx(2 * 1e9 / 15e-3 / 1e9)


def test_single_process_needs_no_collective():
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5


def test_step_bytes_match_the_pages():
    """Second page, table "Bytes decide it before the kernel runs": 288
    experts of NVFP4 w13 + w2 at H=4096, I=2048 are 4.077 GB (2.718 + 1.359)."""
    from nvfp4_block_scaled_gather_gb300.synthetic import CONFIGS
    cfg = CONFIGS["decode_m1"]
    assert bench.expert_bytes(cfg.H, cfg.I) * 288 == 4_076_863_488
    assert bench.expert_bytes(cfg.H, cfg.I) == 14_155_776
    T, G = 1, 8
    assert bench.step_bytes(cfg, G, T) == G * 14_155_776 + 4 * T * cfg.H + 8 * T * cfg.k + 12 * cfg.E


def test_recorded_traffic_is_tied_to_the_kernel_source(tmp_path, monkeypatch):
    """The ncu traffic figure is reported only for the GEMM source it was
    measured on (its translation unit and headers); any change voids it."""
    f = tmp_path / "traffic.txt"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    f.write_text(f"kernel_source_sha256_16: {bench.gemm_source_sha()}\ndram_bytes_per_launch: 123456\n")
    assert bench.recorded_traffic() == 123456
    f.write_text("kernel_source_sha256_16: 0000000000000000\ndram_bytes_per_launch: 123456\n")
    assert bench.recorded_traffic() is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.txt"))
    assert bench.recorded_traffic() is None
