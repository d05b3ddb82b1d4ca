"""Host-side logic of bench.py (CPU only): the multi-rank aggregation over a
world_size-2 gloo group, the throughput arithmetic and the reference arm's
rank handling."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out_q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out_q.put((rank, bench.max_over_ranks(values[rank], world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    values = [3.25, 7.5]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 7.5, 1: 7.5}


def test_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    one = bench.job_throughput(4096, 1, 10, 25.0)
    two = bench.job_throughput(4096, 2, 10, 25.0)
    assert one == pytest.approx(4096 * 10 / 0.025)
    assert two == pytest.approx(2 * one)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "tiny_f32"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_one_contract_line_on_rank_0():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "tiny_f32"], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0


def test_clock_summary_keeps_samples_inside_the_timed_window():
    sys.path.insert(0, ROOT)
    import bench
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.source, cs.error, cs.window = "nvml", None, (10.0, 11.0)
    cs.samples = [(9.5, 2032.0, 2032.0, 200.0, []),                # before the window
                  (10.2, 1900.0, 2032.0, 900.0, ["sw_power_cap"]),
                  (10.6, 1800.0, 2032.0, 950.0, []),
                  (10.9, 2000.0, 2032.0, 800.0, []),
                  (11.5, 600.0, 2032.0, 100.0, ["hw_slowdown"])]    # after it
    s = cs.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1900.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 950.0


def test_clock_sampler_places_smi_lines_by_their_own_timestamps():
    """Lines from `nvidia-smi -lms` reach the pipe in bursts; each sample must
    be placed at the time nvidia-smi took it, not when the line was read."""
    import datetime
    import io
    sys.path.insert(0, ROOT)
    import bench
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.source, cs.error, cs.samples = "nvidia-smi", None, []
    lines = ["2026/12/03 04:55:37.107, 1222, 2032, 590.57, Not Active, Not Active, Not Active, Active\n",
             "2026/12/03 04:55:37.127, 1230, 2032, 600.00, Not Active, Not Active, Not Active, Active\n",
             "garbage line\n"]
    cs.proc = type("P", (), {"stdout": io.StringIO("".join(lines))})()
    cs._read_smi()
    assert len(cs.samples) == 2
    t0 = datetime.datetime(2026, 12, 3, 4, 55, 37, 107000).timestamp()
    assert abs(cs.samples[0][0] - t0) < 1e-3 and abs(cs.samples[1][0] - t0 - 0.02) < 1e-3
    assert cs.samples[0][1:4] == (1222.0, 2032.0, 590.57) and cs.samples[0][4] == ["sw_power_cap"]
    cs.window = (t0 - 0.001, t0 + 0.05)
    s = cs.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 1226.0 and s["reasons"] == ["sw_power_cap"]


def test_recorded_traffic_is_dropped_once_the_kernel_source_changes(tmp_path, monkeypatch):
    """roofline.traffic comes from a committed ncu capture only while the kernel
    source it was taken on is unchanged: a stale hash reads as no figure."""
    sys.path.insert(0, ROOT)
    import bench
    csrc = tmp_path / "csrc"
    csrc.mkdir()
    (csrc / "k.cu").write_text("__global__ void k() {}\n")
    monkeypatch.setattr(bench, "CSRC", str(csrc))
    entry = {"sources": ["k.cu"], "dram_bytes_per_launch": 12345, "source_sha256_16": bench.source_hash(["k.cu"])}
    tf = tmp_path / "traffic.json"
    tf.write_text(json.dumps({"w": entry}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tf))
    assert bench.recorded_traffic("w") == 12345
    assert bench.recorded_traffic("other") is None
    (csrc / "k.cu").write_text("__global__ void k() { /* changed */ }\n")
    assert bench.recorded_traffic("w") is None

