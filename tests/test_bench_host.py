"""bench.py's host logic on CPU: the reference arm's JSON line (the oracle on a
bounded sample), the silent exit of ranks other than 0, the summary of the
clock samples taken during a timed region, and, with two gloo ranks, the
slowest-rank time and whole-job throughput that several replicas report."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _run(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    p = _run({}, "--impl", "reference", "--steps", "1", "--warmup", "0")
    assert p.returncode == 0, p.stderr
    lines = [x for x in p.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["metric"] == "AG-GEMM+GEMM-RS TFLOP/s (qwen32b_mlp_tp8)"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == bench.WORKLOAD


def test_reference_arm_other_ranks_exit_without_work():
    p = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--impl", "reference", "--gpus", "2",
             "--steps", "1", "--warmup", "0")
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def _fake_clocks(tmp_path, lines, start_line=0):
    c = bench.Clocks(0)
    c.path = str(tmp_path / "clocks.csv")
    with open(c.path, "w") as f:
        f.write("".join(x + "\n" for x in lines))
    c.proc = object()          # a sampler ran
    c.start_line = start_line
    return c


def test_clock_summary_takes_loaded_samples_and_reasons(tmp_path):
    row = "0, {sm}, 2070, {pw}, 0x0, {hw}, Not Active, Not Active, {cap}"
    lines = [row.format(sm=900, pw=150.0, hw="Not Active", cap="Not Active"),     # before the region
             row.format(sm=2070, pw=900.5, hw="Not Active", cap="Not Active"),
             row.format(sm=1950, pw=1390.0, hw="Not Active", cap="Active"),
             row.format(sm=2010, pw=1200.0, hw="Not Active", cap="Not Active"),
             row.format(sm=1200, pw=120.0, hw="Not Active", cap="Not Active")]    # idle, ignored
    s = _fake_clocks(tmp_path, lines, start_line=1).summary()
    assert s["samples"] == 4
    assert s["sm_mhz"] == 2010.0          # median of the loaded samples (power above 300 W)
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w_max"] == 1390.0


def test_clock_summary_reports_slowdowns_and_missing_samples(tmp_path):
    row = "0, 1500, 2070, 800, 0x8, Active, Active, Not Active, Not Active"
    s = _fake_clocks(tmp_path, [row]).summary()
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    assert s["sm_mhz"] == 1500.0
    assert _fake_clocks(tmp_path, []).summary()["reasons"] == ["no samples"]
    assert bench.Clocks(0).summary()["reasons"] == ["nvidia-smi unavailable"]   # no sampler ran


def test_peaks_read_the_measured_file():
    pk = bench.peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        assert pk["src"] == "measured" and pk["hbm"] == d["hbm_gbs"] and pk["bf16"] == d["bf16_tflops"]
    else:
        pytest.skip("no measured peaks in this checkout")


def _rank_worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [70.0, 75.5][rank]           # rank 1 is the slower one
        worst = bench.max_over_ranks(local_ms, dist, torch, "cpu")
        q.put((rank, worst, bench.job_tflops(world, 4.0e12, 50, worst)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank_and_the_whole_job():
    import socket
    import torch.multiprocessing as mp
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_rank_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, tflops in res:
        assert worst == 75.5
        # both ranks' 50 steps of 4 TFLOP over the slowest rank's 75.5 ms
        assert tflops == pytest.approx(2 * 4.0e12 * 50 / 75.5e-3 / 1e12)


def test_one_process_needs_no_group():
    assert bench.max_over_ranks(12.5, None, None, "cpu") == 12.5
    assert bench.job_tflops(1, 1e12, 10, 1000.0) == pytest.approx(10.0)
