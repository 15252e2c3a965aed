"""bench.py's host logic on CPU: the reference arm's JSON line (the oracle on a
bounded sample), the silent exit of ranks other than 0, the one-line refusal
of a run on several GPUs, and the summary of the clock samples taken during a
timed region."""
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


def test_several_gpus_print_unavailable_and_touch_no_gpu():
    # the path runs on one GPU: --gpus 2 (launched as two ranks) gives one line
    # from rank 0 with an "unavailable" key, nothing from rank 1, exit 0 on both,
    # and no CUDA call (this host has no GPU, so any would fail)
    for rank, expect_line in ((0, True), (1, False)):
        p = _run({"RANK": str(rank), "WORLD_SIZE": "2", "LOCAL_RANK": str(rank),
                  "CUDA_VISIBLE_DEVICES": ""}, "--gpus", "2", "--steps", "3", "--warmup", "3")
        assert p.returncode == 0, p.stderr
        lines = [x for x in p.stdout.splitlines() if x.strip()]
        if not expect_line:
            assert lines == []
            continue
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "tdg" and d["n_gpus"] == 2 and "one GPU" in d["unavailable"]
        assert "value" not in d
    # the flag alone (one process) is refused the same way
    p = _run({"CUDA_VISIBLE_DEVICES": ""}, "--gpus", "4")
    assert p.returncode == 0 and json.loads(p.stdout.strip())["n_gpus"] == 4
