"""The benchmark's JSON contract on CPU: the reference arm (the oracle, timed on the host) prints
one line with the metric, unit and direction of the GPU arm, its CPU-baseline description and an
end-to-end object with zero transfer bytes; non-zero ranks of a multi-rank launch print nothing."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env=None):
    e = dict(os.environ)
    if env:
        e.update(env)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                         capture_output=True, text=True, timeout=600, env=e)
    assert out.returncode == 0, out.stderr[-2000:]
    return [ln for ln in out.stdout.splitlines() if ln.strip()]


def test_reference_arm_line():
    lines = _run(["--impl", "reference", "--workload", "wgrad_tiny", "--steps", "2", "--warmup", "1"])
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == "MXFP8 grouped wgrad TFLOP/s" and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "wgrad_tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    lines = _run(["--impl", "reference", "--workload", "wgrad_tiny", "--steps", "1", "--warmup", "0"],
                 env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert lines == []


def test_cpu_baseline_sizes_its_sample_from_a_pilot():
    """The default run's CPU baseline: the oracle on a square grad_w block whose side is a
    multiple of 128, sized from the pilot toward the requested seconds, and described."""
    sys.path.insert(0, ROOT)
    import bench
    from moe_grouped_gemm_wgrad_gb300 import synth

    case = synth.wgrad_random(2048, 1024, 1024, [1024, 1024], seed=3)
    cb = bench.cpu_baseline(case, target_s=0.2)
    assert cb["kind"] == "oracle" and cb["unit"] == "TFLOP/s" and cb["cores"] == 1
    assert cb["value"] > 0 and cb["seconds"] > 0
    side = int(cb["sample"].split("grad_w block ")[1].split("x")[0])
    assert side % 128 == 0 and 128 <= side <= 1024
    assert "1024 tokens" in cb["sample"]


def test_clock_sampler_summarises_the_timed_window_without_a_csv():
    """The clock record needs no output folder: samples come through a drained pipe, only
    those inside the marked window are summarised, and active throttle reasons are named."""
    import datetime
    import time

    sys.path.insert(0, ROOT)
    import bench

    now = time.time()
    fmt = "%Y/%m/%d %H:%M:%S.%f"

    def line(t, mhz, cap):
        ts = datetime.datetime.fromtimestamp(t).strftime(fmt)[:-3]
        return f"{ts}, 0, {mhz}, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, {cap}"

    lines = [line(now - 50, 1000, "Not Active")]                    # before the window
    lines += [line(now - 5 + 0.1 * i, 1950 + i, "Active") for i in range(5)]
    lines += [line(now + 50, 500, "Not Active")]                    # after the window
    # many more lines than a pipe buffer holds, then wait to be terminated
    script = ("import sys, time\n"
              f"lines = {lines!r}\n"
              "filler = 'x' * 200\n"
              "for i in range(2000): print(filler)\n"
              "for l in lines: print(l)\n"
              "sys.stdout.flush()\n"
              "time.sleep(60)\n")
    sampler = bench.ClockSampler(0, cmd=[sys.executable, "-c", script], settle_s=0.0)
    deadline = time.time() + 30
    while len(sampler.lines) < 2000 + len(lines) and time.time() < deadline:
        time.sleep(0.05)
    sampler.mark(now - 10, now + 10)                  # the timed step ("step")
    sampler.mark(now - 4.85, now - 4.65, "leg")       # a second window: samples 2 and 3
    summary = sampler.stop()
    assert summary is not None
    leg = summary["leg"]
    assert leg["samples_in_timed_window"] == 2 and leg["sm_mhz"] == 1952.5
    assert summary["all"]["samples"] == 7
    clk = summary["step"]
    assert clk["samples_in_timed_window"] == 5 and clk["samples"] == 5
    assert clk["sm_mhz"] == 1952.0 and clk["sm_max_mhz"] == 2070.0
    assert clk["reasons"] == ["sw_power_cap"]


def test_clock_sampler_without_nvidia_smi_reports_nothing():
    sys.path.insert(0, ROOT)
    import bench

    sampler = bench.ClockSampler(0, cmd=["/nonexistent/nvidia-smi"], settle_s=0.0)
    assert sampler.stop() is None
