"""CPU: bench.py's reference arm (the oracle timed on the host cores) keeps the
bench contract -- one JSON line from rank 0 only, the other ranks exit 0 --
when run alone and under torchrun with two ranks."""

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"]


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check_line(line, n):
    assert line["impl"] == "reference" and line["n_gpus"] == n
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def _env():
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""
    return env


def test_reference_arm_one_gpu():
    r = subprocess.run([sys.executable, "bench.py"] + ARGS, cwd=ROOT, env=_env(),
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 1)


def test_reference_arm_two_ranks_prints_one_line():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2"] + ARGS
    r = subprocess.run(cmd, cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 2)


def test_clock_sampler_with_a_fake_nvidia_smi(tmp_path, monkeypatch):
    """SM clock median, max clock and throttle reasons from nvidia-smi's CSV
    lines (a stand-in script on PATH prints three samples, then waits)."""
    fake = tmp_path / "nvidia-smi"
    fake.write_text(
        "#!/bin/sh\n"
        "echo '0, 2070, 2070, 1201.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active'\n"
        "echo '0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active'\n"
        "echo '0, 2070, 2070, 1100.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active'\n"
        "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", str(tmp_path) + os.pathsep + os.environ["PATH"])
    sys.path.insert(0, ROOT)
    try:
        import bench
    finally:
        sys.path.remove(ROOT)
    import time
    s = bench.ClockSampler(0)
    s.start()
    time.sleep(1.0)
    r = s.stop()
    assert r == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_records_the_timing_rules_reject():
    sys.path.insert(0, ROOT)
    try:
        import bench
    finally:
        sys.path.remove(ROOT)
    rec = lambda mhz, reasons: {"sm_mhz": mhz, "sm_max_mhz": 2070.0, "reasons": reasons, "samples": 9}
    assert not bench.clocks_rejected(None)
    assert not bench.clocks_rejected(rec(2070.0, []))
    assert not bench.clocks_rejected(rec(1500.0, ["sw_power_cap"]))   # power cap: kept
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected(rec(2070.0, [r]))
    assert bench.clocks_rejected(rec(1200.0, []))                      # held low, no reason
    assert not bench.clocks_rejected(rec(1900.0, []))
