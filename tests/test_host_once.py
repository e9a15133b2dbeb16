"""CPU: the per-device, thread-safe set-up table the library's host code uses.

The attention kernels opt into more than 48 KB of shared memory with a
per-device CUDA attribute; the library records that set-up once per device
under a lock (``csrc/host_once.h``).  This test compiles a small C++ program
against that header with g++ (no CUDA involved) and runs it: 16 threads asking
for all 64 device slots run each slot's set-up exactly once, a failed set-up is
retried, and indices outside the table are refused.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_per_device_once_table(tmp_path):
    exe = str(tmp_path / "host_once_test")
    subprocess.run(["g++", "-std=c++17", "-O1", "-pthread",
                    "-I", os.path.join(ROOT, "fp8_vision_encoder_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "cpp", "host_once_test.cpp"), "-o", exe],
                   check=True)
    r = subprocess.run([exe], stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=120)
    assert r.returncode == 0, r.stdout
    assert "host_once ok" in r.stdout


def test_library_keeps_no_unguarded_static_flags():
    """No kernel file keeps a plain ``static bool`` set-up flag (per process,
    unsynchronised); per-device set-up goes through PerDeviceOnce."""
    csrc = os.path.join(ROOT, "fp8_vision_encoder_gb300", "csrc")
    for name in os.listdir(csrc):
        if name.endswith((".cu", ".cuh", ".h")):
            text = open(os.path.join(csrc, name)).read()
            assert "static bool" not in text, name
