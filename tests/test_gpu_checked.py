"""GPU: the bounds-checked build (-DVITFP8_CHECKED) on the edge-case shapes.

The checked build compares every global- and shared-memory index its kernels
compute with the extent the arguments imply and records
VITFP8_ERR_DEVICE_BOUNDS (skipping the access) on a miss, so a kernel that
reads or writes outside its buffers shows up as an error word instead of a
silent wrong value.  This test builds it into libvitfp8_checked.so, runs the
ragged, tiny, 3000-segment, padded, fused-QKV and every-head-dim cases through
it in a subprocess (amax, quantize + un-pad, FP8 and BF16 attention), and
requires: every device error word 0; 4 KB canary bands before and after every
code and output buffer untouched; and codes and outputs bit-identical to the
normal build's (the checks change no result).  The bounds self-test shows the
check itself fires: the checked build records VITFP8_ERR_DEVICE_BOUNDS for an
index one past a buffer (never accessed), the normal build records nothing.
"""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def _build_checked():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_vitfp8_build", os.path.join(ROOT, "fp8_vision_encoder_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build(checked=True)


def test_checked_build_clean_and_identical(tmp_path):
    import fp8_vision_encoder_gb300 as vf
    import checked_cases
    assert torch.cuda.is_available()
    lib = _build_checked()
    out = str(tmp_path / "checked.npz")
    env = dict(os.environ, VITFP8_LIBRARY=lib,
               PYTHONPATH=os.pathsep.join([ROOT, os.path.join(ROOT, "tests")]))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_cases.py"), out],
                       env=env, cwd=ROOT, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:]
    chk = np.load(out)
    ref = checked_cases.run_cases(vf)

    assert int(chk["checked_build"][0]) == 1 and int(ref["checked_build"][0]) == 0
    assert int(chk["selftest_bounds"][0]) == 5       # VITFP8_ERR_DEVICE_BOUNDS
    assert int(ref["selftest_bounds"][0]) == 0
    names = sorted(k for k in ref if k.endswith(".errors"))
    assert len(names) >= 21
    for k in names:
        case = k[:-len(".errors")]
        assert chk[k].tolist() == [0, 0, 0], (case, chk[k].tolist())
        assert ref[k].tolist() == [0, 0, 0], (case, ref[k].tolist())
        assert chk[case + ".bands"].all(), (case, "checked build wrote into a canary band")
        assert ref[case + ".bands"].all(), (case, "normal build wrote into a canary band")
        for part in ("q8", "k8", "v8t", "o", "o16"):
            a, b = chk[case + "." + part], ref[case + "." + part]
            assert a.shape == b.shape and np.array_equal(a, b), (case, part)
