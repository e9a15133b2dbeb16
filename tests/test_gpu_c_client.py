"""GPU: the library driven from plain C through its ABI alone.

tests/c_client/vitfp8_client.c allocates with cudaMalloc, runs dynamic
scaling, quantization and attention for a few forwards, runs the last
forward's codes through each named attention kernel, takes the
calibrate-once scale-file values of the state on the device, and writes the
scale state, the outputs and those values; all are compared with the oracle.
"""

import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import workloads
from oracle import calib as ocalib, quant as oquant, scales as oscales

from gpu_util import assert_attention_ok, compare_attention, np32, oracle_push, state_matches

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _build_client(tmp):
    import fp8_vision_encoder_gb300 as vf
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdir = os.path.dirname(vf.LIB_PATH)
    exe = os.path.join(tmp, "vitfp8_client")
    cc = shutil.which("gcc") or "cc"
    cmd = [cc, "-O2", "-std=c11", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_client", "vitfp8_client.c"), "-o", exe,
           "-L", libdir, "-lvitfp8", "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           "-Wl,-rpath," + libdir + ":" + os.path.join(cuda, "lib64")]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    assert r.returncode == 0, r.stdout
    return exe


def test_plain_c_client_matches_oracle(tmp_path):
    import fp8_vision_encoder_gb300 as vf
    seqlens, H, D, seeds = [64, 192, 17, 0, 300], 2, 80, [3, 4, 5]
    T = sum(seqlens)
    cu = np.cumsum([0] + seqlens).astype(np.int32)
    inp = os.path.join(str(tmp_path), "in.bin")
    ost = oscales.ScaleState()
    with open(inp, "wb") as f:
        f.write(np.array([T, H, D, len(seqlens), len(seeds)], dtype=np.int32).tobytes())
        f.write(cu.tobytes())
        for seed in seeds:
            q, k, v = workloads.make_qkv(seqlens, H, D, seed, True, True)
            for t in (q, k, v):
                f.write(t.contiguous().view(torch.int16).numpy().tobytes())
            oracle_push(ost, q, k, v)
    exe = _build_client(str(tmp_path))
    outp = os.path.join(str(tmp_path), "out.bin")
    r = subprocess.run([exe, inp, outp], stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stdout
    raw = open(outp, "rb").read()
    nst = vf.STATE_BYTES
    s = vf._StateStruct.from_buffer_copy(raw[:nst])
    state = {"hist": [list(s.hist[t]) for t in range(3)], "pos": s.pos, "count": s.count,
             "mode": s.mode, "amax_ref": list(s.amax_ref), "scale": list(s.scale),
             "inv_scale": list(s.inv_scale), "amax_cur": list(s.amax_cur),
             "amax_bits": list(s.amax_bits), "blocks_done": s.blocks_done, "dev_error": s.dev_error}
    state_matches(state, ost)
    nout = T * H * D * 2
    out = torch.from_numpy(np.frombuffer(raw[nst:nst + nout], dtype=np.int16).copy()).view(torch.bfloat16)
    out = out.reshape(T, H, D)
    # calibrate-once from C: float32(ring max) * float32(1.5), bit for bit
    saved = np.frombuffer(raw[nst + nout:nst + nout + 12], dtype=np.float32)
    want = np.asarray(ocalib.saved_values(np.asarray(ost.hist, dtype=np.float32).max(axis=1), 1.5),
                      dtype=np.float32)
    assert np.array_equal(saved.view(np.uint32), want.view(np.uint32)), (saved, want)
    # oracle codes of the last forward (bit-exact with the library's, checked elsewhere)
    codes = [torch.from_numpy(oquant.quantize(np32(x), ost.inv_scale[t]))
             for t, x in enumerate((q, k, v))]
    stats = compare_attention(out, codes[0], codes[1], codes[2], list(ost.scale), [int(x) for x in cu], D)
    assert_attention_ok(stats, "C client", outliers=True)
    # the same codes through vitfp8_attn_varlen_kernel with each named kernel:
    # unit and persistent give the same bits, the two two-tile forms too, and
    # every one is within the bound of the oracle
    kout = np.frombuffer(raw[nst + nout + 12:nst + nout + 12 + 4 * nout], dtype=np.int16).reshape(4, T, H, D)
    assert np.array_equal(kout[0], kout[1]) and np.array_equal(kout[2], kout[3])
    for i, name in enumerate(("unit", "persistent", "two-tile", "persistent two-tile")):
        o = torch.from_numpy(kout[i].copy()).view(torch.bfloat16)
        stats = compare_attention(o, codes[0], codes[1], codes[2], list(ost.scale), [int(x) for x in cu], D)
        assert_attention_ok(stats, "C client, " + name, outliers=True)
