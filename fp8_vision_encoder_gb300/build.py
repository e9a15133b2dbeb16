"""Build libvitfp8.so in-tree with nvcc for sm_103a (no cmake, no torch build).

Usage: ``python fp8_vision_encoder_gb300/build.py`` or ``build()``.  The
translation units compile in parallel; the CUDA runtime is linked statically
so the library loads without a separate libcudart on the path.
"""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libvitfp8.so")
LIB_CHECKED = os.path.join(PKG, "libvitfp8_checked.so")
SOURCES = ["api.cu", "quant.cu", "attn_fp8.cu", "attn_fp8_2tile.cu", "attn_bf16.cu", "attn_noalloc.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: %s\n%s" % (" ".join(cmd), r.stdout))
    return r.stdout


def build(verbose=False, extra_flags=(), checked=False):
    """Compile every CUDA source and link libvitfp8.so next to this file.

    checked=True builds the bounds-checked variant (-DVITFP8_CHECKED) into
    libvitfp8_checked.so instead, from its own object directory.
    """
    build_dir = BUILD + ("_checked" if checked else "")
    lib = LIB_CHECKED if checked else LIB
    flags = list(extra_flags) + (["-DVITFP8_CHECKED"] if checked else [])
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmds.append([nvcc, *ARCH, *FLAGS, *flags, "-c", os.path.join(CSRC, src), "-o", obj])
    with ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        outs = list(ex.map(_run, cmds))
    if verbose:
        for o in outs:
            sys.stdout.write(o)
    tmp = lib + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, extra_flags=("-Xptxas", "-v") if "-v" in sys.argv else (),
                checked="--checked" in sys.argv))
