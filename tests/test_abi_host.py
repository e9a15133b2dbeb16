"""Host-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before launching anything.  No GPU
is needed: every call here fails validation on the host first."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vitfp8.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vitfp8_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def vf():
    import fp8_vision_encoder_gb300 as vf
    return vf


def test_header_declares_the_path_entry_points():
    names = _declared_functions()
    for n in ("vitfp8_amax_update", "vitfp8_set_static_scales", "vitfp8_quantize_unpad",
              "vitfp8_attn_varlen", "vitfp8_scale_state_init"):
        assert n in names


def test_library_exports_every_declared_symbol(vf):
    lib = ctypes.CDLL(vf.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert missing == []


def test_state_struct_size_matches_header_layout(vf):
    # 3x16 floats + 4 int32 + 4x3 floats + 3 uint32 + 1 uint32
    assert vf.STATE_BYTES == 3 * 16 * 4 + 4 * 4 + 4 * 3 * 4 + 3 * 4 + 4


def test_status_strings(vf):
    for code in range(8):
        assert vf._lib.vitfp8_status_string(code)
    assert vf._lib.vitfp8_status_string(99) == b"unknown status"


def test_sizes(vf):
    assert vf.vt_stride(10800) == 10800
    assert vf.vt_stride(257) == 272
    assert vf.vt_stride(0) == 0
    assert vf.workspace_size(3) >= 64 + 4 * 7
    assert vf.workspace_size(3) % 256 == 0


P = ctypes.c_void_p


def test_validation_rejects_without_launch(vf):
    lib = vf._lib
    good = P(1 << 20)           # 16-byte aligned fake device address, never dereferenced
    odd = P((1 << 20) + 4)
    lay = vf.SrcLayout.packed(2, 128)
    st = vf._state_init
    assert st(P(0), P(0)) == 1
    assert vf._set_static(good, 0.0, 1.0, 1.0, P(0)) == 1
    assert vf._set_static(good, float("nan"), 1.0, 1.0, P(0)) == 1
    assert vf._set_static(good, 1.0, float("inf"), 1.0, P(0)) == 1
    assert vf._set_static(good, 1.0, 1.0, -2.0, P(0)) == 1
    # amax: bad D, H, misaligned source, bad strides
    assert vf._amax_update(good, good, good, good, ctypes.byref(lay), good, 1, 10, 2, 12, P(0)) == 1
    assert vf._amax_update(good, good, good, good, ctypes.byref(lay), good, 1, 10, 0, 128, P(0)) == 1
    assert vf._amax_update(good, odd, good, good, ctypes.byref(lay), good, 1, 10, 2, 128, P(0)) == 1
    bad = vf.SrcLayout(0, 0, 0, 13, 128)
    assert vf._amax_update(good, good, good, good, ctypes.byref(bad), good, 1, 10, 2, 128, P(0)) == 1
    assert vf._amax_update(good, good, good, good, ctypes.byref(lay), good, -1, 10, 2, 128, P(0)) == 1
    assert vf._amax_update(good, good, good, good, None, good, 1, 10, 2, 128, P(0)) == 1
    assert vf._amax_update(good, good, good, good, ctypes.byref(lay), good, 1, 10, 2, 264, P(0)) == 2
    # empty input is a successful no-op (nothing launched)
    assert vf._amax_update(good, good, good, good, ctypes.byref(lay), good, 0, 0, 2, 128, P(0)) == 0
    # quantize: D_pad checks
    q = vf._quantize_unpad
    assert q(good, good, good, good, ctypes.byref(lay), good, 1, 10, 2, 128, 120, good, good, good, P(0)) == 1
    assert q(good, good, good, good, ctypes.byref(lay), good, 1, 10, 2, 80, 88, good, good, good, P(0)) == 1
    assert q(good, good, good, good, ctypes.byref(lay), good, 1, 10, 2, 128, 128, P(0), good, good, P(0)) == 1
    assert q(good, good, good, good, ctypes.byref(lay), good, 1, 10, 2, 128, 128, good, odd, good, P(0)) == 1
    # attention
    a = vf._attn
    ws = vf.workspace_size(1)
    args = [good, good, good, good, good, 1, 10, 10, 2, 128, 128, 0.088, good, good, ws, P(0)]

    def call(**kw):
        x = list(args)
        names = ["q8", "k8", "v8t", "st", "cu", "nseq", "maxlen", "T", "H", "D", "Dp", "sm",
                 "out", "ws", "wsb", "stream"]
        for k, v in kw.items():
            x[names.index(k)] = v
        return a(*x)

    assert call(D=256, Dp=256) == 2            # head dim above the kernel's limit
    assert call(D=136, Dp=144) == 2
    assert call(Dp=120) == 1
    assert call(sm=0.0) == 1
    assert call(sm=float("nan")) == 1
    assert call(H=0) == 1
    assert call(out=P(0)) == 1
    assert call(out=odd) == 1
    assert call(ws=P(0)) == 7
    assert call(wsb=ws - 1) == 7
    assert call(nseq=0, T=0) == 0              # empty: no-op
    # calibrate once: margin must be finite and positive, the static state distinct
    cs = vf._calibrated
    assert cs(P(0), 1.5, P(0), P(0), P(0)) == 1
    assert cs(good, 0.0, P(0), P(0), P(0)) == 1
    assert cs(good, float("nan"), P(0), P(0), P(0)) == 1
    assert cs(good, float("inf"), P(0), P(0), P(0)) == 1
    assert cs(good, 1.5, P((1 << 20) + 2), P(0), P(0)) == 1   # d_saved not 4-byte aligned
    assert cs(good, 1.5, P(0), good, P(0)) == 1     # d_static == d_dynamic
    # self-test arguments
    assert vf._selftest_bounds(P(0), 256, P(0)) == 1
    assert vf._selftest_bounds(good, 8, P(0)) == 1
    assert vf._checked_build() in (0, 1)


def test_oracle_and_product_share_no_code():
    """Neither side imports, loads or links the other (static check of the sources)."""
    imp_oracle = re.compile(r"^\s*(from|import)\s+oracle\b", re.M)
    imp_pkg = re.compile(r"^\s*(from|import)\s+fp8_vision_encoder_gb300\b|libvitfp8|CDLL", re.M)
    pkg = os.path.join(ROOT, "fp8_vision_encoder_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not imp_oracle.search(src), f
                assert "oracle/" not in src, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            src = open(os.path.join(ROOT, "oracle", f)).read()
            assert not imp_pkg.search(src), f
