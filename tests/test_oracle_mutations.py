"""CPU: the oracle's pins catch plausible mistakes in the oracle.

Each case plants one mistake in one oracle function -- a wrong exponent bias,
a rounding mode, a dropped saturation, swapped scale factors, a ring of the
wrong length, the other ring order, a missing absolute value, a dropped
softmax scale, a transposed score matrix, a wrong normaliser, keys taken
across segments, a multiplier used as a divisor, a smaller P shift, a
floored P reference, a scale file without its margin or with k and v
swapped, padded rows or strides misplaced -- by rewriting one line of its source (or one
constant), and checks that at least one pin below then fails.  The pins use
only what the E4M3 format, the pages' values and library routines fix (the OCP
value table, ties-to-even at every midpoint, saturation, torch's float8
conversion, a deque of length 16, torch's float64 attention, segment
independence, constant V, two worked P-requantization examples computed by
hand from the E4M3 grid, the page's example scale file); none of them re-runs the oracle's own formula.
With no mistake planted, every pin passes.
"""

import collections
import inspect
import math
import os
import textwrap
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import attention, calib, e4m3, quant, scales

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "e4m3_ocp_values.txt")
SCALE_FILE = os.path.join(os.path.dirname(GOLDEN), "scale_file_example.json")


# ---------------------------------------------------------------- pins

def pin_decode_ocp_values():
    codes, vals = [], []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            c, v = line.split()
            codes.append(int(c, 16))
            vals.append(float(v))
    got = e4m3.decode(np.array(codes, dtype=np.uint8))
    want = np.array(vals)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def pin_encode_roundtrip_and_ties():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = e4m3.decode(codes)
    assert np.array_equal(e4m3.encode(vals), codes)
    pos = np.array(sorted(c for c in range(0x7F)), dtype=np.uint8)   # 0 .. 448, increasing
    v = e4m3.decode(pos)
    mid = (v[:-1] + v[1:]) / 2
    even = np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:])             # the even mantissa of the pair
    assert np.array_equal(e4m3.encode(mid), even)
    inner_lo = v[:-1] + (v[1:] - v[:-1]) * 0.25
    inner_hi = v[:-1] + (v[1:] - v[:-1]) * 0.75
    assert np.array_equal(e4m3.encode(inner_lo), pos[:-1])
    assert np.array_equal(e4m3.encode(inner_hi), pos[1:])


def pin_encode_saturation():
    x = np.array([449.0, 464.0, 1e6, np.inf, -np.inf, -500.0])
    assert np.array_equal(e4m3.encode(x), np.array([0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE], np.uint8))


def pin_encode_torch():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(20000) * np.exp2(rng.uniform(-12, 9, 20000))).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3.encode(x), ref)


def pin_scale_values():
    st = scales.ScaleState()
    st.set_static(224.0, 198.0, 210.0)
    for t, A in enumerate((224, 198, 210)):
        for got, exact in ((st.scale[t], Fraction(A, 448)), (st.inv_scale[t], Fraction(448, A))):
            g = Fraction(float(got))
            ulp = Fraction(float(np.spacing(np.float32(got))))
            assert abs(g - exact) <= ulp / 2


def pin_amax():
    assert scales.amax(np.array([-3.0, 2.0, np.nan], np.float32)) == np.float32(3.0)


def pin_ring_orders():
    rng = np.random.default_rng(2)
    for delayed in (False, True):
        st = scales.ScaleState()
        st.set_ring_order(delayed)
        hist = collections.deque(maxlen=16)
        for _ in range(40):
            a = rng.uniform(0.1, 100.0, 3).astype(np.float32)
            before = max((h[0] for h in hist), default=0.0)
            st.push(a)
            hist.append(a)
            want = before if delayed else max(h[0] for h in hist)
            assert st.amax_ref[0] == np.float32(want)


def _qkv(T, H, D, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(T, H, D, generator=g, dtype=torch.float64).numpy() for _ in range(3)]


def pin_attention_sdpa():
    q, k, v = _qkv(37, 2, 16, 3)
    o = attention.attention_varlen(q, k, v, [0, 37])
    t = lambda a: torch.from_numpy(a).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v))[0].permute(1, 0, 2).numpy()
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)


def pin_attention_segments():
    q, k, v = _qkv(30, 2, 8, 4)
    cu = [0, 10, 22, 30]
    o1 = attention.attention_varlen(q, k, v, cu)
    k2, v2 = k.copy(), v.copy()
    k2[10:22] += 5.0
    v2[10:22] *= -3.0
    o2 = attention.attention_varlen(q, k2, v2, cu)
    assert np.array_equal(o1[:10], o2[:10]) and np.array_equal(o1[22:], o2[22:])


def pin_attention_constant_v():
    q, k, _ = _qkv(25, 1, 8, 5)
    v = np.full((25, 1, 8), 0.37)
    assert np.allclose(attention.attention_varlen(q, k, v, [0, 5, 25]), 0.37, atol=1e-14)


def pin_quant_torch():
    rng = np.random.default_rng(6)
    x = rng.standard_normal(5000).astype(np.float32) * 3
    inv = np.float32(448.0 / 9.5)
    y = np.clip(x * inv, -448, 448)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(quant.quantize(x, inv), ref)


def pin_p8_worked_example():
    # Two keys, scores (3.9 ln 2, 3 ln 2): the power-of-two reference is 2^4,
    # so P' = E4M3(2^(8 - 0.1)) = E4M3(238.86...) = 240 (grid step 16 in
    # [128, 256)) and E4M3(2^7) = 128; with v = (1, 0) the output is 240 / 368.
    L2 = math.log(2.0)
    q = np.array([[[1.0]], [[0.0]]])
    k = np.array([[[3.9 * L2]], [[3.0 * L2]]])
    v = np.array([[[1.0]], [[0.0]]])
    o = attention.attention_varlen_p8(q, k, v, [0, 2], sm_scale=1.0, rows=[0])
    assert abs(o[0, 0, 0] - 240.0 / 368.0) < 1e-15


def pin_p8_far_keys_exact():
    # Scores -j ln 2 (j = 0..16): every weight is a power of two, and with the
    # 2^8 shift the farthest, 2^-8, is still an E4M3 value (two subnormal
    # steps), so the rounded weights are exact and so is the output.
    L2 = math.log(2.0)
    n = 17
    q = np.zeros((n, 1, 1))
    q[0, 0, 0] = 1.0
    k = (-np.arange(n, dtype=np.float64) * L2).reshape(n, 1, 1)
    v = np.zeros((n, 1, 1))
    v[n - 1, 0, 0] = 1.0
    o = attention.attention_varlen_p8(q, k, v, [0, n], sm_scale=1.0, rows=[0])
    exact = 2.0 ** -16 / sum(2.0 ** -j for j in range(n))
    assert abs(o[0, 0, 0] - exact) <= 1e-15 * exact


def pin_scale_file_example():
    # The page's example file: layer 0 holds q 224, k 198, v 210; layer 1
    # q 218, k 195, v 207.  The same entry under the _scale aliases parses alike.
    import json
    d = json.load(open(SCALE_FILE))
    assert calib.parse_file_dict(d) == {0: (224.0, 198.0, 210.0), 1: (218.0, 195.0, 207.0)}
    alias = {"visual.blocks.3.attn.attn": {"q_scale": 1.0, "k_scale": 2.0, "v_scale": 3.0}}
    assert calib.parse_file_dict(alias) == {3: (1.0, 2.0, 3.0)}


def pin_margin():
    # The 1.5 save margin on exactly representable values.
    assert calib.saved_values([100.0, 200.0, 2.0]) == [150.0, 300.0, 3.0]
    assert calib.layer_key(7) == "visual.blocks.7.attn.attn"


def pin_unpad_layouts():
    # A padded batch [B, s_max, H, D] with padding rows of huge values, and a
    # fused [T, 3, H, D] QKV view, against packed rows cut out with numpy
    # slicing: the same codes, padding never read.
    rng = np.random.default_rng(7)
    seqlens, H, D, s_max = [3, 5, 1], 2, 4, 6
    cu = [0, 3, 8, 9]
    packed = rng.standard_normal((9, H, D)).astype(np.float32)
    padded = np.full((3, s_max, H, D), 3.0e4, np.float32)
    for b, L in enumerate(seqlens):
        padded[b, :L] = packed[cu[b]:cu[b + 1]]
    inv = np.float32(10.0)
    want = np.zeros((9, H, 8), np.uint8)
    want[:, :, :D] = quant.quantize(packed, inv)
    lay = quant.SrcLayout.padded_batch(s_max, H, D)
    assert np.array_equal(quant.quantize_unpad(padded.ravel(), lay, cu, H, D, 8, inv), want)
    fused = np.stack([packed * 0 + 7.0, packed, packed * 0 - 7.0], axis=1)   # k in the middle
    lay_f = quant.SrcLayout(0, 0, 3 * H * D, D)
    got = quant.quantize_unpad(fused.ravel()[H * D:], lay_f, cu, H, D, 8, inv)
    assert np.array_equal(got, want)
    # heads 6 elements apart, the 2 between them holding garbage
    wide = np.full((9, H, 6), -3.0e4, np.float32)
    wide[:, :, :D] = packed
    lay_w = quant.SrcLayout(0, 0, H * 6, 6)
    assert np.array_equal(quant.quantize_unpad(wide.ravel(), lay_w, cu, H, D, 8, inv), want)


PINS = [pin_decode_ocp_values, pin_encode_roundtrip_and_ties, pin_encode_saturation,
        pin_encode_torch, pin_scale_values, pin_amax, pin_ring_orders, pin_attention_sdpa,
        pin_attention_segments, pin_attention_constant_v, pin_quant_torch,
        pin_p8_worked_example, pin_p8_far_keys_exact, pin_scale_file_example, pin_margin,
        pin_unpad_layouts]


# ---------------------------------------------------------------- mistakes

MUTANTS = {
    "decode: exponent bias 8": (e4m3, "decode", [("(e - 10)", "(e - 11)")]),
    "decode: subnormals read as zero": (e4m3, "decode", [("np.ldexp(m.astype(np.float64), -9)",
                                                           "np.zeros(m.shape)")]),
    "encode: ties away from zero": (e4m3, "encode", [("q = np.rint(np.ldexp(an_fin, (3 - e)))",
                                                      "q = np.floor(np.ldexp(an_fin, (3 - e)) + 0.5)")]),
    "encode: truncation": (e4m3, "encode", [("q = np.rint(np.ldexp(an_fin, (3 - e)))",
                                             "q = np.trunc(np.ldexp(an_fin, (3 - e)))")]),
    "encode: subnormals flushed": (e4m3, "encode", [("q_sub = np.rint(np.ldexp(np.where(sub, a, 0.0), 9))",
                                                     "q_sub = np.zeros(a.shape)")]),
    "encode: overflow to NaN": (e4m3, "encode", [("code_n = np.where(over, 0x7E, code_n)",
                                                  "code_n = np.where(over, 0x7F, code_n)")]),
    "scales: scale and multiplier swapped": (scales, "scale_pair", [
        ("return np.float32(A / F448), np.float32(F448 / A)", "return np.float32(F448 / A), np.float32(A / F448)")]),
    "amax: no absolute value": (scales, "amax", [("a = np.abs(np.asarray(x, dtype=np.float32).ravel())",
                                                  "a = np.asarray(x, dtype=np.float32).ravel()")]),
    "ring: 15 slots": (scales.ScaleState, "push", [("(self.pos + 1) % RING", "(self.pos + 1) % (RING - 1)")]),
    "ring: scale before the push in push-then-scale": (scales.ScaleState, "push", [
        ("if self.mode == 2:\n    self._scale_from_ring()", "if self.mode in (0, 2):\n    self._scale_from_ring()"),
        ("if self.mode == 0:\n    self._scale_from_ring()", "if False:\n    self._scale_from_ring()")]),
    "attention: softmax scale dropped": (attention, "_attend", [("sc = (q @ k.T) * float(sm_scale)", "sc = (q @ k.T)")]),
    "attention: score matrix transposed": (attention, "_attend", [("sc = (q @ k.T) * float(sm_scale)",
                                                                  "sc = (k @ q.T) * float(sm_scale)")]),
    "attention: normalised by the block total": (attention, "_attend", [
        ("return (p @ v) / p.sum(axis=1, keepdims=True)\n", "return (p @ v) / p.sum()\n")]),
    "attention: keys across segments": (attention, "attention_varlen", [
        ("kh[s:e, h, :], vh[s:e, h, :]", "kh[:, h, :], vh[:, h, :]")]),
    "P requantization: shift 2^4 instead of 2^8": (attention, "P_SHIFT", 4),
    "P requantization: reference from floor": (attention, "_attend", [
        ("M = np.ceil(sc.max(axis=1, keepdims=True) / math.log(2.0))",
         "M = np.floor(sc.max(axis=1, keepdims=True) / math.log(2.0))")]),
    "scale file: margin not applied": (calib, "saved_values", [
        ("return [float(np.float32(x) * np.float32(margin)) for x in a]", "return [float(np.float32(x)) for x in a]")]),
    "scale file: k and v entries swapped": (calib, "parse_file_dict", [
        ('for t in ("q", "k", "v"):', 'for t in ("q", "v", "k"):')]),
    "un-padding: padded rows at b * (s_max - 1)": (quant, "source_rows", [
        ("rows.append(b * layout.s_max + i)", "rows.append(b * (layout.s_max - 1) + i)")]),
    "un-padding: head stride taken as D for every layout": (quant, "gather_valid", [
        ("* layout.head_stride", "* D")]),
    "un-padding: token stride taken as H * D": (quant, "gather_valid", [
        ("idx = (rows[:, None, None] * layout.token_stride", "idx = (rows[:, None, None] * (H * D)")]),
    "quant: multiplier used as divisor": (quant, "quantize", [
        ("np.asarray(x, dtype=np.float32) * np.float32(inv)", "np.asarray(x, dtype=np.float32) / np.float32(inv)")]),
}


def _mutated(owner, name, edits):
    fn = getattr(owner, name)
    src = textwrap.dedent(inspect.getsource(fn))
    for old, new in edits:
        # match indentation-insensitively for multi-line edits
        lines_old = [l.strip() for l in old.split("\n")]
        src_lines = src.split("\n")
        found = False
        for i in range(len(src_lines) - len(lines_old) + 1):
            window = [l.strip() for l in src_lines[i:i + len(lines_old)]]
            if len(lines_old) == 1:
                if lines_old[0] and lines_old[0] in src_lines[i]:
                    src_lines[i] = src_lines[i].replace(old.strip(), new.strip())
                    found = True
                    break
            elif window == lines_old:
                indent = src_lines[i][:len(src_lines[i]) - len(src_lines[i].lstrip())]
                new_lines = new.split("\n")
                base = len(new_lines[0]) - len(new_lines[0].lstrip())
                src_lines[i:i + len(lines_old)] = [indent + l[base:] if l.strip() else l for l in new_lines]
                found = True
                break
        assert found, "mutation site not found in %s: %r" % (name, old)
        src = "\n".join(src_lines)
    module = inspect.getmodule(fn)
    ns = dict(vars(module))
    exec(compile(src, "<mutant of %s>" % name, "exec"), ns)
    return ns[name]


def _failing_pins():
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except Exception:
            failed.append(pin.__name__)
    return failed


def test_every_pin_passes_on_the_oracle():
    assert _failing_pins() == []


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(monkeypatch, mutant):
    owner, name, edits = MUTANTS[mutant]
    new = _mutated(owner, name, edits) if isinstance(edits, list) else edits
    monkeypatch.setattr(owner, name, new)
    monkeypatch.setattr(attention, "_DECODE", None)   # dequant's table is rebuilt afterwards
    failed = _failing_pins()
    assert failed, "no pin caught: " + mutant
