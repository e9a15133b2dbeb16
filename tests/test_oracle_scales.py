"""Pins for the oracle's amax, ring and scale arithmetic (CPU only)."""

import collections
import json
import os
from fractions import Fraction

import numpy as np

from oracle import calib, scales


def _correctly_rounded_f32(fr):
    """Nearest float32 to the exact rational ``fr`` (ties to even), by search."""
    guess = np.float32(float(fr))
    best = None
    for c in (np.nextafter(guess, np.float32(-np.inf)), guess, np.nextafter(guess, np.float32(np.inf))):
        err = abs(Fraction(float(c)) - fr)
        key = (err, int(np.array(c).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_scale_pair_is_one_correctly_rounded_division():
    rng = np.random.default_rng(0)
    for A in list(rng.uniform(1e-3, 1e4, 2000).astype(np.float32)) + [np.float32(224.0), np.float32(198.0)]:
        s, inv = scales.scale_pair(A)
        assert s == _correctly_rounded_f32(Fraction(float(A)) / 448)
        assert inv == _correctly_rounded_f32(Fraction(448) / Fraction(float(A)))


def test_page_static_values():
    # "Scale File Format" example: q 224, k 198, v 210.
    st = scales.ScaleState()
    st.set_static(224.0, 198.0, 210.0)
    assert st.mode == 1
    assert st.scale[0] == np.float32(0.5) and st.inv_scale[0] == np.float32(2.0)
    assert st.scale[1] == np.float32(198.0) / np.float32(448.0)
    assert list(st.amax_ref) == [224.0, 198.0, 210.0]


def test_ring_against_deque_bruteforce():
    rng = np.random.default_rng(5)
    st = scales.ScaleState()
    dq = [collections.deque(maxlen=16) for _ in range(3)]
    for n in range(1, 40):
        a = rng.uniform(0, 100, 3).astype(np.float32)
        st.push(a)
        for t in range(3):
            dq[t].append(a[t])
            assert st.amax_ref[t] == max(dq[t])
            assert sorted(st.hist[t][st.hist[t] > 0]) == sorted(dq[t])
            # slot of push k (1-based) is (k-1) mod 16
            assert st.hist[t][(n - 1) % 16] == a[t]
        assert st.count == min(n, 16)
        assert st.pos == n % 16


def test_ring_push_then_scale_includes_current_forward():
    st = scales.ScaleState()
    st.push([1.0, 2.0, 3.0])
    assert list(st.amax_ref) == [1.0, 2.0, 3.0]
    st.push([10.0, 0.5, 3.0])
    assert list(st.amax_ref) == [10.0, 2.0, 3.0]


def test_ring_wraps_and_forgets_after_16():
    st = scales.ScaleState()
    st.push([100.0, 100.0, 100.0])
    for _ in range(15):
        st.push([1.0, 1.0, 1.0])
    assert st.amax_ref[0] == 100.0
    st.push([1.0, 1.0, 1.0])           # 17th push overwrites the 100
    assert st.amax_ref[0] == 1.0


def test_zero_inf_nan_rules():
    st = scales.ScaleState()
    st.push([0.0, 0.0, 0.0])
    assert list(st.scale) == [1.0, 1.0, 1.0] and list(st.inv_scale) == [1.0, 1.0, 1.0]
    s, inv = scales.scale_pair(np.float32(np.inf))
    assert np.isinf(s) and inv == 0.0
    assert scales.amax(np.array([1.0, np.nan, -3.0])) == 3.0
    assert scales.amax(np.array([1.0, -np.inf])) == np.inf


def test_amax_bruteforce():
    rng = np.random.default_rng(9)
    x = rng.standard_normal(5000).astype(np.float32)
    assert scales.amax(x) == max(abs(float(v)) for v in x)


def test_scale_file_example_parses():
    path = os.path.join(os.path.dirname(__file__), "golden", "scale_file_example.json")
    with open(path) as f:
        d = json.load(f)
    parsed = calib.parse_file_dict(d)
    assert parsed == {0: (224.0, 198.0, 210.0), 1: (218.0, 195.0, 207.0)}


def test_scale_file_aliases_and_roundtrip():
    d = {"visual.blocks.3.attn.attn": {"q_scale": 1.0, "k": 2.0, "v_scale": 3.0}}
    assert calib.parse_file_dict(d) == {3: (1.0, 2.0, 3.0)}
    out = calib.to_file_dict([(10.0, 20.0, 30.0)])
    assert out == {"visual.blocks.0.attn.attn": {"q": 15.0, "k": 30.0, "v": 45.0}}
    assert calib.DEFAULT_MARGIN == 1.5 and calib.CALIB_PASSES == 16


def test_delayed_order_cold_start_uses_unit_scale():
    # Delayed scaling: the first forward sees an empty ring (reading: empty
    # slots hold 0, and a zero ring maximum gives scale = inv = 1).
    st = scales.ScaleState()
    st.set_ring_order(True)
    st.push([100.0, 50.0, 25.0])
    assert st.mode == 2
    assert list(st.amax_ref) == [0.0, 0.0, 0.0]
    assert list(st.scale) == [1.0, 1.0, 1.0] and list(st.inv_scale) == [1.0, 1.0, 1.0]
    assert list(st.hist[:, 0]) == [100.0, 50.0, 25.0] and st.count == 1
    st.push([1.0, 2.0, 3.0])
    assert list(st.amax_ref) == [100.0, 50.0, 25.0]


def test_delayed_order_against_previous_sixteen_bruteforce():
    rng = np.random.default_rng(9)
    st, now = scales.ScaleState(), scales.ScaleState()
    st.set_ring_order(True)
    seen = []
    for n in range(40):
        a = rng.uniform(0, 100, 3).astype(np.float32)
        st.push(a)
        now.push(a)
        prev = seen[-16:]
        for t in range(3):
            want = max((x[t] for x in prev), default=np.float32(0.0))
            assert st.amax_ref[t] == want
            assert (st.scale[t], st.inv_scale[t]) == scales.scale_pair(want)
        # the ring itself is the same as with push-then-scale
        assert np.array_equal(st.hist, now.hist) and st.pos == now.pos and st.count == now.count
        seen.append(a)


def test_ring_order_leaves_static_alone():
    st = scales.ScaleState()
    st.set_static(224.0, 198.0, 210.0)
    st.set_ring_order(True)
    assert st.mode == 1
    st.push([1.0, 1.0, 1.0])
    assert list(st.amax_ref) == [224.0, 198.0, 210.0]
    dyn = scales.ScaleState()
    dyn.set_ring_order(True)
    dyn.set_ring_order(False)
    assert dyn.mode == 0
