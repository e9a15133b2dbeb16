"""GPU: the calibrate-once workflow end to end, and dynamic scaling captured in
one CUDA graph.

Calibration: 16 dynamic forwards per layer on the device, the scale file
built from the ring maxima, loaded back into static states, then one forward
with those states.  Every number is compared with the oracle on the same
inputs: ring maxima and static scale pairs bit for bit, E4M3 codes bit for
bit, attention within the parity tolerances.

Graph capture: the amax + ring update, quantization and attention of one
forward are captured once and replayed over fresh inputs copied into the
captured buffers; the state after every replay and the final codes and
output must equal an eager run of the same sequence exactly.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import calib as ocalib, scales as oscales

from gpu_util import (assert_attention_ok, check_codes, compare_attention, cu_tensor, np32,
                      oracle_push, qkv, state_matches, vt_to_thd)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vf():
    import fp8_vision_encoder_gb300 as vf
    assert torch.cuda.is_available()
    return vf


def test_calibrate_save_load_static(vf, tmp_path):
    from fp8_vision_encoder_gb300 import calibration as cal
    seqlens, H, D, layers = [300, 77, 500], 4, 128, 3
    cu, cul = cu_tensor(seqlens)
    c = cal.Calibrator(layers)
    ost = [oscales.ScaleState() for _ in range(layers)]
    for p in range(cal.CALIBRATION_PASSES):
        for n in range(layers):
            q, k, v = qkv(seqlens, H, D, 1000 * n + p, outliers=True, per_head_std=(n == 1))
            c.observe(n, q, k, v, cu)
            oracle_push(ost[n], q, k, v)
    for n in range(layers):
        state_matches(c.states[n].read(), ost[n])
    doc = c.scale_file()
    assert doc == ocalib.to_file_dict([o.amax_ref for o in ost])
    path = tmp_path / "scales.json"
    cal.save_scale_file(str(path), doc)
    states = cal.static_states(cal.load_scale_file(str(path)), num_layers=layers)
    for n in range(layers):
        ref = oscales.ScaleState()
        ref.set_static(*ocalib.saved_values(ost[n].amax_ref))
        state_matches(states[n].read(), ref)
    # one static forward of layer 2 with the loaded scales
    q, k, v = qkv(seqlens, H, D, 4242, outliers=True)
    q8, k8, v8t = vf.quantize_unpad(states[2], q, k, v, cu)
    out = vf.attn_varlen(q8, k8, v8t, states[2], cu, max(seqlens), D)
    torch.cuda.synchronize()
    ref = oscales.ScaleState()
    ref.set_static(*ocalib.saved_values(ost[2].amax_ref))
    T = sum(seqlens)
    check_codes(q8, q, ref.inv_scale[0], D, D)
    check_codes(vt_to_thd(v8t, T), v, ref.inv_scale[2], D, D)
    stats = compare_attention(out, q8, k8, vt_to_thd(v8t, T), list(ref.scale), cul, D)
    assert_attention_ok(stats, "calibrated static")


def test_scale_file_refuses_short_calibration(vf):
    from fp8_vision_encoder_gb300 import calibration as cal
    seqlens = [64]
    cu, _ = cu_tensor(seqlens)
    c = cal.Calibrator(1)
    q, k, v = qkv(seqlens, 2, 64, 1)
    for _ in range(3):
        c.observe(0, q, k, v, cu)
    with pytest.raises(RuntimeError):
        c.scale_file()
    assert len(c.scale_file(min_passes=3)) == 1


def test_dynamic_forward_replays_from_one_cuda_graph(vf):
    seqlens, H, D = [200, 64, 333], 4, 80
    cu, cul = cu_tensor(seqlens)
    T = sum(seqlens)
    D_pad = vf.default_d_pad(D)
    feeds = [qkv(seqlens, H, D, 70 + i, outliers=(i % 3 == 0), per_head_std=True) for i in range(20)]

    def forward(st, q, k, v, codes, out, ws):
        vf.amax_update(st, q, k, v, cu)
        vf.quantize_unpad(st, q, k, v, cu, D_pad=D_pad, out=codes)
        vf.attn_varlen(*codes, st, cu, max(seqlens), D, out=out, workspace=ws)

    # eager reference
    st_e = vf.ScaleState().init()
    codes_e = vf.alloc_codes(T, H, D_pad)
    out_e = torch.empty((T, H, D), dtype=torch.bfloat16, device="cuda")
    ws_e = vf.Workspace(len(seqlens))
    eager_states, eager_out = [], []
    for f in feeds:
        forward(st_e, *f, codes_e, out_e, ws_e)
        eager_states.append(st_e.buf.clone())
        eager_out.append(out_e.clone())

    # captured
    st = vf.ScaleState().init()
    bufs = [torch.empty_like(t) for t in feeds[0]]
    codes = vf.alloc_codes(T, H, D_pad)
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device="cuda")
    ws = vf.Workspace(len(seqlens))
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        forward(st, *bufs, codes, out, ws)
    torch.cuda.synchronize()
    # capture records work without running it: the state is still fresh
    vf.ScaleState.init(st)
    torch.cuda.synchronize()
    for i, f in enumerate(feeds):
        for b, t in zip(bufs, f):
            b.copy_(t)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(st.buf, eager_states[i]), "state differs after replay %d" % i
        assert torch.equal(out, eager_out[i]), "output differs after replay %d" % i
    assert st.read()["count"] == 16 and ws.error() == 0 and st.device_error() == 0
    # and the last replay agrees with the oracle
    ost = oscales.ScaleState()
    for f in feeds:
        oracle_push(ost, *f)
    state_matches(st.read(), ost)
    stats = compare_attention(out, codes[0], codes[1], vt_to_thd(codes[2], T), list(ost.scale), cul, D)
    assert_attention_ok(stats, "graph replay", outliers=True)


@pytest.mark.parametrize("delayed", [False, True])
def test_device_calibrated_scales_match_oracle(vf, delayed):
    """vitfp8_calibrated_scales: after 16 dynamic forwards, the saved values
    float32(ring max) * float32(margin) come out of the device bit-exact with
    the oracle's, for several margins and either ring order, and the static
    state it sets equals the oracle's static state from those values."""
    seqlens, H, D = [300, 77, 500], 4, 128
    cu, _ = cu_tensor(seqlens)
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    if delayed:
        st.set_ring_order(True)
        ost.set_ring_order(True)
    for p in range(16):
        q, k, v = qkv(seqlens, H, D, 5000 + p, outliers=(p % 3 == 0))
        vf.amax_update(st, q, k, v, cu)
        oracle_push(ost, q, k, v)
    state_matches(st.read(), ost)
    ring_max = np.asarray(ost.hist, dtype=np.float32).max(axis=1)
    for margin in (1.5, 1.0, 2.0, 1.25, 0.75):
        static = vf.ScaleState().init()
        saved = vf.calibrated_scales(st, margin, static)
        torch.cuda.synchronize()
        want = np.asarray(ocalib.saved_values(ring_max, margin), dtype=np.float32)
        assert np.array_equal(saved.cpu().numpy().view(np.uint32), want.view(np.uint32)), margin
        ref = oscales.ScaleState()
        ref.set_static(*want.tolist())
        state_matches(static.read(), ref)
    assert st.device_error() == 0


def test_device_calibrated_scales_empty_ring_is_an_error(vf):
    """A state that saw no forward has no learned scale: the call records
    VITFP8_ERR_INVALID_ARG in that state's error word and leaves the static
    state as it was."""
    st = vf.ScaleState().init()
    static = vf.ScaleState().init().set_static(1.0, 2.0, 3.0)
    before = static.read()
    saved = vf.calibrated_scales(st, 1.5, static)
    torch.cuda.synchronize()
    assert st.device_error() == 1
    assert static.read() == before
    assert saved.cpu().tolist() == [0.0, 0.0, 0.0]
    with pytest.raises(vf.VitFp8Error):
        vf.calibrated_scales(st, float("nan"))
