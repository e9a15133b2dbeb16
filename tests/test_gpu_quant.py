"""GPU parity: amax ring, scales and E4M3 codes must match the oracle bit for bit."""

import numpy as np
import pytest
import torch

import workloads
from oracle import e4m3, quant as oquant, scales as oscales

from gpu_util import (check_codes, cu_tensor, np32, oracle_push, qkv, state_matches, vt_to_thd)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vf():
    import fp8_vision_encoder_gb300 as vf
    assert torch.cuda.is_available()
    return vf


def _all_bf16_patterns(H, D):
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16)
    T = 65536 // (H * D)
    return x.reshape(T, H, D), T


@pytest.mark.parametrize("A", [448.0, 224.0, 198.0, 210.0, 1.0, 3.5e4, 1e-3])
def test_cvt_sweep_all_bf16_patterns(vf, A):
    """Every bf16 bit pattern x scale multiplier: codes equal the oracle's."""
    H, D = 1, 128
    x, T = _all_bf16_patterns(H, D)
    xd = x.cuda()
    cu, _ = cu_tensor([T])
    st = vf.ScaleState().set_static(A, A, A)
    q8, k8, v8t = vf.quantize_unpad(st, xd, xd, xd, cu)
    torch.cuda.synchronize()
    inv = oscales.scale_pair(np.float32(A))[1]
    ref = oquant.quantize(np32(x), inv)
    for got in (q8.cpu().numpy(), k8.cpu().numpy(), vt_to_thd(v8t, T).cpu().numpy()):
        xn = np32(x)
        nan = np.isnan(xn)
        assert np.array_equal(got[~nan], ref[~nan])
        assert np.all((got[nan] & 0x7F) == 0x7F)


def test_static_scales_and_amax_noop(vf):
    seqlens = [64, 192]
    q, k, v = qkv(seqlens, 2, 128, seed=0)
    cu, cul = cu_tensor(seqlens)
    st = vf.ScaleState().init().set_static(224.0, 198.0, 210.0)
    vf.amax_update(st, q, k, v, cu)                    # static: no-op
    ost = oscales.ScaleState()
    ost.set_static(224.0, 198.0, 210.0)
    state_matches(st.read(), ost)


@pytest.mark.parametrize("layout", ["packed", "padded"])
def test_tiny_dynamic_three_forwards(vf, layout):
    w = workloads.WORKLOADS["tiny"]
    cu, cul = cu_tensor(w.seqlens)
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    for seed in w.seeds:
        q, k, v = qkv(w.seqlens, w.H, w.D, seed)
        if layout == "packed":
            src, lay = (q, k, v), None
        else:
            s_max = max(w.seqlens) + 5
            src = [workloads.to_padded(t, w.seqlens, s_max) for t in (q, k, v)]
            lay = vf.SrcLayout.padded_batch(s_max, w.H, w.D)
        vf.amax_update(st, *src, cu, total_tokens=w.T, layout=lay, H=w.H, D=w.D)
        oracle_push(ost, q, k, v)
        state_matches(st.read(), ost)
        q8, k8, v8t = vf.quantize_unpad(st, *src, cu, total_tokens=w.T, layout=lay, H=w.H, D=w.D)
        torch.cuda.synchronize()
        for t, (codes, x) in enumerate(((q8, q), (k8, k), (vt_to_thd(v8t, w.T), v))):
            check_codes(codes, x, ost.inv_scale[t], w.D, w.D)
        assert st.device_error() == 0
    assert ost.count == 3


@pytest.mark.parametrize("D_pad", [80, 96, 128])
def test_hd3_ring_wraps_d80(vf, D_pad):
    """3 x 3600 tokens, 16 heads, d=80, per-head std; 20 forwards wrap the ring."""
    w = workloads.WORKLOADS["hd3"]
    cu, cul = cu_tensor(w.seqlens)
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    for f, seed in enumerate(w.seeds):
        q, k, v = qkv(w.seqlens, w.H, w.D, seed, outliers=False, per_head_std=True)
        vf.amax_update(st, q, k, v, cu)
        oracle_push(ost, q, k, v)
        if f in (0, 15, 16, 19):
            state_matches(st.read(), ost)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu, D_pad=D_pad)
    torch.cuda.synchronize()
    check_codes(q8, q, ost.inv_scale[0], w.D, D_pad)
    check_codes(k8, k, ost.inv_scale[1], w.D, D_pad)
    check_codes(vt_to_thd(v8t, w.T), v, ost.inv_scale[2], w.D, D_pad)
    Tv = vf.vt_stride(w.T)
    assert np.all(v8t[:, :, w.T:Tv].cpu().numpy() == 0)


@pytest.mark.parametrize("D,D_pad", [(256, 256), (200, 256), (8, 16)])
def test_largest_and_smallest_head_dims(vf, D, D_pad):
    """Quantization takes head dims up to 256 (attention stops at 128): the
    largest padded width, a ragged one below it, and the smallest."""
    seqlens, H = [70, 1, 130], 3
    T = sum(seqlens)
    cu, _ = cu_tensor(seqlens)
    q, k, v = qkv(seqlens, H, D, seed=17, per_head_std=True)
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    vf.amax_update(st, q, k, v, cu)
    oracle_push(ost, q, k, v)
    state_matches(st.read(), ost)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu, D_pad=D_pad)
    torch.cuda.synchronize()
    check_codes(q8, q, ost.inv_scale[0], D, D_pad)
    check_codes(k8, k, ost.inv_scale[1], D, D_pad)
    check_codes(vt_to_thd(v8t, T), v, ost.inv_scale[2], D, D_pad)
    with pytest.raises(vf.VitFp8Error):
        vf.quantize_unpad(st, q, k, v, cu, D_pad=D_pad + 16 if D_pad == 256 else 8)


def test_ragged_tokens_and_zero_length_segment(vf):
    seqlens = [1, 127, 0, 129, 33, 200]
    H, D = 3, 64
    q, k, v = qkv(seqlens, H, D, seed=11)
    cu, cul = cu_tensor(seqlens)
    T = sum(seqlens)
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    vf.amax_update(st, q, k, v, cu)
    oracle_push(ost, q, k, v)
    state_matches(st.read(), ost)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
    torch.cuda.synchronize()
    check_codes(q8, q, ost.inv_scale[0], D, D)
    check_codes(vt_to_thd(v8t, T), v, ost.inv_scale[2], D, D)
    assert np.all(v8t[:, :, T:].cpu().numpy() == 0)


def test_strided_fused_qkv_source(vf):
    """q/k/v as views into one fused [T, 3, H, D] buffer (token stride 3*H*D)."""
    seqlens = [100, 37]
    H, D = 4, 128
    q, k, v = qkv(seqlens, H, D, seed=12)
    fused = torch.stack([q, k, v], dim=1).contiguous()
    cu, _ = cu_tensor(seqlens)
    lay = vf.SrcLayout.packed(H, D, token_stride=3 * H * D, head_stride=D)
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    qv, kv, vv = fused[:, 0], fused[:, 1], fused[:, 2]
    vf.amax_update(st, qv, kv, vv, cu, total_tokens=137, layout=lay, H=H, D=D)
    oracle_push(ost, q, k, v)
    state_matches(st.read(), ost)
    q8, k8, v8t = vf.quantize_unpad(st, qv, kv, vv, cu, total_tokens=137, layout=lay, H=H, D=D)
    torch.cuda.synchronize()
    check_codes(k8, k, ost.inv_scale[1], D, D)


def test_padding_rows_never_read(vf):
    seqlens = [10, 50]
    H, D = 2, 128
    q, k, v = qkv(seqlens, H, D, seed=13)
    cu, _ = cu_tensor(seqlens)
    s_max = 64
    pads = [workloads.to_padded(t, seqlens, s_max, fill=3.0e4) for t in (q, k, v)]
    lay = vf.SrcLayout.padded_batch(s_max, H, D)
    st = vf.ScaleState().init()
    vf.amax_update(st, *pads, cu, total_tokens=60, layout=lay, H=H, D=D)
    ost = oscales.ScaleState()
    oracle_push(ost, q, k, v)
    state_matches(st.read(), ost)
    q8, _, _ = vf.quantize_unpad(st, *pads, cu, total_tokens=60, layout=lay, H=H, D=D)
    torch.cuda.synchronize()
    check_codes(q8, q, ost.inv_scale[0], D, D)


def test_bad_seqlens_padded_sets_error_not_fault(vf):
    """cu_seqlens that overruns s_max: rows are skipped and the error word is set."""
    H, D = 2, 128
    q, k, v = qkv([40], H, D, seed=14)
    s_max = 16
    pads = [torch.zeros((2, s_max, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    cu = torch.tensor([0, 20, 40], dtype=torch.int32, device="cuda")   # 20 > s_max
    lay = vf.SrcLayout.padded_batch(s_max, H, D)
    st = vf.ScaleState().init()
    vf.amax_update(st, *pads, cu, total_tokens=40, layout=lay, H=H, D=D)
    assert st.device_error() == 6


def _oracle_code_table(inv):
    """E4M3 code of float32(x) * inv for every bf16 bit pattern x, from the
    oracle's quantize (the code of an element depends on nothing else)."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        return oquant.quantize(x, inv)


def _assert_codes_full(codes_thd, x, inv, chunk=1 << 14):
    """Every code of a [T, H, D] (or strided [T, H, D_pad] view) against the
    oracle, in token chunks so host memory stays bounded."""
    table = _oracle_code_table(inv)
    T = x.shape[0]
    for t0 in range(0, T, chunk):
        xb = x[t0:t0 + chunk].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        got = codes_thd[t0:t0 + chunk].cpu().numpy()
        ref = table[xb]
        mism = np.count_nonzero(got != ref)
        assert mism == 0, "%d code mismatches in tokens %d.." % (mism, t0)


@pytest.mark.parametrize("name", ["micro8k", "qhd3", "uhd3mix"])
def test_full_size_codes_and_amax_exact(vf, name):
    """Full-size workloads: the scale state bit-exact with the oracle's, and
    EVERY code of q, k and v (all T x H x D of each, V through its transposed
    layout) equal to the oracle's quantization of its bf16 input.  qhd3 runs
    as the bench runs it: 16 dynamic calibration forwards, static scales
    1.5 x the calibrated amax, one layer."""
    w = workloads.WORKLOADS[name]
    cu, cul = cu_tensor(w.seqlens)
    gen = lambda seed: workloads.make_qkv(w.seqlens, w.H, w.D, seed, w.outliers, w.per_head_std,
                                          device="cuda")
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    if w.scaling == "static":
        st.set_static(*w.static)
        ost.set_static(*w.static)
        q, k, v = gen(w.seeds[0])
    elif w.scaling == "calibrated":
        for seed in w.calib_seeds:
            q, k, v = gen(seed)
            vf.amax_update(st, q, k, v, cu)
            oracle_push(ost, q, k, v)
        state_matches(st.read(), ost)
        A = [float(np.float32(a) * np.float32(1.5)) for a in ost.amax_ref]
        st.set_static(*A)
        ost.set_static(*A)
        q, k, v = gen(w.layer_seeds[0])
    else:
        q, k, v = gen(w.seeds[0])
        vf.amax_update(st, q, k, v, cu)
        oracle_push(ost, q, k, v)
    state_matches(st.read(), ost)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
    torch.cuda.synchronize()
    assert st.device_error() == 0
    D = w.D
    _assert_codes_full(q8[:, :, :D], q, ost.inv_scale[0])
    _assert_codes_full(k8[:, :, :D], k, ost.inv_scale[1])
    _assert_codes_full(v8t[:, :D, :w.T].permute(2, 0, 1), v, ost.inv_scale[2])
    # head-dim padding and V's token padding are zero codes
    if q8.shape[2] > D:
        assert int(q8[:, :, D:].sum().item()) == 0 and int(k8[:, :, D:].sum().item()) == 0


@pytest.mark.parametrize("split", [False, True])
def test_delayed_ring_order(vf, split):
    # Delayed scaling (mode 2): each forward is quantized with the scale of the
    # ring its predecessors left; state and codes bit-exact with the oracle,
    # through amax_update or through amax_local + ring_push.
    seqlens, H, D = [333, 64, 200], 4, 80
    cu, _ = cu_tensor(seqlens)
    T = sum(seqlens)
    st = vf.ScaleState().init().set_ring_order(True)
    ost = oscales.ScaleState()
    ost.set_ring_order(True)
    for seed in range(20):
        q, k, v = qkv(seqlens, H, D, 500 + seed, outliers=(seed % 3 == 0), per_head_std=True)
        if split:
            vf.ring_push(st, vf.amax_local(st, q, k, v, cu))
        else:
            vf.amax_update(st, q, k, v, cu)
        oracle_push(ost, q, k, v)
        state_matches(st.read(), ost)
        q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
        torch.cuda.synchronize()
        for t, (codes, x) in enumerate(((q8, q), (k8, k), (vt_to_thd(v8t, T), v))):
            check_codes(codes, x, ost.inv_scale[t], D, vf.default_d_pad(D))
    assert st.read()["mode"] == 2 and st.device_error() == 0
    # switching back, and a static state ignoring the order
    st.set_ring_order(False)
    assert st.read()["mode"] == 0
    s2 = vf.ScaleState().init().set_static(224.0, 198.0, 210.0).set_ring_order(True)
    assert s2.read()["mode"] == 1


@pytest.mark.parametrize("padded", [False, True])
def test_head_stride_wider_than_d(vf, padded):
    """Heads not contiguous within a token (head stride 96 > D = 80, the gap
    holding huge values that must never be read): the amax takes the per-head
    path; padded sources add padding rows that must not be read either."""
    seqlens = [70, 0, 130, 9]
    H, D, HS = 3, 80, 96
    T = sum(seqlens)
    q, k, v = qkv(seqlens, H, D, seed=31, outliers=True)
    cu, _ = cu_tensor(seqlens)
    wide = []
    for x in (q, k, v):
        w = torch.full((T, H, HS), 3.0e4, dtype=torch.bfloat16, device="cuda")
        w[:, :, :D] = x
        wide.append(w)
    if padded:
        s_max = 140
        wide = [workloads.to_padded(w, seqlens, s_max, fill=3.0e4) for w in wide]
        lay = vf.SrcLayout(1, 0, s_max, H * HS, HS)
    else:
        lay = vf.SrcLayout.packed(H, D, token_stride=H * HS, head_stride=HS)
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    for rep in range(2):
        vf.amax_update(st, *wide, cu, total_tokens=T, layout=lay, H=H, D=D)
        oracle_push(ost, q, k, v)
        state_matches(st.read(), ost)
    q8, k8, v8t = vf.quantize_unpad(st, *wide, cu, total_tokens=T, layout=lay, H=H, D=D)
    torch.cuda.synchronize()
    check_codes(q8, q, ost.inv_scale[0], D, vf.default_d_pad(D))
    check_codes(vt_to_thd(v8t, T), v, ost.inv_scale[2], D, vf.default_d_pad(D))
