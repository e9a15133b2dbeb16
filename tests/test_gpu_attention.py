"""GPU parity of the FP8 varlen attention kernel against the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

import workloads
from oracle import scales as oscales

from gpu_util import (assert_attention_ok, check_codes, compare_attention, cu_tensor, np32,
                      oracle_push, qkv, sample_rows, vt_to_thd)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vf():
    import fp8_vision_encoder_gb300 as vf
    assert torch.cuda.is_available()
    return vf


def _run(vf, seqlens, H, D, seeds, static=None, D_pad=None, outliers=True, per_head_std=False,
         gen_device="cpu"):
    cu, cul = cu_tensor(seqlens)
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    if static is not None:
        st.set_static(*static)
        ost.set_static(*static)
    for seed in seeds:
        q, k, v = [t.cuda() for t in workloads.make_qkv(seqlens, H, D, seed, outliers, per_head_std,
                                                         device=gen_device)]
        if static is None:
            vf.amax_update(st, q, k, v, cu)
            oracle_push(ost, q, k, v)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu, D_pad=D_pad)
    ws = vf.Workspace(len(seqlens))
    out = vf.attn_varlen(q8, k8, v8t, st, cu, max(seqlens) if seqlens else 0, D, workspace=ws)
    torch.cuda.synchronize()
    assert ws.error() == 0
    T = sum(seqlens)
    return dict(out=out, q8=q8, k8=k8, v8=vt_to_thd(v8t, T), v8t=v8t, scales=list(ost.scale),
                cu=cul, st=st, ws=ws, cu_t=cu, q=q, k=k, v=v)


@pytest.mark.parametrize("outliers", [True, False])
def test_tiny_config(vf, outliers):
    w = workloads.WORKLOADS["tiny"]
    r = _run(vf, w.seqlens, w.H, w.D, w.seeds, outliers=outliers)
    stats = compare_attention(r["out"], r["q8"], r["k8"], r["v8"], r["scales"], r["cu"], w.D)
    assert_attention_ok(stats, "tiny outliers=%s" % outliers, outliers)


@pytest.mark.parametrize("outliers", [True, False])
@pytest.mark.parametrize("D", [64, 80, 128])
def test_ragged_segments(vf, D, outliers):
    seqlens = [1, 127, 128, 129, 300, 17, 0, 5]
    r = _run(vf, seqlens, 3, D, [21], outliers=outliers)
    stats = compare_attention(r["out"], r["q8"], r["k8"], r["v8"], r["scales"], r["cu"], D)
    assert_attention_ok(stats, "ragged D=%d outliers=%s" % (D, outliers), outliers)


@pytest.mark.parametrize("D", [8, 16, 24, 40, 48, 56, 72, 88, 96, 104, 112, 120])
def test_every_head_dim(vf, D):
    """Every other supported head dim (multiples of 8 up to 128) on a ragged
    batch with single-token segments and one segment spanning two key tiles."""
    seqlens = [1, 130, 300, 9, 1]
    r = _run(vf, seqlens, 2, D, [40 + D], outliers=False, per_head_std=True)
    stats = compare_attention(r["out"], r["q8"], r["k8"], r["v8"], r["scales"], r["cu"], D)
    assert_attention_ok(stats, "D=%d" % D)


@pytest.mark.parametrize("factor", [0.25, 3.0])
def test_softmax_scale_argument(vf, factor):
    """sm_scale other than 1/sqrt(D) (a flatter and a sharper softmax; the
    sharper one moves the row reference on more tiles)."""
    D = 128
    r = _run(vf, [300, 1000, 77], 2, D, [61], outliers=False)
    sm_scale = factor / math.sqrt(D)
    out = vf.attn_varlen(r["q8"], r["k8"], r["v8t"], r["st"], r["cu_t"], 1000, D, sm_scale=sm_scale,
                         workspace=r["ws"])
    torch.cuda.synchronize()
    assert r["ws"].error() == 0
    stats = compare_attention(out, r["q8"], r["k8"], r["v8"], r["scales"], r["cu"], D,
                              sm_scale=sm_scale)
    assert_attention_ok(stats, "sm_scale x%.2f" % factor)


@pytest.mark.parametrize("H", [1, 40])
def test_one_head_and_many_heads(vf, H):
    """One head, and 40 heads (the whole-row quantization takes 2 tokens per
    block then), on a ragged batch."""
    r = _run(vf, [300, 65, 1], H, 64, [81], outliers=False, per_head_std=True)
    stats = compare_attention(r["out"], r["q8"], r["k8"], r["v8"], r["scales"], r["cu"], 64)
    assert_attention_ok(stats, "H=%d" % H)


def test_saturating_static_scales(vf):
    """Static values far below the data's magnitude (A = 0.5 for unit-normal
    data with x20 outliers): most codes saturate to +-448; attention on those
    codes still matches the oracle on the same codes."""
    r = _run(vf, [300, 129], 2, 128, [71], static=(0.5, 0.5, 0.5), outliers=True)
    q8 = r["q8"].cpu().numpy()
    assert np.mean((q8 & 0x7F) == 0x7E) > 0.3
    stats = compare_attention(r["out"], r["q8"], r["k8"], r["v8"], r["scales"], r["cu"], 128)
    assert_attention_ok(stats, "saturating static", outliers=True)


def test_all_zero_inputs(vf):
    """q = k = v = 0 in dynamic mode: amax 0, so scale = multiplier = 1, every
    code 0x00, uniform attention over zeros: the output is exactly 0."""
    seqlens, H, D = [200, 17], 2, 128
    cu, _ = cu_tensor(seqlens)
    z = torch.zeros((sum(seqlens), H, D), dtype=torch.bfloat16, device="cuda")
    st = vf.ScaleState().init()
    vf.amax_update(st, z, z, z, cu)
    q8, k8, v8t = vf.quantize_unpad(st, z, z, z, cu)
    out = vf.attn_varlen(q8, k8, v8t, st, cu, 200, D)
    torch.cuda.synchronize()
    s = st.read()
    assert s["scale"] == [1.0, 1.0, 1.0] and s["inv_scale"] == [1.0, 1.0, 1.0] and s["count"] == 1
    assert int(q8.count_nonzero()) == 0 and int(v8t.count_nonzero()) == 0
    assert int(out.count_nonzero()) == 0 and st.device_error() == 0


def test_d80_padded_codes(vf):
    r = _run(vf, [200, 333], 2, 80, [5], D_pad=96, per_head_std=True, outliers=False)
    stats = compare_attention(r["out"], r["q8"], r["k8"], r["v8"], r["scales"], r["cu"], 80)
    assert_attention_ok(stats, "d80 D_pad=96")


@pytest.mark.parametrize("outliers", [True, False])
def test_single_long_segment_static(vf, outliers):
    r = _run(vf, [2000], 4, 128, [0], static=(224.0, 198.0, 210.0), outliers=outliers)
    rows = sample_rows(r["cu"], 300)
    stats = compare_attention(r["out"], r["q8"], r["k8"], r["v8"], r["scales"], r["cu"], 128, rows)
    assert_attention_ok(stats, "2000 static outliers=%s" % outliers, outliers, literal=not outliers)


def test_rescale_path_late_large_score(vf):
    """A key in a late tile scores far above everything before it: O is rescaled."""
    seqlens = [1000]
    H, D = 1, 128
    cu, cul = cu_tensor(seqlens)
    g = torch.Generator().manual_seed(3)
    q = torch.randn(1000, H, D, generator=g) * 0.3
    k = torch.randn(1000, H, D, generator=g) * 0.3
    v = torch.randn(1000, H, D, generator=g)
    k[900] = q.mean(dim=0) * 40.0       # aligned with the average query, large
    q, k, v = [t.to(torch.bfloat16).cuda() for t in (q, k, v)]
    st = vf.ScaleState().init()
    vf.amax_update(st, q, k, v, cu)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
    out = vf.attn_varlen(q8, k8, v8t, st, cu, 1000, D)
    torch.cuda.synchronize()
    sc = st.read()["scale"]
    stats = compare_attention(out, q8, k8, vt_to_thd(v8t, 1000), sc, cul, D)
    assert_attention_ok(stats, "rescale", outliers=True)


def test_constant_v_is_reproduced(vf):
    """All value codes equal: every output equals that value (weights sum to one)."""
    seqlens = [77, 300]
    H, D = 2, 128
    cu, cul = cu_tensor(seqlens)
    q, k, _ = qkv(seqlens, H, D, seed=8)
    v = torch.full_like(q, 0.75)
    st = vf.ScaleState().init()
    vf.amax_update(st, q, k, v, cu)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
    out = vf.attn_varlen(q8, k8, v8t, st, cu, 300, D)
    torch.cuda.synchronize()
    assert torch.allclose(out.float(), torch.full_like(out.float(), 0.75), rtol=2 ** -7, atol=0)


def test_deterministic_and_no_cross_segment_leakage(vf):
    seqlens = [300, 129, 500]
    H, D = 2, 128
    r = _run(vf, seqlens, H, D, [7])
    out1 = r["out"].clone()
    out2 = vf.attn_varlen(r["q8"], r["k8"], r["v8t"], r["st"], r["cu_t"], 500, D)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    # perturb segment 1's keys and values: segments 0 and 2 must not move a bit
    k8 = r["k8"].clone()
    v8t = r["v8t"].clone()
    k8[300:429] = (k8[300:429].to(torch.int32) ^ 0x11).to(torch.uint8) & 0x77
    v8t[:, :, 300:429] = 0x38
    out3 = vf.attn_varlen(r["q8"], k8, v8t, r["st"], r["cu_t"], 500, D)
    torch.cuda.synchronize()
    a = out1.view(torch.int16)
    b = out3.view(torch.int16)
    assert torch.equal(a[:300], b[:300]) and torch.equal(a[429:], b[429:])
    assert not torch.equal(a[300:429], b[300:429])


def test_bad_seqlens_reports_and_writes_nothing(vf):
    H, D = 2, 128
    T = 64
    q8 = torch.zeros((T, H, D), dtype=torch.uint8, device="cuda")
    v8t = torch.zeros((H, D, vf.vt_stride(T)), dtype=torch.uint8, device="cuda")
    st = vf.ScaleState().init()
    out = torch.full((T, H, D), 7.0, dtype=torch.bfloat16, device="cuda")
    for bad in ([0, 40, 30, 64], [0, 32, 60], [1, 32, 64]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        ws = vf.Workspace(len(bad) - 1)
        vf.attn_varlen(q8, q8, v8t, st, cu, 64, D, out=out, workspace=ws)
        assert ws.error() == 6
    assert torch.all(out.float() == 7.0)


def test_empty_inputs_are_noops(vf):
    st = vf.ScaleState().init()
    cu = torch.zeros(1, dtype=torch.int32, device="cuda")
    e = torch.empty((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    vf.amax_update(st, e, e, e, cu)
    q8, k8, v8t = vf.quantize_unpad(st, e, e, e, cu)
    out = vf.attn_varlen(q8, k8, v8t, st, cu, 0, 128)
    torch.cuda.synchronize()
    assert out.shape == (0, 2, 128)
    assert st.read()["count"] == 0


@pytest.mark.parametrize("name,outliers", [("micro8k", True), ("micro8k", False), ("hd3", False),
                                           ("qhd3", True), ("qhd3", False), ("uhd3mix", True)])
def test_full_size_sampled_rows(vf, name, outliers):
    """Full-size workloads in the bench's launch configuration, sampled query rows.

    Each workload runs as specified; the "outliers=False" cases rerun the same
    shapes with pure unit-normal inputs for the literal tolerance."""
    w = workloads.WORKLOADS[name]
    cu, cul = cu_tensor(w.seqlens)
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    gen = lambda seed: workloads.make_qkv(w.seqlens, w.H, w.D, seed, outliers and w.outliers,
                                          w.per_head_std, device="cuda")
    if w.scaling == "static":
        st.set_static(*w.static)
        ost.set_static(*w.static)
        q, k, v = gen(w.seeds[0])
    elif w.scaling == "calibrated":
        for seed in w.calib_seeds:
            q, k, v = gen(seed)
            vf.amax_update(st, q, k, v, cu)
            oracle_push(ost, q, k, v)
        A = [float(np.float32(a) * np.float32(1.5)) for a in st.read()["amax_ref"]]
        st.set_static(*A)
        ost.set_static(*A)
        q, k, v = gen(w.layer_seeds[0])
    else:
        for seed in w.seeds:        # hd3: all 20 forwards, so the 16-entry ring wraps
            q, k, v = gen(seed)
            vf.amax_update(st, q, k, v, cu)
            oracle_push(ost, q, k, v)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
    out = vf.attn_varlen(q8, k8, v8t, st, cu, w.max_seqlen, w.D)
    torch.cuda.synchronize()
    rows = sample_rows(cul, 48, seed=1)
    stats = compare_attention(out, q8, k8, vt_to_thd(v8t, w.T), list(ost.scale), cul, w.D, rows)
    has_outliers = outliers and w.outliers
    # the literal bound (max |error| <= 2e-2) holds for unit-normal inputs on the long shapes
    literal = (not has_outliers) and name in ("micro8k", "qhd3")
    assert_attention_ok(stats, "%s outliers=%s" % (name, has_outliers), has_outliers, literal)


def test_buffers_beyond_2_gib():
    """272 segments of 4096 tokens x 16 heads x d = 128 (T = 1 114 112): each
    code buffer holds 2.28e9 elements and each bf16 source twice that in
    bytes, so the last segment's element offsets pass 2^31 (64-bit index
    arithmetic in the quantization, the tensor maps and the output stores).  Codes of the first and last segments
    are checked bit for bit and sampled rows of both against the oracle."""
    import fp8_vision_encoder_gb300 as vf
    H, D, L, B = 16, 128, 4096, 272
    T = L * B
    cu, _ = cu_tensor([L] * B)
    st = vf.ScaleState().init().set_static(224.0, 198.0, 210.0)
    ost = oscales.ScaleState()
    ost.set_static(224.0, 198.0, 210.0)
    g = torch.Generator(device="cuda").manual_seed(2024)
    src = []
    for _ in range(3):
        x = torch.empty((T, H, D), dtype=torch.bfloat16, device="cuda")
        for c in range(0, T, 1 << 16):       # draw in 64 Ki-token chunks (bounded scratch)
            x[c:c + (1 << 16)] = torch.randn((1 << 16, H, D), device="cuda", generator=g).to(torch.bfloat16)
        src.append(x)
    q, k, v = src
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
    ws = vf.Workspace(B)
    out = vf.attn_varlen(q8, k8, v8t, st, cu, L, D, workspace=ws)
    torch.cuda.synchronize()
    assert ws.error() == 0 and st.device_error() == 0
    assert (T - L) * H * D > 2 ** 31
    rng = np.random.default_rng(3)
    for s in (0, B - 1):
        a, b = s * L, (s + 1) * L
        check_codes(q8[a:b], q[a:b], ost.inv_scale[0], D, D)
        check_codes(vt_to_thd(v8t[:, :, a:b], L), v[a:b], ost.inv_scale[2], D, D)
        rows = np.sort(rng.choice(L, 24, replace=False))
        stats = compare_attention(out[a:b], q8[a:b], k8[a:b], vt_to_thd(v8t[:, :, a:b], L),
                                  list(ost.scale), [0, L], D, rows)
        assert_attention_ok(stats, "segment %d of %d" % (s, B), literal=True)


def test_bounded_wait_expires_into_a_status(vf):
    """A wait on a barrier nothing arrives on gives up after its limit and
    reports VITFP8_ERR_DEVICE_TIMEOUT through the workspace error word; the
    context stays usable and the next call clears the word."""
    import time
    ws = vf.Workspace(1)
    t0 = time.time()
    vf.selftest_bounded_wait(ws)
    assert ws.error() == 4          # VITFP8_ERR_DEVICE_TIMEOUT (this read synchronises)
    assert 0.1 < time.time() - t0 < 30
    r = _run(vf, [64, 192], 2, 128, [0], outliers=False)
    assert r["ws"].error() == 0
    stats = compare_attention(r["out"], r["q8"], r["k8"], r["v8"], r["scales"], r["cu"], 128)
    assert_attention_ok(stats, "after the timeout self-test")
    # the same workspace, reused by an attention call, is cleared as well
    cu, _ = cu_tensor([64, 192])
    vf.attn_varlen(r["q8"], r["k8"], r["v8t"], r["st"], cu, 192, 128, workspace=ws)
    assert ws.error() == 0


def test_more_segments_than_the_sorted_work_list():
    """3000 segments of 0..24 tokens: past 2048 segments the work list keeps
    the natural order instead of sorting longest first; every row checked."""
    import fp8_vision_encoder_gb300 as vf
    rng = np.random.default_rng(8)
    seqlens = [int(x) for x in rng.integers(0, 25, 3000)]
    r = _run(vf, seqlens, 3, 64, [9], outliers=False)
    stats = compare_attention(r["out"], r["q8"], r["k8"], r["v8"], r["scales"], r["cu"], 64)
    assert_attention_ok(stats, "3000 segments")
