"""GPU parity of the BF16 comparison attention kernel against the fp64 oracle.

The oracle is the exact softmax attention of the oracle module evaluated in
fp64 on the very bf16 values the kernel reads.
"""

import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oattn

from gpu_util import (TOL_BF16_MAX_VREL, TOL_BF16_REL_RMS, TOL_MAX_ABS, cu_tensor, np32,
                      sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vf():
    import fp8_vision_encoder_gb300 as vf
    assert torch.cuda.is_available()
    return vf


def _check(vf, out, q, k, v, cul, rows=None, literal=False, tag="", sm_scale=None):
    T, H, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    qn, kn, vn = np32(q), np32(k), np32(v)
    if rows is None:
        rows = np.arange(T)
    rows = np.unique(np.asarray(rows, dtype=np.int64))
    ref = oattn.attention_varlen(qn, kn, vn, cul, sm_scale, rows)[rows]
    got = out[torch.from_numpy(rows).to(out.device)].float().cpu().numpy().astype(np.float64)
    err = got - ref
    v_max = float(np.abs(vn).max()) if vn.size else 0.0
    v_rms = float(np.sqrt(np.mean(vn.astype(np.float64) ** 2))) if vn.size else 1.0
    max_abs = float(np.abs(err).max())
    rel_rms = float(np.sqrt(np.mean(err ** 2)) / v_rms)
    msg = "%s max_abs=%.3e (bound %.3e) rel_rms=%.3e" % (
        tag, max_abs, TOL_BF16_MAX_VREL * max(1.0, v_max), rel_rms)
    print(msg)
    assert max_abs <= TOL_BF16_MAX_VREL * max(1.0, v_max), msg
    assert rel_rms <= TOL_BF16_REL_RMS, msg
    if literal:
        assert max_abs <= TOL_MAX_ABS, msg


def _run(vf, seqlens, H, D, seed, outliers=True, per_head_std=False, device="cpu"):
    cu, cul = cu_tensor(seqlens)
    q, k, v = [t.cuda() for t in workloads.make_qkv(seqlens, H, D, seed, outliers, per_head_std,
                                                     device=device)]
    ws = vf.Workspace(len(seqlens))
    out = vf.attn_varlen_bf16(q, k, v, cu, max(seqlens) if seqlens else 0, workspace=ws)
    torch.cuda.synchronize()
    assert ws.error() == 0
    return out, q, k, v, cu, cul


@pytest.mark.parametrize("outliers", [True, False])
def test_tiny_config(vf, outliers):
    w = workloads.WORKLOADS["tiny"]
    out, q, k, v, cu, cul = _run(vf, w.seqlens, w.H, w.D, w.seeds[-1], outliers)
    _check(vf, out, q, k, v, cul, tag="tiny outliers=%s" % outliers)


@pytest.mark.parametrize("outliers", [True, False])
@pytest.mark.parametrize("D", [64, 72, 80, 128])
def test_ragged_segments(vf, D, outliers):
    seqlens = [1, 127, 128, 129, 300, 17, 0, 5]
    out, q, k, v, cu, cul = _run(vf, seqlens, 3, D, 21, outliers)
    _check(vf, out, q, k, v, cul, tag="ragged D=%d outliers=%s" % (D, outliers))


@pytest.mark.parametrize("factor", [0.25, 3.0])
def test_softmax_scale_argument(vf, factor):
    """sm_scale other than 1/sqrt(D): a flatter and a sharper softmax."""
    seqlens, D = [300, 1000, 77], 128
    cu, cul = cu_tensor(seqlens)
    q, k, v = [t.cuda() for t in workloads.make_qkv(seqlens, 2, D, 61, False, False)]
    sm_scale = factor / math.sqrt(D)
    ws = vf.Workspace(len(seqlens))
    out = vf.attn_varlen_bf16(q, k, v, cu, 1000, sm_scale=sm_scale, workspace=ws)
    torch.cuda.synchronize()
    assert ws.error() == 0
    _check(vf, out, q, k, v, cul, tag="sm_scale x%.2f" % factor, sm_scale=sm_scale)


@pytest.mark.parametrize("D", [8, 16, 24, 40, 48, 56, 88, 96, 104, 112, 120])
def test_every_head_dim(vf, D):
    seqlens = [1, 130, 300, 9, 1]
    out, q, k, v, cu, cul = _run(vf, seqlens, 2, D, 40 + D, outliers=False, per_head_std=True)
    _check(vf, out, q, k, v, cul, tag="D=%d" % D)


def test_single_token_segments_copy_v(vf):
    """A segment of one token attends only to itself: o = v exactly."""
    seqlens = [1] * 37
    out, q, k, v, cu, cul = _run(vf, seqlens, 2, 128, 4)
    assert torch.equal(out.view(torch.int16), v.view(torch.int16))


def test_constant_v_is_reproduced(vf):
    seqlens = [77, 300]
    cu, _ = cu_tensor(seqlens)
    q, k, _ = [t.cuda() for t in workloads.make_qkv(seqlens, 2, 128, 8, True, False)]
    v = torch.full_like(q, 0.75)
    out = vf.attn_varlen_bf16(q, k, v, cu, 300)
    torch.cuda.synchronize()
    assert torch.allclose(out.float(), torch.full_like(out.float(), 0.75), rtol=2 ** -8, atol=0)


def test_rescale_path_late_large_score(vf):
    seqlens = [1000]
    H, D = 1, 128
    cu, cul = cu_tensor(seqlens)
    g = torch.Generator().manual_seed(3)
    q = torch.randn(1000, H, D, generator=g) * 0.3
    k = torch.randn(1000, H, D, generator=g) * 0.3
    v = torch.randn(1000, H, D, generator=g)
    k[900] = q.mean(dim=0) * 40.0
    q, k, v = [t.to(torch.bfloat16).cuda() for t in (q, k, v)]
    out = vf.attn_varlen_bf16(q, k, v, cu, 1000)
    torch.cuda.synchronize()
    _check(vf, out, q, k, v, cul, tag="rescale")


def test_deterministic_and_no_cross_segment_leakage(vf):
    seqlens = [300, 129, 500]
    out1, q, k, v, cu, cul = _run(vf, seqlens, 2, 128, 7)
    out2 = vf.attn_varlen_bf16(q, k, v, cu, 500)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    k2, v2 = k.clone(), v.clone()
    k2[300:429] = -k2[300:429] * 3.0
    v2[300:429] = 5.0
    out3 = vf.attn_varlen_bf16(q, k2, v2, cu, 500)
    torch.cuda.synchronize()
    a, b = out1.view(torch.int16), out3.view(torch.int16)
    assert torch.equal(a[:300], b[:300]) and torch.equal(a[429:], b[429:])
    assert not torch.equal(a[300:429], b[300:429])


def test_bad_seqlens_reports_and_writes_nothing(vf):
    H, D, T = 2, 128, 64
    q = torch.zeros((T, H, D), dtype=torch.bfloat16, device="cuda")
    out = torch.full((T, H, D), 7.0, dtype=torch.bfloat16, device="cuda")
    for bad in ([0, 40, 30, 64], [0, 32, 60], [1, 32, 64]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        ws = vf.Workspace(len(bad) - 1)
        vf.attn_varlen_bf16(q, q, q, cu, 64, out=out, workspace=ws)
        assert ws.error() == 6
    assert torch.all(out.float() == 7.0)


def test_empty_inputs_are_noops(vf):
    cu = torch.zeros(1, dtype=torch.int32, device="cuda")
    e = torch.empty((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    out = vf.attn_varlen_bf16(e, e, e, cu, 0)
    torch.cuda.synchronize()
    assert out.shape == (0, 2, 128)


@pytest.mark.parametrize("name,outliers", [("micro8k", True), ("micro8k", False), ("hd3", False),
                                           ("qhd3", False), ("uhd3mix", True)])
def test_full_size_sampled_rows(vf, name, outliers):
    """Full-size workloads in the bench's launch configuration, sampled query rows."""
    w = workloads.WORKLOADS[name]
    cu, cul = cu_tensor(w.seqlens)
    seed = w.layer_seeds[0] if w.scaling == "calibrated" else w.seeds[0]
    q, k, v = workloads.make_qkv(w.seqlens, w.H, w.D, seed, outliers and w.outliers,
                                 w.per_head_std, device="cuda")
    out = vf.attn_varlen_bf16(q, k, v, cu, w.max_seqlen)
    torch.cuda.synchronize()
    rows = sample_rows(cul, 48, seed=1)
    has_outliers = outliers and w.outliers
    literal = (not has_outliers) and name in ("micro8k", "qhd3")
    _check(vf, out, q, k, v, cul, rows, literal, "%s outliers=%s" % (name, has_outliers))


def test_buffers_beyond_2_gib(vf):
    """272 segments of 4096 tokens x 16 heads x d = 128: the last segment's
    element offsets in the bf16 q/k/v/out buffers pass 2^31."""
    H, D, L, B = 16, 128, 4096, 272
    T = L * B
    cu, _ = cu_tensor([L] * B)
    g = torch.Generator(device="cuda").manual_seed(77)
    src = []
    for _ in range(3):
        x = torch.empty((T, H, D), dtype=torch.bfloat16, device="cuda")
        for c in range(0, T, 1 << 16):
            x[c:c + (1 << 16)] = torch.randn((1 << 16, H, D), device="cuda", generator=g).to(torch.bfloat16)
        src.append(x)
    q, k, v = src
    ws = vf.Workspace(B)
    out = vf.attn_varlen_bf16(q, k, v, cu, L, workspace=ws)
    torch.cuda.synchronize()
    assert ws.error() == 0
    assert (T - L) * H * D > 2 ** 31
    rng = np.random.default_rng(4)
    for s in (0, B - 1):
        a, b = s * L, (s + 1) * L
        rows = np.sort(rng.choice(L, 24, replace=False))
        _check(vf, out[a:b], q[a:b], k[a:b], v[a:b], [0, L], rows=rows, literal=True,
               tag="segment %d of %d" % (s, B))


def test_more_segments_than_the_sorted_work_list(vf):
    rng = np.random.default_rng(8)
    seqlens = [int(x) for x in rng.integers(0, 25, 3000)]
    out, q, k, v, cu, cul = _run(vf, seqlens, 3, 64, 9, outliers=False)
    _check(vf, out, q, k, v, cul, tag="3000 segments")
