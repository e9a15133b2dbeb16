"""GPU parity of the FP8 attention kernel's key-range split.

When a call's work items (one per 128-query tile of a (segment, head)) leave
a last wave that fills at most half the GPU, the plan cuts each item of that
wave into k parts of consecutive 256-key tiles, one CTA per part, and the
part that finishes last combines them by exact powers of two.  These tests
check, on the device's own SM count:

* that the plan's decision (first split item, parts per item, read back from
  the workspace header) is the rule stated here (``expected_split``), so the
  cases below really run the split path;
* the output of split items against the fp64 oracle, element by element,
  under the same bound as every other attention case;
* that the result does not depend on which part finishes last (bit-identical
  across runs).
"""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import assert_attention_ok, compare_attention, cu_tensor, oracle_push, vt_to_thd
from oracle import scales as oscales

pytestmark = pytest.mark.gpu

from split_rule import BN, ROWS, expected_split


@pytest.fixture(scope="module")
def vf():
    import fp8_vision_encoder_gb300 as vf
    assert torch.cuda.is_available()
    return vf


def nsm():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _run(vf, seqlens, H, D, seed, outliers=True, kernel="unit"):
    cu, cul = cu_tensor(seqlens)
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    q, k, v = workloads.make_qkv(seqlens, H, D, seed, outliers, False, device="cpu")
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    vf.amax_update(st, q, k, v, cu)
    oracle_push(ost, q, k, v)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
    ws = vf.Workspace(len(seqlens))
    out = vf.attn_varlen(q8, k8, v8t, st, cu, max(seqlens), D, workspace=ws, kernel=kernel)
    torch.cuda.synchronize()
    assert ws.error() == 0
    hdr = ws.buf[:20].view(torch.int32).cpu().tolist()   # error, items, nseq, split_first, split_k
    return dict(out=out, q8=q8, k8=k8, v8t=v8t, v8=vt_to_thd(v8t, sum(seqlens)),
                scales=list(ost.scale), cu=cul, cu_t=cu, st=st, hdr=hdr)


@pytest.mark.parametrize("D,outliers", [(128, True), (128, False), (80, True), (64, False)])
def test_every_item_split(vf, D, outliers):
    """One 2048-token segment, 2 heads: 32 items, all in the last wave, each
    cut into 4 parts of 2 key tiles (on 152 SMs)."""
    seqlens, H = [2048], 2
    N, sfirst, k = expected_split(seqlens, H, nsm())
    assert k >= 2 and sfirst == 0
    r = _run(vf, seqlens, H, D, 60 + D, outliers)
    assert r["hdr"][1:] == [N, 1, sfirst, k]
    stats = compare_attention(r["out"], r["q8"], r["k8"], r["v8"], r["scales"], r["cu"], D)
    assert_attention_ok(stats, "split D=%d" % D, outliers)


def test_last_wave_only_split(vf):
    """A long segment fills nsm - 2 items and a 600-token one adds 5 more, so
    the last wave holds 3 items (the 600-token segment's last three query
    tiles, 3 key tiles each): only those are split, into 3 parts."""
    n_sm = nsm()
    seqlens, H, D = [ROWS * (n_sm - 2), 600], 1, 64
    N, sfirst, k = expected_split(seqlens, H, n_sm)
    assert (N, sfirst, k) == (n_sm + 3, n_sm, 3)
    r = _run(vf, seqlens, H, D, 71)
    assert r["hdr"][1:] == [N, 2, sfirst, k]
    s0 = seqlens[0]
    rows = np.concatenate([np.arange(s0, s0 + 600),                       # every row of the short segment
                           np.random.default_rng(3).choice(s0, 200, replace=False)])
    stats = compare_attention(r["out"], r["q8"], r["k8"], r["v8"], r["scales"], r["cu"], D, rows=rows)
    assert_attention_ok(stats, "last wave split", True)


def test_split_ragged_and_deterministic(vf):
    """Ragged segments with unaligned starts whose items have 3 to 6 key tiles
    (and an empty segment), all in the last wave; further runs give
    bit-identical outputs."""
    seqlens, H, D = [1500, 0, 900, 700, 513], 1, 128
    N, sfirst, k = expected_split(seqlens, H, nsm())
    assert k >= 2
    r1 = _run(vf, seqlens, H, D, 72)
    assert r1["hdr"][1:] == [N, len(seqlens), sfirst, k]
    stats = compare_attention(r1["out"], r1["q8"], r1["k8"], r1["v8"], r1["scales"], r1["cu"], D)
    assert_attention_ok(stats, "ragged split", True)
    outs = []
    for _ in range(3):
        ws = vf.Workspace(len(seqlens))
        outs.append(vf.attn_varlen(r1["q8"], r1["k8"], r1["v8t"], r1["st"], r1["cu_t"], max(seqlens), D,
                                   workspace=ws, kernel="unit"))
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), r1["out"].view(torch.int16))
