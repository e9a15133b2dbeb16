"""The FP8 attention call runs one of two kernels, chosen by max_seqlen: a
persistent one (one CTA per SM walking the work units, for segments of up to
6144 tokens when there is more than one wave of work items) and one with a
CTA per work item (longer segments, or a single wave).  Both do the
same arithmetic for every unit, so their outputs are bit-identical.  max_seqlen
is only an upper bound on the segment lengths, so passing a larger one runs
the other kernel on the same inputs; the first call of each case runs the
persistent kernel and is also checked against the fp64 oracle.
"""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import assert_attention_ok, compare_attention, cu_tensor, oracle_push, vt_to_thd
from oracle import scales as oscales

pytestmark = pytest.mark.gpu

PERSISTENT_MAX = 6144


@pytest.fixture(scope="module")
def vf():
    import fp8_vision_encoder_gb300 as vf
    assert torch.cuda.is_available()
    return vf


# Every case has more work items than a GB300 has SMs (the persistent kernel
# runs only then: with a single wave there is no next unit to overlap).
CASES = [
    ("ragged", [1, 127, 128, 129, 300, 17, 0, 5], 16, 128),
    ("hd_like", [3600, 3600, 3600], 4, 80),
    ("split_last_wave", [2048], 12, 128),          # 192 items: the last 40 split in 3
    ("many_short", [256] * 200, 4, 64),            # ~5 units per CTA
    ("near_threshold", [6000, 100, 44], 4, 128),
]


@pytest.mark.parametrize("name,seqlens,H,D", CASES, ids=[c[0] for c in CASES])
def test_kernels_agree_bitwise(vf, name, seqlens, H, D):
    assert max(seqlens) <= PERSISTENT_MAX
    cu, cul = cu_tensor(seqlens)
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    q, k, v = [t.cuda() for t in workloads.make_qkv(seqlens, H, D, 90 + len(name), True, False, device="cpu")]
    vf.amax_update(st, q, k, v, cu)
    oracle_push(ost, q, k, v)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
    outs = []
    for max_seqlen in (max(seqlens), 1 << 20):
        ws = vf.Workspace(len(seqlens))
        outs.append(vf.attn_varlen(q8, k8, v8t, st, cu, max_seqlen, D, workspace=ws))
        torch.cuda.synchronize()
        assert ws.error() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    T = sum(seqlens)
    rows = None
    if T > 4000:
        rows = np.random.default_rng(5).choice(T, 1500, replace=False)
    stats = compare_attention(outs[0], q8, k8, vt_to_thd(v8t, T), list(ost.scale), cul, D, rows=rows)
    assert_attention_ok(stats, name, True)


@pytest.mark.parametrize("name,seqlens,H,D", CASES, ids=[c[0] for c in CASES])
def test_bf16_kernels_agree_bitwise(vf, name, seqlens, H, D):
    """The BF16 path has the same two kernels and the same choice."""
    cu, cul = cu_tensor(seqlens)
    q, k, v = [t.cuda() for t in workloads.make_qkv(seqlens, H, D, 190 + len(name), True, False, device="cpu")]
    outs = []
    for max_seqlen in (max(seqlens), 1 << 20):
        ws = vf.Workspace(len(seqlens))
        outs.append(vf.attn_varlen_bf16(q, k, v, cu, max_seqlen, workspace=ws))
        torch.cuda.synchronize()
        assert ws.error() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))



def _random_batches():
    """Seeded random batches with more work items than SMs: up to 60
    segments of 1..6000 tokens, 1..16 heads, a head dim of 32..128."""
    rng = np.random.default_rng(2024)
    out = []
    while len(out) < 6:
        n = int(rng.integers(1, 61))
        seqlens = [int(x) for x in rng.integers(1, 6001, size=n)]
        if rng.random() < 0.3:
            seqlens[int(rng.integers(0, n))] = 0
        H = int(rng.integers(1, 17))
        D = int(rng.choice([32, 64, 80, 128]))
        items = sum(-(-L // 128) for L in seqlens) * H
        if items > 200 and sum(seqlens) * H * D < 40_000_000:
            out.append((seqlens, H, D))
    return out


@pytest.mark.parametrize("case", range(6))
def test_random_batches_agree(vf, case):
    """FP8 and BF16: the persistent kernel (max_seqlen = the true maximum) and
    the per-item kernel (a larger bound) give the same bits on random batches."""
    seqlens, H, D = _random_batches()[case]
    cu, cul = cu_tensor(seqlens)
    q, k, v = [t.cuda() for t in workloads.make_qkv(seqlens, H, D, 500 + case, True, False, device="cpu")]
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    vf.amax_update(st, q, k, v, cu)
    oracle_push(ost, q, k, v)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
    for bf16 in (False, True):
        outs = []
        for max_seqlen in (max(seqlens), 1 << 20):
            ws = vf.Workspace(len(seqlens))
            if bf16:
                outs.append(vf.attn_varlen_bf16(q, k, v, cu, max_seqlen, workspace=ws))
            else:
                outs.append(vf.attn_varlen(q8, k8, v8t, st, cu, max_seqlen, D, workspace=ws))
            torch.cuda.synchronize()
            assert ws.error() == 0
        assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16)), (case, bf16)
        assert torch.isfinite(outs[0].float()).all()
        if not bf16:
            T = sum(seqlens)
            rows = np.random.default_rng(case).choice(T, min(T, 300), replace=False)
            stats = compare_attention(outs[0], q8, k8, vt_to_thd(v8t, T), list(ost.scale), cul, D, rows=rows)
            assert_attention_ok(stats, "random batch %d" % case, True)
