"""The FP8 attention call runs one of four kernels (the library's choice, or
the one named by ``kernel=``):

* "unit": one CTA per 128-query work item;
* "persistent": one CTA per SM walking the same work items;
* "two_tile": one CTA per 256-query unit, two query tiles sharing each key
  tile (one S buffer for d > 80, one per tile for d <= 80);
* "two_tile_persistent": one CTA per SM walking the same 256-query units.

The unit and persistent kernels do the same arithmetic for every item, so
their outputs are bit-identical, and so are the two two-tile kernels.  The
two-tile kernels move a row's reference at 128-key boundaries; their outputs
are checked against the fp64 oracle under the same bound as every other
case, and against the unit kernel (almost all outputs identical).  The BF16 path has the unit and persistent kernels,
chosen by max_seqlen (an upper bound on the segment lengths, so a larger one
runs the other kernel on the same inputs).
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


def nsm():
    return torch.cuda.get_device_properties(0).multi_processor_count


CASES = [
    ("ragged", [1, 127, 128, 129, 300, 17, 0, 5], 16, 128),
    ("hd_like", [3600, 3600, 3600], 4, 80),
    ("split_last_wave", [2048], 12, 128),          # 192 items: the last 40 split in 3
    ("many_short", [256] * 200, 4, 64),            # ~5 units per CTA
    ("near_threshold", [6000, 100, 44], 4, 128),
    ("d40_ragged", [255, 256, 257, 513, 1], 3, 40),
    ("d96", [1000, 300], 2, 96),
]


def _codes(vf, seqlens, H, D, seed):
    cu, cul = cu_tensor(seqlens)
    st = vf.ScaleState().init()
    ost = oscales.ScaleState()
    q, k, v = [t.cuda() for t in workloads.make_qkv(seqlens, H, D, seed, True, False, device="cpu")]
    vf.amax_update(st, q, k, v, cu)
    oracle_push(ost, q, k, v)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
    return dict(cu=cu, cul=cul, st=st, scales=list(ost.scale), q=q, k=k, v=v, q8=q8, k8=k8, v8t=v8t)


def _run(vf, c, seqlens, D, kernel):
    ws = vf.Workspace(len(seqlens))
    out = vf.attn_varlen(c["q8"], c["k8"], c["v8t"], c["st"], c["cu"], max(seqlens), D, workspace=ws,
                         kernel=kernel)
    torch.cuda.synchronize()
    assert ws.error() == 0
    return out


def _oracle_check(c, out, seqlens, D, name, nrows=1500):
    T = sum(seqlens)
    rows = None
    if T > 4000:
        rows = np.random.default_rng(5).choice(T, nrows, replace=False)
    stats = compare_attention(out, c["q8"], c["k8"], vt_to_thd(c["v8t"], T), c["scales"], c["cul"], D,
                              rows=rows)
    assert_attention_ok(stats, name, True)


def _close_to(a, b):
    """Two-tile against unit outputs: almost all bits equal, the rest within
    a few bf16 ulps of the output's scale."""
    eq = (a.view(torch.int16) == b.view(torch.int16)).float().mean().item()
    diff = (a.float() - b.float()).abs()
    scale = b.float().abs().amax(dim=-1, keepdim=True).clamp_min(1.0)
    assert eq >= 0.95, eq
    assert (diff <= scale * 2.0 ** -5).all(), diff.max().item()


@pytest.mark.parametrize("name,seqlens,H,D", CASES, ids=[c[0] for c in CASES])
def test_kernels_agree(vf, name, seqlens, H, D):
    c = _codes(vf, seqlens, H, D, 90 + len(name))
    unit = _run(vf, c, seqlens, D, "unit")
    pers = _run(vf, c, seqlens, D, "persistent")
    assert torch.equal(unit.view(torch.int16), pers.view(torch.int16))
    two = _run(vf, c, seqlens, D, "two_tile")
    two_p = _run(vf, c, seqlens, D, "two_tile_persistent")
    assert torch.equal(two.view(torch.int16), two_p.view(torch.int16))
    _oracle_check(c, pers, seqlens, D, name)
    _oracle_check(c, two, seqlens, D, name + " two-tile")
    _close_to(two, unit)


def test_auto_runs_the_rule(vf):
    """attn_varlen without a kernel gives the bits of the kernel the stated rule names."""
    for seqlens, H, D in (([3600] * 3, 16, 80), ([300, 200], 2, 128), ([1024] * 8, 16, 64),
                          ([1024] * 8, 5, 64), ([8192], 16, 128)):
        c = _codes(vf, seqlens, H, D, 7)
        name = vf.attn_kernel_for(len(seqlens), max(seqlens), sum(seqlens), H, nsm())
        auto = _run(vf, c, seqlens, D, "auto")
        named = _run(vf, c, seqlens, D, name)
        assert torch.equal(auto.view(torch.int16), named.view(torch.int16)), name


def test_unknown_kernel_rejected(vf):
    c = _codes(vf, [64], 1, 64, 3)
    with pytest.raises(ValueError):
        _run(vf, c, [64], 64, "fastest")


@pytest.mark.parametrize("name,seqlens,H,D", CASES[:5], ids=[c[0] for c in CASES[:5]])
def test_bf16_kernels_agree_bitwise(vf, name, seqlens, H, D):
    """The BF16 path has the unit and persistent kernels, chosen by max_seqlen."""
    assert max(seqlens) <= PERSISTENT_MAX
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
    """FP8: unit and persistent kernels bit-identical, the two-tile kernel on
    sampled rows against the oracle; BF16: its two kernels bit-identical."""
    seqlens, H, D = _random_batches()[case]
    c = _codes(vf, seqlens, H, D, 500 + case)
    unit = _run(vf, c, seqlens, D, "unit")
    pers = _run(vf, c, seqlens, D, "persistent")
    assert torch.equal(unit.view(torch.int16), pers.view(torch.int16)), case
    two = _run(vf, c, seqlens, D, "two_tile")
    two_p = _run(vf, c, seqlens, D, "two_tile_persistent")
    assert torch.equal(two.view(torch.int16), two_p.view(torch.int16)), case
    T = sum(seqlens)
    rows = np.random.default_rng(case).choice(T, min(T, 300), replace=False)
    for out, tag in ((unit, "unit"), (two, "two-tile")):
        assert torch.isfinite(out.float()).all()
        stats = compare_attention(out, c["q8"], c["k8"], vt_to_thd(c["v8t"], T), c["scales"], c["cul"], D,
                                  rows=rows)
        assert_attention_ok(stats, "random batch %d %s" % (case, tag), True)
    _close_to(two, unit)
    outs = []
    for max_seqlen in (max(seqlens), 1 << 20):
        ws = vf.Workspace(len(seqlens))
        outs.append(vf.attn_varlen_bf16(c["q"], c["k"], c["v"], c["cu"], max_seqlen, workspace=ws))
        torch.cuda.synchronize()
        assert ws.error() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16)), case
