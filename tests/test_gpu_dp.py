"""GPU: the data-parallel split of dynamic scaling, on one GPU.

amax_local + ring_push must equal amax_update bit for bit, and two shards of a
batch (two stand-in ranks, their values combined with an elementwise max in
place of the all-reduce) must leave every rank's state equal to amax_update
over the whole batch -- and to the oracle.
"""

import numpy as np
import pytest
import torch

from oracle import scales as oscales

from gpu_util import cu_tensor, oracle_push, qkv, state_matches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vf():
    import fp8_vision_encoder_gb300 as vf
    assert torch.cuda.is_available()
    return vf


def test_local_plus_push_equals_update(vf):
    seqlens, H, D = [300, 77, 500, 64], 4, 80
    cu, _ = cu_tensor(seqlens)
    a = vf.ScaleState().init()
    b = vf.ScaleState().init()
    ost = oscales.ScaleState()
    for seed in range(18):   # the ring wraps
        q, k, v = qkv(seqlens, H, D, 40 + seed, outliers=(seed % 2 == 0), per_head_std=True)
        vf.amax_update(a, q, k, v, cu)
        vals = vf.amax_local(b, q, k, v, cu)
        torch.cuda.synchronize()
        assert vals[3].item() == 1.0
        assert torch.equal(vals[:3].cpu(), torch.tensor(a.read()["amax_cur"], dtype=torch.float32))
        vf.ring_push(b, vals)
        torch.cuda.synchronize()
        assert torch.equal(a.buf, b.buf)
        oracle_push(ost, q, k, v)
        state_matches(b.read(), ost)


@pytest.mark.parametrize("world", [2, 3])
def test_shards_reduced_equal_whole_batch(vf, world):
    from fp8_vision_encoder_gb300 import dp
    seqlens, H, D = [300, 77, 500, 64, 129], 2, 128
    cu, _ = cu_tensor(seqlens)
    whole = vf.ScaleState().init()
    ranks = [vf.ScaleState().init() for _ in range(world)]
    parts = dp.shard_segments(seqlens, world)
    for seed in range(20):
        q, k, v = qkv(seqlens, H, D, 7 * seed + 1, outliers=True)
        vf.amax_update(whole, q, k, v, cu)
        vals = []
        for r in range(world):
            rcu, ranges = dp.shard_cu_seqlens(seqlens, parts[r])
            if ranges:
                idx = torch.cat([torch.arange(s, e) for s, e in ranges]).cuda()
                qs, ks, vs = (x.index_select(0, idx).contiguous() for x in (q, k, v))
            else:
                qs, ks, vs = (x[:0] for x in (q, k, v))
            rcu_t = torch.tensor(rcu, dtype=torch.int32, device="cuda")
            vals.append(vf.amax_local(ranks[r], qs, ks, vs, rcu_t, total_tokens=rcu[-1], H=H, D=D))
        red = torch.stack(vals).max(dim=0).values     # the all-reduce(MAX)
        for r in range(world):
            vf.ring_push(ranks[r], red.clone())
        torch.cuda.synchronize()
        for r in range(world):
            assert torch.equal(ranks[r].buf, whole.buf), "rank %d after forward %d" % (r, seed)


def test_static_and_empty(vf):
    seqlens, H, D = [64, 32], 2, 64
    cu, _ = cu_tensor(seqlens)
    q, k, v = qkv(seqlens, H, D, 3)
    st = vf.ScaleState().init().set_static(224.0, 198.0, 210.0)
    before = st.buf.clone()
    vals = vf.amax_local(st, q, k, v, cu)
    vf.ring_push(st, vals)
    torch.cuda.synchronize()
    assert vals.cpu().tolist() == [0.0, 0.0, 0.0, 0.0]
    assert torch.equal(st.buf, before)
    # a rank without tokens contributes zeros and pushes nothing by itself
    dyn = vf.ScaleState().init()
    before = dyn.buf.clone()
    cu0 = torch.zeros(1, dtype=torch.int32, device="cuda")
    vals = vf.amax_local(dyn, q[:0], k[:0], v[:0], cu0, total_tokens=0, H=H, D=D)
    vf.ring_push(dyn, vals)
    torch.cuda.synchronize()
    assert vals.cpu().tolist() == [0.0, 0.0, 0.0, 0.0]
    assert torch.equal(dyn.buf, before)
    with pytest.raises(ValueError):
        vf.ring_push(dyn, torch.zeros(3, device="cuda"))


def test_dp_helper_without_group_equals_update(vf):
    from fp8_vision_encoder_gb300 import dp
    seqlens, H, D = [128, 256], 2, 128
    cu, _ = cu_tensor(seqlens)
    a = vf.ScaleState().init()
    b = vf.ScaleState().init()
    for seed in range(3):
        q, k, v = qkv(seqlens, H, D, seed)
        vf.amax_update(a, q, k, v, cu)
        dp.amax_update_dp(b, q, k, v, cu)
    torch.cuda.synchronize()
    assert torch.equal(a.buf, b.buf)
