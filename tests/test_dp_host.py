"""Data-parallel host logic on CPU: segment sharding, and the dynamic-scaling
exchange run by two gloo ranks.

The ranks compute their local amax with the oracle (no GPU here), combine
them through the library's all-reduce helper, and push into oracle ring
states; both rings must equal the single-process ring of the whole batch.
"""

import itertools
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import workloads
from oracle import scales as oscales


@pytest.fixture(scope="module")
def dp():
    from fp8_vision_encoder_gb300 import dp
    return dp


def _cost(seqlens, part):
    return sum(int(seqlens[i]) ** 2 for i in part)


def test_shard_covers_every_segment_once(dp):
    rng = np.random.default_rng(1)
    for _ in range(50):
        n = int(rng.integers(0, 12))
        seqlens = [int(x) for x in rng.integers(0, 5000, n)]
        for w in (1, 2, 3, 8):
            parts = dp.shard_segments(seqlens, w)
            assert len(parts) == w
            flat = sorted(i for p in parts for i in p)
            assert flat == list(range(n))
            assert all(p == sorted(p) for p in parts)


def test_shard_balance_within_lpt_bound(dp):
    # Longest-processing-time-first is within 4/3 - 1/(3m) of the optimum
    # (Graham); the optimum is brute-forced on small cases.
    rng = np.random.default_rng(2)
    for _ in range(40):
        n = int(rng.integers(1, 8))
        seqlens = [int(x) for x in rng.integers(1, 3000, n)]
        for w in (2, 3):
            parts = dp.shard_segments(seqlens, w)
            got = max(_cost(seqlens, p) for p in parts)
            best = min(max(sum(int(seqlens[i]) ** 2 for i in range(n) if a[i] == r) for r in range(w))
                       for a in itertools.product(range(w), repeat=n))
            assert got <= (4 / 3 - 1 / (3 * w)) * best + 1e-9


def test_shard_examples(dp):
    # three equal QHD images on two ranks: two on rank 0, one on rank 1
    assert dp.shard_segments([14400] * 3, 2) == [[0, 2], [1]]
    assert dp.shard_segments([5], 3) == [[0], [], []]
    assert dp.shard_segments([], 2) == [[], []]
    with pytest.raises(ValueError):
        dp.shard_segments([1], 0)


def test_shard_cu_seqlens(dp):
    cu, ranges = dp.shard_cu_seqlens([3, 5, 7, 2], [1, 3])
    assert cu == [0, 5, 7]
    assert ranges == [(3, 8), (15, 17)]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, seqlens, H, D, seeds, out_dir):
    import torch.distributed as dist
    from fp8_vision_encoder_gb300 import dp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = dp.shard_segments(seqlens, world)[rank]
        _, ranges = dp.shard_cu_seqlens(seqlens, mine)
        st = oscales.ScaleState()
        for seed in seeds:
            q, k, v = workloads.make_qkv(seqlens, H, D, seed, True, True)
            vals = torch.zeros(4, dtype=torch.float32)
            if ranges:
                idx = torch.cat([torch.arange(a, b) for a, b in ranges])
                for t, x in enumerate((q, k, v)):
                    vals[t] = float(oscales.amax(x[idx].float().numpy()))
                vals[3] = 1.0
            dp.allreduce_amax(vals)
            if vals[3] > 0:
                st.push(vals[:3].numpy())
        np.savez(os.path.join(out_dir, "rank%d.npz" % rank), hist=st.hist, pos=st.pos,
                 count=st.count, amax_ref=st.amax_ref, scale=st.scale, inv_scale=st.inv_scale)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("seqlens", [[300, 77, 500, 64, 129], [200]])
def test_two_gloo_ranks_keep_identical_rings(tmp_path, seqlens):
    H, D, seeds, world = 2, 64, list(range(18)), 2
    mp.start_processes(_rank_main, args=(world, _free_port(), seqlens, H, D, seeds, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    ref = oscales.ScaleState()
    for seed in seeds:
        q, k, v = workloads.make_qkv(seqlens, H, D, seed, True, True)
        ref.push([oscales.amax(x.float().numpy()) for x in (q, k, v)])
    for r in range(world):
        got = np.load(os.path.join(str(tmp_path), "rank%d.npz" % r))
        assert np.array_equal(got["hist"], ref.hist)
        assert int(got["pos"]) == ref.pos and int(got["count"]) == ref.count
        for f in ("amax_ref", "scale", "inv_scale"):
            assert np.array_equal(got[f], getattr(ref, f)), f
