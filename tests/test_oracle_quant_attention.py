"""Pins for the oracle's quantize/un-pad and attention (CPU only)."""

import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention, e4m3, quant, scales


def _bf16_np(t):
    return t.float().numpy()


def test_unpad_padded_equals_packed_and_ignores_pad_rows():
    seqlens = [5, 11, 3]
    H, D = 2, 16
    q, _, _ = workloads.make_qkv(seqlens, H, D, seed=4)
    cu = np.cumsum([0] + seqlens)
    s_max = 13
    pad = workloads.to_padded(q, seqlens, s_max, fill=30000.0)
    a = quant.gather_valid(_bf16_np(q).ravel(), quant.SrcLayout.packed(H, D), cu, H, D)
    b = quant.gather_valid(_bf16_np(pad).ravel(), quant.SrcLayout.padded_batch(s_max, H, D), cu, H, D)
    assert np.array_equal(a, b)
    assert scales.amax(b) < 30000.0


def test_strided_source_view():
    # q as a view into a fused [T, 3, H, D] buffer: token stride 3*H*D.
    seqlens = [7, 9]
    H, D = 3, 8
    q, k, v = workloads.make_qkv(seqlens, H, D, seed=6)
    fused = torch.stack([q, k, v], dim=1).contiguous()      # [T, 3, H, D]
    cu = np.cumsum([0] + seqlens)
    lay = quant.SrcLayout(0, 0, 3 * H * D, D)
    flat = _bf16_np(fused).ravel()
    got_k = quant.gather_valid(flat[H * D:], lay, cu, H, D)
    assert np.array_equal(got_k, _bf16_np(k))


def test_quantize_matches_torch_and_pads_zero():
    seqlens = [17, 40]
    H, D, D_pad = 2, 24, 32
    q, _, _ = workloads.make_qkv(seqlens, H, D, seed=7)
    cu = np.cumsum([0] + seqlens)
    inv = np.float32(448.0) / scales.amax(_bf16_np(q))
    codes = quant.quantize_unpad(_bf16_np(q).ravel(), quant.SrcLayout.packed(H, D), cu, H, D, D_pad, inv)
    assert codes.shape == (57, H, D_pad)
    assert np.all(codes[:, :, D:] == 0)
    y = (q.float() * torch.tensor(inv)).clamp(-448, 448)
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[:, :, :D], ref)
    # the tensor's amax maps exactly to +-448 under its own dynamic scale
    assert np.abs(e4m3.decode(codes[:, :, :D])).max() == 448.0


def _rand_qkv(T, H, D, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, H, D)), rng.standard_normal((T, H, D)),
            rng.standard_normal((T, H, D)))


def test_attention_matches_bruteforce_loops():
    cu = [0, 3, 8, 9]
    q, k, v = _rand_qkv(9, 2, 4, seed=1)
    a = attention.attention_varlen(q, k, v, cu)
    b = attention.attention_bruteforce(q, k, v, cu)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


def test_attention_rows_are_convex_weights():
    # V = one-hot rows: o_i is the softmax row itself -> non-negative, sums to 1.
    L, D = 6, 8
    q, k, _ = _rand_qkv(L, 1, D, seed=2)
    v = np.zeros((L, 1, L))
    v[np.arange(L), 0, np.arange(L)] = 1.0
    o = attention.attention_varlen(q, k, v, [0, L], sm_scale=1 / math.sqrt(D))
    assert np.all(o >= 0)
    assert np.allclose(o.sum(axis=2), 1.0, atol=1e-14)


def test_constant_v_reproduces_v():
    q, k, _ = _rand_qkv(20, 2, 8, seed=3)
    v = np.ones((20, 2, 8)) * 0.37
    o = attention.attention_varlen(q, k, v, [0, 12, 20])
    assert np.allclose(o, 0.37, atol=1e-14)


def test_key_permutation_invariance_within_segment():
    q, k, v = _rand_qkv(30, 2, 8, seed=4)
    cu = [0, 10, 30]
    o1 = attention.attention_varlen(q, k, v, cu)
    perm = np.arange(30)
    perm[10:] = 10 + np.random.default_rng(0).permutation(20)
    o2 = attention.attention_varlen(q, k[perm], v[perm], cu)
    assert np.allclose(o1, o2, atol=1e-13)


def test_zero_cross_segment_leakage():
    q, k, v = _rand_qkv(30, 2, 8, seed=5)
    cu = [0, 10, 22, 30]
    o1 = attention.attention_varlen(q, k, v, cu)
    k2, v2 = k.copy(), v.copy()
    k2[10:22] += 5.0
    v2[10:22] *= -3.0
    o2 = attention.attention_varlen(q, k2, v2, cu)
    assert np.array_equal(o1[:10], o2[:10]) and np.array_equal(o1[22:], o2[22:])
    assert not np.allclose(o1[10:22], o2[10:22])


def test_single_segment_matches_torch_sdpa_float64():
    q, k, v = _rand_qkv(37, 3, 16, seed=6)
    o = attention.attention_varlen(q, k, v, [0, 37])
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[0].permute(1, 0, 2).numpy()
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_sampled_rows_equal_full_rows():
    q, k, v = _rand_qkv(40, 2, 8, seed=7)
    cu = [0, 15, 40]
    full = attention.attention_varlen(q, k, v, cu)
    rows = [0, 3, 14, 15, 39]
    part = attention.attention_varlen(q, k, v, cu, rows=rows)
    assert np.array_equal(part[rows], full[rows])
    assert np.isnan(part[1]).all()


def test_zero_padded_head_dim_leaves_codes_attention_unchanged():
    seqlens = [9, 14]
    H, D = 2, 16
    q, k, v = workloads.make_qkv(seqlens, H, D, seed=8)
    cu = np.cumsum([0] + seqlens)
    lay = quant.SrcLayout.packed(H, D)
    sc = [np.float32(1.0)] * 3
    c16 = [quant.quantize_unpad(_bf16_np(t).ravel(), lay, cu, H, D, D, np.float32(20.0)) for t in (q, k, v)]
    c32 = [quant.quantize_unpad(_bf16_np(t).ravel(), lay, cu, H, D, 32, np.float32(20.0)) for t in (q, k, v)]
    o16 = attention.attention_fp8(*c16, sc, cu, D)
    qh = attention.dequant(c32[0], 1.0)
    kh = attention.dequant(c32[1], 1.0)
    vh = attention.dequant(c32[2], 1.0)
    o32 = attention.attention_varlen(qh, kh, vh, cu, sm_scale=1 / math.sqrt(D))
    assert np.allclose(o16, o32[:, :, :D], atol=1e-13)
    assert np.all(o32[:, :, D:] == 0)


def test_p8_exact_when_p_is_representable():
    # Scores whose exponentials are powers of two: rounding P changes nothing.
    L = 8
    q = np.zeros((L, 1, 2))
    k = np.zeros((L, 1, 2))
    q[:, 0, 0] = 1.0
    k[:, 0, 0] = -np.log(2.0) * (np.arange(L) % 3)      # s in {0, -ln2, -2ln2}
    v = np.random.default_rng(0).standard_normal((L, 1, 4))
    a = attention.attention_varlen(q, k, v, [0, L], sm_scale=1.0)
    b = attention.attention_varlen_p8(q, k, v, [0, L], sm_scale=1.0)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-13)


def test_p8_error_within_e4m3_bound_and_nonzero():
    q, k, v = _rand_qkv(64, 2, 16, seed=9)
    cu = [0, 64]
    a = attention.attention_varlen(q, k, v, cu)
    b = attention.attention_varlen_p8(q, k, v, cu)
    # Each weight p_j/l moves by at most a factor (1 +- 2^-4)/(1 -+ 2^-4) and both
    # weight sets sum to one, so |b - a| <= (2^-3 / (1 - 2^-4)) * (max v - min v) / 2.
    rng_v = v.max(axis=0, keepdims=True) - v.min(axis=0, keepdims=True)
    bound = (2.0 ** -3 / (1 - 2.0 ** -4)) * rng_v / 2 + 1e-12
    assert np.all(np.abs(b - a) <= bound)
    rel = np.sqrt(np.mean((b - a) ** 2)) / np.sqrt(np.mean(a ** 2))
    assert 1e-3 < rel < 6e-2


def test_p8_weights_sum_to_one():
    # Constant V comes back exactly and one-hot V rows sum to one: the rounded
    # weights are normalised by their own sum.
    L, D = 40, 8
    q, k, _ = _rand_qkv(L, 1, D, seed=11)
    v = np.full((L, 1, 4), -1.75)
    o = attention.attention_varlen_p8(q, k, v, [0, L])
    assert np.allclose(o, -1.75, rtol=0, atol=1e-14)
    v1 = np.zeros((L, 1, L))
    v1[np.arange(L), 0, np.arange(L)] = 1.0
    o1 = attention.attention_varlen_p8(q, k, v1, [0, L])
    assert np.allclose(o1.sum(axis=2), 1.0, atol=1e-14)
    # and every weight is an E4M3-representable value over the common sum
    w = o1[:, 0, :] * (1.0 / o1[:, 0, :].max(axis=1, keepdims=True))
    assert np.all(w >= 0)


def test_p8_underflow_drops_far_keys():
    # Keys 20 binades below the maximum give 2^8 p = 2^-12 < 2^-10 (half the
    # smallest E4M3 subnormal): they round to zero and o is the top key's value.
    L = 6
    q = np.zeros((L, 1, 1))
    k = np.zeros((L, 1, 1))
    q[:, 0, 0] = 1.0
    k[:, 0, 0] = -20 * np.log(2.0)
    k[2, 0, 0] = 0.0
    v = np.arange(L, dtype=np.float64).reshape(L, 1, 1) + 0.5
    o = attention.attention_varlen_p8(q, k, v, [0, L], sm_scale=1.0)
    assert np.all(o == 2.5)
    # 17 binades below: 2^-9 is the smallest subnormal and survives
    k[:, 0, 0] = -17 * np.log(2.0)
    k[2, 0, 0] = 0.0
    o = attention.attention_varlen_p8(q, k, v, [0, L], sm_scale=1.0)
    w_far = 2.0 ** -9
    expect = (2.5 * 256 + w_far * (v[:, 0, 0].sum() - 2.5)) / (256 + 5 * w_far)
    assert np.allclose(o, expect, rtol=1e-12)


def test_p8_does_not_depend_on_reference_power_of_two():
    # Shifting every score of a row by a multiple of ln 2 shifts P by a power of
    # two and must leave the rounded result unchanged.
    q, k, v = _rand_qkv(16, 1, 8, seed=10)
    cu = [0, 16]
    o1 = attention.attention_varlen_p8(q, k, v, cu, sm_scale=1.0)
    q2 = np.concatenate([q, np.ones((16, 1, 1))], axis=2)
    k2 = np.concatenate([k, np.full((16, 1, 1), 3 * np.log(2.0))], axis=2)
    o2 = attention.attention_varlen_p8(q2, k2, v, cu, sm_scale=1.0)
    assert np.allclose(o1, o2, rtol=1e-10, atol=1e-12)
