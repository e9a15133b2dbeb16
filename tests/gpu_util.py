"""Helpers shared by the GPU parity tests (test infrastructure).

The CUDA path runs through the C ABI (via the thin binding); the oracle runs on
CPU copies of the very same seeded inputs.
"""

import math

import numpy as np
import torch

import workloads
from oracle import attention as oattn
from oracle import quant as oquant
from oracle import scales as oscales

# Tolerances (derivation in the design notes, section "Tolerances"):
#
# * Literal bound, unit-normal inputs on the benchmark shapes (long segments):
#   max-abs 2e-2 and relative RMS 1e-2, the RMS error taken relative to the
#   RMS of the dequantized value inputs (the inputs' unit scale).
# * Every case: relative RMS 1e-2 as above, and max-abs at most 2^-4 of
#   max(1, max|o_ref|).  2^-4 is E4M3's relative half-ulp: with few keys per
#   row (short segments) or a few dominant keys (x20 outliers) the rounding of
#   the P weights is not averaged out, and outputs with outliers reach tens.
# * Against the oracle variant that requantizes P exactly as specified
#   (E4M3(2^8 p) on the row's power-of-two maximum, weights normalised by their
#   rounded sum), output rounded to bf16: relative RMS 2e-3 without outliers;
#   1e-2 with outliers, where the online reference is lower than the final one
#   for early tiles and keeps mass that the final-reference model underflows.
#
# BF16 comparison path (bf16 inputs, P rounded to bf16 and normalised by the
# sum of the rounded weights): each rounded weight p~_j = p_j (1 + d_j) with
# |d_j| <= 2^-9, so o - o_ref = sum_j w_j (d_j - d_mean) v_j / (1 + d_mean) is
# at most 2^-8 max|v|, plus 2^-9 |o| <= 2^-9 max|v| from the output rounding;
# the test allows 2^-7 max(1, max|v|) (margin for the fp32 sums and the
# tensor-core accumulation), and relative RMS 2e-3 of RMS(v).
TOL_BF16_MAX_VREL = 2.0 ** -7
TOL_BF16_REL_RMS = 2e-3
TOL_MAX_ABS = 2e-2
TOL_REL_RMS = 1e-2
TOL_MAX_NORM = 2.0 ** -4
TOL_P8_REL_RMS = 2e-3
TOL_P8_REL_RMS_OUTLIERS = 1e-2


def np32(t):
    return t.detach().float().cpu().numpy()


def vt_to_thd(v8t, T):
    """[H, D_pad, Tv] transposed V codes -> [T, H, D_pad]."""
    return v8t[:, :, :T].permute(2, 0, 1).contiguous()


def oracle_codes(x, inv):
    return oquant.quantize(np32(x), inv)


def check_codes(vf_codes, x, inv, D, D_pad):
    """Bit-exact comparison of [T, H, D_pad] codes against the oracle."""
    got = vf_codes.cpu().numpy()
    ref = oracle_codes(x, inv)
    assert got.shape[2] == D_pad
    mism = np.count_nonzero(got[:, :, :D] != ref)
    assert mism == 0, "%d code mismatches" % mism
    assert np.all(got[:, :, D:] == 0)


def sample_rows(cu, per_segment, seed=0):
    """Seeded sample of query rows: first, last and random rows of every segment."""
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(len(cu) - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        if e - s <= per_segment:
            rows.extend(range(s, e))
        else:
            pick = set(rng.choice(np.arange(s, e), per_segment - 2, replace=False).tolist())
            pick.update([s, e - 1])
            rows.extend(sorted(pick))
    return np.array(rows, dtype=np.int64)


def value_rms(v8, scale, D):
    """RMS of the dequantized value codes [T, H, >=D] (exact, via a code histogram)."""
    counts = np.bincount(np.ascontiguousarray(v8[:, :, :D]).ravel(), minlength=256).astype(np.float64)
    vals = oattn.dequant(np.arange(256, dtype=np.uint8), scale)
    vals = np.where(np.isnan(vals), 0.0, vals)
    return float(np.sqrt((counts * vals ** 2).sum() / counts.sum()))


def compare_attention(out, q8, k8, v8, scales, cu, D, rows=None, sm_scale=None):
    """Return (max_abs, rel_rms, p8_rel_rms, err/|o|) on the given rows.

    max_abs is max|o - o_ref| (and max_norm that over max(1, max|o_ref|)); rel_rms is
    RMS(o - o_ref) / RMS(v_hat); p8_rel_rms compares with the
    P-rounding oracle variant rounded to bf16, relative to RMS of that output.
    """
    T = q8.shape[0]
    q8n, k8n, v8n = q8.cpu().numpy(), k8.cpu().numpy(), v8.cpu().numpy()
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if rows is None:
        rows = np.arange(T)
    rows = np.unique(np.asarray(rows, dtype=np.int64))
    ref = oattn.attention_fp8(q8n, k8n, v8n, scales, cu, D, sm_scale, rows)
    ref8 = oattn.attention_fp8(q8n, k8n, v8n, scales, cu, D, sm_scale, rows, p_round=True)
    got = out[torch.from_numpy(rows).to(out.device)].float().cpu().numpy().astype(np.float64)
    v_rms = value_rms(v8n, scales[2], D)
    err = got - ref
    max_abs = float(np.abs(err).max())
    max_norm = max_abs / max(1.0, float(np.abs(ref).max()))
    rel_rms = float(np.sqrt(np.mean(err ** 2)) / v_rms)
    ref8_bf = torch.from_numpy(ref8).to(torch.bfloat16).double().numpy()
    p8 = float(np.sqrt(np.mean((got - ref8_bf) ** 2)) / np.sqrt(np.mean(ref8 ** 2)))
    ref_rel = float(np.sqrt(np.mean(err ** 2)) / np.sqrt(np.mean(ref ** 2)))
    return dict(max_abs=max_abs, max_norm=max_norm, rel_rms=rel_rms, p8=p8, ref_rel=ref_rel)


def assert_attention_ok(stats, tag="", outliers=False, literal=False):
    msg = ("%s max_abs=%.3e max_norm=%.3e rel_rms=%.3e p8_rel_rms=%.3e (err/|o| %.3e)"
           % (tag, stats["max_abs"], stats["max_norm"], stats["rel_rms"], stats["p8"], stats["ref_rel"]))
    print(msg)
    if literal:
        assert not outliers
        assert stats["max_abs"] <= TOL_MAX_ABS, msg
    assert stats["max_norm"] <= TOL_MAX_NORM, msg
    assert stats["rel_rms"] <= TOL_REL_RMS, msg
    assert stats["p8"] <= (TOL_P8_REL_RMS_OUTLIERS if outliers else TOL_P8_REL_RMS), msg


def state_matches(st_dict, ost):
    """Bit-exact comparison of the device state with the oracle's ScaleState."""
    f32 = lambda a: np.asarray(a, dtype=np.float32)
    assert np.array_equal(f32(st_dict["hist"]), ost.hist)
    assert st_dict["pos"] == ost.pos and st_dict["count"] == ost.count
    assert st_dict["mode"] == ost.mode
    assert np.array_equal(f32(st_dict["amax_ref"]), ost.amax_ref)
    assert np.array_equal(f32(st_dict["scale"]), ost.scale)
    assert np.array_equal(f32(st_dict["inv_scale"]), ost.inv_scale)
    if ost.mode == 0:
        assert np.array_equal(f32(st_dict["amax_cur"]), ost.amax_cur)
    assert st_dict["amax_bits"] == [0, 0, 0] and st_dict["blocks_done"] == 0
    assert st_dict["dev_error"] == 0


def oracle_push(ost, q, k, v):
    ost.push([oscales.amax(np32(q)), oscales.amax(np32(k)), oscales.amax(np32(v))])


def cu_tensor(seqlens, device="cuda"):
    cu = [0]
    for L in seqlens:
        cu.append(cu[-1] + L)
    return torch.tensor(cu, dtype=torch.int32, device=device), cu


def qkv(seqlens, H, D, seed, outliers=True, per_head_std=False, device="cuda"):
    return [t.to(device) for t in workloads.make_qkv(seqlens, H, D, seed, outliers, per_head_std)]
