"""Helpers shared by the GPU parity tests (test infrastructure).

The CUDA path runs through the C ABI (via the thin binding); the oracle runs on
CPU copies of the very same seeded inputs.
"""

import math

import numpy as np
import torch

import workloads
from oracle import attention as oattn
from oracle import e4m3
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
# * Against the oracle variant that requantizes P as reading 12 specifies,
#   element by element: |o - o*| within the per-element bound of
#   p8_reference_and_bound (median about 2^-8 of the output's RMS; derived
#   from fp32 scores and sums, the exp2 error, the online reference and the
#   bf16 output).
# * Against the same variant
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
# Relative error allowed in an implementation's 2^y before E4M3 rounding (fp32
# scores from the tensor core, the fp32 product with the scale, ex2.approx):
# a weight whose exact value lies within this relative distance of a rounding
# midpoint may round either way (see p8_reference_and_bound).
P8_FLIP_DELTA = 2.0 ** -14


def p8_reference_and_bound(q8, k8, v8, scales, cu, D, sm_scale, rows, delta=P8_FLIP_DELTA):
    """The reading-12 model o* = sum P* v / sum P* (fp64) on the given rows, and
    a per-element bound on how far an implementation of the same reading may
    deviate from it.  Returns (o*, bound), both [len(rows), H, D] in the order
    of the sorted rows.

    An implementation differs from the model in four ways, each bounded here:

    * Rounding flips.  It computes 2^y with a small relative error (fp32
      scores and scale products, a hardware exp2), so a weight z = 2^y whose
      exact value lies within relative ``delta`` of a midpoint between two E4M3
      values may round to the other neighbour: |dP| <= ulp(z).
    * Online reference.  Its power-of-two reference may lag the row maximum
      (weights scaled up by 2^k, O and l rescaled exactly), which changes
      nothing in E4M3's normal range but may round a weight below 2^-6 (the
      subnormal range) differently: |dP| <= 2^-9 there.
    * With perturbations dP_k of total U = sum |dP_k|, o' - o* =
      sum dP_k (v_k - o*) / (l* + sum dP_k), so
      |o' - o*| <= sum |dP_k| (|v_k| + |o*|) / (l* - U).
    * fp32 accumulation of O and l over L keys (relative error at most
      L 2^-24 of the sums of magnitudes each), and the final product and
      bf16 rounding (2^-8 |o*| covers the half-ulp 2^-9 and the fp32 steps).
    """
    T, H = q8.shape[0], q8.shape[1]
    rows = np.unique(np.asarray(rows, dtype=np.int64))
    o_all = np.full((rows.size, H, D), np.nan)
    b_all = np.full((rows.size, H, D), np.nan)
    ln2 = math.log(2.0)
    cu = [int(c) for c in cu]
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        sel = rows[(rows >= s) & (rows < e)]
        if sel.size == 0:
            continue
        pos = np.searchsorted(rows, sel)
        L = e - s
        for h in range(H):
            q = oattn.dequant(q8[sel, h, :D], scales[0])
            k = oattn.dequant(k8[s:e, h, :D], scales[1])
            v = oattn.dequant(v8[s:e, h, :D], scales[2])
            sc = (q @ k.T) * float(sm_scale)
            M = np.ceil(sc.max(axis=1, keepdims=True) / ln2)
            z = np.ldexp(np.exp(sc - M * ln2), oattn.P_SHIFT)
            P = e4m3.decode(e4m3.encode(z))
            l = P.sum(axis=1)
            o = (P @ v) / l[:, None]
            normal = z >= 2.0 ** -6
            _, Ex = np.frexp(np.where(normal, z, 1.0))
            ulp = np.ldexp(1.0, Ex - 1 - 3)
            t = np.where(normal, z, 1.0) / ulp
            dist = np.abs(t - np.floor(t) - 0.5) * ulp
            u = np.where(normal & (dist <= delta * z), ulp, 0.0) + np.where(normal, 0.0, 2.0 ** -9)
            U = u.sum(axis=1)
            absv = np.abs(v)
            dev = (u @ absv + U[:, None] * np.abs(o)) / np.maximum(l - U, 0.5 * l)[:, None]
            gamma = L * 2.0 ** -24
            acc = 2.0 * gamma * ((P @ absv) / l[:, None] + np.abs(o))
            o_all[pos, h, :] = o
            b_all[pos, h, :] = dev + acc + 2.0 ** -8 * np.abs(o) + 1e-30
    return o_all, b_all


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
    o8, bound = p8_reference_and_bound(q8n, k8n, v8n, scales, cu, D, sm_scale, rows)
    _, bound16 = p8_reference_and_bound(q8n, k8n, v8n, scales, cu, D, sm_scale, rows, 2.0 ** -16)
    ratio = np.abs(got - o8) / bound
    return dict(max_abs=max_abs, max_norm=max_norm, rel_rms=rel_rms, p8=p8, ref_rel=ref_rel,
                p8_bound_ratio=float(ratio.max()),
                p8_bound_ratio_d16=float((np.abs(got - o8) / bound16).max()),
                p8_max_abs=float(np.abs(got - o8).max()),
                p8_bound_median_rel=float(np.median(bound) / np.sqrt(np.mean(o8 ** 2))))


def assert_attention_ok(stats, tag="", outliers=False, literal=False):
    msg = ("%s max_abs=%.3e max_norm=%.3e rel_rms=%.3e p8_rel_rms=%.3e (err/|o| %.3e) "
           "vs p8 model: max_abs=%.3e, max |err|/bound=%.3f (%.3f with delta 2^-16; "
           "median bound / RMS(o) %.2e)"
           % (tag, stats["max_abs"], stats["max_norm"], stats["rel_rms"], stats["p8"], stats["ref_rel"],
              stats["p8_max_abs"], stats["p8_bound_ratio"], stats["p8_bound_ratio_d16"],
              stats["p8_bound_median_rel"]))
    print(msg)
    # Element by element against the reading-12 model: within the deviation
    # that model admits (flips of weights next to an E4M3 midpoint,
    # subnormal-range weights under a lagging reference, fp32 sums, bf16).
    assert stats["p8_bound_ratio"] <= 1.0, msg
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
