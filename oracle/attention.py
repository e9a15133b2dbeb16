"""Variable-length non-causal attention in float64 on dequantized E4M3 codes.

Sources:

* "FP8 ViT Encoder Attention", intro: Q/K/V are quantized to FP8 and then
  handed to the attention call; Performance: the attention kernel measured at
  head_dim 128, seq_len 8192.
* "FP8 vision encoder attention" (Sonar), Requirements: packed
  variable-length image batches with per-tensor FP8 scales.

Readings taken where the pages are silent:

* Segments are delimited by cu_seqlens (segment b holds packed tokens
  cu_seqlens[b] .. cu_seqlens[b+1]-1).  Attention is non-causal inside a
  segment and no token attends across a segment boundary (ViT encoder).
* Dequantisation: x_hat = decode(code) * scale_t, scale_t = A_t / 448.
* Scores use the true head dim D (D_pad columns are zeros and do not count):
  s_ij = sm_scale * sum_{d<D} q_hat_id k_hat_jd, sm_scale = 1/sqrt(D) unless
  given.
* Output o_i = sum_j p_ij v_hat_j with p = softmax_j(s) (max-subtracted).

``attention_varlen`` is that plain definition.  ``attention_varlen_p8`` adds
the one rounding step the FP8 hot path takes inside the softmax -- P is
requantized to E4M3 before the P.V product -- under this reading:

  p_ij  = exp(s_ij - M_i ln 2),  M_i = ceil(max_j s_ij / ln 2)  (p_ij <= 1),
  P'_ij = E4M3(2^8 p_ij)         (row maximum lands in (128, 256], below 448),
  o_i   = sum_j P'_ij v_hat_j / sum_j P'_ij,

i.e. the row sum adds the same rounded values, so the weights applied to V sum
to one.  The reference is a power of two, so within E4M3's normal range the
rounded significands do not depend on which power of two an online softmax
happens to use.
"""

import math

import numpy as np

from . import e4m3

P_SHIFT = 8  # P' = E4M3(2^8 p), p <= 1

_DECODE = None


def dequant(codes, scale):
    """float64 values of E4M3 codes times the float32 scale.

    Decoding goes through a 256-entry table of ``e4m3.decode`` (the same
    closed form, evaluated once per code).
    """
    global _DECODE
    if _DECODE is None:
        _DECODE = e4m3.decode(np.arange(256, dtype=np.uint8))
    return _DECODE[np.asarray(codes, dtype=np.uint8)] * np.float64(np.float32(scale))


def _segments(cu_seqlens):
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return [(int(cu[b]), int(cu[b + 1])) for b in range(len(cu) - 1)]


def _rows_by_segment(cu_seqlens, rows):
    """Map each requested packed row to its segment; None means all rows."""
    segs = _segments(cu_seqlens)
    if rows is None:
        return [(s, e, np.arange(s, e)) for s, e in segs]
    rows = np.asarray(rows, dtype=np.int64)
    out = []
    for s, e in segs:
        sel = rows[(rows >= s) & (rows < e)]
        if sel.size:
            out.append((s, e, sel))
    return out


def _attend(q, k, v, sm_scale, p_round):
    """One (segment, head) block: q [r, D], k [L, D], v [L, Dv] float64 -> [r, Dv]."""
    sc = (q @ k.T) * float(sm_scale)
    if p_round:
        # Power-of-two reference 2^M, M = ceil(rowmax / ln 2); P' = E4M3(2^8 p).
        M = np.ceil(sc.max(axis=1, keepdims=True) / math.log(2.0))
        p = np.exp(sc - M * math.log(2.0))
        pq = e4m3.decode(e4m3.encode(np.ldexp(p, P_SHIFT)))
        return (pq @ v) / pq.sum(axis=1, keepdims=True)
    m = sc.max(axis=1, keepdims=True)
    p = np.exp(sc - m)
    return (p @ v) / p.sum(axis=1, keepdims=True)


def attention_varlen(qh, kh, vh, cu_seqlens, sm_scale=None, rows=None, p_round=False):
    """o[T, H, Dv] float64 (rows not requested stay NaN when ``rows`` is given).

    qh, kh, vh: float64 [T, H, D] dequantized values (only the true D columns).
    """
    qh = np.asarray(qh, dtype=np.float64)
    kh = np.asarray(kh, dtype=np.float64)
    vh = np.asarray(vh, dtype=np.float64)
    T, H, D = qh.shape
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    out = np.full((T, H, vh.shape[2]), np.nan, dtype=np.float64)
    for s, e, sel in _rows_by_segment(cu_seqlens, rows):
        for h in range(H):
            out[sel, h, :] = _attend(qh[sel, h, :], kh[s:e, h, :], vh[s:e, h, :], sm_scale, p_round)
    return out


def attention_varlen_p8(qh, kh, vh, cu_seqlens, sm_scale=None, rows=None):
    """Same as ``attention_varlen`` with P rounded to E4M3 significand precision."""
    return attention_varlen(qh, kh, vh, cu_seqlens, sm_scale, rows, p_round=True)


def attention_fp8(q8, k8, v8, scales, cu_seqlens, D, sm_scale=None, rows=None, p_round=False):
    """Attention on packed [T, H, D_pad] E4M3 codes with per-tensor scales (q, k, v).

    Returns [T, H, D], or [len(rows), H, D] in the order of the sorted ``rows``
    when rows are given.  Dequantizes one (segment, head) slice at a time, so
    full-size workloads fit in host memory; the arithmetic is that of
    ``attention_varlen``.
    """
    T, H = q8.shape[0], q8.shape[1]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if rows is not None:
        rows = np.unique(np.asarray(rows, dtype=np.int64))
    n = T if rows is None else rows.size
    out = np.full((n, H, D), np.nan, dtype=np.float64)
    for s, e, sel in _rows_by_segment(cu_seqlens, rows):
        pos = sel if rows is None else np.searchsorted(rows, sel)
        for h in range(H):
            q = dequant(q8[sel, h, :D], scales[0])
            k = dequant(k8[s:e, h, :D], scales[1])
            v = dequant(v8[s:e, h, :D], scales[2])
            out[pos, h, :] = _attend(q, k, v, sm_scale, p_round)
    return out


def attention_bruteforce(qh, kh, vh, cu_seqlens, sm_scale=None):
    """Pure-Python loops, no BLAS: for tiny inputs only (an independent check)."""
    qh = np.asarray(qh, dtype=np.float64)
    kh = np.asarray(kh, dtype=np.float64)
    vh = np.asarray(vh, dtype=np.float64)
    T, H, D = qh.shape
    Dv = vh.shape[2]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    out = np.zeros((T, H, Dv))
    for s, e in _segments(cu_seqlens):
        for h in range(H):
            for i in range(s, e):
                scores = []
                for j in range(s, e):
                    acc = 0.0
                    for d in range(D):
                        acc += float(qh[i, h, d]) * float(kh[j, h, d])
                    scores.append(acc * sm_scale)
                mx = max(scores)
                w = [math.exp(x - mx) for x in scores]
                tot = sum(w)
                for d in range(Dv):
                    acc = 0.0
                    for jj, j in enumerate(range(s, e)):
                        acc += w[jj] * float(vh[j, h, d])
                    out[i, h, d] = acc / tot
    return out
