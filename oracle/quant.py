"""Quantize + un-pad: source rows -> packed [T, H, D_pad] E4M3 codes.

Sources:

* "FP8 ViT Encoder Attention", intro: Q/K/V are quantized on the fly to FP8
  before the attention call; note: the quantization launches come together
  with "un-padding".
* "FP8 vision encoder attention" (Sonar), Requirements: packed
  variable-length image batches.

Readings taken where the pages are silent:

* What un-padding removes.  The source is either a padded batch (segment b's
  token i at row b * s_max + i; rows i >= L_b are ignored) or packed rows
  (segment b's token i at row cu_seqlens[b] + i).  Element (row, h, d) sits
  at row * token_stride + h * head_stride + d.  The output is always the packed
  token order [T, H, D_pad] with T = cu_seqlens[-1]; head-dim entries
  D..D_pad-1 are written as code 0x00.  Padded rows never enter the amax.
* Quantize operation: y = float32(x) * inv (one IEEE float32 multiply, round
  to nearest even), then E4M3 encode of y (round to nearest even, saturating).
"""

import numpy as np

from . import e4m3


class SrcLayout:
    """Where the valid source rows live (mirrors ``vitfp8_src_layout``)."""

    def __init__(self, padded, s_max, token_stride, head_stride):
        self.padded = int(padded)
        self.s_max = int(s_max)
        self.token_stride = int(token_stride)
        self.head_stride = int(head_stride)

    @staticmethod
    def packed(H, D):
        return SrcLayout(0, 0, H * D, D)

    @staticmethod
    def padded_batch(s_max, H, D):
        return SrcLayout(1, s_max, H * D, D)


def source_rows(layout, cu_seqlens):
    """Source row index of every packed token t in [0, T)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    rows = []
    for b in range(len(cu) - 1):
        L = int(cu[b + 1] - cu[b])
        i = np.arange(L, dtype=np.int64)
        if layout.padded:
            rows.append(b * layout.s_max + i)
        else:
            rows.append(cu[b] + i)
    if not rows:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate(rows)


def gather_valid(src_flat, layout, cu_seqlens, H, D):
    """Packed [T, H, D] float32 view of the valid source elements."""
    src = np.asarray(src_flat, dtype=np.float32).ravel()
    rows = source_rows(layout, cu_seqlens)
    idx = (rows[:, None, None] * layout.token_stride
           + np.arange(H, dtype=np.int64)[None, :, None] * layout.head_stride
           + np.arange(D, dtype=np.int64)[None, None, :])
    return src[idx]


def quantize(x, inv):
    """E4M3 codes of float32(x) * float32(inv), same shape as x."""
    y = np.asarray(x, dtype=np.float32) * np.float32(inv)  # IEEE float32 RN multiply
    return e4m3.encode(y)


def quantize_unpad(src_flat, layout, cu_seqlens, H, D, D_pad, inv):
    """Packed [T, H, D_pad] uint8 codes; entries d >= D are 0x00."""
    x = gather_valid(src_flat, layout, cu_seqlens, H, D)
    codes = quantize(x, inv)
    out = np.zeros((x.shape[0], H, D_pad), dtype=np.uint8)
    out[:, :, :D] = codes
    return out
