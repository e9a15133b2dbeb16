"""Seeded synthetic workloads shaped like the pages' ViT-encoder attention.

This module holds only shapes, seeds and random-number draws.  It contains
none of the path's arithmetic (no amax, no scaling, no quantization, no
attention), so both the CPU oracle and the CUDA path consume its tensors.

Shapes follow the pages' measurements: "FP8 ViT Encoder Attention",
Performance (kernel at head_dim 128, seq_len 8192; encoder forward with
3 images per request at HD 720x1280, QHD 1440x2560 and 4K 2160x3840).  At
16-pixel patches those images are 45x80, 90x160 and 135x240 patches, i.e.
3600, 14400 and 32400 tokens.  The real images and datasets are not used:
these draws stand in for them.

Recipe (every draw comes from one ``torch.Generator`` per forward, seeded
with the forward's seed, tensors drawn in the order q, k, v):

* values ~ N(0, 1) in float32, then rounded to bf16 (round to nearest even);
* "per-head std": before each tensor's normals, sigma_h ~ U[0.5, 2] per
  head is drawn and the head's values are multiplied by it;
* "outliers": after each tensor's normals, round(0.001 * N) flat positions
  are drawn uniformly (with replacement; a position drawn twice is scaled
  once) and those entries are multiplied by 20 before the bf16 rounding.
"""

import torch

HD_TOKENS = 45 * 80        # 720x1280 at 16-px patches
QHD_TOKENS = 90 * 160      # 1440x2560
UHD_TOKENS = 135 * 240     # 2160x3840


class Workload:
    def __init__(self, name, seqlens, H, D, outliers, per_head_std, scaling,
                 seeds, static=None, calib_seeds=(), layer_seeds=(), desc=""):
        self.name = name
        self.seqlens = list(seqlens)
        self.H = H
        self.D = D
        self.outliers = outliers
        self.per_head_std = per_head_std
        self.scaling = scaling          # "dynamic" | "static" | "calibrated"
        self.seeds = list(seeds)        # forwards run through dynamic scaling
        self.static = static            # (q, k, v) file values for "static"
        self.calib_seeds = list(calib_seeds)
        self.layer_seeds = list(layer_seeds)
        self.desc = desc

    @property
    def T(self):
        return sum(self.seqlens)

    @property
    def cu_seqlens(self):
        cu = [0]
        for L in self.seqlens:
            cu.append(cu[-1] + L)
        return cu

    @property
    def max_seqlen(self):
        return max(self.seqlens) if self.seqlens else 0

    def flops(self, D=None):
        """Algorithmic attention flops 4 * sum(L^2) * H * D (true D)."""
        D = self.D if D is None else D
        return 4 * sum(L * L for L in self.seqlens) * self.H * D


WORKLOADS = {
    "tiny": Workload(
        "tiny", [64, 192], 2, 128, True, False, "dynamic", [0, 1, 2],
        desc="2 images (64, 192 tokens), 2 heads, d=128, outliers, 3 dynamic forwards"),
    "micro8k": Workload(
        "micro8k", [8192], 16, 128, True, False, "static", [0],
        static=(224.0, 198.0, 210.0),
        desc="1 x 8192 tokens, 16 heads, d=128, outliers, static scales 224/198/210"),
    "hd3": Workload(
        "hd3", [HD_TOKENS] * 3, 16, 80, False, True, "dynamic",
        [100 + f for f in range(20)],
        desc="3 x HD (3600 tokens), 16 heads, d=80, per-head std, 20 dynamic forwards"),
    "qhd3": Workload(
        "qhd3", [QHD_TOKENS] * 3, 16, 128, True, False, "calibrated", [],
        calib_seeds=[200 + f for f in range(16)],
        layer_seeds=[300 + l for l in range(24)],
        desc="3 x QHD (14400 tokens), 16 heads, d=128, outliers, 24 layers, static = 1.5 x calibrated"),
    "uhd3mix": Workload(
        "uhd3mix", [UHD_TOKENS] * 3 + [1024, HD_TOKENS, 8192], 16, 128, True, False,
        "dynamic", [400],
        desc="3 x 4K (32400 tokens) + 1024 + 3600 + 8192, 16 heads, d=128, outliers, dynamic"),
}


def make_qkv(seqlens, H, D, seed, outliers=True, per_head_std=False, device="cpu"):
    """Packed bf16 q, k, v of shape [T, H, D] for one forward."""
    T = sum(seqlens)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = []
    n = T * H * D
    for _ in range(3):
        sig = None
        if per_head_std:
            sig = 0.5 + 1.5 * torch.rand(H, generator=g, device=device)
        x = torch.randn(T, H, D, generator=g, device=device, dtype=torch.float32)
        if sig is not None:
            x *= sig.view(1, H, 1)
        if outliers and n > 0:
            k = int(round(0.001 * n))
            if k > 0:
                idx = torch.randint(0, n, (k,), generator=g, device=device)
                flat = x.view(-1)
                flat[idx] = flat[idx] * 20.0
        out.append(x.to(torch.bfloat16))
    return out


def workload_qkv(w, seed, device="cpu"):
    return make_qkv(w.seqlens, w.H, w.D, seed, w.outliers, w.per_head_std, device)


def to_padded(x, seqlens, s_max, fill=30000.0):
    """Padded-batch copy [B, s_max, H, D] of packed x; pad rows hold ``fill``.

    A large fill value makes any leak of padded rows into the amax or the
    codes visible.
    """
    B = len(seqlens)
    H, D = x.shape[1], x.shape[2]
    out = torch.full((B, s_max, H, D), fill, dtype=x.dtype, device=x.device)
    s = 0
    for b, L in enumerate(seqlens):
        out[b, :L] = x[s:s + L]
        s += L
    return out
