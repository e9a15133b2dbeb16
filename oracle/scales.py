"""Per-tensor amax, the 16-entry amax ring, and static scales (float32, exact).

Sources:

* "FP8 ViT Encoder Attention", Usage: with no scale file, dynamic scaling is
  used -- a 16-entry circular buffer of observed Q/K/V amax values drives
  per-forward scale updates.
* "FP8 vision encoder attention" (Sonar), Enable FP8 attention: the observed
  Q/K/V maximum values are recorded in a 16-entry circular buffer and the
  scales are updated during each forward pass.
* "FP8 ViT Encoder Attention", Scale File Format and Calibrate-Once workflow:
  static per-layer values q/k/v (e.g. 224, 198, 210), saved with a x1.5
  margin "to leave headroom against activation outliers".

Readings taken where the pages are silent:

* A scale value is an amax-like magnitude A: the dequantisation factor is
  A/448 and the quantisation multiplier is 448/A (only under this reading
  does multiplying by 1.5 leave headroom).
* Granularity is per tensor (one value each for q, k and v per layer per
  forward, over all valid tokens, heads and head-dim entries).
* Ring order is push-then-scale: the current forward's amax enters the ring
  before the scale is taken, so the current tensor never saturates.
* Empty slots hold 0.0.  If the ring maximum is 0 the scale and multiplier are
  both 1.0 (every code is then +-0 whatever the scale).
* Amax follows fmax semantics: NaN inputs are ignored, +inf propagates (scale
  becomes inf and the multiplier 0).
* scale = A / 448 and inv = 448 / A are each one IEEE float32 division.
"""

import numpy as np

RING = 16
F448 = np.float32(448.0)
TENSORS = ("q", "k", "v")


def amax(x):
    """max |x| over all elements, float32, NaN ignored (fmax semantics)."""
    a = np.abs(np.asarray(x, dtype=np.float32).ravel())
    a = a[~np.isnan(a)]
    if a.size == 0:
        return np.float32(0.0)
    return np.float32(a.max())


def scale_pair(A):
    """(scale, inv) = (A/448, 448/A) in float32, with the A == 0 rule."""
    A = np.float32(A)
    if A == 0:
        return np.float32(1.0), np.float32(1.0)
    with np.errstate(divide="ignore", over="ignore"):
        return np.float32(A / F448), np.float32(F448 / A)


class ScaleState:
    """Host model of one layer's scale state (mirrors the device struct)."""

    def __init__(self):
        self.hist = np.zeros((3, RING), dtype=np.float32)
        self.pos = 0
        self.count = 0
        self.mode = 0  # 0 dynamic (push, then scale), 1 static, 2 dynamic delayed
        self.amax_ref = np.zeros(3, dtype=np.float32)
        self.scale = np.ones(3, dtype=np.float32)
        self.inv_scale = np.ones(3, dtype=np.float32)
        self.amax_cur = np.zeros(3, dtype=np.float32)

    def _scale_from_ring(self):
        for t in range(3):
            A = np.float32(self.hist[t].max())
            self.amax_ref[t] = A
            self.scale[t], self.inv_scale[t] = scale_pair(A)

    def push(self, amaxes):
        """Dynamic mode, one forward.  Mode 0 follows the push-then-scale
        reading: the forward's amax enters the ring, then the scale is taken
        from the ring including it.  Mode 2 is delayed scaling: the scale is
        taken from the ring as the earlier forwards left it, then the
        forward's amax enters the ring.  Static mode ignores the call."""
        if self.mode == 1:
            return
        if self.mode == 2:
            self._scale_from_ring()
        for t in range(3):
            self.amax_cur[t] = np.float32(amaxes[t])
            self.hist[t, self.pos] = np.float32(amaxes[t])
        self.pos = (self.pos + 1) % RING
        self.count = min(self.count + 1, RING)
        if self.mode == 0:
            self._scale_from_ring()

    def set_ring_order(self, delayed):
        """Choose push-then-scale (False) or delayed scaling (True) for a
        dynamic state; a static state is left as it is."""
        if self.mode != 1:
            self.mode = 2 if delayed else 0

    def set_static(self, q, k, v):
        """Static mode: the file's per-layer values become A for q, k, v."""
        self.mode = 1
        for t, s in enumerate((q, k, v)):
            A = np.float32(s)
            self.amax_ref[t] = A
            self.scale[t], self.inv_scale[t] = scale_pair(A)
