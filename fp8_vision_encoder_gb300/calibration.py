"""Calibrate once, then run with static scales: the host side of the scale file.

"FP8 ViT Encoder Attention", Calibrate-Once, Reuse Workflow: run the encoder
with dynamic scaling for 16 forward passes, then save each attention layer's
learned per-tensor scales multiplied by a save margin (default 1.5) and load
them back as static scales in later runs.  Same page, Scale File Format: a
JSON object with one entry per attention layer, keyed
"visual.blocks.<N>.attn.attn", whose value holds "q", "k" and "v" (the names
"q_scale", "k_scale" and "v_scale" are accepted too).  "FP8 vision encoder
attention" (Sonar), Create static scales: the file is written after 16
forwards.

Reading used here: the learned scale of a tensor is its 16-entry ring maximum
A (the amax-like magnitude that static mode takes back, scale = A / 448), and
the saved value is the float32 product float32(A) * float32(margin).

The device work (amax, ring, static states) runs through the library's C ABI;
this module only reads ring maxima back and formats / parses the file.
"""

import json
import re

import numpy as np

from . import ScaleState, amax_update

CALIBRATION_PASSES = 16
SAVE_MARGIN = 1.5
TENSORS = ("q", "k", "v")
_KEY_RE = re.compile(r"^visual\.blocks\.(\d+)\.attn\.attn$")


def layer_name(n):
    """Scale-file key of attention layer ``n``."""
    return "visual.blocks.%d.attn.attn" % int(n)


def margin_scaled(amax, margin=SAVE_MARGIN):
    """float32(A) * float32(margin), one float32 multiply per tensor."""
    a = np.asarray(amax, dtype=np.float32).reshape(3)
    return tuple(float(x) for x in a * np.float32(margin))


def make_scale_file(per_layer_amax, margin=SAVE_MARGIN):
    """Scale-file dict for layers 0..n-1 from their (A_q, A_k, A_v) ring maxima."""
    doc = {}
    for n, amax in enumerate(per_layer_amax):
        doc[layer_name(n)] = dict(zip(TENSORS, margin_scaled(amax, margin)))
    return doc


def parse_scale_file(doc):
    """{layer index: (q, k, v)} from a scale-file dict.

    Each entry must give every tensor exactly once, under its short name or
    its "_scale" alias; any other key shape is an error (ValueError).
    """
    if not isinstance(doc, dict):
        raise ValueError("a scale file is a JSON object")
    layers = {}
    for key, entry in doc.items():
        m = _KEY_RE.match(key)
        if m is None:
            raise ValueError("not an attention-layer key: %r" % (key,))
        if not isinstance(entry, dict):
            raise ValueError("%s: entry must be an object" % key)
        vals = []
        for t in TENSORS:
            names = [n for n in (t, t + "_scale") if n in entry]
            if len(names) != 1:
                raise ValueError("%s: give exactly one of %r / %r" % (key, t, t + "_scale"))
            vals.append(float(entry[names[0]]))
        layers[int(m.group(1))] = tuple(vals)
    return layers


def save_scale_file(path, doc):
    with open(path, "w") as f:
        json.dump(doc, f, indent=2, sort_keys=True)


def load_scale_file(path):
    """Parse a scale file on disk -> {layer index: (q, k, v)}."""
    with open(path) as f:
        return parse_scale_file(json.load(f))


def static_states(layers, num_layers=None, device="cuda", stream=None):
    """One static ScaleState per layer 0..num_layers-1 from parsed file values.

    A layer missing from the file is an error: static mode has no fallback scale.
    """
    n = (max(layers) + 1 if layers else 0) if num_layers is None else num_layers
    missing = [layer_name(i) for i in range(n) if i not in layers]
    if missing:
        raise KeyError("scale file has no entry for %s" % ", ".join(missing))
    states = []
    for i in range(n):
        st = ScaleState(device).init(stream)
        st.set_static(*layers[i], stream=stream)
        states.append(st)
    return states


class Calibrator:
    """Dynamic-mode scale states for ``num_layers`` attention layers.

    Call ``observe(layer, q, k, v, cu_seqlens)`` once per layer and forward
    (it runs the amax + ring update on the device and returns the layer's
    state, ready for the forward's quantization); after the calibration
    forwards, ``scale_file()`` reads the ring maxima back and builds the file.
    """

    def __init__(self, num_layers, device="cuda", stream=None):
        self.states = [ScaleState(device).init(stream) for _ in range(num_layers)]
        self.passes = [0] * num_layers

    def observe(self, layer, q, k, v, cu_seqlens, **kwargs):
        st = self.states[layer]
        amax_update(st, q, k, v, cu_seqlens, **kwargs)
        self.passes[layer] += 1
        return st

    def ring_maxima(self):
        """Per layer (A_q, A_k, A_v): the ring maxima (synchronising reads)."""
        return [tuple(st.read()["amax_ref"]) for st in self.states]

    def scale_file(self, margin=SAVE_MARGIN, min_passes=CALIBRATION_PASSES):
        short = [i for i, p in enumerate(self.passes) if p < min_passes]
        if short:
            raise RuntimeError("layers %r saw fewer than %d calibration forwards" % (short, min_passes))
        return make_scale_file(self.ring_maxima(), margin)
