"""Calibrate-once workflow and the scale-file format (host logic, plain Python).

Sources:

* "FP8 ViT Encoder Attention", Calibrate-Once, Reuse Workflow: calibration
  runs dynamic scaling for 16 passes and then dumps the learned scales; saved
  scales are multiplied by a save margin whose default is 1.5.
* Same page, Scale File Format: one entry per attention layer keyed
  "visual.blocks.N.attn.attn" holding {"q": .., "k": .., "v": ..}; the keys
  q_scale / k_scale / v_scale are accepted as aliases.
* "FP8 vision encoder attention" (Sonar), Create static scales: the file is
  written after 16 forward passes.

Readings: the "learned scale" of a tensor is the ring maximum A_t after the
16 calibration forwards (the amax-like magnitude that static mode takes back
in); the margin is applied as one float32 multiply.
"""

import numpy as np

DEFAULT_MARGIN = 1.5
CALIB_PASSES = 16
ALIASES = {"q": ("q", "q_scale"), "k": ("k", "k_scale"), "v": ("v", "v_scale")}


def layer_key(n):
    return "visual.blocks.%d.attn.attn" % n


def saved_values(amax_ref, margin=DEFAULT_MARGIN):
    """float32(A_t) * float32(margin) for t in q, k, v."""
    a = np.asarray(amax_ref, dtype=np.float32)
    return [float(np.float32(x) * np.float32(margin)) for x in a]


def to_file_dict(per_layer_amax, margin=DEFAULT_MARGIN):
    """{layer_key(n): {"q":.., "k":.., "v":..}} for a list of per-layer (A_q, A_k, A_v)."""
    out = {}
    for n, a in enumerate(per_layer_amax):
        q, k, v = saved_values(a, margin)
        out[layer_key(n)] = {"q": q, "k": k, "v": v}
    return out


def parse_file_dict(d):
    """{layer index: (q, k, v)} from a scale-file dict, accepting the aliases."""
    out = {}
    for key, entry in d.items():
        parts = key.split(".")
        if len(parts) != 5 or parts[0] != "visual" or parts[1] != "blocks" or parts[3:] != ["attn", "attn"]:
            raise ValueError("unexpected scale-file key %r" % key)
        n = int(parts[2])
        vals = []
        for t in ("q", "k", "v"):
            found = [entry[a] for a in ALIASES[t] if a in entry]
            if len(found) != 1:
                raise ValueError("layer %r: need exactly one of %r" % (key, ALIASES[t]))
            vals.append(float(found[0]))
        out[n] = tuple(vals)
    return out
