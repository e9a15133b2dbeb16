"""CPU oracle for the FP8 ViT-encoder attention path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously-correct
restatement of what the hot path computes.  It is imported only by ``tests/``,
by ``__graft_entry__.smoke()`` and by the CPU-baseline legs of ``bench.py``.
The product (the CUDA library and its Python binding) never imports, calls or
links anything here, and nothing here imports the product.

Sources followed (page title, section):

* "FP8 ViT Encoder Attention" (vLLM docs) -- intro (Q/K/V quantized on the fly
  to FP8 before the attention call), note (quantization launches plus
  un-padding), Usage (dynamic scaling from a 16-entry circular buffer of
  observed Q/K/V amax values), Calibrate-Once workflow and Scale File Format
  (static per-layer q/k/v values, save margin 1.5).
* "FP8 vision encoder attention" (Sonar) -- Requirements (packed
  variable-length image batches, per-tensor FP8), Enable FP8 attention.
* OCP 8-bit Floating Point Specification (OFP8), E4M3 encoding -- the pages
  only say "FP8"; E4M3 with maximum 448 is the reading this oracle takes.

Modules:

* ``e4m3``      -- bit-exact E4M3 encode (round-to-nearest-even, saturating)
                   and decode.
* ``scales``    -- per-tensor amax, 16-entry amax ring, static scales.
* ``quant``     -- quantize + un-pad into the packed [T, H, D_pad] code layout.
* ``attention`` -- fp64 variable-length non-causal attention on dequantized
                   codes, plus the variant that rounds P to E4M3 precision.
* ``calib``     -- calibrate-once workflow and the scale-file JSON format.
"""

from . import e4m3, scales, quant, attention, calib  # noqa: F401
