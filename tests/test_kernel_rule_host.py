"""CPU: the rule that picks the FP8 attention kernel (vitfp8_attn_kernel_for,
a host-only function of the library).

The rule is restated here from its statement in the header, with its
constants read from the sources; the library's answers are compared with the
restatement over a grid of sizes, and pinned on the pages' workloads on a
152-SM GB300.
"""

import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp8_vision_encoder_gb300", "csrc")


def _const(name):
    text = open(os.path.join(CSRC, "internal.cuh")).read()
    m = re.search(r"constexpr\s+(?:int|double)\s+%s\s*=\s*([0-9.]+);" % name, text)
    assert m, name
    return float(m.group(1))


LONG_SEQLEN = _const("kTwoTileLongSeqlen")
MIN_WAVES = _const("kTwoTileMinWaves")
MAX_TAIL = _const("kTwoTileMaxTail")
PERSISTENT_MAX = _const("kPersistentMaxSeqlen")


def expected_kernel(nseq, max_seqlen, T, H, nsm):
    if nsm <= 0 or nseq <= 0 or T <= 0 or H <= 0:
        return "unit"
    w = H * (T + 128.0 * nseq) / 256.0 / nsm
    if w >= MIN_WAVES and (max_seqlen < LONG_SEQLEN or math.ceil(w) <= w * (1.0 + MAX_TAIL)):
        return "two_tile_persistent" if max_seqlen <= PERSISTENT_MAX else "two_tile"
    items = (-(-T // 128) + nseq) * H
    if max_seqlen <= PERSISTENT_MAX and items > nsm:
        return "persistent"
    return "unit"


@pytest.fixture(scope="module")
def vf():
    import fp8_vision_encoder_gb300 as vf
    return vf


def test_constants():
    assert (LONG_SEQLEN, MIN_WAVES, MAX_TAIL, PERSISTENT_MAX) == (2048, 2.0, 0.12, 6144)


def test_pages_workloads_on_152_sms(vf):
    import workloads
    want = {"tiny": "unit", "micro8k": "unit", "hd3": "two_tile_persistent", "qhd3": "two_tile",
            "uhd3mix": "two_tile"}
    for name, k in want.items():
        w = workloads.WORKLOADS[name]
        assert vf.attn_kernel_for(len(w.seqlens), w.max_seqlen, w.T, w.H, 152) == k, name
    # many short segments: the persistent two-tile kernel
    assert vf.attn_kernel_for(8, 1024, 8192, 16, 152) == "two_tile_persistent"
    assert vf.attn_kernel_for(200, 256, 51200, 4, 152) == "two_tile_persistent"
    # short segments but under two waves of 256-query units: the one-tile kernels
    assert vf.attn_kernel_for(8, 1024, 8192, 2, 152) == "unit"
    assert vf.attn_kernel_for(8, 1024, 8192, 5, 152) == "persistent"
    # a last wave a third full: one CTA per item (8192 tokens, 16 heads: 3.4 waves of units)
    assert vf.attn_kernel_for(1, 8192, 8192, 16, 152) == "unit"
    # degenerate sizes
    assert vf.attn_kernel_for(0, 0, 0, 16, 152) == "unit"
    assert vf.attn_kernel_for(3, 14400, 43200, 16, 0) == "unit"


def test_library_matches_the_restated_rule(vf):
    n = 0
    for nsm in (100, 132, 148, 152, 160):
        for H in (1, 2, 4, 12, 16, 32):
            for L in (100, 1024, 2047, 2048, 3600, 6144, 6145, 8192, 14400, 32400):
                for nseq in (1, 2, 3, 7, 40):
                    T = L * nseq - (L // 3 if nseq > 1 else 0)
                    assert vf.attn_kernel_for(nseq, L, T, H, nsm) == expected_kernel(nseq, L, T, H, nsm), \
                        (nseq, L, T, H, nsm)
                    n += 1
    assert n == 5 * 6 * 10 * 5
