"""CPU: the key-range split rule the GPU tests check the plan against.

The rule's constants are read from the kernel sources, so the restatement in
``split_rule.py`` cannot drift from them; the examples fix its behaviour on
fixed SM counts; the workspace size covers the split's partial results.
"""

import os
import re

from split_rule import BN, MAX_K, MAX_PARTS, ROWS, expected_split

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp8_vision_encoder_gb300", "csrc")


def _const(path, name):
    text = open(os.path.join(CSRC, path)).read()
    m = re.search(r"constexpr\s+(?:int|size_t)\s+%s\s*=\s*([0-9 *]+);" % name, text)
    assert m, name
    return eval(m.group(1))


def test_constants_match_the_sources():
    assert _const("internal.cuh", "kSplitMaxK") == MAX_K
    assert _const("internal.cuh", "kSplitMaxParts") == MAX_PARTS
    assert _const("attn_fp8.cu", "BN") == BN
    assert _const("attn_fp8.cu", "BM") == ROWS


def test_rule_examples():
    # a full last wave is not split
    assert expected_split([ROWS * 152], 1, 152) == (152, 152, 1)
    # 3 items left over, each segment tile count allows 3 parts
    assert expected_split([ROWS * 150, 600], 1, 152) == (155, 152, 3)
    # 32 items, all in the last wave: 4 parts (MAX_K)
    assert expected_split([2048], 2, 152) == (32, 0, 4)
    # one key tile per segment: nothing to split
    assert expected_split([64, 192], 2, 152) == (6, 6, 1)
    # a last wave more than half full is not split
    assert expected_split([ROWS * 100], 1, 152) == (100, 100, 1)
    # 3xHD: 1392 items, the last 24 in 4 parts
    assert expected_split([3600] * 3, 16, 152) == (1392, 1368, 4)
    # empty segments are skipped when the parts are counted
    assert expected_split([1500, 0, 900, 700, 513], 1, 152) == (31, 0, 3)
    # other SM counts
    assert expected_split([2048], 2, 148) == (32, 0, 4)
    assert expected_split([3600] * 3, 16, 132) == (1392, 1392, 1)   # 72 left: more than half of 132


def test_parts_never_exceed_the_slots():
    for n_sm in (100, 132, 148, 152, 160, 264):
        for L in (300, 1000, 2048, 3600, 8192):
            for H in (1, 2, 3, 16):
                N, sfirst, k = expected_split([L, L // 2 + 1], H, n_sm)
                if k > 1:
                    assert (N - sfirst) * k <= MAX_PARTS
                    assert 2 * (N - sfirst) <= n_sm


def test_workspace_covers_the_partial_results():
    import fp8_vision_encoder_gb300 as vf
    part_bytes = _const("internal.cuh", "kSplitPartBytes")
    assert vf.workspace_size(3) >= 64 + 16 * 3 + 1024 + MAX_PARTS * part_bytes
