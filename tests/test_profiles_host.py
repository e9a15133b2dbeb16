"""CPU: every committed ncu summary under profiles/ describes the kernel sources
as they stand.  Each summary names the files its kernel is built from and a
prefix of the SHA-256 over them; bench.py reports the summary's DRAM traffic
only while that hash matches, so a kernel edited after its capture would
silently lose its `traffic` figure."""

import hashlib
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp8_vision_encoder_gb300", "csrc")
PROFILES = os.path.join(ROOT, "profiles")


def _summaries():
    out = []
    for name in sorted(os.listdir(PROFILES)):
        text = open(os.path.join(PROFILES, name)).read()
        m = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)\s*\(([^)]*)\)", text)
        if m:
            files = re.findall(r"[\w.]+\.(?:cuh|cu)\b", m.group(2))
            out.append((name, m.group(1), files, text))
    return out


def test_summaries_exist():
    names = [s[0] for s in _summaries()]
    for want in ("attn_fp8_qhd3.md", "attn_bf16_qhd3.md", "quant_qhd3.md", "amax_qhd3.md"):
        assert want in names


@pytest.mark.parametrize("summary", _summaries(), ids=lambda s: s[0])
def test_summary_hash_matches_sources(summary):
    name, sha, files, text = summary
    assert files, name
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    assert h.hexdigest().startswith(sha), "%s was captured from other sources" % name
    assert re.search(r"dram_bytes_per_launch:\s*\d+", text), name
    assert "--clock-control none" in text, name
