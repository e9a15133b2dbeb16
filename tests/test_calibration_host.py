"""Host side of the calibrate-once workflow (CPU only).

The library's scale-file writer and reader are checked against the page's
example file (tests/golden), against the oracle's own file logic, and on the
error cases the format implies.
"""

import json
import os

import numpy as np
import pytest

from oracle import calib as ocalib

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scale_file_example.json")


@pytest.fixture(scope="module")
def cal():
    from fp8_vision_encoder_gb300 import calibration
    return calibration


def test_page_example_parses_to_its_values(cal):
    # "FP8 ViT Encoder Attention", Scale File Format: layer 0 q/k/v 224/198/210,
    # layer 1 218/195/207.
    layers = cal.load_scale_file(GOLDEN)
    assert layers == {0: (224.0, 198.0, 210.0), 1: (218.0, 195.0, 207.0)}
    with open(GOLDEN) as f:
        assert layers == ocalib.parse_file_dict(json.load(f))


def test_defaults_follow_the_pages(cal):
    assert cal.CALIBRATION_PASSES == 16
    assert cal.SAVE_MARGIN == 1.5
    assert cal.layer_name(23) == "visual.blocks.23.attn.attn"


def test_margin_is_one_float32_multiply(cal):
    rng = np.random.default_rng(3)
    for a in rng.uniform(1e-3, 3e4, (200, 3)).astype(np.float32):
        got = cal.margin_scaled(a)
        for t in range(3):
            want = np.float32(a[t]) * np.float32(1.5)
            assert np.float32(got[t]) == want
            # exact product a * 3/2 rounded once to float32
            assert np.float32(got[t]) == np.float32(float(a[t]) * 1.5)
    assert cal.margin_scaled([149.33333, 1.0, 2.0], margin=2.0)[1:] == (2.0, 4.0)


def test_writer_matches_oracle_file_dict(cal):
    rng = np.random.default_rng(11)
    per_layer = [tuple(rng.uniform(0.5, 500.0, 3).astype(np.float32)) for _ in range(24)]
    for margin in (1.5, 1.0, 1.25):
        assert cal.make_scale_file(per_layer, margin) == ocalib.to_file_dict(per_layer, margin)


def test_roundtrip_through_json(cal, tmp_path):
    rng = np.random.default_rng(7)
    per_layer = [tuple(rng.uniform(0.5, 500.0, 3).astype(np.float32)) for _ in range(5)]
    doc = cal.make_scale_file(per_layer)
    path = tmp_path / "scales.json"
    cal.save_scale_file(str(path), doc)
    layers = cal.load_scale_file(str(path))
    assert sorted(layers) == list(range(5))
    for n, a in enumerate(per_layer):
        assert layers[n] == cal.margin_scaled(a)


def test_aliases_accepted(cal):
    doc = {"visual.blocks.3.attn.attn": {"q_scale": 1.0, "k": 2.0, "v_scale": 3.0}}
    assert cal.parse_scale_file(doc) == {3: (1.0, 2.0, 3.0)}
    assert ocalib.parse_file_dict(doc) == {3: (1.0, 2.0, 3.0)}


@pytest.mark.parametrize("doc", [
    {"visual.blocks.0.attn.attn": {"q": 1.0, "q_scale": 1.0, "k": 2.0, "v": 3.0}},   # twice
    {"visual.blocks.0.attn.attn": {"q": 1.0, "k": 2.0}},                             # v missing
    {"visual.blocks.x.attn.attn": {"q": 1.0, "k": 2.0, "v": 3.0}},                   # not an index
    {"blocks.0.attn.attn": {"q": 1.0, "k": 2.0, "v": 3.0}},                          # wrong key
    {"visual.blocks.0.attn.qkv": {"q": 1.0, "k": 2.0, "v": 3.0}},                    # wrong module
])
def test_malformed_files_rejected(cal, doc):
    with pytest.raises(ValueError):
        cal.parse_scale_file(doc)
    with pytest.raises(ValueError):
        ocalib.parse_file_dict(doc)


def test_non_object_rejected(cal):
    with pytest.raises(ValueError):
        cal.parse_scale_file([1, 2, 3])
    with pytest.raises(ValueError):
        cal.parse_scale_file({"visual.blocks.0.attn.attn": [1, 2, 3]})


def test_static_states_requires_every_layer(cal):
    # Fails on the host before any device allocation.
    with pytest.raises(KeyError):
        cal.static_states({0: (1.0, 2.0, 3.0), 2: (1.0, 2.0, 3.0)})
