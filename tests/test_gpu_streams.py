"""GPU: two layers' forwards on two CUDA streams at once.

Every call is stream-ordered and keeps its state in caller-owned device memory
(scale state, workspace), so two layers driven on two streams without any
ordering between them must give exactly what they give one after the other on
one stream: outputs and scale states bit for bit.  One layer runs dynamic
scaling (amax, ring, quantize, attention), the other static scales, with
different shapes and head dims.
"""

import pytest
import torch

from gpu_util import cu_tensor, qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vf():
    import fp8_vision_encoder_gb300 as vf
    assert torch.cuda.is_available()
    return vf


LAYERS = (
    # seqlens, H, D, dynamic, first input seed
    ([700, 1500, 33], 4, 128, True, 500),
    ([2048, 129], 8, 80, False, 600),
)
FORWARDS = 6


def _prepare(vf, layer):
    seqlens, H, D, dynamic, seed0 = layer
    cu, _ = cu_tensor(seqlens)
    T = sum(seqlens)
    inputs = [qkv(seqlens, H, D, seed0 + f, outliers=(f % 2 == 0)) for f in range(FORWARDS)]
    codes = vf.alloc_codes(T, H, vf.default_d_pad(D))
    outs = [torch.empty((T, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(FORWARDS)]
    return dict(seqlens=seqlens, H=H, D=D, dynamic=dynamic, cu=cu, inputs=inputs, codes=codes,
                outs=outs, ws=vf.Workspace(len(seqlens)))


def _new_state(vf, L, stream, st=None):
    st = (st or vf.ScaleState()).init(stream=stream)
    if not L["dynamic"]:
        st.set_static(96.0, 120.0, 80.0, stream=stream)
    return st


def _forward(vf, L, st, f, stream):
    q, k, v = L["inputs"][f]
    if L["dynamic"]:
        vf.amax_update(st, q, k, v, L["cu"], stream=stream)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, L["cu"], out=L["codes"], stream=stream)
    vf.attn_varlen(q8, k8, v8t, st, L["cu"], max(L["seqlens"]), L["D"], out=L["outs"][f],
                   workspace=L["ws"], stream=stream)


def test_two_layers_on_two_streams_equal_one_stream(vf):
    layers = [_prepare(vf, layer) for layer in LAYERS]
    torch.cuda.synchronize()

    # One stream, one layer after the other.
    ref_states, ref_outs = [], []
    for L in layers:
        st = _new_state(vf, L, None)
        for f in range(FORWARDS):
            _forward(vf, L, st, f, None)
        torch.cuda.synchronize()
        ref_states.append(st.read())
        ref_outs.append([o.clone() for o in L["outs"]])
        assert st.device_error() == 0 and L["ws"].error() == 0
    for L in layers:
        for o in L["outs"]:
            o.zero_()
    torch.cuda.synchronize()

    # Two streams, forwards interleaved on the host, no ordering between them.
    # (The state buffers are zero-filled on the current stream before the two
    # streams wait for it.)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    blank = [vf.ScaleState() for _ in layers]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    states = [_new_state(vf, L, s, b) for L, s, b in zip(layers, streams, blank)]
    for f in range(FORWARDS):
        for L, st, s in zip(layers, states, streams):
            _forward(vf, L, st, f, s)
    torch.cuda.synchronize()

    for L, st, rs, ro in zip(layers, states, ref_states, ref_outs):
        assert st.read() == rs
        for f in range(FORWARDS):
            assert torch.equal(L["outs"][f], ro[f]), "forward %d differs" % f
        assert st.device_error() == 0 and L["ws"].error() == 0
