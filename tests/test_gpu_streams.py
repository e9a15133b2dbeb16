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


def test_attention_from_two_host_threads(vf):
    """Two host threads, each driving FP8 and BF16 attention on its own stream
    with its own workspace, at the same time (the binding's ctypes calls
    release the GIL, so the library's host code runs concurrently, including
    its once-per-device set-up when these are the process's first attention
    calls): every output is bit-identical to the same call made alone."""
    import threading

    cases = [([900, 300], 4, 128, 701), ([1500, 64, 700], 2, 80, 702)]
    prepared = []
    for seqlens, H, D, seed in cases:
        cu, _ = cu_tensor(seqlens)
        q, k, v = qkv(seqlens, H, D, seed)
        st = vf.ScaleState().init()
        vf.amax_update(st, q, k, v, cu)
        q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
        prepared.append(dict(seqlens=seqlens, D=D, cu=cu, q=q, k=k, v=v, st=st,
                             q8=q8, k8=k8, v8t=v8t))
    torch.cuda.synchronize()

    results = [dict() for _ in prepared]
    errors = []
    streams = [torch.cuda.Stream() for _ in prepared]
    start = threading.Barrier(len(prepared))
    REPS = 12

    def run(i):
        P = prepared[i]
        try:
            torch.cuda.set_device(0)
            ws = vf.Workspace(len(P["seqlens"]))
            s = streams[i]
            fp8 = [torch.empty_like(P["q"]) for _ in range(REPS)]
            bf16 = [torch.empty_like(P["q"]) for _ in range(REPS)]
            start.wait()
            for r in range(REPS):
                vf.attn_varlen(P["q8"], P["k8"], P["v8t"], P["st"], P["cu"], max(P["seqlens"]),
                               P["D"], out=fp8[r], workspace=ws, stream=s)
                vf.attn_varlen_bf16(P["q"], P["k"], P["v"], P["cu"], max(P["seqlens"]),
                                    out=bf16[r], workspace=ws, stream=s)
            s.synchronize()
            results[i] = dict(fp8=fp8, bf16=bf16, err=ws.error(stream=s))
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(prepared))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    assert all(not t.is_alive() for t in threads)

    for P, R in zip(prepared, results):
        ref8 = vf.attn_varlen(P["q8"], P["k8"], P["v8t"], P["st"], P["cu"], max(P["seqlens"]), P["D"])
        ref16 = vf.attn_varlen_bf16(P["q"], P["k"], P["v"], P["cu"], max(P["seqlens"]))
        torch.cuda.synchronize()
        assert R["err"] == 0
        for r in range(REPS):
            assert torch.equal(R["fp8"][r].view(torch.int16), ref8.view(torch.int16)), "fp8 rep %d" % r
            assert torch.equal(R["bf16"][r].view(torch.int16), ref16.view(torch.int16)), "bf16 rep %d" % r
