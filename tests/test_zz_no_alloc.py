"""GPU check of vitfp8_attn_varlen_noalloc, the attention entry point for
callers that cannot allocate device memory (a plugin handed only raw
pointers, a serving host with a pool fixed at start-up, a loop that cannot
afford cudaMalloc's possible device synchronisation).

It must produce what vitfp8_attn_varlen produces with a caller workspace.  Two
calls in a row with different segment structures also show that the shared
built-in scratch is rewritten by every call.  This file is collected last so
that a run stopping at the first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_util import TOL_MAX_ABS, cu_tensor

pytestmark = pytest.mark.gpu


def _inputs(vf, seqlens, H, D, seed):
    cu, _ = cu_tensor(seqlens)
    q, k, v = [t.cuda() for t in workloads.make_qkv(seqlens, H, D, seed, True, False)]
    st = vf.ScaleState().init()
    vf.amax_update(st, q, k, v, cu)
    q8, k8, v8t = vf.quantize_unpad(st, q, k, v, cu)
    return cu, st, q8, k8, v8t


def _call_noalloc(vf, q8, k8, v8t, st, cu, max_seqlen, D, out):
    """Direct C-ABI call (ctypes), no binding helper in between."""
    fn = vf._lib.vitfp8_attn_varlen_noalloc
    fn.restype = ctypes.c_int
    P = ctypes.c_void_p
    T, H, D_pad = q8.shape
    stream = torch.cuda.current_stream().cuda_stream
    return fn(P(q8.data_ptr()), P(k8.data_ptr()), P(v8t.data_ptr()), st.ptr,
              P(cu.data_ptr()), ctypes.c_int32(cu.numel() - 1), ctypes.c_int32(max_seqlen),
              ctypes.c_int32(T), ctypes.c_int32(H), ctypes.c_int32(D), ctypes.c_int32(D_pad),
              ctypes.c_float(1.0 / np.sqrt(D)), P(out.data_ptr()), P(stream))


def test_noalloc_matches_workspace_entry_point_twice():
    import fp8_vision_encoder_gb300 as vf
    assert torch.cuda.is_available()
    # the third case's items are all split over several CTAs (key-range split);
    # the fourth has more work items than SMs, so the persistent kernel runs it
    cases = [([300, 129, 500], 2, 128, 31), ([1, 64, 700, 17, 3600], 3, 80, 32), ([2048], 2, 128, 34),
             ([3600, 3600, 3600], 4, 80, 35)]
    for seqlens, H, D, seed in cases:
        cu, st, q8, k8, v8t = _inputs(vf, seqlens, H, D, seed)
        T = sum(seqlens)
        ref = vf.attn_varlen(q8, k8, v8t, st, cu, max(seqlens), D)
        out = torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        status = _call_noalloc(vf, q8, k8, v8t, st, cu, max(seqlens), D, out)
        torch.cuda.synchronize()
        assert status == 0, vf._lib.vitfp8_status_string(status)
        diff = (out.float() - ref.float()).abs().max().item()
        assert diff <= TOL_MAX_ABS, diff
        # same kernel, same inputs: the results are in fact bit-identical
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_noalloc_rejects_too_many_segments():
    import fp8_vision_encoder_gb300 as vf
    n = vf.NOALLOC_MAX_SEQS + 1
    seqlens = [1] * n
    cu, st, q8, k8, v8t = _inputs(vf, seqlens, 1, 64, 33)
    out = torch.zeros((n, 1, 64), dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(vf, q8, k8, v8t, st, cu, 1, 64, out) == 2   # VITFP8_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def test_noalloc_after_a_call_with_malformed_seqlens():
    """A call whose device-side check fails (non-monotonic cu_seqlens) leaves
    its output unwritten and puts "no work" into the shared scratch; the next
    valid call must still compute everything, bit-identical to the workspace
    entry point."""
    import fp8_vision_encoder_gb300 as vf
    seqlens, H, D = [300, 129, 500], 2, 128
    cu, st, q8, k8, v8t = _inputs(vf, seqlens, H, D, 34)
    T = sum(seqlens)
    bad = torch.tensor([0, 400, 300, T], dtype=torch.int32, device="cuda")  # 400 > 300
    out_bad = torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(vf, q8, k8, v8t, st, bad, max(seqlens), D, out_bad) == 0
    torch.cuda.synchronize()
    assert torch.isnan(out_bad.float()).all(), "the rejected call wrote output"

    ref = vf.attn_varlen(q8, k8, v8t, st, cu, max(seqlens), D)
    out = torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(vf, q8, k8, v8t, st, cu, max(seqlens), D, out) == 0
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
