"""Host-side argument checks of the Python binding (CPU only): buffers the
library would otherwise address by raw pointer are rejected, before any
launch, when their dtype, shape, layout or device is wrong."""

import pytest
import torch


@pytest.fixture(scope="module")
def vf():
    import fp8_vision_encoder_gb300 as vf
    return vf


def test_code_buffers_checked(vf):
    T, H, Dp = 40, 2, 64
    q8 = torch.empty((T, H, Dp), dtype=torch.uint8)
    k8 = torch.empty((T, H, Dp), dtype=torch.uint8)
    v8t = torch.empty((H, Dp, vf.vt_stride(T)), dtype=torch.uint8)
    with pytest.raises(ValueError, match="k8"):
        vf._check_codes(q8, torch.empty((T, H, Dp + 16), dtype=torch.uint8), v8t)
    with pytest.raises(ValueError, match="v8t"):
        vf._check_codes(q8, k8, torch.empty((H, Dp, T), dtype=torch.uint8))   # Tv must be 48
    with pytest.raises(ValueError, match="v8t"):
        vf._check_codes(q8, k8, v8t.to(torch.int8))
    with pytest.raises(ValueError, match="on the GPU"):
        vf._check_codes(q8, k8, v8t)                                          # right shapes, CPU
    with pytest.raises(ValueError, match="contiguous"):
        vf._need(torch.empty((H, T, Dp), dtype=torch.uint8).transpose(0, 1), torch.uint8, (T, H, Dp), "q8")


def test_cu_seqlens_checked(vf):
    for bad in (torch.zeros(3, dtype=torch.int64), torch.zeros((2, 2), dtype=torch.int32),
                torch.zeros(0, dtype=torch.int32)):
        with pytest.raises(ValueError, match="cu_seqlens"):
            vf._cu_info(bad)
    with pytest.raises(ValueError, match="on the GPU"):
        vf._cu_info(torch.zeros(3, dtype=torch.int32))


def test_ring_push_values_checked(vf):
    st = object.__new__(vf.ScaleState)
    with pytest.raises(ValueError):
        vf.ring_push(st, torch.zeros(4, dtype=torch.float32))              # not on the GPU
    with pytest.raises(ValueError):
        vf.ring_push(st, torch.zeros(3, dtype=torch.float32))
