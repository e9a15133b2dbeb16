"""Python binding of libvitfp8 (FP8 ViT-encoder attention for GB300).

Argument marshalling only: every step of the path runs in the CUDA library
(``libvitfp8.so``, built by ``fp8_vision_encoder_gb300.build``).  PyTorch
provides device memory and streams.  There is no CPU fallback: importing this
package raises if the library has not been built.

Typical layer (dynamic scaling)::

    st = ScaleState(device)                  # one per attention layer
    st.init()
    amax_update(st, q, k, v, cu_seqlens)     # ring push + scales
    q8, k8, v8t = quantize_unpad(st, q, k, v, cu_seqlens)
    o = attn_varlen(q8, k8, v8t, st, cu_seqlens, max_seqlen, D)

Static scaling replaces ``init`` + ``amax_update`` with ``st.set_static(q, k, v)``.
"""

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# VITFP8_LIBRARY may name another build of the same library (the tests load
# the bounds-checked build, libvitfp8_checked.so, this way in a subprocess).
LIB_PATH = os.environ.get("VITFP8_LIBRARY") or os.path.join(_HERE, "libvitfp8.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libvitfp8.so is not built (expected at %s); build it with "
        "`python fp8_vision_encoder_gb300/build.py`" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

VITFP8_OK = 0
STATUS_NAMES = {
    0: "VITFP8_OK", 1: "VITFP8_ERR_INVALID_ARG", 2: "VITFP8_ERR_UNSUPPORTED",
    3: "VITFP8_ERR_CUDA", 4: "VITFP8_ERR_DEVICE_TIMEOUT", 5: "VITFP8_ERR_DEVICE_BOUNDS",
    6: "VITFP8_ERR_BAD_SEQLENS", 7: "VITFP8_ERR_WORKSPACE",
}
RING = 16
# FP8 attention kernels (vitfp8_attn_varlen_kernel); "auto" lets the library pick.
ATTN_KERNELS = {"auto": 0, "unit": 1, "persistent": 2, "two_tile": 3, "two_tile_persistent": 4}
E4M3_MAX = 448.0
MAX_HEAD_DIM = 128


class VitFp8Error(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = _lib.vitfp8_status_string(status).decode()
        super().__init__("%s: %s (%s)" % (where, STATUS_NAMES.get(status, status), msg))


class SrcLayout(ctypes.Structure):
    """Mirror of ``vitfp8_src_layout`` (where the valid source rows live)."""
    _fields_ = [("padded", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("s_max", ctypes.c_int64), ("token_stride", ctypes.c_int64),
                ("head_stride", ctypes.c_int64)]

    @staticmethod
    def packed(H, D, token_stride=None, head_stride=None):
        return SrcLayout(0, 0, 0, H * D if token_stride is None else token_stride,
                         D if head_stride is None else head_stride)

    @staticmethod
    def padded_batch(s_max, H, D):
        return SrcLayout(1, 0, s_max, H * D, D)


class _StateStruct(ctypes.Structure):
    """Mirror of ``vitfp8_scale_state`` (for reading a state back to the host)."""
    _fields_ = [("hist", (ctypes.c_float * RING) * 3), ("pos", ctypes.c_int32),
                ("count", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("dev_error", ctypes.c_int32), ("amax_ref", ctypes.c_float * 3),
                ("scale", ctypes.c_float * 3), ("inv_scale", ctypes.c_float * 3),
                ("amax_cur", ctypes.c_float * 3), ("amax_bits", ctypes.c_uint32 * 3),
                ("blocks_done", ctypes.c_uint32)]


STATE_BYTES = ctypes.sizeof(_StateStruct)

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_f32 = ctypes.c_float


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


_lib.vitfp8_status_string.restype = ctypes.c_char_p
_lib.vitfp8_status_string.argtypes = [ctypes.c_int]
_version = _sig("vitfp8_version", _i32, [])
_state_init = _sig("vitfp8_scale_state_init", ctypes.c_int, [_vp, _vp])
_set_static = _sig("vitfp8_set_static_scales", ctypes.c_int, [_vp, _f32, _f32, _f32, _vp])
_amax_update = _sig("vitfp8_amax_update", ctypes.c_int,
                    [_vp, _vp, _vp, _vp, ctypes.POINTER(SrcLayout), _vp, _i32, _i32, _i32, _i32, _vp])
_set_ring_order = _sig("vitfp8_set_ring_order", ctypes.c_int, [_vp, _i32, _vp])
_amax_local = _sig("vitfp8_amax_local", ctypes.c_int,
                   [_vp, _vp, _vp, _vp, ctypes.POINTER(SrcLayout), _vp, _i32, _i32, _i32, _i32, _vp,
                    _vp])
_ring_push = _sig("vitfp8_ring_push", ctypes.c_int, [_vp, _vp, _vp])
_quantize_unpad = _sig("vitfp8_quantize_unpad", ctypes.c_int,
                       [_vp, _vp, _vp, _vp, ctypes.POINTER(SrcLayout), _vp, _i32, _i32, _i32, _i32,
                        _i32, _vp, _vp, _vp, _vp])
_vt_stride = _sig("vitfp8_vt_stride", ctypes.c_int64, [_i32])
_ws_size = _sig("vitfp8_attn_workspace_size", ctypes.c_size_t, [_i32])
_attn = _sig("vitfp8_attn_varlen", ctypes.c_int,
             [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp,
              ctypes.c_size_t, _vp])
_attn_kernel = _sig("vitfp8_attn_varlen_kernel", ctypes.c_int,
                    [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp,
                     ctypes.c_size_t, _i32, _vp])
_attn_kernel_for = _sig("vitfp8_attn_kernel_for", _i32, [_i32, _i32, _i32, _i32, _i32])
_attn_noalloc = _sig("vitfp8_attn_varlen_noalloc", ctypes.c_int,
                     [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp])
_attn_bf16 = _sig("vitfp8_attn_varlen_bf16", ctypes.c_int,
                  [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, ctypes.c_size_t,
                   _vp])
NOALLOC_MAX_SEQS = 4096
_selftest_wait = _sig("vitfp8_selftest_bounded_wait", ctypes.c_int, [_vp, ctypes.c_size_t, _vp])
_calibrated = _sig("vitfp8_calibrated_scales", ctypes.c_int,
                   [_vp, ctypes.c_float, _vp, _vp, _vp])
_selftest_bounds = _sig("vitfp8_selftest_bounds_check", ctypes.c_int, [_vp, ctypes.c_size_t, _vp])
_checked_build = _sig("vitfp8_checked_build", ctypes.c_int32, [])
_get_err = _sig("vitfp8_get_device_error", ctypes.c_int, [_vp, ctypes.POINTER(_i32), _vp])
_get_ws_err = _sig("vitfp8_get_workspace_error", ctypes.c_int, [_vp, ctypes.POINTER(_i32), _vp])


def version():
    return _version()


def _check(status, where):
    if status != VITFP8_OK:
        raise VitFp8Error(status, where)


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def vt_stride(T):
    return int(_vt_stride(int(T)))


def workspace_size(num_seqs):
    return int(_ws_size(int(num_seqs)))


def _need_shape(t, dtype, shape, name):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or tuple(t.shape) != tuple(shape):
        raise ValueError("%s must be a %s tensor of shape %s" % (name, dtype, tuple(shape)))


def _need_placed(t, name):
    if not t.is_contiguous() or not t.is_cuda:
        raise ValueError("%s must be contiguous and on the GPU" % name)


def _need(t, dtype, shape, name):
    """Raise ValueError unless t is a contiguous CUDA tensor of this dtype and shape
    (the library sees raw pointers and cannot check buffer sizes itself)."""
    _need_shape(t, dtype, shape, name)
    _need_placed(t, name)


def _check_codes(q8, k8, v8t):
    """q8, k8: uint8 [T, H, D_pad]; v8t: uint8 [H, D_pad, vt_stride(T)]."""
    if not isinstance(q8, torch.Tensor) or q8.dim() != 3:
        raise ValueError("q8 must be a uint8 tensor [T, H, D_pad]")
    T, H, D_pad = q8.shape
    want = ((q8, (T, H, D_pad), "q8"), (k8, (T, H, D_pad), "k8"), (v8t, (H, D_pad, vt_stride(T)), "v8t"))
    for t, shape, name in want:
        _need_shape(t, torch.uint8, shape, name)
    for t, _, name in want:
        _need_placed(t, name)
    return T, H, D_pad


def _cu_info(cu_seqlens):
    if (not isinstance(cu_seqlens, torch.Tensor) or cu_seqlens.dtype != torch.int32
            or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1):
        raise ValueError("cu_seqlens must be a 1-D int32 tensor [num_seqs + 1]")
    if not cu_seqlens.is_contiguous() or not cu_seqlens.is_cuda:
        raise ValueError("cu_seqlens must be contiguous and on the GPU")
    return cu_seqlens.numel() - 1


class ScaleState:
    """One layer's device-resident FP8 scale state (``vitfp8_scale_state``)."""

    def __init__(self, device="cuda"):
        self.buf = torch.zeros(STATE_BYTES, dtype=torch.uint8, device=device)

    @property
    def ptr(self):
        return _ptr(self.buf)

    def init(self, stream=None):
        _check(_state_init(self.ptr, _stream(stream)), "vitfp8_scale_state_init")
        return self

    def set_static(self, q, k, v, stream=None):
        _check(_set_static(self.ptr, float(q), float(k), float(v), _stream(stream)),
               "vitfp8_set_static_scales")
        return self

    def set_ring_order(self, delayed, stream=None):
        """Dynamic mode: push-then-scale (delayed=False) or delayed scaling (True)."""
        _check(_set_ring_order(self.ptr, 1 if delayed else 0, _stream(stream)),
               "vitfp8_set_ring_order")
        return self

    def read(self):
        """Host snapshot of the state (synchronising copy) as a dict of lists."""
        raw = bytes(self.buf.cpu().numpy().tobytes())
        s = _StateStruct.from_buffer_copy(raw)
        return {
            "hist": [list(s.hist[t]) for t in range(3)], "pos": s.pos, "count": s.count,
            "mode": s.mode, "dev_error": s.dev_error, "amax_ref": list(s.amax_ref),
            "scale": list(s.scale), "inv_scale": list(s.inv_scale),
            "amax_cur": list(s.amax_cur), "amax_bits": list(s.amax_bits),
            "blocks_done": s.blocks_done,
        }

    def device_error(self, stream=None):
        out = _i32(0)
        _check(_get_err(self.ptr, ctypes.byref(out), _stream(stream)), "vitfp8_get_device_error")
        return out.value


def _layout_for(q, layout, H, D):
    if layout is not None:
        return layout
    if q.dim() != 3 or not q.is_contiguous():
        raise ValueError("pass a SrcLayout for non-contiguous or padded sources")
    return SrcLayout.packed(H, D)


def amax_update(state, q, k, v, cu_seqlens, total_tokens=None, layout=None, H=None, D=None,
                stream=None):
    """Dynamic scaling for one forward (no-op in static mode)."""
    nseq = _cu_info(cu_seqlens)
    H = q.shape[-2] if H is None else H
    D = q.shape[-1] if D is None else D
    T = q.shape[0] if total_tokens is None else total_tokens
    lay = _layout_for(q, layout, H, D)
    _check(_amax_update(state.ptr, _ptr(q), _ptr(k), _ptr(v), ctypes.byref(lay), _ptr(cu_seqlens),
                        nseq, int(T), int(H), int(D), _stream(stream)), "vitfp8_amax_update")


def amax_local(state, q, k, v, cu_seqlens, total_tokens=None, layout=None, H=None, D=None,
               out=None, stream=None):
    """Data-parallel step 1: this rank's (amax_q, amax_k, amax_v, any_tokens) as a
    float32[4] device tensor; the ring is not touched."""
    nseq = _cu_info(cu_seqlens)
    H = q.shape[-2] if H is None else H
    D = q.shape[-1] if D is None else D
    T = q.shape[0] if total_tokens is None else total_tokens
    lay = _layout_for(q, layout, H, D)
    if out is None:
        out = torch.empty(4, dtype=torch.float32, device=q.device)
    _need(out, torch.float32, (4,), "out")
    _check(_amax_local(state.ptr, _ptr(q), _ptr(k), _ptr(v), ctypes.byref(lay), _ptr(cu_seqlens),
                       nseq, int(T), int(H), int(D), _ptr(out), _stream(stream)),
           "vitfp8_amax_local")
    return out


def ring_push(state, vals, stream=None):
    """Data-parallel step 3: push reduced float32[4] values into the ring."""
    if vals.dtype != torch.float32 or vals.numel() != 4 or not vals.is_cuda:
        raise ValueError("vals must be a float32[4] CUDA tensor")
    _check(_ring_push(state.ptr, _ptr(vals), _stream(stream)), "vitfp8_ring_push")


def alloc_codes(T, H, D_pad, device="cuda"):
    q8 = torch.empty((T, H, D_pad), dtype=torch.uint8, device=device)
    k8 = torch.empty((T, H, D_pad), dtype=torch.uint8, device=device)
    v8t = torch.empty((H, D_pad, vt_stride(T)), dtype=torch.uint8, device=device)
    return q8, k8, v8t


def default_d_pad(D):
    return (D + 15) // 16 * 16


def quantize_unpad(state, q, k, v, cu_seqlens, total_tokens=None, D_pad=None, layout=None,
                   H=None, D=None, out=None, stream=None):
    """Quantize + un-pad q, k, v in one launch -> (q8, k8 [T,H,D_pad], v8t [H,D_pad,Tv])."""
    nseq = _cu_info(cu_seqlens)
    H = q.shape[-2] if H is None else H
    D = q.shape[-1] if D is None else D
    T = q.shape[0] if total_tokens is None else total_tokens
    D_pad = default_d_pad(D) if D_pad is None else D_pad
    lay = _layout_for(q, layout, H, D)
    if out is None:
        q8, k8, v8t = alloc_codes(T, H, D_pad, q.device)
    else:
        q8, k8, v8t = out
        if tuple(q8.shape) != (T, H, D_pad):
            raise ValueError("out[0] must have shape %s" % ((T, H, D_pad),))
        _check_codes(q8, k8, v8t)
    _check(_quantize_unpad(state.ptr, _ptr(q), _ptr(k), _ptr(v), ctypes.byref(lay),
                           _ptr(cu_seqlens), nseq, int(T), int(H), int(D), int(D_pad), _ptr(q8),
                           _ptr(k8), _ptr(v8t), _stream(stream)), "vitfp8_quantize_unpad")
    return q8, k8, v8t


class Workspace:
    """Device workspace for the attention work list (caller-owned)."""

    def __init__(self, num_seqs, device="cuda"):
        self.nbytes = workspace_size(num_seqs)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)

    def error(self, stream=None):
        out = _i32(0)
        _check(_get_ws_err(_ptr(self.buf), ctypes.byref(out), _stream(stream)),
               "vitfp8_get_workspace_error")
        return out.value


def calibrated_scales(dynamic_state, margin=1.5, static_state=None, stream=None):
    """Saved scale-file values float32(A) * float32(margin) of a calibrated
    dynamic state (A = its ring maximum per tensor), computed on the device;
    returns a device float32 tensor [3] (q, k, v).  With ``static_state`` that
    state is also set to static mode with those values."""
    out = torch.empty(3, dtype=torch.float32, device=dynamic_state.buf.device)
    _check(_calibrated(dynamic_state.ptr, float(margin), _ptr(out),
                       static_state.ptr if static_state is not None else None, _stream(stream)),
           "vitfp8_calibrated_scales")
    return out


def checked_build():
    """True when the loaded library is the bounds-checked build."""
    return bool(_checked_build())


def selftest_bounds_check(workspace, stream=None):
    """Run the bounds-check self-test (records VITFP8_ERR_DEVICE_BOUNDS in the
    workspace error word in the checked build, nothing in the normal one)."""
    _check(_selftest_bounds(_ptr(workspace.buf), workspace.nbytes, _stream(stream)),
           "vitfp8_selftest_bounds_check")


def selftest_bounded_wait(workspace, stream=None):
    """Run the kernels' bounded wait on a barrier nothing arrives on; afterwards
    workspace.error() reads VITFP8_ERR_DEVICE_TIMEOUT (the wait gave up)."""
    _check(_selftest_wait(_ptr(workspace.buf), workspace.nbytes, _stream(stream)),
           "vitfp8_selftest_bounded_wait")


def attn_kernel_for(num_seqs, max_seqlen, T, H, num_sms):
    """Name of the kernel attn_varlen runs for these sizes on a GPU with num_sms SMs."""
    k = _attn_kernel_for(int(num_seqs), int(max_seqlen), int(T), int(H), int(num_sms))
    return {v: n for n, v in ATTN_KERNELS.items()}[k]


def attn_varlen(q8, k8, v8t, state, cu_seqlens, max_seqlen, D, sm_scale=None, out=None,
                workspace=None, stream=None, kernel="auto"):
    """FP8 varlen attention -> bf16 [T, H, D].

    kernel: "auto" (the library's choice), "unit", "persistent", "two_tile" or
    "two_tile_persistent" (vitfp8_attn_varlen_kernel)."""
    nseq = _cu_info(cu_seqlens)
    T, H, D_pad = _check_codes(q8, k8, v8t)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=q8.device)
    _need(out, torch.bfloat16, (T, H, D), "out")
    if workspace is None:
        workspace = Workspace(nseq, q8.device)
    if kernel not in ATTN_KERNELS:
        raise ValueError("kernel must be one of %s" % sorted(ATTN_KERNELS))
    if kernel == "auto":
        _check(_attn(_ptr(q8), _ptr(k8), _ptr(v8t), state.ptr, _ptr(cu_seqlens), nseq, int(max_seqlen),
                     int(T), int(H), int(D), int(D_pad), float(sm_scale), _ptr(out),
                     _ptr(workspace.buf), workspace.nbytes, _stream(stream)), "vitfp8_attn_varlen")
    else:
        _check(_attn_kernel(_ptr(q8), _ptr(k8), _ptr(v8t), state.ptr, _ptr(cu_seqlens), nseq,
                            int(max_seqlen), int(T), int(H), int(D), int(D_pad), float(sm_scale),
                            _ptr(out), _ptr(workspace.buf), workspace.nbytes, ATTN_KERNELS[kernel],
                            _stream(stream)), "vitfp8_attn_varlen_kernel")
    return out


def attn_varlen_bf16(q, k, v, cu_seqlens, max_seqlen, sm_scale=None, out=None, workspace=None,
                     stream=None):
    """BF16 varlen attention on bf16 [T, H, D] q, k, v -> bf16 [T, H, D]."""
    nseq = _cu_info(cu_seqlens)
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.shape != q.shape:
            raise ValueError("q, k, v must be contiguous bf16 tensors of one shape [T, H, D]")
    T, H, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=q.device)
    _need(out, torch.bfloat16, (T, H, D), "out")
    if workspace is None:
        workspace = Workspace(nseq, q.device)
    _check(_attn_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), nseq, int(max_seqlen), int(T),
                      int(H), int(D), float(sm_scale), _ptr(out), _ptr(workspace.buf),
                      workspace.nbytes, _stream(stream)), "vitfp8_attn_varlen_bf16")
    return out


def attn_varlen_noalloc(q8, k8, v8t, state, cu_seqlens, max_seqlen, D, sm_scale=None, out=None,
                        stream=None):
    """FP8 varlen attention through the entry point that allocates nothing.

    For callers that cannot allocate device memory: the work list lives in a
    fixed device array inside the library (at most NOALLOC_MAX_SEQS segments).
    ``out`` should be passed pre-allocated by such callers.
    """
    nseq = _cu_info(cu_seqlens)
    T, H, D_pad = _check_codes(q8, k8, v8t)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=q8.device)
    _need(out, torch.bfloat16, (T, H, D), "out")
    _check(_attn_noalloc(_ptr(q8), _ptr(k8), _ptr(v8t), state.ptr, _ptr(cu_seqlens), nseq,
                         int(max_seqlen), int(T), int(H), int(D), int(D_pad), float(sm_scale),
                         _ptr(out), _stream(stream)), "vitfp8_attn_varlen_noalloc")
    return out
