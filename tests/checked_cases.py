"""Cases run against both builds of the library for the checked-build test.

Test infrastructure, imported by ``tests/test_gpu_checked.py``: in the test
process with the normal library, and in a subprocess with
``VITFP8_LIBRARY`` pointing at the bounds-checked build.  Every code and
output buffer is the middle of a larger allocation whose bands before and
after hold a canary pattern; each case reports its codes, outputs, the
device error words and whether the bands are intact.
"""

import numpy as np
import torch

import workloads

BAND = 4096          # canary bytes on each side of every code and output buffer
CANARY = 0xA5


def _guarded(nbytes):
    buf = torch.full((nbytes + 2 * BAND,), CANARY, dtype=torch.uint8, device="cuda")
    return buf, buf[BAND:BAND + nbytes]


def _bands_ok(buf):
    return bool((buf[:BAND] == CANARY).all().item() and (buf[-BAND:] == CANARY).all().item())


def _cu(seqlens):
    cu = [0]
    for L in seqlens:
        cu.append(cu[-1] + L)
    return torch.tensor(cu, dtype=torch.int32, device="cuda")


def _case(vf, name, seqlens, H, D, seed, dynamic=True, layout="packed", kernel="auto"):
    T = sum(seqlens)
    Dp = vf.default_d_pad(D)
    Tv = vf.vt_stride(T)
    cu = _cu(seqlens)
    q, k, v = [t.cuda() for t in workloads.make_qkv(seqlens, H, D, seed, True, False)]
    lay = None
    qs, ks, vs = q, k, v
    if layout == "padded":
        s_max = max(seqlens) + 3
        qs, ks, vs = [workloads.to_padded(x, seqlens, s_max).cuda() for x in (q, k, v)]
        lay = vf.SrcLayout.padded_batch(s_max, H, D)
    elif layout == "fused":
        fused = torch.stack([q, k, v], dim=1).contiguous()
        qs, ks, vs = fused[:, 0], fused[:, 1], fused[:, 2]
        lay = vf.SrcLayout.packed(H, D, token_stride=3 * H * D, head_stride=D)

    st = vf.ScaleState().init()
    if dynamic:
        for f in range(2):
            vf.amax_update(st, qs, ks, vs, cu, total_tokens=T, layout=lay, H=H, D=D)
    else:
        st.set_static(96.0, 120.0, 80.0)
    bq, q8 = _guarded(T * H * Dp)
    bk, k8 = _guarded(T * H * Dp)
    bv, v8t = _guarded(H * Dp * Tv)
    q8, k8, v8t = q8.view(T, H, Dp), k8.view(T, H, Dp), v8t.view(H, Dp, Tv)
    vf.quantize_unpad(st, qs, ks, vs, cu, total_tokens=T, D_pad=Dp, layout=lay, H=H, D=D,
                      out=(q8, k8, v8t))
    ws = vf.Workspace(len(seqlens))
    bo, o = _guarded(T * H * D * 2)
    o = o.view(torch.bfloat16).view(T, H, D)
    vf.attn_varlen(q8, k8, v8t, st, cu, max(seqlens), D, out=o, workspace=ws, kernel=kernel)
    ws16 = vf.Workspace(len(seqlens))
    bo16, o16 = _guarded(T * H * D * 2)
    o16 = o16.view(torch.bfloat16).view(T, H, D)
    vf.attn_varlen_bf16(q, k, v, cu, max(seqlens), out=o16, workspace=ws16)
    torch.cuda.synchronize()
    return {
        name + ".q8": q8.cpu().numpy(), name + ".k8": k8.cpu().numpy(), name + ".v8t": v8t.cpu().numpy(),
        name + ".o": o.view(torch.int16).cpu().numpy(), name + ".o16": o16.view(torch.int16).cpu().numpy(),
        name + ".errors": np.array([st.device_error(), ws.error(), ws16.error()], dtype=np.int32),
        name + ".bands": np.array([_bands_ok(b) for b in (bq, bk, bv, bo, bo16)], dtype=np.int32),
    }


def run_cases(vf):
    rng = np.random.default_rng(7)
    short = rng.integers(1, 40, size=3000).tolist()
    cases = [
        ("ragged", [1, 127, 128, 129, 300], 2, 128, 41, True, "packed"),
        ("tiny", [64, 192], 2, 128, 0, True, "packed"),
        ("short3000", short, 2, 64, 42, False, "packed"),
        ("padded", [5, 300, 77], 3, 80, 43, True, "padded"),
        ("fused", [257, 31], 4, 128, 44, True, "fused"),
        ("split", [2048, 600], 2, 128, 45, True, "packed"),   # every item's key range split
        ("long", [7000, 300], 1, 128, 46, True, "packed"),    # one CTA per work item (segments > 6144)
        ("psplit", [2048], 12, 128, 47, True, "packed"),      # persistent kernel, last wave split
        # two-tile kernel: one S buffer (d = 128), one per tile (d = 80, 40)
        ("tt128", [300, 1000, 129, 1], 2, 128, 48, True, "packed", "two_tile"),
        ("tt80", [600, 77, 256], 3, 80, 49, True, "padded", "two_tile"),
        ("tt40", [3, 130, 61, 700], 2, 40, 50, True, "packed", "two_tile"),
        ("ttp", [700, 1, 256, 300, 1500], 4, 128, 51, True, "packed", "two_tile_persistent"),
        ("ttp80", [511, 0, 257], 6, 80, 52, True, "packed", "two_tile_persistent"),
    ]
    for D in range(8, 129, 8):
        cases.append(("d%d" % D, [3, 130, 61], 2, D, 100 + D, D % 16 == 0, "packed"))
    out = {}
    for c in cases:
        out.update(_case(vf, *c))
    ws = vf.Workspace(0)
    vf.selftest_bounds_check(ws)
    out["selftest_bounds"] = np.array([ws.error()], dtype=np.int32)
    out["checked_build"] = np.array([int(vf.checked_build())], dtype=np.int32)
    return out


if __name__ == "__main__":
    import sys
    import fp8_vision_encoder_gb300 as vf
    np.savez(sys.argv[1], **run_cases(vf))
