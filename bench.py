"""Benchmark of the FP8 ViT-encoder attention hot path on GB300.

One step = one encoder forward of the workload: for every layer, quantize +
un-pad Q/K/V (one launch) and run FP8 variable-length attention (work-list
launch + attention launch).  Default workload: 3 QHD images packed
(3 x 14400 tokens), 16 heads, head_dim 128, 24 layers, static scales = 1.5 x
the amax calibrated over 16 dynamic forwards.  Metric: algorithmic attention
TFLOP/s (4 * sum L^2 * H * D per layer) including the quantization time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...    # the CPU oracle on a bounded sample

Prints ONE JSON line (rank 0).  Under torchrun every rank runs its own copy of
the workload on its own GPU (independent layers, no collective on the data
path); the reported value is all ranks' work over the slowest rank's time.
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "FP8 varlen ViT-attention TFLOPS incl. quant (3×QHD, d=128); % of FP8 peak"
FP8_PER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor-core ratio


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# Source files each profiled kernel is compiled from (the summaries under
# profiles/ record a hash over them).
ATTN_FP8_SOURCES = ["attn_fp8.cu", "attn_fp8_2tile.cu", "attn_common.cuh", "checked.cuh", "internal.cuh", "ptx.cuh"]
QUANT_SOURCES = ["quant.cu", "checked.cuh", "internal.cuh", "ptx.cuh"]


def _fp8_kernel(vf, seqlens, H, dev):
    """Name of the FP8 attention kernel the library picks for these segments."""
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    return vf.attn_kernel_for(len(seqlens), max(seqlens), sum(seqlens), H, nsm)


def _profile_traffic(md_name, sources):
    """DRAM bytes per launch from a committed ncu summary, if the kernel is unchanged."""
    import hashlib
    import re
    try:
        text = open(os.path.join(ROOT, "profiles", md_name)).read()
        m = hashlib.sha256()
        for src in sources:
            with open(os.path.join(ROOT, "fp8_vision_encoder_gb300", "csrc", src), "rb") as f:
                m.update(f.read())
        sha = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text).group(1)
        if sha != m.hexdigest()[:len(sha)]:
            return None
        return int(re.search(r"dram_bytes_per_launch:\s*(\d+)", text).group(1))
    except (OSError, AttributeError, ValueError):
        return None


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


L2_FLUSH_BYTES = 256 << 20   # twice the GB300's L2


def flush_l2(buf, value=1):
    """Evict the L2 outside a timed span: write a buffer twice its size, then
    read it all back, so that the lines left in the L2 are clean.  (After the
    write alone the L2 holds ~129 MB of dirty lines, and the next kernel pays
    for writing them back: ~15 us on the first kernel of a short span.)"""
    buf.fill_(value)
    buf.view(torch.int32).max()


def clocks_rejected(clocks):
    """True for a clock record the timing rules reject: hw_slowdown,
    hw_thermal_slowdown or sw_thermal_slowdown active, or the median SM clock
    under 80 % of the maximum with no reason active (a clock lock left behind).
    sw_power_cap alone is kept."""
    if not clocks:
        return False
    if {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"} & set(clocks["reasons"]):
        return True
    mx = clocks.get("sm_max_mhz") or 0.0
    return not clocks["reasons"] and mx > 0 and clocks["sm_mhz"] < 0.8 * mx


# ----------------------------------------------------------------------------- workload
class Runner:
    """Holds a workload's device buffers and runs one step through the C ABI."""

    def __init__(self, vf, w, device, layers=None):
        self.vf = vf
        self.w = w
        self.dev = device
        self.cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=device)
        self.D_pad = vf.default_d_pad(w.D)
        gen = lambda seed: workloads.make_qkv(w.seqlens, w.H, w.D, seed, w.outliers,
                                              w.per_head_std, device=device)
        if w.scaling == "calibrated":
            # Calibrate once: 16 dynamic forwards, then static = 1.5 x ring max.
            st = vf.ScaleState(device).init()
            for seed in w.calib_seeds:
                q, k, v = gen(seed)
                vf.amax_update(st, q, k, v, self.cu)
            A = st.read()["amax_ref"]
            self.static = [float(np.float32(a) * np.float32(1.5)) for a in A]
            seeds = w.layer_seeds if layers is None else w.layer_seeds[:layers]
            self.dynamic = False
        elif w.scaling == "static":
            self.static = list(w.static)
            seeds = w.seeds
            self.dynamic = False
        else:
            self.static = None
            seeds = w.seeds[-1:]
            self.dynamic = True
        self.inputs = [gen(s) for s in seeds]
        self.states = []
        for _ in self.inputs:
            st = vf.ScaleState(device)
            st.init()
            if self.static is not None:
                st.set_static(*self.static)
            self.states.append(st)
        self.codes = vf.alloc_codes(w.T, w.H, self.D_pad, device)
        self.out = torch.empty((w.T, w.H, w.D), dtype=torch.bfloat16, device=device)
        self.ws = vf.Workspace(len(w.seqlens), device)
        self.layers = len(self.inputs)
        self.flops_layer = w.flops()
        self.launches_layer = 3 + (1 if self.dynamic else 0)

    def layer(self, i, stream, ev=None):
        vf, w = self.vf, self.w
        q, k, v = self.inputs[i]
        st = self.states[i]
        if ev is not None:
            ev[0].record(stream)
        if self.dynamic:
            vf.amax_update(st, q, k, v, self.cu, stream=stream)
        vf.quantize_unpad(st, q, k, v, self.cu, D_pad=self.D_pad, out=self.codes, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        q8, k8, v8t = self.codes
        vf.attn_varlen(q8, k8, v8t, st, self.cu, w.max_seqlen, w.D, out=self.out,
                       workspace=self.ws, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    def step(self, stream, evs=None):
        for i in range(self.layers):
            self.layer(i, stream, None if evs is None else evs[i])


def _quant_bytes(w, dynamic):
    n = w.T * w.H * w.D
    return 3 * n * (5 if dynamic else 3)


# ----------------------------------------------------------------------------- cpu baseline
def cpu_oracle_sample(w, seconds_budget=12.0, rows_per_block=None, blocks=None, seed=0):
    """Time the oracle (as it stands) on whole (segment, head) blocks of one layer.

    Each block: E4M3-quantize that head's q/k/v slices of the segment with the
    layer's scales, then fp64 attention for its queries over all its keys.
    Returns (TFLOP/s of algorithmic attention flops, cores, description).
    """
    from oracle import attention as oattn
    from oracle import quant as oquant
    from oracle import scales as oscales

    q, k, v = workloads.make_qkv(w.seqlens, w.H, w.D, seed, w.outliers, w.per_head_std, device="cpu")
    st = oscales.ScaleState()
    st.push([oscales.amax(t.float().numpy()) for t in (q, k, v)])
    order = [(b, h) for b in range(len(w.seqlens)) for h in range(w.H)]
    cu = w.cu_seqlens
    flops = 0.0
    done = 0
    t0 = time.perf_counter()
    for b, h in order:
        s, e = cu[b], cu[b + 1]
        L = e - s
        R = L if rows_per_block is None else min(L, rows_per_block)
        qs = q[s:s + R, h:h + 1].float().numpy()
        ks = k[s:e, h:h + 1].float().numpy()
        vs = v[s:e, h:h + 1].float().numpy()
        c = [oquant.quantize(x, st.inv_scale[t]) for t, x in enumerate((qs, ks, vs))]
        _attend_block(oattn, c, st.scale, R, L, w.D)
        flops += 4.0 * R * L * w.D
        done += 1
        if (blocks is not None and done >= blocks) or (blocks is None and
                                                        time.perf_counter() - t0 > seconds_budget):
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    rows_desc = "all queries" if rows_per_block is None else "%d queries" % rows_per_block
    desc = ("%d of %d (segment, head) blocks of one %s layer: E4M3 quantize of the block's "
            "q/k/v slices + fp64 attention (%s x all keys of the segment)"
            % (done, len(order), w.name, rows_desc))
    return flops / dt / 1e12, cores, desc, dt


def _attend_block(oattn, c, scales, R, L, D):
    """fp64 attention of R queries against L keys of one (segment, head) block."""
    q = oattn.dequant(c[0][:, 0, :D], scales[0])
    k = oattn.dequant(c[1][:, 0, :D], scales[1])
    v = oattn.dequant(c[2][:, 0, :D], scales[2])
    return oattn._attend(q, k, v, 1.0 / math.sqrt(D), False)


# ----------------------------------------------------------------------------- main
def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    w = workloads.WORKLOADS[args.workload]
    vals = []
    desc = ""
    cores = 0
    total = 0.0
    for i in range(args.warmup + args.steps):
        v, cores, desc, dt = cpu_oracle_sample(w, rows_per_block=1024, blocks=1, seed=i)
        if i >= args.warmup:
            vals.append(v)
            total += dt
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.desc},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "per step: " + desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# Image sizes of the pages' encoder measurements ("FP8 ViT Encoder Attention",
# Performance: HD, FullHD, QHD, 4K, 3 images per request) at 16-px patches.
# 1080 px is not a multiple of 16: 67 patch rows are taken (the partial row
# dropped), i.e. 67 x 120 = 8040 patches.
SWEEP_SIZES = [("HD 720x1280", 45 * 80), ("FullHD 1080x1920", 67 * 120),
               ("QHD 1440x2560", 90 * 160), ("4K 2160x3840", 135 * 240)]


def resolution_sweep(vf, dev, stream, reps, head_dims=(80, 128), H=16, images=3, echo=True):
    """One attention layer per image size: FP8 with dynamic scaling (amax +
    quant + attention), FP8 with static scales (quant + attention) and the BF16
    path, each timed alone with CUDA events and L2 flushed before every rep;
    returns (and with ``echo`` prints) one record per (size, head_dim)."""
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    rows = []
    for D in head_dims:
        for name, L in SWEEP_SIZES:
            seqlens = [L] * images
            T = sum(seqlens)
            cu = torch.tensor([i * L for i in range(images + 1)], dtype=torch.int32, device=dev)
            q, k, v = workloads.make_qkv(seqlens, H, D, 900 + D, True, False, device=dev)
            D_pad = vf.default_d_pad(D)
            codes = vf.alloc_codes(T, H, D_pad, dev)
            out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
            wsp = vf.Workspace(images, dev)
            st_dyn = vf.ScaleState(dev).init()
            st_sta = vf.ScaleState(dev).init().set_static(224.0, 198.0, 210.0)
            attn = lambda st: vf.attn_varlen(*codes, st, cu, L, D, out=out, workspace=wsp, stream=stream)
            quant = lambda st: vf.quantize_unpad(st, q, k, v, cu, D_pad=D_pad, out=codes, stream=stream)
            arms = {
                "fp8_dynamic": lambda: (vf.amax_update(st_dyn, q, k, v, cu, stream=stream),
                                        quant(st_dyn), attn(st_dyn)),
                "fp8_static": lambda: (quant(st_sta), attn(st_sta)),
                "fp8_attn_only": lambda: attn(st_sta),
                "bf16": lambda: vf.attn_varlen_bf16(q, k, v, cu, L, out=out, workspace=wsp,
                                                    stream=stream),
            }
            res = {}
            for arm, fn in arms.items():
                for _ in range(3):
                    fn()
                times = []
                for _ in range(reps):
                    flush_l2(flush)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    fn()
                    e1.record(stream)
                    torch.cuda.synchronize(dev)
                    times.append(e0.elapsed_time(e1) * 1e3)
                res[arm] = statistics.median(times)
            assert wsp.error() == 0
            flops = 4 * images * L * L * H * D
            row = {
                "sweep": name, "tokens_per_image": L, "images": images, "heads": H, "head_dim": D,
                "fp8_kernel": _fp8_kernel(vf, [L] * images, H, dev),
                **{k2 + "_us": round(v2, 1) for k2, v2 in res.items()},
                "fp8_dynamic_vs_bf16": round(res["bf16"] / res["fp8_dynamic"], 3),
                "fp8_static_vs_bf16": round(res["bf16"] / res["fp8_static"], 3),
                "fp8_attn_tflops": round(flops / res["fp8_attn_only"] / 1e6, 1),
                "bf16_tflops": round(flops / res["bf16"] / 1e6, 1)}
            rows.append(row)
            if echo:
                print(json.dumps(row), flush=True)
            del q, k, v, codes, out
    return rows


# The other configurations of the workload list, reported beside the headline
# one (which sets `value`): tiny packed varlen, the 8192-token kernel
# microbench, 3 HD images at d = 80 and 3 4K images plus mixed segments.
PER_CONFIG = ["tiny", "micro8k", "hd3", "uhd3mix"]


def per_config_block(vf, dev, stream, peaks, peak_kind, reps=None):
    """One layer of each PER_CONFIG workload as `bench.py --workload NAME` runs
    it (dynamic scaling = amax + ring + quantize; static = quantize), FP8
    attention and the BF16 path on the same inputs; each arm timed alone with
    CUDA events, the L2 flushed (a 256 MB write read back, outside the timed
    span) before every rep, median of the reps."""
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    fp8_peak = peaks["bf16_tflops_sustained"] * FP8_PER_BF16
    bf16_peak = peaks["bf16_tflops_sustained"]
    block = {}
    for name in PER_CONFIG:
        w = workloads.WORKLOADS[name]
        run = Runner(vf, w, dev, layers=1)
        q, k, v = run.inputs[0]
        st = run.states[0]
        q8, k8, v8t = run.codes

        def quant():
            if run.dynamic:
                vf.amax_update(st, q, k, v, run.cu, stream=stream)
            vf.quantize_unpad(st, q, k, v, run.cu, D_pad=run.D_pad, out=run.codes, stream=stream)

        arms = {
            "quant": quant,
            "fp8_attn": lambda: vf.attn_varlen(q8, k8, v8t, st, run.cu, w.max_seqlen, w.D,
                                               out=run.out, workspace=run.ws, stream=stream),
            "bf16_attn": lambda: vf.attn_varlen_bf16(q, k, v, run.cu, w.max_seqlen, out=run.out,
                                                     workspace=run.ws, stream=stream),
        }
        n = reps if reps is not None else (5 if w.flops() > 1e13 else 15)
        res = {}
        for arm, fn in arms.items():
            for _ in range(3):
                fn()
            times = []
            for _ in range(n):
                with torch.cuda.stream(stream):
                    flush_l2(flush)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                times.append(e0.elapsed_time(e1) * 1e3)
            res[arm] = statistics.median(times)
        assert run.ws.error() == 0 and st.device_error() == 0
        flops = w.flops()
        qbytes = _quant_bytes(w, run.dynamic)
        fp8_tf = flops / res["fp8_attn"] / 1e6
        bf16_tf = flops / res["bf16_attn"] / 1e6
        layer_us = res["quant"] + res["fp8_attn"]
        block[name] = {
            "workload": w.desc, "scaling": "dynamic" if run.dynamic else "static",
            "tokens": w.T, "heads": w.H, "head_dim": w.D, "flops": flops,
            "fp8_kernel": _fp8_kernel(vf, w.seqlens, w.H, dev),
            "fp8_attn_us": round(res["fp8_attn"], 1), "fp8_attn_tflops": round(fp8_tf, 1),
            "fp8_attn_frac_of_peak": round(fp8_tf / fp8_peak, 4),
            "quant_us": round(res["quant"], 1), "quant_bytes": qbytes,
            "quant_gbs": round(qbytes / res["quant"] / 1e3, 1),
            "quant_frac_of_hbm": round(qbytes / res["quant"] / 1e3 / peaks["hbm_gbs"], 4),
            "layer_us": round(layer_us, 1), "layer_tflops_incl_quant": round(flops / layer_us / 1e6, 1),
            "bf16_attn_us": round(res["bf16_attn"], 1), "bf16_tflops": round(bf16_tf, 1),
            "bf16_frac_of_peak": round(bf16_tf / bf16_peak, 4),
            "fp8_vs_bf16_attn": round(res["bf16_attn"] / res["fp8_attn"], 3),
            "fp8_with_quant_vs_bf16": round(res["bf16_attn"] / layer_us, 3),
            "reps": n}
        del run, q, k, v, q8, k8, v8t, st
        torch.cuda.empty_cache()
    block["_peaks"] = {"fp8": fp8_peak, "bf16": bf16_peak, "hbm_gbs": peaks["hbm_gbs"],
                       "source": "%s bf16 sustained x %.0f for FP8; %s HBM copy"
                                 % (peak_kind, FP8_PER_BF16, peak_kind),
                       "l2": "flushed (256 MB write, read back) before every rep, outside the timed span"}
    return block


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qhd3", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--layers", type=int, default=None, help="limit layers (qhd3 only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-bf16", action="store_true", help="skip the BF16 comparison column")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload block and the resolution sweep block")
    ap.add_argument("--sweep", action="store_true",
               help="per image size: FP8 (dynamic / static, with quant) vs BF16 layer time, then exit")
    ap.add_argument("--sweep-reps", type=int, default=7)
    args = ap.parse_args()
    ws, rank, local = _dist()
    if args.impl == "reference":
        return run_reference(args, ws, rank)

    import fp8_vision_encoder_gb300 as vf

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    if args.sweep:
        resolution_sweep(vf, dev, torch.cuda.current_stream(dev), args.sweep_reps)
        return 0

    w = workloads.WORKLOADS[args.workload]
    run = Runner(vf, w, dev, layers=args.layers)
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(3, args.warmup)):
        run.step(stream)
    torch.cuda.synchronize(dev)

    # Every layer reads its own inputs.  A step whose inputs take at least
    # twice the L2 leaves nothing in it for the next step; a smaller one gets
    # the L2 flushed (a write of twice its size) before every timed step,
    # outside the timed spans, which are then summed.
    step_bytes = 3 * w.T * w.H * w.D * 2 * run.layers
    flush = (torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
             if step_bytes < L2_FLUSH_BYTES else None)

    def timed_region():
        # Per-kernel events ride along on the timed steps.
        marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps if flush is not None else 1)]
        evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)]
                for _ in range(run.layers)] for _ in range(args.steps)]
        sampler = ClockSampler(local)
        if pg:
            pg.barrier()
        torch.cuda.synchronize(dev)
        sampler.start()
        time.sleep(0.3)
        if flush is None:
            marks[0][0].record(stream)
            for s in range(args.steps):
                run.step(stream, evs[s])
            marks[0][1].record(stream)
        else:
            for s in range(args.steps):
                with torch.cuda.stream(stream):
                    flush_l2(flush, s & 0xFF)
                marks[s][0].record(stream)
                run.step(stream, evs[s])
                marks[s][1].record(stream)
        torch.cuda.synchronize(dev)
        clocks = sampler.stop()
        if pg:
            pg.barrier()
        ms = sum(a.elapsed_time(b) for a, b in marks)
        if pg:
            t = torch.tensor([ms], device=dev)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            ms = float(t.item())
        quant_ms = [e[0].elapsed_time(e[1]) for st in evs for e in st]
        attn_ms = [e[1].elapsed_time(e[2]) for st in evs for e in st]
        return ms, clocks, quant_ms, attn_ms

    ms, clocks, quant_ms, attn_ms = timed_region()
    # A region that saw a hardware or thermal slowdown, or SM clocks held well
    # below their maximum with no reason given, is timed once more (all ranks
    # agree first); the first attempt's clock record stays in the line.
    bad = clocks_rejected(clocks)
    if pg:
        t = torch.tensor([1.0 if bad else 0.0], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        bad = t.item() > 0
    first_clocks = None
    if bad:
        first_clocks = clocks
        ms, clocks, quant_ms, attn_ms = timed_region()
    assert run.ws.error() == 0, "attention workspace reported a device error"

    flops_step = run.flops_layer * run.layers
    value = ws * flops_step * args.steps / (ms * 1e-3) / 1e12
    peaks, peak_kind = _peaks()
    fp8_peak = peaks["bf16_tflops_sustained"] * FP8_PER_BF16
    attn_avg = statistics.mean(attn_ms)
    quant_avg = statistics.mean(quant_ms)
    achieved = run.flops_layer / (attn_avg * 1e-3) / 1e12
    qbytes = _quant_bytes(w, run.dynamic)
    quant_gbs = qbytes / (quant_avg * 1e-3) / 1e9

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3", "data": "synthetic",
        "config": {"workload": w.desc, "name": w.name, "tokens": w.T, "segments": w.seqlens[:8],
                   "heads": w.H, "head_dim": w.D, "layers": run.layers,
                   "static_scales": run.static,
                   "l2": (("inputs larger than L2 (each layer reads its own %.0f MB of bf16 q/k/v)"
                           % (3 * w.T * w.H * w.D * 2 / 1e6)) if flush is None else
                          ("L2 flushed (a %d MB write, read back) before every timed step, outside the timed "
                           "spans; a step reads %.0f MB of bf16 q/k/v" % (L2_FLUSH_BYTES >> 20,
                                                                          step_bytes / 1e6))),
                   "parallelism": "replicas" if ws > 1 else "single",
                   "fp8_kernel": _fp8_kernel(vf, w.seqlens, w.H, dev)},
        "frac_of_fp8_peak": value / fp8_peak,
        "roofline": {"bound": "tensor", "kernel": "attn_fp8 (work-list + attention launch)",
                     "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": achieved / fp8_peak,
                     "traffic": (_profile_traffic("attn_fp8_qhd3.md", ATTN_FP8_SOURCES)
                                 if w.name == "qhd3" else None),
                     "algorithmic_bytes": 3 * w.T * w.H * w.D + 2 * w.T * w.H * w.D,
                     "peak_source": "%s bf16 sustained x %.0f (fp8/bf16 nominal ratio)"
                                    % (peak_kind, FP8_PER_BF16)},
        "quant_roofline": {"bound": "hbm", "achieved": quant_gbs, "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": quant_gbs / peaks["hbm_gbs"],
                           "algorithmic_bytes": qbytes, "peak_source": peak_kind,
                           "traffic": (_profile_traffic("quant_qhd3.md", QUANT_SOURCES)
                                       if w.name == "qhd3" and not run.dynamic else None)},
        "breakdown_us": {"quant": 1e3 * quant_avg, "attn": 1e3 * attn_avg},
        "gpu_launches": run.launches_layer * run.layers * args.steps,
        "clocks": clocks if first_clocks is None else dict(clocks, rejected_first_attempt=first_clocks),
    }

    # the BF16 path built the same way, on the same layers (timed separately)
    if not args.no_bf16:
        line["bf16_path"] = bf16_column(vf, run, stream, dev, args.steps, peaks, peak_kind,
                                        1e3 * attn_avg, 1e3 * (attn_avg + quant_avg))

    # end to end through the public API with host buffers
    if not args.no_e2e:
        line["e2e"] = e2e(vf, run, stream, dev, args.e2e_steps, max(3, args.warmup), ws, pg)
    # The other workloads and the resolution sweep, beside the headline line
    # (one GPU; after the timed region, so they do not touch its numbers).
    if rank == 0 and ws == 1 and not args.no_per_config and args.workload == "qhd3":
        del run.inputs
        torch.cuda.empty_cache()
        line["per_config"] = per_config_block(vf, dev, stream, peaks, peak_kind)
        line["sweep"] = resolution_sweep(vf, dev, stream, reps=5, echo=False)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, cores, desc, dt = cpu_oracle_sample(w)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": dt}
    if rank == 0:
        print(json.dumps(line))
    if pg:
        pg.destroy_process_group()
    return 0


def bf16_column(vf, run, stream, dev, steps, peaks, peak_kind, fp8_attn_us, fp8_layer_us):
    """BF16 attention (vitfp8_attn_varlen_bf16) on each layer's bf16 q, k, v.

    Same layers, same output buffer and workspace as the FP8 step; no scales
    and no quantization.  Timed with CUDA events on the launching stream.
    """
    w = run.w

    def one_step(evs=None):
        for i, (q, k, v) in enumerate(run.inputs):
            if evs is not None:
                evs[i][0].record(stream)
            vf.attn_varlen_bf16(q, k, v, run.cu, w.max_seqlen, out=run.out, workspace=run.ws,
                                stream=stream)
            if evs is not None:
                evs[i][1].record(stream)

    for _ in range(3):
        one_step()
    torch.cuda.synchronize(dev)
    n = max(1, min(steps, 3))
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(run.layers)]
           for _ in range(n)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for s_ in range(n):
        one_step(evs[s_])
    stop.record(stream)
    torch.cuda.synchronize(dev)
    assert run.ws.error() == 0, "attention workspace reported a device error (bf16)"
    ms = start.elapsed_time(stop) / n
    attn_us = 1e3 * statistics.mean(e[0].elapsed_time(e[1]) for st in evs for e in st)
    bf16_peak = peaks["bf16_tflops_sustained"]
    achieved = run.flops_layer / (attn_us * 1e-6) / 1e12
    return {"value": run.flops_layer * run.layers / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": ms, "attn_us": attn_us, "dtype": "bf16",
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16_peak,
                         "unit": "TFLOP/s", "frac": achieved / bf16_peak,
                         "peak_source": "%s bf16 sustained" % peak_kind},
            "fp8_attn_speedup": attn_us / fp8_attn_us,
            "fp8_with_quant_speedup": attn_us / fp8_layer_us}


def e2e(vf, run, stream, dev, steps, warmup, ws, pg):
    """Same metric with pinned host inputs copied in and the output copied out every layer.

    The copies run on their own streams and overlap the compute of the
    neighbouring layers (inputs of layer i+1 come in while layer i runs, the
    output of layer i goes out while layer i+1 runs), with two device buffers
    for each; the timed region ends when the last output has reached the host.
    """
    w = run.w
    host_in = []
    for trio in run.inputs:
        hs = []
        for t in trio:
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            hs.append(h)
        host_in.append(hs)
    host_out = [torch.empty(run.out.shape, dtype=run.out.dtype).pin_memory() for _ in range(2)]
    dev_in = [[torch.empty_like(t) for t in run.inputs[0]] for _ in range(2)]
    dev_out = [torch.empty_like(run.out) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in[0]) * run.layers
    d2h = host_out[0].numel() * host_out[0].element_size() * run.layers
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready = [ev(), ev()]      # inputs of the buffer landed
    in_free = [ev(), ev()]       # compute done with the buffer's inputs
    out_ready = [ev(), ev()]     # output buffer written
    out_free = [ev(), ev()]      # output buffer copied to the host

    def load(i):
        b = i % 2
        s_in.wait_event(in_free[b])
        with torch.cuda.stream(s_in):
            for d, h in zip(dev_in[b], host_in[i]):
                d.copy_(h, non_blocking=True)
        in_ready[b].record(s_in)

    def one_step():
        for b in range(2):
            in_free[b].record(stream)
            out_free[b].record(stream)
        load(0)
        for i in range(run.layers):
            b = i % 2
            if i + 1 < run.layers:
                load(i + 1)
            stream.wait_event(in_ready[b])
            stream.wait_event(out_free[b])
            q, k, v = dev_in[b]
            st = run.states[i]
            if run.dynamic:
                vf.amax_update(st, q, k, v, run.cu, stream=stream)
            vf.quantize_unpad(st, q, k, v, run.cu, D_pad=run.D_pad, out=run.codes, stream=stream)
            in_free[b].record(stream)
            q8, k8, v8t = run.codes
            vf.attn_varlen(q8, k8, v8t, st, run.cu, w.max_seqlen, w.D, out=dev_out[b],
                           workspace=run.ws, stream=stream)
            out_ready[b].record(stream)
            s_out.wait_event(out_ready[b])
            with torch.cuda.stream(s_out):
                host_out[b].copy_(dev_out[b], non_blocking=True)
            out_free[b].record(s_out)
        stream.wait_stream(s_out)

    # Warm-up: the first pass over a freshly pinned host buffer is several
    # times slower than later ones (256 ms against 69 ms for a 24-layer step),
    # so the copies get the same warm-up steps as the compute.
    for _ in range(warmup):
        one_step()
    torch.cuda.synchronize(dev)

    # The host link alone, for reading the number: one layer's inputs in and
    # one output out, each direction timed by itself, best of three (the host
    # side is shared, so a single copy can land in someone else's burst).
    def link_gbs(copy, nbytes, s):
        best = 0.0
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            with torch.cuda.stream(s):
                copy()
            e1.record(s)
            torch.cuda.synchronize(dev)
            best = max(best, nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
        return best

    h2d_link = link_gbs(lambda: [d.copy_(h, non_blocking=True) for d, h in zip(dev_in[0], host_in[0])],
                        h2d // run.layers, s_in)
    d2h_link = link_gbs(lambda: host_out[0].copy_(dev_out[0], non_blocking=True), d2h // run.layers,
                        s_out)
    if pg:
        pg.barrier()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    marks[0].record(stream)
    for i in range(steps):
        one_step()
        marks[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    ms = marks[0].elapsed_time(marks[-1])
    step_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(steps)]
    if pg:
        t = torch.tensor([ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms = float(t.item())
    val = ws * run.flops_layer * run.layers * steps / (ms * 1e-3) / 1e12
    return {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "warmup": warmup, "ms_per_step": ms / steps,
            "step_ms": [round(x, 2) for x in step_ms],
            "median_ms_per_step": statistics.median(step_ms),
            "value_at_median_step": ws * run.flops_layer * run.layers / (statistics.median(step_ms) * 1e-3) / 1e12,
            "link_gbs": {"h2d": h2d_link, "d2h": d2h_link,
                         "step_floor_ms": h2d / (h2d_link * 1e6)},
            "copies": "pinned host buffers; H2D, compute and D2H on three streams, overlapped across layers"}


if __name__ == "__main__":
    sys.exit(main())
