#!/usr/bin/env python3
"""Benchmark of the convolution hot path on GB300: one step = one decoder pass over synthetic data.

The step runs every stage of the path through the library's C ABI:
  * taesd  - TAESD-like 2D chain, NCHW f16, N=4, 3x256x256: 3->64, 3x 64->64, 64->64 stride 2,
             2x 64->64 at 128x128, all with bias + ReLU (conv_stack_forward, 7 layers);
  * stack  - causal 3x3x3 stack, NDHWC bf16: two chained 128->128 layers with ReLU over 4 frames
             (+2 carried) at 352x624 (conv_stack_forward with per-layer carries);
  * l3     - causal 256->128 over 4 frames (+2 carried) at 176x312 (conv_forward);
  * head   - conv_out head: causal 256->12 over 4 frames (+2 carried) at 352x624, bias, clamp to
             [-1,1], 2x2 unpatchify to 4x704x1248 RGB (conv_forward: the stencil head, the temporal
             sums of the nine taps on the tensor cores and the nine spatial taps in the epilogue;
             the single-pass form and the two-pass forms are timed beside it).
value = total convolution FLOP of the step / step time (TFLOP/s, whole job over all ranks).
Also reported: decoder-stack ms per frame (stack + l3 + head over the 4 frames), per-stage times,
every configuration's time-based roofline (``configs``: the step's stages and layers, plus the
16->16 64x64 conv and the causal 256->256 layer timed alone with L2 flushed between launches), the
roofline fraction of the dominant kernel, peak device memory (the step, and a pass-by-pass decoder
against one long pass for 16 to 64 frames), an end-to-end number with host buffers, the SM clocks
seen during the timed region, and the CPU oracle timed on a bounded sample.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own replica of the step (weak scaling, no collective on the
data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "conv TFLOP/s & HBM GB/s vs roofline; decoder-stack ms/frame, 1 GB300"
WORKLOAD = ("decoder pass: TAESD-like 2D chain (N=4, 3x256x256, 7 convs, NCHW f16) + causal 3x3x3 "
            "stack (2x 128->128 @4+2x352x624, 256->128 @4+2x176x312, NDHWC bf16) + conv_out head "
            "(256->12 @4+2x352x624, clamp, 2x2 unpatchify)")
FRAMES = 4
STAGES = ["taesd", "stack", "l3", "head"]
AB_STAGES = ["head_fused", "head_two_pass", "head_split"]
SINGLE_STAGES = ["conv16", "conv256"]
# dram__bytes_read.sum + dram__bytes_write.sum of one launch of each kernel at the benchmark's size,
# from one ncu capture of that launch of the current code (each kernel's summary under profiles/; the
# TAESD entry is its stage's eight launches; the 256->256 layer's was taken back to back, L2-warm)
DRAM_BYTES = {"conv16": 337408.0, "taesd": 157752576.0, "conv256": 46769408.0, "stack_128": 644807936.0,
              "l3": 260427776.0, "head": 700393472.0}


def layer_descs():
    """The descriptors (keyword arguments of x3x3_convolution_gb300.make_desc) of every layer this
    benchmark runs, by stage: the step's four stages and the two single-layer configurations timed
    beside it (the 16->16 64x64 NCHW f16 conv and the causal 256->256 4+2x88x156 layer). The full-size
    parity tests build their plans from these, so they cover the launch configurations timed here."""
    from x3x3_convolution_gb300.synth import TAESD_CHAIN
    taesd, H, W = [], 256, 256
    for ci, co, s in TAESD_CHAIN:
        taesd.append(dict(dims=2, N=4, C_in=ci, C_out=co, H=H, W=W, stride=s, layout="NCHW", dtype="f16",
                          act="relu"))
        H, W = (H - 1) // s + 1, (W - 1) // s + 1
    stack = [dict(dims=3, N=1, C_in=128, C_out=128, H=352, W=624, D=FRAMES, act="relu") for _ in range(2)]
    return {"taesd": taesd, "stack": stack,
            "l3": dict(dims=3, N=1, C_in=256, C_out=128, H=176, W=312, D=FRAMES, act="none"),
            "head": dict(dims=3, N=1, C_in=256, C_out=12, H=352, W=624, D=FRAMES, act="clamp", unpatchify2x2=True),
            "conv16": dict(dims=2, N=1, C_in=16, C_out=16, H=64, W=64, layout="NCHW", dtype="f16", act="relu"),
            "conv256": dict(dims=3, N=1, C_in=256, C_out=256, H=88, W=156, D=FRAMES, act="none")}


def flop2d(N, Ci, Co, Ho, Wo):
    return 2.0 * N * Ci * Co * 9 * Ho * Wo


def flop3d(Ci, Co, D, H, W):
    return 2.0 * Ci * Co * 27 * D * H * W


def stage_cost():
    """FLOP and algorithmic bytes (input read once incl. carried frames, output written once,
    weights, bias) of each stage."""
    from x3x3_convolution_gb300.synth import TAESD_CHAIN
    f_taesd, b_taesd, H, W = 0.0, 0.0, 256, 256
    for ci, co, s in TAESD_CHAIN:
        Ho, Wo = (H - 1) // s + 1, (W - 1) // s + 1
        f_taesd += flop2d(4, ci, co, Ho, Wo)
        b_taesd += 2.0 * (4 * ci * H * W + 4 * co * Ho * Wo + co * ci * 9 + co)
        H, W = Ho, Wo
    b_l1 = 2.0 * (6 * 352 * 624 * 128 + 4 * 352 * 624 * 128 + 128 * 128 * 27 + 128)
    flops = {"taesd": f_taesd, "stack": 2 * flop3d(128, 128, 4, 352, 624), "l3": flop3d(256, 128, 4, 176, 312),
             "head": flop3d(256, 12, 4, 352, 624)}
    nbytes = {"taesd": b_taesd, "stack": 2 * b_l1,
              "l3": 2.0 * (6 * 176 * 312 * 256 + 4 * 176 * 312 * 128 + 256 * 128 * 27 + 128),
              "head": 2.0 * (6 * 352 * 624 * 256 + 4 * 352 * 624 * 12 + 256 * 12 * 27 + 12)}
    return flops, nbytes


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """SM clocks and clock-event (throttle) reasons sampled during the timed region: NVML read through
    ctypes every millisecond from a background thread (the timed region of a short run lasts only tens
    of milliseconds), else nvidia-smi every 200 ms. Read-only: no setting of the GPU is touched."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits (nvml.h): SwPowerCap, HwSlowdown, SwThermalSlowdown, HwThermalSlowdown
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.nvml = None
        self.handle = None
        self.samples = []
        self.stop_flag = None
        self.thread = None
        try:
            import ctypes
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            ok = False
            try:
                import torch
                pr = torch.cuda.get_device_properties(gpu_index)
                bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0".encode()
                ok = lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) == 0
            except Exception:
                ok = False
            if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            self.nvml, self.handle = lib, h
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except Exception:
            self.nvml = None

    def _poll(self):
        import ctypes
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0 and \
                    self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0 and \
                    self.reasons_fn(self.handle, ctypes.byref(rs)) == 0:
                self.samples.append((clk.value, mx.value, rs.value))
            time.sleep(0.001)

    def start(self):
        if self.nvml is not None:
            import threading
            self.samples = []
            self.stop_flag = threading.Event()
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.nvml is not None:
            self.stop_flag.set()
            self.thread.join(timeout=5)
            if not self.samples:
                return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "source": "nvml"}
            reasons = sorted({name for _, _, r in self.samples for bit, name in self.REASON_BITS.items() if r & bit})
            return {"sm_mhz": statistics.median(c for c, _, _ in self.samples),
                    "sm_max_mhz": max(m for _, m, _ in self.samples), "reasons": reasons,
                    "samples": len(self.samples), "source": "nvml, 1 ms"}
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi, 200 ms"}


class Workload:
    """All layers of the decoder pass, with packed weights, inputs, carries and outputs on the GPU."""

    def __init__(self, device, seed_base=0):
        import torch
        import x3x3_convolution_gb300 as x3
        from x3x3_convolution_gb300 import synth
        dev = device
        descs = layer_descs()
        xt, layers = synth.taesd_chain(seed=1002 + seed_base)
        convs = [x3.Conv(x3.make_desc(**dd), L.w.torch(dev), L.b.torch(dev)) for dd, L in zip(descs["taesd"], layers)]
        self.taesd = x3.ConvStack(convs)
        self.taesd_x = xt.torch(dev)
        self.taesd_y = torch.empty(convs[-1].out_shape(), dtype=torch.float16, device=dev)
        st = synth.conv3d_stack(seed=1004 + seed_base)
        sc = []
        for dd, L in zip(descs["stack"], st["layers"]):
            sc.append(x3.Conv(x3.make_desc(**dd), L.w.torch(dev), L.b.torch(dev)))
        self.stack = x3.ConvStack(sc)
        self.stack_x = st["x"].torch(dev)
        self.stack_carries = [c.torch(dev).contiguous() for c in st["carries"]]
        self.stack_y = torch.empty(sc[-1].out_shape(), dtype=torch.bfloat16, device=dev)
        L3 = st["L3"]
        self.l3 = x3.Conv(x3.make_desc(**descs["l3"]), L3.w.torch(dev), L3.b.torch(dev))
        self.l3_x = st["x3"].torch(dev)
        self.l3_c = st["carry3"].torch(dev)
        self.l3_y = torch.empty(self.l3.out_shape(), dtype=torch.bfloat16, device=dev)
        hx, hc, HL = synth.head(seed=1005 + seed_base)
        head_desc = dict(D=FRAMES, act="clamp", unpatchify2x2=True)
        # the step's head: the library's default (the stencil head: one kernel, G kept in fp32 on chip)
        self.head = x3.Conv(x3.make_desc(**descs["head"]), HL.w.torch(dev), HL.b.torch(dev))
        self.head_x = hx.torch(dev)
        self.head_c = hc.torch(dev)
        self.head_y = torch.empty(self.head.out_shape(), dtype=torch.bfloat16, device=dev)
        # A/B forms of the head, not part of the step: the single pass (kw folded into M), the two
        # passes with an fp32 G plane and with a bf16 one (the page's value path)
        self.head_fused = x3.Conv(x3.make_desc(3, 1, 256, 12, 352, 624, kernel="igemm", **head_desc),
                                  HL.w.torch(dev), HL.b.torch(dev))
        self.head_fused_y = torch.empty(self.head_fused.out_shape(), dtype=torch.bfloat16, device=dev)
        self.head2 = x3.Conv(x3.make_desc(3, 1, 256, 12, 352, 624, kernel="head_two_pass", **head_desc),
                             HL.w.torch(dev), HL.b.torch(dev))
        self.head2_y = torch.empty(self.head2.out_shape(), dtype=torch.bfloat16, device=dev)
        self.head_split = x3.Conv(x3.make_desc(3, 1, 256, 12, 352, 624, kernel="head_split", **head_desc),
                                  HL.w.torch(dev), HL.b.torch(dev))
        self.head_split_y = torch.empty(self.head_split.out_shape(), dtype=torch.bfloat16, device=dev)
        # kernels per step: layout conversion + 7 TAESD convs, 2 stack convs and their 2 carry copies,
        # l3, the head
        self.kernels_per_step = 1 + len(convs) + 2 * len(sc) + 1 + 1
        self.plans = {"taesd": [x3.conv_plan_describe(c.plan) for c in convs],
                      "stack": x3.conv_plan_describe(sc[0].plan),
                      "l3": x3.conv_plan_describe(self.l3.plan),
                      "head": x3.conv_plan_describe(self.head.plan)}
        self.carry_valid = False

    def inputs(self):
        return [self.taesd_x, self.stack_x, self.l3_x, self.head_x]

    def outputs(self):
        return [self.taesd_y, self.stack_y, self.l3_y, self.head_y]

    def stage(self, i, stream):
        """Stage i of the step alone (0 taesd, 1 stack, 2 l3, 3 head)."""
        if i == 0:
            self.taesd(self.taesd_x, out=self.taesd_y, stream=stream)
        elif i == 1:
            self.stack(self.stack_x, carries=self.stack_carries, carry_valid=self.carry_valid, out=self.stack_y,
                       stream=stream)
            self.carry_valid = True
        elif i == 2:
            self.l3(self.l3_x, self.l3_c, out=self.l3_y, stream=stream)
        else:
            self.head(self.head_x, self.head_c, out=self.head_y, stream=stream)

    def step(self, stream, ev=None):
        """One decoder pass; ev: optional 5 CUDA events recorded between the stages."""
        if ev:
            ev[0].record(stream)
        self.taesd(self.taesd_x, out=self.taesd_y, stream=stream)
        if ev:
            ev[1].record(stream)
        self.stack(self.stack_x, carries=self.stack_carries, carry_valid=self.carry_valid, out=self.stack_y,
                   stream=stream)
        self.carry_valid = True
        if ev:
            ev[2].record(stream)
        self.l3(self.l3_x, self.l3_c, out=self.l3_y, stream=stream)
        if ev:
            ev[3].record(stream)
        self.head(self.head_x, self.head_c, out=self.head_y, stream=stream)
        if ev:
            ev[4].record(stream)


def time_alone(fn, stream, reps, flush):
    """Mean device time (ms) of fn() over `reps` launches, each bracketed by its own CUDA events on
    `stream`, with a write of `flush` (larger than L2) between launches, outside the events."""
    import torch
    for _ in range(3):
        fn()
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    for e0, e1 in pairs:
        flush.add_(1)
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in pairs)


def roof_entry(ms, flop, nbytes, peaks, timing, dram=None, frames=None):
    """Time-based roofline of one kernel or stage: t_roof = max(bytes / HBM peak, FLOP / bf16 peak),
    frac = t_roof / t_measured; the bound is the larger of the two terms."""
    t = ms * 1e-3
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flop / (peaks["bf16_tflops"] * 1e12)
    e = {"ms": ms, "tflops": flop / t / 1e12, "gbs": nbytes / t / 1e9, "gflop": flop / 1e9, "alg_mb": nbytes / 1e6,
         "bound": "hbm" if t_hbm >= t_tc else "tensor", "t_roof_ms": max(t_hbm, t_tc) * 1e3,
         "frac": max(t_hbm, t_tc) / t, "frac_tensor": flop / t / 1e12 / peaks["bf16_tflops"],
         "frac_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"], "timing": timing,
         "dram_bytes_ncu": dram}
    if frames:
        e["ms_per_frame"] = ms / frames
    return e


def single_layer_configs(dev, stream, peaks, reps=20):
    """The two single-layer configurations, each timed alone with L2 flushed between launches: the
    16->16 64x64 NCHW f16 conv (bias, ReLU) and the causal 256->256 layer over 4+2 x 88x156."""
    import torch
    import x3x3_convolution_gb300 as x3
    from x3x3_convolution_gb300 import synth
    descs = layer_descs()
    x1, L1 = synth.conv2d_single(seed=1001)
    c1 = x3.Conv(x3.make_desc(**descs["conv16"]), L1.w.torch(dev), L1.b.torch(dev))
    x1d = x1.torch(dev)
    y1 = torch.empty(c1.out_shape(), dtype=torch.float16, device=dev)
    x3_, cr3, L3 = synth.conv3d_single(seed=1003)
    c3 = x3.Conv(x3.make_desc(**descs["conv256"]), L3.w.torch(dev), L3.b.torch(dev))
    x3d, cr3d = x3_.torch(dev), cr3.torch(dev)
    y3 = torch.empty(c3.out_shape(), dtype=torch.bfloat16, device=dev)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)  # 256 MB, twice the L2
    ms1 = time_alone(lambda: c1(x1d, out=y1, stream=stream), stream, reps, flush)
    ms3 = time_alone(lambda: c3(x3d, cr3d, out=y3, stream=stream), stream, reps, flush)
    f1, b1 = flop2d(1, 16, 16, 64, 64), 2.0 * (16 * 64 * 64 * 2 + 16 * 16 * 9 + 16)
    f3 = flop3d(256, 256, 4, 88, 156)
    b3 = 2.0 * (6 * 88 * 156 * 256 + 4 * 88 * 156 * 256 + 256 * 256 * 27 + 256)
    timing = f"alone, {reps} launches, L2 flushed between launches (256 MB write)"
    return {"conv16_64x64": dict(roof_entry(ms1, f1, b1, peaks, timing, DRAM_BYTES["conv16"]),
                                 note="launch-latency bound: 0.27 MB, far below a launch's fixed cost"),
            "causal256_4x88x156": dict(roof_entry(ms3, f3, b3, peaks, timing, DRAM_BYTES["conv256"], frames=FRAMES),
                                       plan=x3.conv_plan_describe(c3.plan))}


def pass_memory_curve(wl, dev):
    """Peak device memory of the causal 128->128 stack (the step's two layers, 352x624, 4 frames per
    pass) decoding T = 16, 32 and 64 frames pass by pass from pinned host memory (PassDecoder: one pass
    of frames, the histories and the two workspace buffers on the device), against one pass over all T
    frames with the whole sequence, its intermediates and its output on the device at once."""
    import torch
    import x3x3_convolution_gb300 as x3
    from x3x3_convolution_gb300.video import PassDecoder
    convs = wl.stack.layers
    out = []
    for passes in (4, 8, 16):
        T = FRAMES * passes
        x = torch.zeros((1, T, 352, 624, 128), dtype=torch.bfloat16).pin_memory()
        torch.cuda.synchronize()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        dec = PassDecoder(convs, FRAMES)
        y = dec.decode(x)
        torch.cuda.synchronize()
        peak_pass = torch.cuda.max_memory_allocated() - base
        del dec, y
        longc = [x3.Conv(x3.make_desc(3, 1, 128, 128, 352, 624, D=T, act={0: "none", 1: "relu", 2: "clamp"}[c.desc.act]),
                         torch.zeros((128, 128, 3, 3, 3), dtype=torch.bfloat16, device=dev),
                         torch.zeros(128, dtype=torch.bfloat16, device=dev)) for c in convs]
        torch.cuda.synchronize()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        st = x3.ConvStack(longc)
        xd = x.to(dev)
        yd = st(xd)
        torch.cuda.synchronize()
        peak_long = torch.cuda.max_memory_allocated() - base
        del st, xd, yd, longc, x
        torch.cuda.empty_cache()
        out.append({"frames": T, "passes": passes, "pass_decoder_gib": peak_pass / 2 ** 30,
                    "one_pass_gib": peak_long / 2 ** 30})
    return out


def cpu_baseline(target_s=12.0):
    """The oracle, as it stands, on the host cores, on a bounded sample of the dominant stage: the
    causal 128->128 layer at 352x624 restricted to a band of output rows of one frame."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(77)
    C, W = 128, 624
    w = (rng.standard_normal((C, C, 3, 3, 3)) * 0.03).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, C).astype(np.float32)

    def run(rows):
        x = rng.standard_normal((1, 1, rows, W, C)).astype(np.float32)
        c = rng.standard_normal((1, 2, rows, W, C)).astype(np.float32)
        t0 = time.perf_counter()
        oracle.conv3d_causal(x, w, b, carry=c, act="relu", layout="NDHWC")
        return time.perf_counter() - t0

    dt = run(4)
    rows = int(max(4, min(352, 4 * target_s / max(dt, 1e-3))))
    dt = run(rows)
    fl = flop3d(C, C, 1, rows, W)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.threads_used(), "kind": "oracle",
            "sample": f"causal 128->128 3x3x3 layer, 1 output frame x {rows} rows x 624 cols (of 4 x 352 x 624), "
                      f"{fl / 1e9:.1f} GFLOP in {dt:.1f} s", "seconds": dt}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def reduce_max(world, value):
    from x3x3_convolution_gb300 import dist as xd
    return xd.max_over_ranks(value) if world > 1 else value


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_stage_rate(stage, seconds, rng):
    """The oracle's FLOP rate on a band of output rows of one stage of the step, sized to take about
    `seconds`; returns (FLOP/s, description)."""
    import numpy as np
    import oracle

    def band3d(C_in, C_out, H, W, act, rows):
        w = (rng.standard_normal((C_out, C_in, 3, 3, 3)) / np.sqrt(27 * C_in)).astype(np.float32)
        b = rng.uniform(-0.1, 0.1, C_out).astype(np.float32)
        x = rng.standard_normal((1, 1, rows, W, C_in)).astype(np.float32)
        c = rng.standard_normal((1, 2, rows, W, C_in)).astype(np.float32)
        t0 = time.perf_counter()
        oracle.conv3d_causal(x, w, b, carry=c, act=act, layout="NDHWC")
        return time.perf_counter() - t0, flop3d(C_in, C_out, 1, rows, W)

    def band2d(C_in, C_out, H, W, rows):
        w = (rng.standard_normal((C_out, C_in, 3, 3)) / np.sqrt(9 * C_in)).astype(np.float32)
        b = rng.uniform(-0.1, 0.1, C_out).astype(np.float32)
        x = rng.uniform(-1, 1, (1, C_in, rows, W)).astype(np.float32)
        t0 = time.perf_counter()
        oracle.conv2d(x, w, b, act="relu")
        return time.perf_counter() - t0, flop2d(1, C_in, C_out, rows, W)

    shapes = {"taesd": lambda r: band2d(64, 64, 256, 256, r), "stack": lambda r: band3d(128, 128, 352, 624, "relu", r),
              "l3": lambda r: band3d(256, 128, 176, 312, "none", r), "head": lambda r: band3d(256, 12, 352, 624, "clamp", r)}
    limit = {"taesd": 256, "stack": 352, "l3": 176, "head": 352}[stage]
    dt, fl = shapes[stage](2)
    rows = int(max(2, min(limit, 2 * seconds / max(dt, 1e-4))))
    dt, fl = shapes[stage](rows)
    return fl / dt, f"{stage}: {rows} rows, {fl / 1e9:.2f} GFLOP in {dt:.2f} s"


def run_reference(args, rank):
    """The oracle as the reference arm: rank 0 times it on the host cores, each step a bounded sample
    of every stage of the workload (a band of output rows of one frame per stage); other ranks do
    nothing. `value` is the workload's throughput at the sampled per-stage FLOP rates (each stage's
    full FLOP count over its rate), `ms_per_step` the time a step's samples took, and the time one
    whole step of the workload would take at those rates is reported beside them."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    rng = np.random.default_rng(77)
    fl, _ = stage_cost()
    per_step_s = min(12.0, 150.0 / (args.steps + args.warmup))
    for _ in range(args.warmup):
        for st in STAGES:
            oracle_stage_rate(st, per_step_s / len(STAGES) / 4, rng)
    step_ms, sample_ms, notes = [], [], []
    for _ in range(args.steps):
        t = 0.0
        t0 = time.perf_counter()
        for st in STAGES:
            rate, note = oracle_stage_rate(st, per_step_s / len(STAGES), rng)
            t += fl[st] / rate
            notes.append(note)
        sample_ms.append((time.perf_counter() - t0) * 1e3)
        step_ms.append(t * 1e3)
    ms = float(np.mean(step_ms))
    value = sum(fl.values()) / (ms * 1e-3) / 1e12
    sample = ("each step: the oracle on a band of output rows of one frame of every stage (" +
              "; ".join(notes[-len(STAGES):]) + "); value = the workload's FLOP over its time at the "
              "sampled per-stage FLOP rates")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": float(np.mean(sample_ms)),
            "full_step_ms_at_sampled_rates": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "note": "CPU oracle (plain fp32 loops) on bounded samples of the workload"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads_used(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_stage(wl, args, stream, fl, nb):
    """Warm up, then time `steps` runs of one stage alone (CUDA events); one JSON line."""
    import torch
    if args.stage in SINGLE_STAGES:
        import x3x3_convolution_gb300 as x3
        from x3x3_convolution_gb300 import synth
        dd = layer_descs()[args.stage]
        if args.stage == "conv16":
            x, L = synth.conv2d_single(seed=1001)
            carry = None
            flop, nbytes = flop2d(1, 16, 16, 64, 64), 2.0 * (16 * 64 * 64 * 2 + 16 * 16 * 9 + 16)
        else:
            x, c, L = synth.conv3d_single(seed=1003)
            carry = c.torch(stream.device)
            flop = flop3d(256, 256, 4, 88, 156)
            nbytes = 2.0 * (6 * 88 * 156 * 256 + 4 * 88 * 156 * 256 + 256 * 256 * 27 + 256)
        conv = x3.Conv(x3.make_desc(**dd), L.w.torch(stream.device), L.b.torch(stream.device))
        xd = x.torch(stream.device)
        out = torch.empty(conv.out_shape(), dtype=xd.dtype, device=xd.device)
        run = lambda: conv(xd, carry, out=out, stream=stream)
        for _ in range(args.warmup):
            run()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        print(json.dumps({"stage": args.stage, "ms": ms, "tflops": flop / (ms * 1e-3) / 1e12,
                          "gbs": nbytes / (ms * 1e-3) / 1e9, "note": "back to back (L2-warm)",
                          "plan": x3.conv_plan_describe(conv.plan)}), flush=True)
        return
    fn = {"taesd": lambda: wl.taesd(wl.taesd_x, out=wl.taesd_y, stream=stream),
          "stack": lambda: wl.stack(wl.stack_x, carries=wl.stack_carries, carry_valid=True, out=wl.stack_y,
                                    stream=stream),
          "l3": lambda: wl.l3(wl.l3_x, wl.l3_c, out=wl.l3_y, stream=stream),
          "head": lambda: wl.head(wl.head_x, wl.head_c, out=wl.head_y, stream=stream),
          "head_fused": lambda: wl.head_fused(wl.head_x, wl.head_c, out=wl.head_fused_y, stream=stream),
          "head_two_pass": lambda: wl.head2(wl.head_x, wl.head_c, out=wl.head2_y, stream=stream),
          "head_split": lambda: wl.head_split(wl.head_x, wl.head_c, out=wl.head_split_y, stream=stream)}[args.stage]
    for _ in range(args.warmup):
        fn()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    key = "head" if args.stage.startswith("head") else args.stage
    print(json.dumps({"stage": args.stage, "ms": ms, "tflops": fl[key] / (ms * 1e-3) / 1e12,
                      "gbs": nb[key] / (ms * 1e-3) / 1e9, "plan": wl.plans[key]}), flush=True)


def head_ab(wl, stream, reps=10):
    """The step's head (the stencil head), the single-pass head, the two passes with fp32 and with
    bf16 G, each timed alone (CUDA events, after warm-up), and the largest differences from the
    single pass."""
    import torch
    out = {}
    for name, conv, y in (("stencil", wl.head, wl.head_y), ("fused", wl.head_fused, wl.head_fused_y),
                          ("split_f32", wl.head_split, wl.head_split_y), ("two_pass_bf16", wl.head2, wl.head2_y)):
        for _ in range(3):
            conv(wl.head_x, wl.head_c, out=y, stream=stream)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            conv(wl.head_x, wl.head_c, out=y, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        out[name + "_ms"] = e0.elapsed_time(e1) / reps
    out["max_abs_diff_stencil"] = float((wl.head_fused_y.float() - wl.head_y.float()).abs().max())
    out["max_abs_diff_split_f32"] = float((wl.head_fused_y.float() - wl.head_split_y.float()).abs().max())
    out["max_abs_diff_two_pass_bf16"] = float((wl.head_fused_y.float() - wl.head2_y.float()).abs().max())
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-memory", action="store_true", help="skip the pass-decoder peak-memory curve")
    ap.add_argument("--stage", choices=STAGES + AB_STAGES + SINGLE_STAGES, default=None,
                    help="run only this stage per step (for profiler captures); prints its per-launch time")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    import torch
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    barrier(world)
    import x3x3_convolution_gb300 as x3
    from x3x3_convolution_gb300 import dist as xd
    try:
        x3.load()
        loaded = True
    except Exception:
        loaded = False
    if not (xd.agree_all(loaded) if world > 1 else loaded):  # every rank runs the kernels, or none does
        raise RuntimeError("the CUDA library did not load on every rank")

    dev = f"cuda:{local}"
    wl = Workload(dev, seed_base=rank)
    stream = torch.cuda.current_stream()
    fl, nb = stage_cost()
    total_flop = sum(fl.values())

    if args.stage:
        run_stage(wl, args, stream, fl, nb)
        return
    for _ in range(args.warmup):
        wl.step(stream)
    torch.cuda.synchronize()
    st = x3.conv_device_status(1)
    if st != x3.X3_OK:
        raise RuntimeError(f"device status after warm-up: {st} {x3.conv_last_error()}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    torch.cuda.reset_peak_memory_stats()
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    if clocks.nvml is None:
        time.sleep(0.3)  # nvidia-smi needs a moment to start its 200 ms loop
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # the timed steps carry no events between their stages: an event between two launches would keep
    # the next stage's first kernel from starting early (programmatic dependent launch) as it does
    # inside a stage; the stage times come from a second run of the same steps with those events
    t0.record(stream)
    for k in range(args.steps):
        wl.step(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    step_peak = torch.cuda.max_memory_allocated()
    barrier(world)
    ms_per_step = reduce_max(world, t0.elapsed_time(t1)) / args.steps
    for k in range(args.steps):
        wl.step(stream, evs[k])
    torch.cuda.synchronize()
    stage_ms = {name: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs) for i, name in enumerate(STAGES)}
    ms_with_stage_events = statistics.mean(e[0].elapsed_time(e[len(STAGES)]) for e in evs)
    st = x3.conv_device_status(1)
    if st != x3.X3_OK:
        raise RuntimeError(f"device status after the timed steps: {st} {x3.conv_last_error()}")

    e2e = None
    if not args.no_e2e:
        # end to end through host buffers: every step copies each stage's input in from pinned host
        # memory and its output back out, inside the timed region. The copies run on their own
        # streams (one per direction) so that a stage's input transfer overlaps the previous stage's
        # kernels; events order each stage after its input and each buffer's reuse after its last
        # reader.
        hin = [t.cpu().pin_memory() for t in wl.inputs()]
        hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in wl.outputs()]
        h2d = sum(t.numel() * t.element_size() for t in hin)
        d2h = sum(t.numel() * t.element_size() for t in hout)
        din, dout = wl.inputs(), wl.outputs()
        copy_in, copy_out = torch.cuda.Stream(), torch.cuda.Stream()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        n_e2e = max(3, min(args.steps, 10))
        done_prev, out_prev = [None] * 4, [None] * 4
        barrier(world)
        e0.record(stream)
        copy_in.wait_stream(stream)
        copy_out.wait_stream(stream)
        for _ in range(n_e2e):
            ev_in = []
            for i in range(4):
                if done_prev[i] is not None:
                    copy_in.wait_event(done_prev[i])       # the previous step's stage i has read its input
                with torch.cuda.stream(copy_in):
                    din[i].copy_(hin[i], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_in)
                ev_in.append(ev)
            for i in range(4):
                stream.wait_event(ev_in[i])
                if out_prev[i] is not None:
                    stream.wait_event(out_prev[i])         # the previous step's output i is copied out
                wl.stage(i, stream)
                ev = torch.cuda.Event()
                ev.record(stream)
                done_prev[i] = ev
            for i in range(4):
                copy_out.wait_event(done_prev[i])
                with torch.cuda.stream(copy_out):
                    hout[i].copy_(dout[i], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_out)
                out_prev[i] = ev
        stream.wait_stream(copy_in)
        stream.wait_stream(copy_out)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(world, e0.elapsed_time(e1)) / n_e2e
        e2e = {"value": world * total_flop / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": n_e2e}

    ab = head_ab(wl, stream)
    peaks = load_peaks()
    # dominant kernel: the causal 128->128 tcgen05 implicit GEMM, launched twice per step by the stack
    # stage; its per-launch time is the stage time over 2 (the stage also holds the two 2-frame carry
    # copies, kernels that run beside the second half of each layer)
    launch_ms = stage_ms["stack"] / 2
    achieved = fl["stack"] / 2 / (launch_ms * 1e-3) / 1e12
    # the timed region lasts milliseconds (ms_per_step x steps), not the seconds under the power cap of
    # the sustained figure: the burst figure is the peak; the SM clock seen meanwhile is in `clocks`
    peak = peaks["bf16_tflops"]
    timed_ms = ms_per_step * args.steps
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                # dram__bytes_read.sum + dram__bytes_write.sum of one launch of this kernel, from an ncu
                # capture of that launch (algorithmic: 563.2 MB)
                "traffic": DRAM_BYTES["stack_128"],
                "kernel": "igemm_cl_kernel (channels-last, swapped operands, 128-byte swizzle) causal 128->128 @4+2x352x624",
                "peak_source": f"{peaks['source']} bf16_tflops (burst; the timed region lasts {timed_ms:.0f} ms)",
                "launch_ms": launch_ms, "sm_mhz_during": clk.get("sm_mhz"),
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
    stages = {}
    for k in STAGES:
        stages[k] = roof_entry(stage_ms[k], fl[k], nb[k], peaks, "inside the step")
    configs = {"taesd_chain_n4_256": dict(stages["taesd"], ms_per_image=stage_ms["taesd"] / 4,
                                          dram_bytes_ncu=DRAM_BYTES["taesd"]),
               "causal128_stack_4x352x624": dict(roof_entry(stage_ms["stack"] / 2, fl["stack"] / 2, nb["stack"] / 2,
                                                            peaks, "inside the step: stack stage / 2",
                                                            DRAM_BYTES["stack_128"], frames=FRAMES),
                                                 stack_ms_per_frame=stage_ms["stack"] / FRAMES),
               "causal256to128_4x176x312": roof_entry(stage_ms["l3"], fl["l3"], nb["l3"], peaks, "inside the step",
                                                      DRAM_BYTES["l3"], frames=FRAMES),
               "head_256to12_4x352x624": roof_entry(stage_ms["head"], fl["head"], nb["head"], peaks, "inside the step",
                                                    DRAM_BYTES["head"], frames=FRAMES)}
    configs.update(single_layer_configs(dev, stream, peaks))
    line = {
        "metric": METRIC, "value": world * total_flop / (ms_per_step * 1e-3) / 1e12, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16/f16 (fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (each step streams ~3 GB; no explicit flush)",
                   "frames_per_pass": FRAMES},
        "ms_per_step_with_stage_events": ms_with_stage_events,
        "decoder_ms_per_frame": (stage_ms["stack"] + stage_ms["l3"] + stage_ms["head"]) / FRAMES,
        "stages": stages, "configs": configs, "roofline": roofline, "gpu_launches": wl.kernels_per_step * args.steps,
        "clocks": clk, "e2e": e2e, "head_variants": ab,
        "plans": {k: (v if k != "taesd" else [p.get("kernel") for p in v]) for k, v in wl.plans.items()},
    }
    line["peak_memory"] = {"step_gib": step_peak / 2 ** 30,
                           "note": "torch.cuda.max_memory_allocated over the timed steps: every input, output, "
                                   "weight and workspace of the step's workload (plus the A/B head forms' weights)"}
    if not args.no_memory:
        line["peak_memory"]["pass_decoder"] = pass_memory_curve(wl, dev)
    if rank == 0 and not args.no_cpu_baseline:
        cb = cpu_baseline()
        line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
