#!/usr/bin/env python3
"""Benchmark of the DCN core op (forward + backward) on one or more GPUs.

A step is one pass of the whole op over one batch: the fused forward and the
backward (grad_input, grad_offset, grad_mask) at the FlashInternImage-T
stage-1 shape (N=64, 56x56, C=64, G=4, gc=16, 3x3, DCNv4 weights, float16
storage), on seeded synthetic inputs already resident in HBM.

  value     = ideal bytes of the step / device time of the step, in GB/s, over
              all ranks (each rank runs its own batch: weak scaling)
  ideal     = every tensor the op reads or writes, counted once
  e2e       = the same metric with the inputs copied from pinned host memory
              and every result copied back inside each timed step, steps
              streamed so that copies and compute overlap (the one-at-a-time
              figure beside it as "serial")
  roofline  = the dominant phase (the backward call) against the measured HBM
              copy bandwidth; the forward kernel's own roofline beside it
  images/s  = FlashInternImage-T core-op throughput: 64 images over the sum of
              depth x step time of the four stages
  cpu_baseline = the oracle (plain binary64 loops) on the host cores, on a
              bounded sample of the same workload
  projections = the layers around the core at the workload's shape, beside
              the step: the offset/mask and output projections (dcn_linear),
              the centre feature scale (forward and backward) and the offset
              branch's feature step (dcn_dwconv_ln_gelu, 5 x 5)

L2 is flushed (a write of twice its size) before every timed step, outside
the step's events.  ``--impl reference`` times the oracle alone, on the host.
Run under torchrun for N > 1 (one process per GPU).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from deformable_convolution_03_b300 import binding as B  # noqa: E402
from deformable_convolution_03_b300.replicas import (  # noqa: E402
    aggregate_gbs, max_over_ranks, rank_seed)
from deformable_convolution_03_b300.inputs import (  # noqa: E402
    DTYPES, T_DEPTHS, WORKLOADS, Workload, ideal_bytes, make_dwconv_inputs, make_inputs)

# The depthwise kernel of the offset branch's feature step (dw_kernel_size 5,
# page "没有CUDA内核也能跑：InternImage-G的DCNv3纯PyTorch回退实现逐行解读", section 一).
DW_KERNEL = 5

METRIC = "DCN core fwd/bwd GB/s and % of HBM roofline; images/s at FlashInternImage-T shapes"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6400.0

# DRAM traffic per call (dram__bytes_read.sum + dram__bytes_write.sum of the
# call's kernels in an ncu capture of `bench.py --profile-step --workload W`),
# keyed by phase and workload, with the sha1 of the kernel sources it was
# taken on (the kernels' and the planner's, with the switches' defaults): a
# changed source voids the figure.  The backward's memset of its
# float32 accumulator is not a kernel and is not counted.
FWD_SRCS = ("dcn_fwd_tma.cu", "dcn_fwd.cu", "dcn_common.cuh", "dcn_api.cu", "dcn_options.h")
BWD_SRCS = ("dcn_bwd_split.cu", "dcn_bwd.cu", "dcn_common.cuh", "dcn_api.cu", "dcn_options.h")
_F, _B = "194dd595571d", "8ef9c1baf1f9"
TRAFFIC = {
    "fwd@v3_tiny_f32": {"bytes": 60_160, "sha": _F},
    "bwd@v3_tiny_f32": {"bytes": 51_968, "sha": _B},
    "fwd@t_stage1_f16": {"bytes": 72_210_176, "sha": _F},
    "bwd@t_stage1_f16": {"bytes": 269_116_160, "sha": _B},
    "fwd@t_stage1_bf16": {"bytes": 72_225_024, "sha": _F},
    "bwd@t_stage1_bf16": {"bytes": 268_785_664, "sha": _B},
    "fwd@t_stage2_bf16": {"bytes": 34_699_008, "sha": _F},
    "bwd@t_stage2_bf16": {"bytes": 105_152_512, "sha": _B},
    "fwd@t_stage3_bf16": {"bytes": 17_317_120, "sha": _F},
    "bwd@t_stage3_bf16": {"bytes": 23_797_504, "sha": _B},
    "fwd@t_stage4_bf16": {"bytes": 8_687_104, "sha": _F},
    "bwd@t_stage4_bf16": {"bytes": 11_940_608, "sha": _B},
    "fwd@g_stage1_bf16": {"bytes": 66_867_456, "sha": _F},
    "bwd@g_stage1_bf16": {"bytes": 309_864_192, "sha": _B},
    "fwd@g_stage1_rc_bf16": {"bytes": 62_951_936, "sha": _F},
    "bwd@g_stage1_rc_bf16": {"bytes": 298_695_424, "sha": _B},
    "fwd@fb28_f32": {"bytes": 72_508_928, "sha": _F},
    "bwd@fb28_f32": {"bytes": 153_240_576, "sha": _B},
    "fwd@fb28_s2d2_f32": {"bytes": 35_062_272, "sha": _F},
    "bwd@fb28_s2d2_f32": {"bytes": 67_902_208, "sha": _B},
}


def src_sha(names) -> str:
    h = hashlib.sha1()
    for name in names:
        path = os.path.join(ROOT, "deformable_convolution_03_b300", "csrc", name)
        h.update(open(path, "rb").read())
    return h.hexdigest()[:12]


def traffic_for(key: str, srcs):
    rec = TRAFFIC.get(key)
    if not rec or rec["sha"] != src_sha(srcs):
        return None
    return rec["bytes"]


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(path))["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---- clocks during the timed region (NVML reads only) ------------------------

class ClockSampler:
    """SM clock and throttle reasons of the benchmarked GPU, sampled in a
    background thread while the timed steps run (reads only; the GPU is found
    by UUID, so the index NVML uses does not matter).  Falls back to
    nvidia-smi's query loop when NVML is unavailable."""
    REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "sw_power_cap": 0x4, "hw_power_brake_slowdown": 0x80}
    SMI = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
           "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
           "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev, period: float = 0.02):
        self.period = period
        self.samples, self.reasons = [], set()
        self.max_mhz, self.error, self.nv, self.proc = None, None, None, None
        self._stop = threading.Event()
        self._t = None
        self.uuid = None
        try:
            u = str(torch.cuda.get_device_properties(dev).uuid)
            self.uuid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception as e:  # pragma: no cover - depends on the torch build
            self.error = f"uuid: {e}"
        try:
            import pynvml
            pynvml.nvmlInit()
            self.h = pynvml.nvmlDeviceGetHandleByUUID(self.uuid)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.nv = pynvml
        except Exception as e:
            self.error = f"nvml: {e}"

    def _run(self):
        get_reasons = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
                r = get_reasons(self.h)
                for k, bit in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(k)
            except Exception as e:
                self.error = f"nvml sample: {e}"
            time.sleep(self.period)

    def __enter__(self):
        if self.nv is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        elif self.uuid:
            import subprocess
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.SMI}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            # the first sample marks that the query loop is running
            self.first = self.proc.stdout.readline()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t is not None:
            self._t.join()
        if self.proc is not None:
            self.proc.terminate()
            out, _ = self.proc.communicate()
            out = getattr(self, "first", "") + out
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for row in out.splitlines():
                f = [x.strip() for x in row.split(",")]
                if len(f) < 6:
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for name, v in zip(names, f[2:]):
                    if v.lower().startswith("active"):
                        self.reasons.add(name)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"],
                    "error": self.error}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


# ---- one workload on the device ----------------------------------------------

def merged_stride(P: int) -> int:
    """Row stride of the merged offset/mask tensor: 3P rounded up to 16 elements."""
    return (3 * P + 15) // 16 * 16


class Case:
    """Device tensors, outputs and workspace of one workload.  layout "merged"
    feeds offsets and masks as DCNv4's single offset/mask tensor."""

    def __init__(self, w: Workload, dev, rank: int = 0, layout: str = "separate"):
        self.w, self.dev, self.layout = w, dev, layout
        t = make_inputs(w, seed=rank_seed(w.seed, rank), grad=True)
        if layout == "merged":
            rs = self.stride = merged_stride(w.P)
            o, m = t.pop("offset"), t.pop("mask")
            pad = torch.zeros(o.shape[:4] + (rs - 3 * w.P,), dtype=o.dtype)
            t["offset_mask"] = torch.cat([o.flatten(-2), m, pad], -1).contiguous()
        self.host = t
        self.p = B.Params(dtype=B.TORCH_TO_DCN[DTYPES[w.dtype]], **w.params())
        self.x = {k: v.to(dev) for k, v in t.items()}
        self.out = torch.empty(w.N, w.H_out, w.W_out, w.C, dtype=DTYPES[w.dtype], device=dev)
        self.gi = torch.empty_like(self.x["input"])
        if layout == "merged":
            self.go = torch.empty_like(self.x["offset_mask"])
            self.gm = None
        else:
            self.go = torch.empty_like(self.x["offset"])
            self.gm = torch.empty_like(self.x["mask"])
        self.ws_bytes = B.dcn_core_bwd_workspace(self.p)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev)

    def fwd(self, x=None, res=None):
        x = x or self.x
        out = (res or self.results())[0]
        if self.layout == "merged":
            B.dcn_core_fwd_om(self.p, x["input"], x["offset_mask"], self.stride, out)
        else:
            B.dcn_core_fwd(self.p, x["input"], x["offset"], x["mask"], out)

    def bwd(self, x=None, res=None):
        x = x or self.x
        r = res or self.results()
        if self.layout == "merged":
            B.dcn_core_bwd_om(self.p, x["grad_out"], x["input"], x["offset_mask"], self.stride,
                              r[1], r[2], self.ws, self.ws_bytes)
        else:
            B.dcn_core_bwd(self.p, x["grad_out"], x["input"], x["offset"], x["mask"], r[1],
                           r[2], r[3], self.ws, self.ws_bytes)

    def results(self):
        """output, grad_input, grad_offset (or grad_offset_mask), grad_mask."""
        return [t for t in (self.out, self.gi, self.go, self.gm) if t is not None]

    def ideal(self) -> dict:
        """Ideal bytes; the merged tensor is counted with its padding."""
        ib = ideal_bytes(self.w)
        if self.layout == "merged":
            es = torch.empty((), dtype=DTYPES[self.w.dtype]).element_size()
            rows = self.w.N * self.w.H_out * self.w.W_out * self.w.G
            sep = rows * 3 * self.w.P * es
            mer = rows * self.stride * es
            ib = {"fwd": ib["fwd"] - sep + mer, "bwd": ib["bwd"] - 2 * sep + 2 * mer}
        return ib

    def launches_per_step(self) -> int:
        # forward kernel; backward kernel (both halves in one launch, or the
        # single-pass kernel for float32); the rounding kernel of 16-bit grad_input
        return 2 + (1 if self.ws_bytes else 0)


def timed_steps(case: Case, steps: int, flush, phases=("fwd", "bwd")):
    """Per-step, per-phase device times (ms), each step after an L2 flush
    (none when flush is None: the warm-cache reading)."""
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(phases) + 1)]
          for _ in range(steps)]
    for k in range(steps):
        if flush is not None:
            flush.zero_()
        ev[k][0].record()
        for j, ph in enumerate(phases):
            getattr(case, ph)()
            ev[k][j + 1].record()
    torch.cuda.synchronize()
    return {ph: [ev[k][j].elapsed_time(ev[k][j + 1]) for k in range(steps)]
            for j, ph in enumerate(phases)}


def e2e_steps(case: Case, steps: int, flush: torch.Tensor):
    """The step through host buffers, one at a time: pinned inputs in, the
    forward and backward, every result out, then the next step."""
    hin = {k: v.pin_memory() for k, v in case.host.items()}
    hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in case.results()]
    dev = {k: torch.empty_like(v) for k, v in case.x.items()}
    h2d = sum(v.numel() * v.element_size() for v in hin.values())
    d2h = sum(v.numel() * v.element_size() for v in hout)
    times = []
    for k in range(steps + 2):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for key in dev:
            dev[key].copy_(hin[key], non_blocking=True)
        case.fwd(dev)
        case.bwd(dev)
        for h, d in zip(hout, case.results()):
            h.copy_(d, non_blocking=True)
        b.record()
        b.synchronize()
        if k >= 2:
            times.append(a.elapsed_time(b))
    return times, h2d, d2h


def e2e_pipelined(case: Case, steps: int, flush: torch.Tensor) -> float:
    """The same steps streamed: every step still copies its inputs in from
    pinned host memory and all its results out, but on three streams with two
    device buffer sets, so that step k+1's inputs travel in and step k-1's
    results travel out while step k computes (the host link's two directions
    and the GPU work overlap).  L2 is flushed before each step's compute, on
    the compute stream.  Returns ms per step over all steps (device events
    from the first upload to the last download) and the last step's results
    as they arrived in host memory."""
    hin = {k: v.pin_memory() for k, v in case.host.items()}
    bufs = [{k: torch.empty_like(v) for k, v in case.x.items()} for _ in range(2)]
    res = [[torch.empty_like(t) for t in case.results()] for _ in range(2)]
    hout = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in case.results()]
            for _ in range(2)]
    s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    e_in = [ev() for _ in range(steps)]
    e_c = [ev() for _ in range(steps)]
    e_out = [ev() for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(s_in)
    for k in range(steps):
        j = k % 2
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(e_c[k - 2])        # buffer set j's inputs are consumed
            for key, d in bufs[j].items():
                d.copy_(hin[key], non_blocking=True)
            e_in[k].record(s_in)
        with torch.cuda.stream(s_c):
            s_c.wait_event(e_in[k])
            if k >= 2:
                s_c.wait_event(e_out[k - 2])       # result set j has been read out
            flush.zero_()
            case.fwd(bufs[j], res[j])
            case.bwd(bufs[j], res[j])
            e_c[k].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(e_c[k])
            for h, d in zip(hout[j], res[j]):
                h.copy_(d, non_blocking=True)
            e_out[k].record(s_out)
    end.record(s_out)
    end.synchronize()
    return start.elapsed_time(end) / steps, hout[(steps - 1) % 2]


def projections(w: Workload, dev, flush, reps: int, peak: float) -> dict:
    """The layers around the core at the workload's shape: DCNv4's merged
    offset/mask projection (C -> G x row stride, P = 9 rows padded to 32) and
    the output projection (C -> C) by dcn_linear, the centre feature scale's
    mix (dcn_center_feature_scale, forward and backward) and the offset
    branch's feature step (dcn_dwconv_ln_gelu), on synthetic inputs and
    weights, each timed alone with L2 flushed (outputs allocated beforehand,
    so that a call's host side stays shorter than the flush before it),
    against HBM on their ideal bytes (each tensor read or written once); and
    the forward with its
    projection in one launch (dcn_core_fwd_proj), and the forward with the
    centre feature scale in its epilogue (dcn_core_fwd_cfs), and the forward
    with the output projection in its epilogue (dcn_core_fwd_out), each beside
    the same work as separate launches."""
    dt = DTYPES[w.dtype]
    M, C = w.N * w.H_out * w.W_out, w.C
    rs = 32 if w.P == 9 else ((3 * w.P + 7) // 8) * 8
    g = torch.Generator().manual_seed(77)
    out = {}
    for name, n_out in (("offset_mask", w.G * rs), ("output_proj", C)):
        x = (torch.rand(M, C, generator=g) * 2 - 1).to(dt).to(dev)
        wt = (torch.randn(n_out, C, generator=g) / C ** 0.5).to(dt).to(dev)
        b = torch.randn(n_out, generator=g).to(dt).to(dev)
        y = torch.empty(M, n_out, dtype=dt, device=dev)
        ms = _time_alone(lambda: B.dcn_linear(x, wt, b, y), flush, reps)
        es = torch.empty(0, dtype=dt).element_size()
        ideal = (M * C + n_out * C + n_out + M * n_out) * es
        gbs = ideal / (ms * 1e-3) / 1e9
        out[name] = {"shape": f"{M}x{C} -> {n_out}", "ms": round(ms, 5), "GB/s": round(gbs, 1),
                     "frac_hbm": round(gbs / peak, 4), "ideal_bytes": ideal}
    # the centre feature scale: its gate logits (C -> G), then the mix of the
    # core's output with x_proj, forward and backward
    es = torch.empty(0, dtype=dt).element_size()
    core, xp, go = ((torch.rand(M, C, generator=g) * 2 - 1).to(dt).to(dev) for _ in range(3))
    lg = torch.randn(M, w.G, generator=g).to(dt).to(dev)
    o1, o2, o3 = (torch.empty_like(core) for _ in range(3))
    ol = torch.empty_like(lg)
    gates = {
        "cfs_forward": (lambda: B.dcn_center_feature_scale(core, xp, lg, o1, w.G),
                        (3 * M * C + M * w.G) * es),
        "cfs_backward": (lambda: B.dcn_center_feature_scale_bwd(go, core, xp, lg, o2, o3, ol, w.G),
                         (5 * M * C + 2 * M * w.G) * es),
    }
    for name, (fn, ideal) in gates.items():
        ms = _time_alone(fn, flush, reps)
        gbs = ideal / (ms * 1e-3) / 1e9
        out[name] = {"shape": f"{M}x{C}, {w.G} gates", "ms": round(ms, 5), "GB/s": round(gbs, 1),
                     "frac_hbm": round(gbs / peak, 4), "ideal_bytes": ideal}
    # the offset branch's feature step on the core's input: 5 x 5 depthwise
    # convolution, LayerNorm and GELU in one pass (x read once, x1 written once)
    t = make_dwconv_inputs(w.N, w.H, w.W, C, DW_KERNEL, w.dtype, seed=78)
    t = {key: v.to(dev) for key, v in t.items()}
    ideal = (2 * w.N * w.H * w.W * C + (DW_KERNEL ** 2 + 3) * C) * es
    x1 = torch.empty_like(t["x"])
    ms = _time_alone(lambda: B.dcn_dwconv_ln_gelu(t["x"], t["weight"], t["bias"], t["gamma"],
                                                  t["beta"], x1, 1e-6), flush, reps)
    gbs = ideal / (ms * 1e-3) / 1e9
    out["dwconv_ln_gelu"] = {"shape": f"{w.N}x{w.H}x{w.W}x{C}, k{DW_KERNEL}", "ms": round(ms, 5),
                             "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peak, 4),
                             "ideal_bytes": ideal}
    # the forward with DCNv4's merged offset/mask projection in its launch
    # (features of C channels, rows of rs), beside the same work as two
    # launches: the projection into the merged tensor, then the core on it
    if es == 2 and C % 64 == 0 and C <= 256:
        p = B.Params(dtype=B.TORCH_TO_DCN[dt], **w.params())
        inp = make_inputs(w)["input"].to(dev)
        feat = (torch.rand(w.N, w.H_out, w.W_out, C, generator=g) * 2 - 1).to(dt).to(dev)
        wt = (torch.randn(w.G * rs, C, generator=g) / C ** 0.5).to(dt).to(dev)
        bo = torch.randn(w.G * rs, generator=g).to(dt).to(dev)
        y = torch.empty(w.N, w.H_out, w.W_out, C, dtype=dt, device=dev)
        rows = torch.empty(w.N, w.H_out, w.W_out, w.G, rs, dtype=dt, device=dev)
        fused = _time_alone(lambda: B.dcn_core_fwd_proj(p, inp, feat, wt, bo, rs, y, None), flush,
                            reps)
        two = _time_alone(lambda: (B.dcn_linear(feat.reshape(-1, C), wt, bo,
                                                rows.reshape(-1, w.G * rs)),
                                   B.dcn_core_fwd_om(p, inp, rows, rs, y)), flush, reps)
        out["forward_with_projection"] = {
            "shape": f"{M}x{C} -> {w.G}x{rs} rows, then the core", "ms": round(fused, 5),
            "two_launches_ms": round(two, 5)}
    # the core forward with the centre feature scale (x_proj = the core's
    # input) in its epilogue, beside the core forward and the gate as two
    # launches; ideal bytes: the core's plus the logits'
    if w.H_out == w.H and w.W_out == w.W and w.stride_h == 1 and w.stride_w == 1:
        p = B.Params(dtype=B.TORCH_TO_DCN[dt], **w.params())
        t = {key: v.to(dev) for key, v in make_inputs(w).items()}
        lgu = torch.randn(w.N, w.H_out, w.W_out, w.G, generator=g).to(dt).to(dev)
        y = torch.empty(w.N, w.H_out, w.W_out, C, dtype=dt, device=dev)
        fused = _time_alone(lambda: B.dcn_core_fwd_cfs(p, t["input"], t["offset"], t["mask"], lgu,
                                                       y), flush, reps)
        two = _time_alone(lambda: (B.dcn_core_fwd(p, t["input"], t["offset"], t["mask"], y),
                                   B.dcn_center_feature_scale(y.reshape(M, C),
                                                              t["input"].reshape(M, C),
                                                              lgu.reshape(M, w.G), y.reshape(M, C),
                                                              w.G)), flush, reps)
        ideal = ideal_bytes(w)["fwd"] + M * w.G * es
        gbs = ideal / (fused * 1e-3) / 1e9
        out["forward_with_cfs"] = {"shape": f"{M} pixels x {w.G} gates, the core's workload",
                                   "ms": round(fused, 5), "two_launches_ms": round(two, 5),
                                   "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peak, 4),
                                   "ideal_bytes": ideal}
    # the core forward with the output projection (C -> C, then the bias) in
    # its epilogue, after the centre feature scale where the output keeps the
    # input's size, beside the same work as launches of their own (the core,
    # the gate, dcn_linear); ideal bytes: the core's with y for its output,
    # plus the weight, the bias and the logits
    if es == 2 and C == 64:
        p = B.Params(dtype=B.TORCH_TO_DCN[dt], **w.params())
        t = {key: v.to(dev) for key, v in make_inputs(w).items()}
        same = w.H_out == w.H and w.W_out == w.W and w.stride_h == 1 and w.stride_w == 1
        lgu = torch.randn(w.N, w.H_out, w.W_out, w.G, generator=g).to(dt).to(dev) if same else None
        wt = (torch.randn(C, C, generator=g) / C ** 0.5).to(dt).to(dev)
        bo = torch.randn(C, generator=g).to(dt).to(dev)
        core = torch.empty(w.N, w.H_out, w.W_out, C, dtype=dt, device=dev)
        y = torch.empty_like(core)
        fused = _time_alone(lambda: B.dcn_core_fwd_out(p, t["input"], t["offset"], t["mask"], lgu,
                                                       wt, bo, y), flush, reps)

        def two():
            if same:
                B.dcn_core_fwd_cfs(p, t["input"], t["offset"], t["mask"], lgu, core)
            else:
                B.dcn_core_fwd(p, t["input"], t["offset"], t["mask"], core)
            B.dcn_linear(core.reshape(M, C), wt, bo, y.reshape(M, C))

        sep = _time_alone(two, flush, reps)
        ideal = ideal_bytes(w)["fwd"] + (C * C + C + (M * w.G if same else 0)) * es
        gbs = ideal / (fused * 1e-3) / 1e9
        out["forward_with_output_projection"] = {
            "shape": f"{M} pixels, {C} -> {C}" + (f", {w.G} gates first" if same else ""),
            "ms": round(fused, 5), "two_launches_ms": round(sep, 5), "GB/s": round(gbs, 1),
            "frac_hbm": round(gbs / peak, 4), "ideal_bytes": ideal}
    return out


def _time_alone(fn, flush, reps: int) -> float:
    """Median ms of fn over reps calls, each after an L2 flush, by CUDA events on
    the current stream (three untimed calls first).  All reps are queued before
    one synchronisation, as the timed steps are, so that the device always has
    the next flush and call waiting and a slow host moment is not timed."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for e0, e1 in ev:
        flush.zero_()
        e0.record()
        fn()
        e1.record()
    torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)


def images_per_s(dev, flush, reps: int):
    """FlashInternImage-T core op: 64 images / sum_i depth_i * t_i (fwd, fwd+bwd)."""
    per_stage = []
    for i, depth in enumerate(T_DEPTHS, start=1):
        w = WORKLOADS[f"t_stage{i}_bf16"]
        c = Case(w, dev)
        for _ in range(3):
            c.fwd()
            c.bwd()
        t = timed_steps(c, reps, flush)
        per_stage.append((depth, statistics.median(t["fwd"]), statistics.median(t["bwd"])))
        del c
    fwd_s = sum(d * f for d, f, _ in per_stage) / 1e3
    step_s = sum(d * (f + b) for d, f, b in per_stage) / 1e3
    return {"fwd": 64 / fwd_s, "fwd_bwd": 64 / step_s,
            "stages_ms": [{"depth": d, "fwd": round(f, 5), "bwd": round(b, 5)}
                          for d, f, b in per_stage]}


# ---- the oracle on the host --------------------------------------------------

class OracleTimer:
    """The oracle's forward + backward on a seeded random sample of output
    pixels of the workload (all of their groups, points and channels).  The
    throughput is scaled to the metric's unit by the fraction of output pixels
    processed: ideal bytes x (sample / all pixels) / time."""

    def __init__(self, w: Workload):
        import numpy as np
        import oracle
        oracle.build()
        self.o, self.w = oracle, w
        t = make_inputs(w, grad=True)
        self.f = {k: v.to(torch.float64).numpy() for k, v in t.items()}
        self.q = oracle.Params(coord_f32=1, **w.params())
        self.total = w.N * w.H_out * w.W_out
        self.perm = np.random.default_rng(1234).permutation(self.total)
        ib = ideal_bytes(w)
        self.step_bytes = ib["fwd"] + ib["bwd"]
        self.cores = self.all_cores = oracle.max_threads()

    def set_cores(self, n: int) -> None:
        self.o.set_threads(n)
        self.cores = n

    def run(self, npix: int) -> float:
        pix = self.perm[:npix]
        f = self.f
        t0 = time.perf_counter()
        self.o.forward_pixels(self.q, f["input"], f["offset"], f["mask"], pix)
        self.o.backward_pixels(self.q, f["grad_out"], f["input"], f["offset"], f["mask"], pix)
        return time.perf_counter() - t0

    def size_for(self, seconds: float) -> int:
        n = min(self.total, 64)
        dt = self.run(n)
        while dt < 0.2 and n < self.total:
            n = min(self.total, n * 4)
            dt = self.run(n)
        return int(max(16, min(self.total, n * seconds / max(dt, 1e-6))))

    def gbs(self, npix: int, seconds: float) -> float:
        return self.step_bytes * npix / self.total / seconds / 1e9

    def describe(self, npix: int, seconds: float) -> str:
        return (f"forward+backward of {npix} random output pixels of {self.total} "
                f"({100.0 * npix / self.total:.2f}% of {self.w.name}) in {seconds:.2f} s, "
                f"{self.cores} threads")


def run_reference(args, rank, world):
    """The reference arm: the oracle on the host cores, same metric and workload;
    each step a bounded sample sized so that all steps end within minutes."""
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    ot = OracleTimer(w)
    per_step = max(0.01, min(args.ref_budget, 150.0 / (args.steps + args.warmup)))
    npix = ot.size_for(per_step)
    times = []
    for k in range(args.warmup + args.steps):
        dt = ot.run(npix)
        if k >= args.warmup:
            times.append(dt)
    total_t = sum(times)
    value = ot.gbs(npix * len(times), total_t)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ot.step_bytes / (value * 1e9) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {**config_of(w, args.gpus), "layout": args.layout},
        "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": ot.cores,
                         "kind": "oracle",
                         "sample": "each step: " + ot.describe(npix, total_t / len(times))},
        "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def profile_step(w: Workload, dev, layout: str) -> int:
    """One step of the workload bracketed for a profiler started with
    --profile-from-start off (after two warm-up steps)."""
    case = Case(w, dev, 0, layout)
    for _ in range(2):
        case.fwd()
        case.bwd()
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    case.fwd()
    case.bwd()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    return 0


def profile_proj(dev) -> int:
    """The layers around the core, one call each bracketed for a profiler:
    FlashInternImage-T stage 1's merged offset/mask projection (200704 x 64 ->
    128) and output projection (-> 64) in float16, InternImage-G stage 1's
    512 -> 512 projection (32768 rows) in bfloat16, and the centre feature
    scale forward and backward at stage 1 (200704 x 64, 4 gates, float16), and
    the offset branch's feature step (5 x 5 depthwise convolution, LayerNorm,
    GELU) at T stage 1 (64 x 56 x 56 x 64, float16) and G stage 1
    (2 x 128 x 128 x 512, bfloat16), and at T stage 1 in float16 the forward
    with its offset/mask projection in one launch (64 -> 4 x 32 rows), with the
    centre feature scale in its epilogue, and with the gate and the output
    projection (64 -> 64) in its epilogue."""
    g = torch.Generator().manual_seed(1)
    calls = []
    for M, K, N, dt in ((200704, 64, 128, torch.float16), (200704, 64, 64, torch.float16),
                        (32768, 512, 512, torch.bfloat16)):
        x = (torch.rand(M, K, generator=g) * 2 - 1).to(dt).to(dev)
        wt = (torch.randn(N, K, generator=g) / K ** 0.5).to(dt).to(dev)
        b = torch.randn(N, generator=g).to(dt).to(dev)
        calls.append(lambda x=x, wt=wt, b=b: B.linear(x, wt, b))
    M, C, G = 200704, 64, 4
    core, xp, go = ((torch.rand(M, C, generator=g) * 2 - 1).half().to(dev) for _ in range(3))
    lg = torch.randn(M, G, generator=g).half().to(dev)
    calls.append(lambda: B.center_feature_scale(core, xp, lg))
    calls.append(lambda: B.center_feature_scale_backward(go, core, xp, lg))
    for N, H, C, dt in ((64, 56, 64, "f16"), (2, 128, 512, "bf16")):
        t = {key: v.to(dev) for key, v in
             make_dwconv_inputs(N, H, H, C, DW_KERNEL, dt, seed=2).items()}
        calls.append(lambda t=t: B.dwconv_ln_gelu(t["x"], t["weight"], t["bias"], t["gamma"],
                                                  t["beta"]))
    # the forward with its offset/mask projection in one launch, stage 1
    w = WORKLOADS["t_stage1_f16"]
    p = B.Params(dtype=B.DCN_F16, **w.params())
    inp = make_inputs(w)["input"].to(dev)
    feat = (torch.rand(w.N, w.H_out, w.W_out, 64, generator=g) * 2 - 1).half().to(dev)
    wt = (torch.randn(w.G * 32, 64, generator=g) / 8).half().to(dev)
    bo = torch.randn(w.G * 32, generator=g).half().to(dev)
    y = torch.empty(w.N, w.H_out, w.W_out, w.C, dtype=torch.float16, device=dev)
    calls.append(lambda: B.dcn_core_fwd_proj(p, inp, feat, wt, bo, 32, y, None))
    # the forward with the centre feature scale in its epilogue, and with the
    # gate and then the output projection (64 -> 64) in its epilogue, stage 1
    t = {key: v.to(dev) for key, v in make_inputs(w).items()}
    lgu = torch.randn(w.N, w.H_out, w.W_out, w.G, generator=g).half().to(dev)
    wo = (torch.randn(64, 64, generator=g) / 8).half().to(dev)
    bw = torch.randn(64, generator=g).half().to(dev)
    yc = torch.empty_like(y)
    yo = torch.empty_like(y)
    calls.append(lambda: B.dcn_core_fwd_cfs(p, t["input"], t["offset"], t["mask"], lgu, yc))
    calls.append(lambda: B.dcn_core_fwd_out(p, t["input"], t["offset"], t["mask"], lgu, wo, bw,
                                            yo))
    for f in calls:
        f()
        f()
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    for f in calls:
        f()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    return 0


def config_of(w: Workload, n: int) -> dict:
    return {"workload": w.name,
            "shape": f"N={w.N} H=W={w.H} C={w.C} G={w.G} gc={w.gc} k{w.kernel_h}x{w.kernel_w} "
                     f"s{w.stride_h} p{w.pad_h} d{w.dilation_h} P={w.P}",
            "op": "DCNv3 (softmax)" if w.softmax else "DCNv4 (raw mask)",
            "step": "forward + backward (grad_input, grad_offset, grad_mask)",
            "storage": w.dtype, "accumulate": "f32",
            "global_batch": w.N * n, "per_gpu_batch": w.N, "parallelism": f"replicas x{n}",
            "inputs": f"input U(-1,1), offsets N(0,{w.offset_std}) px, mask N(0,1), grad N(0,1)",
            "l2": "flushed before every timed step (write of 2x L2)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="t_stage1_f16")
    ap.add_argument("--layout", default="separate", choices=["separate", "merged"],
                    help="offsets and masks as two tensors, or as DCNv4's one offset/mask tensor")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle timing")
    ap.add_argument("--no-stages", action="store_true", help="skip the T-stage images/s sweep")
    ap.add_argument("--no-proj", action="store_true",
                    help="skip the projections around the core (dcn_linear)")
    ap.add_argument("--profile-step", action="store_true",
                    help="for a profiler: two warm-up steps, then one step (forward + backward) "
                         "between cudaProfilerStart and cudaProfilerStop; no timing")
    ap.add_argument("--profile-proj", action="store_true",
                    help="for a profiler: the projections and the centre feature scale around the "
                         "core, two warm-up calls each, then one call each between "
                         "cudaProfilerStart and cudaProfilerStop")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=8.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    w = WORKLOADS[args.workload]
    if args.profile_step:
        return profile_step(w.with_(backward=True), dev, args.layout)
    if args.profile_proj:
        return profile_proj(dev)
    case = Case(w, dev, rank, args.layout)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)

    for _ in range(args.warmup):
        flush.zero_()
        case.fwd()
        case.bwd()
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    wall0 = time.perf_counter()
    with ClockSampler(dev) as clk:
        t = timed_steps(case, args.steps, flush)
    barrier()
    wall = time.perf_counter() - wall0

    fwd_ms = statistics.mean(t["fwd"])
    bwd_ms = statistics.mean(t["bwd"])
    step_ms, fwd_ms, bwd_ms = max_over_ranks([fwd_ms + bwd_ms, fwd_ms, bwd_ms], dist, dev)

    # secondary reading after the timed region: the same steps without the
    # flush, so that what the previous step left in L2 is reused
    warm_steps = min(args.steps, 200)
    tw = timed_steps(case, warm_steps, None)
    warm = {"fwd_median": round(statistics.median(tw["fwd"]), 5),
            "bwd_median": round(statistics.median(tw["bwd"]), 5), "steps": warm_steps,
            "how": "no L2 flush between steps (secondary; the headline flushes)"}

    ib = case.ideal()
    step_bytes = ib["fwd"] + ib["bwd"]
    value = aggregate_gbs(step_bytes, world, step_ms)

    # end to end through host buffers
    e2e = None
    if args.e2e_steps > 0:
        e2e_t, h2d, d2h = e2e_steps(case, args.e2e_steps, flush)
        serial_ms = max_over_ranks([statistics.median(e2e_t)], dist, dev)[0]
        e2e_pipelined(case, 3, flush)  # warm-up: streams, pinned buffers
        pipe_ms = max_over_ranks([e2e_pipelined(case, args.e2e_steps, flush)[0]], dist, dev)[0]
        e2e = {"value": round(aggregate_gbs(step_bytes, world, pipe_ms), 3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(pipe_ms, 4),
               "how": "every step copies its inputs in from pinned host memory and every result "
                      "out; steps streamed over three streams with two device buffer sets, so a "
                      "step's compute overlaps the next step's upload and the previous step's "
                      "download; L2 flushed before each step's compute",
               "serial": {"value": round(aggregate_gbs(step_bytes, world, serial_ms), 3),
                          "ms_per_step": round(serial_ms, 4),
                          "how": "one step at a time: upload, compute, download, then the next"}}

    peak, peak_kind = hbm_peak()
    fwd_gbs = ib["fwd"] / (fwd_ms * 1e-3) / 1e9
    bwd_gbs = ib["bwd"] / (bwd_ms * 1e-3) / 1e9
    dominant = "bwd" if bwd_ms >= fwd_ms else "fwd"
    roof = {
        "bwd": {"bound": "hbm", "achieved": round(bwd_gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(bwd_gbs / peak, 4),
                "traffic": traffic_for(f"bwd@{w.name}", BWD_SRCS) if args.layout == "separate" else None,
                "phase": "dcn_core_bwd: workspace memset + bwd_both_kernel + round_kernel",
                "ms": round(bwd_ms, 5), "peak_source": f"{peak_kind} HBM copy bandwidth"},
        "fwd": {"bound": "hbm", "achieved": round(fwd_gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(fwd_gbs / peak, 4),
                "traffic": traffic_for(f"fwd@{w.name}", FWD_SRCS) if args.layout == "separate" else None,
                "phase": "dcn_core_fwd: fwd_tile_kernel (TMA-staged)", "ms": round(fwd_ms, 5),
                "peak_source": f"{peak_kind} HBM copy bandwidth"},
    }

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {**config_of(w, world), "layout": args.layout},
        "roofline": {**roof[dominant], "kernel": dominant},
        "roofline_fwd": roof["fwd"],
        "phases_ms": {"fwd": round(fwd_ms, 5), "bwd": round(bwd_ms, 5),
                      "fwd_median": round(statistics.median(t["fwd"]), 5),
                      "bwd_median": round(statistics.median(t["bwd"]), 5),
                      "fwd_min": round(min(t["fwd"]), 5), "bwd_min": round(min(t["bwd"]), 5),
                      "warm_l2": warm},
        "ideal_bytes": {"fwd": ib["fwd"], "bwd": ib["bwd"]},
        "e2e": e2e,
        "gpu_launches": args.steps * case.launches_per_step(),
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 3),
    }
    if rank == 0 and not args.no_proj:
        line["projections"] = projections(w, dev, flush, reps=200, peak=peak)
    if rank == 0 and not args.no_stages:
        line["images_per_s"] = images_per_s(dev, flush, reps=200)
    if rank == 0 and world == 1 and not args.no_cpu:
        ot = OracleTimer(w)
        npix = ot.size_for(args.cpu_budget)
        dt = ot.run(npix)
        line["cpu_baseline"] = {"value": round(ot.gbs(npix, dt), 5), "unit": UNIT,
                                "cores": ot.cores, "kind": "oracle",
                                "sample": ot.describe(npix, dt),
                                "nproc": os.cpu_count()}
        # the same oracle on one core, on a sample sized for the same budget
        ot.set_cores(1)
        n1 = ot.size_for(args.cpu_budget / 2)
        dt1 = ot.run(n1)
        line["cpu_baseline"]["one_core"] = {"value": round(ot.gbs(n1, dt1), 5), "unit": UNIT,
                                            "cores": 1, "sample": ot.describe(n1, dt1)}
        ot.set_cores(ot.all_cores)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
