"""Benchmark of one MoE prefill layer (quantize-scatter -> group gather -> grouped
MMQ gate/up -> hidden re-quantization -> grouped MMQ down -> top-k combine) on
GB300, through the library's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Prints one JSON line.  A step is one whole layer over the T=8192 workload
(d=2048, f=768, E=512, K=10, Q8_0 weights, Zipf-skewed routing) by default.
Inputs are resident in HBM when the timed region starts; L2 is flushed by a
512 MB write between steps (outside the per-step CUDA events).  Per-stage CUDA
events give the phase table, the quantizer GB/s and the dominant kernel's
roofline.  ``e2e`` repeats the measurement through ``MoeLayer.forward_host``
with every step's inputs copied from pinned host memory and its output read
back inside the timed region (steps queued back to back, each one's copies
overlapping its neighbours' layers; also reported: each call waited for, and
the copies in line on one stream).
``--impl reference`` times the CPU oracle (single thread, host cores) on a
bounded token sample of the same workload instead.
Under torchrun each rank runs its own replica (weak scaling, no collective on
the data path); the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_workloads as mw  # noqa: E402

METRIC = "MoE prefill layer tokens/s at T=8192 (1 GB300) + % roofline; quantize GB/s"
DEFAULT_CONFIG = mw.T8192.name
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """SM clock and clock-event reasons sampled every 5 ms through NVML (the
    driver's libnvidia-ml, via ctypes) while the timed region runs; falls back
    to nvidia-smi (200 ms) when NVML cannot be loaded."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, pci_bus_id: str | None = None):
        self.index = index
        self.pci = pci_bus_id
        self.samples = []
        self.max_mhz = 0.0
        self.reasons = set()
        self._stop = None
        self._thread = None
        self._smi = None

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        rc = 1
        if self.pci:  # the device this process uses, whatever CUDA_VISIBLE_DEVICES says
            rc = lib.nvmlDeviceGetHandleByPciBusId_v2(self.pci.encode(), ctypes.byref(h))
        if rc != 0 and lib.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return lib, h, fn

    def start(self):
        import ctypes
        import threading
        try:
            lib, h, reasons_fn = self._nvml()
        except (OSError, AttributeError):
            self._start_smi()
            return
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1 = NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        self._stop = threading.Event()

        def loop():
            clk = ctypes.c_uint()
            rs = ctypes.c_ulonglong()
            while not self._stop.is_set():
                if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                    self.samples.append(float(clk.value))
                if reasons_fn(h, ctypes.byref(rs)) == 0:
                    for bit, name in self.REASONS.items():
                        if rs.value & bit:
                            self.reasons.add(name)
                self._stop.wait(0.005)

        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()

    def _start_smi(self):
        self.path = os.path.join("/tmp", f"moe_bench_clocks_{os.getpid()}.csv")
        fields = ("index,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.fh = open(self.path, "w")
            self._smi = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={fields}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except OSError:
            self._smi = None

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=2)
            src = "nvml"
        elif self._smi is not None:
            self._smi.terminate()
            try:
                self._smi.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._smi.kill()
            self.fh.close()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            with open(self.path) as fh:
                for line in fh:
                    parts = [p.strip() for p in line.split(",")]
                    try:
                        self.samples.append(float(parts[1]))
                        self.max_mhz = max(self.max_mhz, float(parts[2]))
                    except (ValueError, IndexError):
                        continue
                    for n, v in zip(names, parts[3:7]):
                        if v.lower() == "active":
                            self.reasons.add(n)
            os.unlink(self.path)
            src = "nvidia-smi"
        else:
            return None
        if not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples), "source": src}


def pci_bus_id(dev):
    import torch
    p = torch.cuda.get_device_properties(dev)
    try:
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except AttributeError:
        return None


# ------------------------------------------------------------ bytes / ops --

# FP32 operations per block-scale partial in the MMQ epilogue: fma(dW*dX, I, acc)
# is a multiply and an FMA; Q4_1 adds fma(mW, sX, acc), Q2_K two such FMAs (one
# per 16-value half).
ALU_OPS_PER_PARTIAL = {0: 2, 1: 3, 2: 2, 3: 4}  # by weight type (Q8_0, Q4_1, Q2_0, Q2_K)
FP32_LANES_PER_SM = 128
MAX_SM_MHZ = 2070.0  # GB300 maximum SM clock


def alu_peak_ops(sms: int, mhz: float = MAX_SM_MHZ) -> float:
    """FP32 operations per second, an FMA counted as one operation: SMs x 128
    lanes x clock."""
    return sms * FP32_LANES_PER_SM * mhz * 1e6


def layer_accounting(cfg, n_active: int, rec_bytes: int, R: int):
    """Per stage (bytes, flops): the algorithmic bytes each stage must move (every
    tensor read or written once) and, for the two MMQ stages, the flops of their
    block dots (2 per multiply-add of routed rows only).  Also the layer's total
    algorithmic bytes and ops."""
    T, d, f, K = cfg.T, cfg.d, cfg.f, cfg.K
    # bytes per q8_1 value: int8 plus (d, s) fp16 per 32, or (d, s, s_lo, s_hi) (D2S6, Q2_K)
    q8 = 1.25 if cfg.wtype == mw.Q2_K else 1.125
    w_gu = n_active * rec_bytes * 2.0 / 3.0  # gate and up matrices of the routed experts
    w_dn = n_active * rec_bytes / 3.0
    stages = {
        "slot_map": (T * K * 4 * 4, 0.0),
        "quantize_scatter": (T * d * 4 + R * d * q8 + T * K * 4, 0.0),
        "group_gather": (2 * n_active * rec_bytes, 0.0),
        "mmq_gateup": (R * d * q8 + w_gu + R * f * 4, 2.0 * R * 2 * f * d),
        "requant_hidden": (R * f * 4 + R * f * q8, 0.0),
        "mmq_down": (R * f * q8 + w_dn + R * d * 4, 2.0 * R * d * f),
        "combine_topk": (R * d * 4 + T * d * 4 + T * K * 8, 0.0),
    }
    total_bytes = (T * d * 4 + 2 * R * d * q8 + 2 * R * f * 4 + 2 * R * f * q8 + 2 * R * d * 4
                   + T * d * 4 + 6 * R * 4 + 3 * n_active * rec_bytes)
    ops = 2.0 * R * 3 * f * d
    return stages, total_bytes, ops


def stage_roofline(bytes_, flops, sec, hbm_gbs, tensor_tflops, peak_src):
    """The roofline of one kernel: the slower of its algorithmic bytes at the
    measured HBM copy rate and its flops at the measured bf16 tensor rate (the
    fp16 MMA these kernels issue runs at the bf16 rate); achieved and peak in
    that bound's unit; frac = roofline time / event time."""
    t_hbm = bytes_ / (hbm_gbs * 1e9)
    t_tc = flops / (tensor_tflops * 1e12) if flops else 0.0
    if t_tc > t_hbm:
        return {"bound": "tensor", "achieved": round(flops / sec / 1e12, 2),
                "peak": round(tensor_tflops, 1), "unit": "TFLOP/s", "frac": round(t_tc / sec, 4),
                "algorithmic_flops": flops, "algorithmic_bytes": int(bytes_),
                "peak_source": f"{peak_src} bf16 (burst)"}
    return {"bound": "hbm", "achieved": round(bytes_ / sec / 1e9, 1), "peak": round(hbm_gbs, 1),
            "unit": "GB/s", "frac": round(t_hbm / sec, 4), "algorithmic_bytes": int(bytes_),
            **({"algorithmic_flops": flops} if flops else {}),
            "peak_source": f"{peak_src} copy"}


def mmq_tensor_flops(cfg, R: int, stage: str) -> float:
    """Flops of the integer block dots of an MMQ stage (2 per multiply-add)."""
    return 2.0 * R * (2 * cfg.f * cfg.d if stage == "mmq_gateup" else cfg.d * cfg.f)


def alu_partials(cfg, R: int) -> float:
    """Block-scale partials of the layer: one per output element per 32-block."""
    return R * 2.0 * cfg.f * (cfg.d // 32) + R * 1.0 * cfg.d * (cfg.f // 32)


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of a
# stage's main kernel, from one ncu capture (summaries under profiles/), valid
# only while the kernel's code is the code that was profiled: "code_sha256_16"
# hashes the source with its comments and blank lines removed (code_digest), so
# a comment edit keeps the figure and any code change drops it.
PROFILED_TRAFFIC = {
    ("mmq_gateup", "T8192_d2048_f768_E512_K10_q8_0_zipf"): {
        "source": "quantized_routed_expert_q8_gb300/csrc/mmq_tc.cu",
        "code_sha256_16": "a3765f4cd7855d9f", "bytes": 609651200 + 254658304},
    ("mmq_down", "T8192_d2048_f768_E512_K10_q8_0_zipf"): {
        "source": "quantized_routed_expert_q8_gb300/csrc/mmq_fold.cu",
        "code_sha256_16": "3426d9a626cde64a", "bytes": 275820544 + 666888704},
    ("quantize_scatter", "T32768_d2048_f768_E512_K10_q4_1"): {
        "source": "quantized_routed_expert_q8_gb300/csrc/quantize.cu",
        "code_sha256_16": "217e4c4ac0275670", "bytes": 270006272 + 694668800},
    ("requant_hidden", "T8192_d2048_f768_E512_K10_q8_0_zipf"): {
        "source": "quantized_routed_expert_q8_gb300/csrc/quantize.cu",
        "code_sha256_16": "217e4c4ac0275670", "bytes": 251683584 + 14620672},
}


def code_digest(text: str) -> str:
    """sha256 prefix of C/CUDA source without comments and blank lines."""
    import hashlib
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def profiled_traffic(stage: str, workload: str):
    rec = PROFILED_TRAFFIC.get((stage, workload))
    if not rec:
        return None
    try:
        digest = code_digest(open(os.path.join(ROOT, rec["source"])).read())
    except OSError:
        return None
    return rec["bytes"] if rec["code_sha256_16"] == digest else None


# ------------------------------------------------------------ multi-rank --

def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The slowest rank's time is the job's time: all-reduce MAX of a per-rank
    scalar (a no-op on one rank)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank runs its own replica of the workload."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


# -------------------------------------------------------------- GPU arm --

def run_gpu(args, rank, world, local_rank):
    import torch

    import quantized_routed_expert_q8_gb300 as m

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg = mw.CONFIGS[args.config]
    wl = mw.make_workload(cfg)
    T, K, E, d, f = cfg.T, cfg.K, cfg.E, cfg.d, cfg.f
    R = T * K
    arena = torch.from_numpy(wl.arena).to(dev)
    x = torch.from_numpy(wl.x).to(dev)
    ids = torch.from_numpy(wl.ids).to(dev)
    w = torch.from_numpy(wl.w).to(dev)
    layer = m.MoeLayer(cfg.wtype, E, d, f, K, T, arena, wl.rec_bytes, wl.arena_stride, dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    stage_names = ["slot_map", "quantize_scatter", "group_gather", "mmq_gateup",
                   "requant_hidden", "mmq_down", "combine_topk"]
    q_scatter, q_gather, q_requant = m.quantizers(cfg.wtype)

    def step(evs=None):
        L = layer
        calls = [
            lambda: m.moe_build_slot_map(ids, E, L.offsets, L.slot, L.src, L.active, L.n_active,
                                         L.ws),
            lambda: q_scatter(x, L.slot, K, R, L.q, L.ds),
            lambda: m.moe_group_gather_active(L.arena, L.rec_bytes, L.arena_stride, L.active,
                                              L.n_active, E, L.group_buf, L.slot_stride),
            lambda: m.moe_grouped_mmq_gateup(L.wtype, L.group_buf, L.slot_stride, L.active,
                                             L.n_active, L.offsets, E, L.q, L.ds, R, d, f, L.h,
                                             L.ws),
            lambda: q_requant(L.h, R, f, L.hq, L.hds),
            lambda: m.moe_grouped_mmq_down(L.wtype, L.group_buf, L.slot_stride, L.active,
                                           L.n_active, L.offsets, E, L.hq, L.hds, R, d, f, L.y,
                                           L.ws),
            lambda: m.moe_combine_topk(L.y, R, L.slot, w, T, K, d, L.out),
        ]
        for i, c in enumerate(calls):
            if evs is not None:
                evs[i].record(stream)
            c()
        if evs is not None:
            evs[len(calls)].record(stream)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize(dev)
    assert m.moe_device_error(layer.ws) == 0
    n_active = int(layer.n_active.item())

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank, pci_bus_id(dev)) if rank == 0 else None
    if sampler:
        sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = m.moe_launch_count()
    t_wall = time.perf_counter()
    for s in range(args.steps):
        flush.fill_(s & 0xFF)
        step(events[s])
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    launches = m.moe_launch_count() - launches0
    clocks = sampler.stop() if sampler else None
    stage_ms = np.array([[ev[i].elapsed_time(ev[i + 1]) for i in range(7)] for ev in events])
    step_ms = stage_ms.sum(axis=1)
    ms = max_over_ranks(float(step_ms.mean()), dist, dev)

    # end to end through the public API: pinned host inputs in, output out
    hx = torch.from_numpy(wl.x).pin_memory()
    hids = torch.from_numpy(wl.ids).pin_memory()
    hw = torch.from_numpy(wl.w).pin_memory()
    hout = torch.empty((T, d), dtype=torch.float32).pin_memory()
    dx = torch.empty_like(x)
    dids = torch.empty_like(ids)
    dw = torch.empty_like(w)

    def e2e_serial():
        # the copies in line with the layer on one stream
        dx.copy_(hx, non_blocking=True)
        dids.copy_(hids, non_blocking=True)
        dw.copy_(hw, non_blocking=True)
        out = layer.forward(dx, dids, dw)
        hout.copy_(out, non_blocking=True)

    def e2e_overlapped():
        # MoeLayer.forward_host: x copied in token slices while the routing map
        # and the gather run, out copied back per combined slice; the stream
        # waits for the copies back
        layer.forward_host(hx, hids, hw, hout)

    def time_e2e_pipelined():
        # forward_host calls back to back (wait=False): one call's copies overlap
        # the neighbouring calls' layers; every call still uploads its inputs and
        # downloads its output, and the timed region ends when the last
        # download has landed.  The L2 flush before each call runs on the layer's
        # stream inside the region, bracketed by its own events; its duration is
        # taken out, as the per-stage events leave it out of the device time.
        for _ in range(max(1, args.warmup)):
            layer.forward_host(hx, hids, hw, hout, wait=False)
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        fl = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        a.record(stream)
        for s in range(args.steps):
            fl[s][0].record(stream)
            flush.fill_(s & 0xFF)
            fl[s][1].record(stream)
            last = layer.forward_host(hx, hids, hw, hout, wait=False)
        stream.wait_event(last)
        b.record(stream)
        torch.cuda.synchronize(dev)
        flush_ms = sum(f0.elapsed_time(f1) for f0, f1 in fl)
        return max_over_ranks((a.elapsed_time(b) - flush_ms) / args.steps, dist, dev)

    def time_e2e(fn):
        for _ in range(max(1, args.warmup)):
            fn()
        torch.cuda.synchronize(dev)
        times = []
        for s in range(args.steps):
            flush.fill_(s & 0xFF)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b))
        return max_over_ranks(float(np.mean(times)), dist, dev)

    e2e_serial_ms = time_e2e(e2e_serial)
    ref_out = hout.clone()
    e2e_call_ms = time_e2e(e2e_overlapped)
    e2e_same = bool(torch.equal(hout, ref_out))
    hout.fill_(float("nan"))
    e2e_ms = time_e2e_pipelined()
    e2e_same = e2e_same and bool(torch.equal(hout, ref_out))
    assert m.moe_device_error(layer.ws) == 0

    if rank != 0:
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return None

    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tc = float(peaks["bf16_tflops"])  # burst: every kernel here runs well under a second
    stages, total_bytes, ops = layer_accounting(cfg, n_active, wl.rec_bytes, R)
    mean_stage = stage_ms.mean(axis=0)
    phases = {n: round(float(v), 4) for n, v in zip(stage_names, mean_stage)}
    stage_roof = {n: dict(ms=round(float(v), 4),
                          **stage_roofline(*stages[n], float(v) / 1e3, hbm, tc, peak_src),
                          traffic=profiled_traffic(n, cfg.name))
                  for n, v in zip(stage_names, mean_stage)}
    dom = int(np.argmax(mean_stage))
    dom_name = stage_names[dom]
    roof = {k: v for k, v in stage_roof[dom_name].items() if k not in ("ms", "traffic")}
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    alu_peak = alu_peak_ops(sms)
    t_roof = max(total_bytes / (hbm * 1e9), ops / (tc * 1e12))
    # the CUDA-core floor of the per-block-scaling kernel (stage 4's kernel):
    # one multiply and one FMA per block-scale partial (+ one FMA for Q4_1)
    gu_partials = R * 2.0 * f * (d // 32)
    t_alu_gu = gu_partials * ALU_OPS_PER_PARTIAL[cfg.wtype] / alu_peak
    qs_sec = mean_stage[1] / 1e3
    qs_gbs = stages["quantize_scatter"][0] / qs_sec / 1e9
    value = weak_scaling_value(world, T, ms)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8 x int8 block dots, fp32 scales and accumulation",
        "data": "synthetic: seeded N(0,1) activations and router logits, N(0,0.02) weights "
                "quantized to " + mw.WTYPE_NAMES[cfg.wtype],
        "config": dict(cfg.describe(), l2="flushed between steps (512 MB write)",
                       n_active_experts=n_active, mmq_path=mmq_path()),
        "roofline": {"kernel": dom_name, **roof,
                     "traffic": profiled_traffic(dom_name, cfg.name)},
        "alu_floor": {"kernel": "mmq_gateup (per-block scaling on the CUDA cores)",
                      "ms": round(t_alu_gu * 1e3, 4),
                      "frac": round(t_alu_gu * 1e3 / float(mean_stage[3]), 4),
                      "peak_source": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x "
                                     f"{MAX_SM_MHZ:.0f} MHz"},
        "layer_roofline": {"t_roofline_ms": round(t_roof * 1e3, 4),
                           "frac": round(t_roof * 1e3 / ms, 4),
                           "algorithmic_bytes": int(total_bytes), "ops": ops,
                           "bound": "hbm" if total_bytes / hbm / 1e9 >= ops / tc / 1e12 else "tensor",
                           "peak_source": f"{peak_src} copy and bf16 (burst)"},
        "stages": stage_roof,
        "quantize_scatter": {"GB/s": round(qs_gbs, 1), "frac_of_hbm": round(qs_gbs / hbm, 4),
                             "bytes": int(stages["quantize_scatter"][0])},
        "phases_ms": phases,
        "phases_median_ms": {n: round(float(v), 4)
                             for n, v in zip(stage_names, np.median(stage_ms, axis=0))},
        "ms_per_step_median": round(float(np.median(step_ms)), 4),
        "e2e": {"value": round(weak_scaling_value(world, T, e2e_ms), 1), "unit": "tokens/s",
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": int(wl.x.nbytes + wl.ids.nbytes + wl.w.nbytes),
                "d2h_bytes_per_step": int(T * d * 4),
                "api": "MoeLayer.forward_host, calls back to back (copies overlapped with "
                       "the layer and with the neighbouring calls; L2 flushed before each "
                       "call, its own duration not counted)",
                "per_call_ms_per_step": round(e2e_call_ms, 4),
                "serial_ms_per_step": round(e2e_serial_ms, 4),
                "bytes_identical_to_serial": e2e_same},
        "gpu_launches": int(launches),
        "wall_s_timed": round(t_wall, 3),
        "clocks": clocks,
    }
    if not args.no_ab:
        # after the timed region: these calls reuse the layer's buffers
        line["ab"] = ab_compare(m, layer, x, ids, flush, K)
        try:  # the fused calls take the tensor-core shapes only
            line["fused"] = fused_compare(m, layer, x, ids, w, flush)
        except m.MoeError as e:
            line["fused"] = {"unavailable": str(e)}
    if args.streamed:
        line["streamed"] = streamed_measure(m, layer, wl, x, ids, w, flush, args, ms, n_active)
    if world == 1 and not args.no_quantize_large:
        # the quantizer alone on the workload whose 268 MB input exceeds L2
        line["quantize_scatter_large"] = quantize_measure(args, dev)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return line


QUANTIZE_LARGE = mw.T32768.name


def quantize_measure(args, dev, reps: int = 20):
    """Stage 2 alone on the T=32768 Q4_1 workload (x = 268 MB > L2): only the
    quantizer's buffers (x, slot, q, ds) on the device; CUDA events around each
    call, L2 flushed between calls; GB/s of its algorithmic bytes."""
    import torch

    import quantized_routed_expert_q8_gb300 as m

    cfg = mw.CONFIGS[QUANTIZE_LARGE]
    T, K, E, d = cfg.T, cfg.K, cfg.E, cfg.d
    R = T * K
    x = torch.from_numpy(mw.activations(cfg)).to(dev)
    ids_h, _ = mw.topk_softmax(mw.routing_logits(cfg), K)
    ids = torch.from_numpy(ids_h).to(dev)
    i32 = dict(dtype=torch.int32, device=dev)
    off, slot, src = torch.zeros(E + 1, **i32), torch.zeros(R, **i32), torch.zeros(R, **i32)
    act, na = torch.zeros(E, **i32), torch.zeros(1, **i32)
    ws = torch.zeros(m.moe_workspace_size(T, K, E, cfg.d, cfg.f), dtype=torch.uint8, device=dev)
    m.moe_workspace_init(ws)
    m.moe_build_slot_map(ids, E, off, slot, src, act, na, ws)
    q = torch.empty((R, d), dtype=torch.int8, device=dev)
    ds = torch.empty((R, d // 32, 2), dtype=torch.int16, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        m.moe_quantize_scatter_q8_1(x, slot, K, R, q, ds)
    times = []
    for i in range(reps):
        flush.fill_(i & 0xFF)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        m.moe_quantize_scatter_q8_1(x, slot, K, R, q, ds)
        b.record(stream)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    assert m.moe_device_error(ws) == 0
    peaks, peak_src = load_peaks()
    nbytes = T * d * 4 + R * d * 1.125 + T * K * 4
    sec = float(np.mean(times)) / 1e3
    gbs = nbytes / sec / 1e9
    del x, q, ds, flush, ws
    torch.cuda.empty_cache()
    return {"workload": cfg.name, "ms": round(sec * 1e3, 4), "GB/s": round(gbs, 1),
            "frac_of_hbm": round(gbs / float(peaks["hbm_gbs"]), 4), "bytes": int(nbytes),
            "reps": reps, "peak_source": f"{peak_src} copy"}


def streamed_measure(m, layer, wl, x, ids, w, flush, args, resident_ms, n_active):
    """The layer with the expert records in pinned host memory, streamed over
    NVLink-C2C through the device staging ring: per-step time (CUDA events on
    the compute stream, the call's own synchronization included) and the
    host-to-device bytes it moved."""
    import torch

    host_arena = torch.from_numpy(wl.arena).pin_memory()

    def step():
        layer.forward_streamed(host_arena, x, ids, w, ring_groups=args.ring_groups)

    for _ in range(max(2, args.warmup)):
        step()
    torch.cuda.synchronize()
    times = []
    for s in range(args.steps):
        flush.fill_(s & 0xFF)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        step()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    assert m.moe_device_error(layer.ws) == 0
    t = float(np.mean(times))
    h2d = n_active * wl.rec_bytes
    return {"ms_per_step": round(t, 4), "tokens/s": round(wl.cfg.T / t * 1e3, 1),
            "ring_groups": args.ring_groups, "h2d_bytes_per_step": int(h2d),
            "h2d_GB/s_over_step": round(h2d / t / 1e6, 1),
            "vs_resident_ms": round(t / resident_ms, 3)}


def fused_compare(m, layer, x, ids, w, flush, reps: int = 10):
    """The fused epilogues against the seven calls: the whole layer each way,
    and each fused call against the two calls it replaces.  Each fused call runs
    on the kernel its two calls use by default (gate/up: per-block scaling;
    down: folded scales), so the layer's bytes must not change."""
    import torch

    L = layer
    T, K = ids.shape
    R, E, d, f = T * K, L.E, L.d, L.f

    def timed(fn):
        for _ in range(3):
            fn()
        tot = 0.0
        for i in range(reps):
            flush.fill_(i & 0xFF)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
        return tot / reps

    t_layer = timed(lambda: L.forward(x, ids, w))
    ref = L.out[:T].clone()
    hq_ref, y_ref = L.hq.clone(), L.y.clone()
    t_layer_f = timed(lambda: L.forward(x, ids, w, fused=True))
    same = bool(torch.equal(L.out[:T], ref) and torch.equal(L.hq, hq_ref)
                and torch.equal(L.y, y_ref))

    def gu_requant():
        m.moe_grouped_mmq_gateup(L.wtype, L.group_buf, L.slot_stride, L.active, L.n_active,
                                 L.offsets, E, L.q, L.ds, R, d, f, L.h, L.ws)
        m.quantizers(L.wtype)[2](L.h, R, f, L.hq, L.hds)

    def gu_fused():
        m.moe_grouped_mmq_gateup_q8_1(L.wtype, L.group_buf, L.slot_stride, L.active, L.n_active,
                                      L.offsets, E, L.q, L.ds, R, d, f, L.hq, L.hds, L.ws)

    def down_combine():
        m.moe_grouped_mmq_down(L.wtype, L.group_buf, L.slot_stride, L.active, L.n_active,
                               L.offsets, E, L.hq, L.hds, R, d, f, L.y, L.ws)
        m.moe_combine_topk(L.y, R, L.slot, w, T, K, d, L.out)

    def down_fused():
        m.moe_grouped_mmq_down_combine(L.wtype, L.group_buf, L.slot_stride, L.active, L.n_active,
                                       L.offsets, E, L.hq, L.hds, R, d, f, L.src, L.slot, w, T, K,
                                       L.y, L.out, L.ws)

    res = {"layer_ms": round(t_layer, 4), "layer_fused_ms": round(t_layer_f, 4),
           "gateup_requant_ms": round(timed(gu_requant), 4),
           "gateup_q8_1_ms": round(timed(gu_fused), 4),
           "down_combine_ms": round(timed(down_combine), 4),
           "down_combine_fused_ms": round(timed(down_fused), 4),
           "bytes_identical": same}
    assert m.moe_device_error(L.ws) == 0
    return res


def ab_compare(m, layer, x, ids, flush, K, reps: int = 10):
    """The pages' own comparisons on this GPU, each checked for byte identity:
    per-row gather quantization (each token row quantized again for each of its
    K expert rows) against quantize-once-and-scatter, and the expert gather as
    one launch per expert, one per group of 16, and one device-driven launch."""
    import torch

    L = layer
    T, d = x.shape
    R = T * K
    E = L.E
    m.moe_build_slot_map(ids, E, L.offsets, L.slot, L.src, L.active, L.n_active, L.ws)
    torch.cuda.synchronize()
    n_active = int(L.n_active.item())
    active = L.active[:n_active].cpu().tolist()

    def timed(fn):
        for _ in range(3):
            fn()
        tot = 0.0
        for i in range(reps):
            flush.fill_(i & 0xFF)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
        return tot / reps

    q2, ds2 = torch.empty_like(L.q), torch.empty_like(L.ds)
    q_scatter, q_gather, _ = m.quantizers(L.wtype)
    t_scatter = timed(lambda: q_scatter(x, L.slot, K, R, L.q, L.ds))
    t_gather = timed(lambda: q_gather(x, L.src, R, q2, ds2))
    q_same = bool(torch.equal(L.q[:R], q2[:R]) and torch.equal(L.ds[:R], ds2[:R]))

    ss = L.slot_stride
    used = n_active * ss

    def per_expert():
        for p, e in enumerate(active):
            base = (p // 16) * 16 * ss
            m.moe_group_gather(L.arena, L.rec_bytes, L.arena_stride, [e], p % 16,
                               L.group_buf[base:], ss)

    def per_group():
        for g0 in range(0, n_active, 16):
            m.moe_group_gather(L.arena, L.rec_bytes, L.arena_stride, active[g0:g0 + 16], 0,
                               L.group_buf[g0 * ss:], ss)

    def device():
        m.moe_group_gather_active(L.arena, L.rec_bytes, L.arena_stride, L.active, L.n_active, E,
                                  L.group_buf, ss)

    t_dev = timed(device)
    ref = L.group_buf[:used].clone()
    t_group = timed(per_group)
    same_group = bool(torch.equal(L.group_buf[:used], ref))
    t_expert = timed(per_expert)
    same_expert = bool(torch.equal(L.group_buf[:used], ref))
    return {
        "quantize": {"scatter_ms": round(t_scatter, 4), "per_row_gather_ms": round(t_gather, 4),
                     "gather_over_scatter": round(t_gather / t_scatter, 3),
                     "bytes_identical": q_same},
        "group_gather": {"n_active_experts": n_active,
                         "one_device_launch_ms": round(t_dev, 4),
                         "per_group_of_16_ms": round(t_group, 4),
                         "per_group_launches": (n_active + 15) // 16,
                         "per_expert_ms": round(t_expert, 4), "per_expert_launches": n_active,
                         "bytes_identical": same_group and same_expert},
    }


def mmq_path() -> str:
    """The MMQ kernels the run used: the CUDA-core kernel, one tensor-core kernel
    for both stages, or the default (per-block scaling for gate/up, folded
    scales for down)."""
    v = os.environ.get("MOE_MMQ_PATH", "")
    return v if v in ("simt", "blockscale", "fold") else "default"


def run_stage(args):
    """One stage of the layer, timed alone on its own inputs (a full layer is run
    once first to produce them).  Used for profiler captures of one kernel."""
    import torch

    import quantized_routed_expert_q8_gb300 as m

    cfg = mw.CONFIGS[args.config]
    T, K, E, d, f = cfg.T, cfg.K, cfg.E, cfg.d, cfg.f
    R = T * K
    dev = torch.device("cuda", 0)
    if args.stage == "quantize_scatter":
        # only the quantizer's own buffers: x, slot, q, ds (keeps profiler captures small)
        x = torch.from_numpy(mw.activations(cfg)).to(dev)
        ids_h, _ = mw.topk_softmax(mw.routing_logits(cfg), K)
        ids = torch.from_numpy(ids_h).to(dev)
        i32 = dict(dtype=torch.int32, device=dev)
        off, slot, src = torch.zeros(E + 1, **i32), torch.zeros(R, **i32), torch.zeros(R, **i32)
        act, na = torch.zeros(E, **i32), torch.zeros(1, **i32)
        ws = torch.zeros(m.moe_workspace_size(T, K, E, d, f), dtype=torch.uint8, device=dev)
        m.moe_workspace_init(ws)
        m.moe_build_slot_map(ids, E, off, slot, src, act, na, ws)
        q = torch.empty((R, d), dtype=torch.int8, device=dev)
        ds = torch.empty((R, d // 32, m.ds_halves(cfg.wtype)), dtype=torch.int16, device=dev)
        scatter = m.quantizers(cfg.wtype)[0]
        return _time_stage(args, cfg, lambda: scatter(x, slot, K, R, q, ds),
                           ws, int(na.item()), 0)
    wl = mw.make_workload(cfg)
    # only the routed experts' records go to the device (ids renumbered to them),
    # so a profiler capture holds ~1-2 GB instead of the whole expert arena
    used = [int(e) for e in np.unique(wl.ids)]  # Python ints: e * st exceeds int32
    st = wl.arena_stride
    arena_h = np.concatenate([wl.arena[e * st:(e + 1) * st] for e in used])
    ids_h = np.searchsorted(used, wl.ids).astype(np.int32)
    E = len(used)
    arena = torch.from_numpy(arena_h).to(dev)
    x = torch.from_numpy(wl.x).to(dev)
    ids = torch.from_numpy(ids_h).to(dev)
    w = torch.from_numpy(wl.w).to(dev)
    L = m.MoeLayer(cfg.wtype, E, d, f, K, T, arena, wl.rec_bytes, st, dev)
    L.forward(x, ids, w)
    calls = {
        "slot_map": lambda: m.moe_build_slot_map(ids, E, L.offsets, L.slot, L.src, L.active,
                                                 L.n_active, L.ws),
        "quantize_scatter": lambda: m.quantizers(cfg.wtype)[0](x, L.slot, K, R, L.q, L.ds),
        "group_gather": lambda: m.moe_group_gather_active(L.arena, L.rec_bytes, L.arena_stride,
                                                          L.active, L.n_active, E, L.group_buf,
                                                          L.slot_stride),
        "mmq_gateup": lambda: m.moe_grouped_mmq_gateup(L.wtype, L.group_buf, L.slot_stride,
                                                       L.active, L.n_active, L.offsets, E, L.q,
                                                       L.ds, R, d, f, L.h, L.ws),
        "requant_hidden": lambda: m.quantizers(cfg.wtype)[2](L.h, R, f, L.hq, L.hds),
        "mmq_down": lambda: m.moe_grouped_mmq_down(L.wtype, L.group_buf, L.slot_stride, L.active,
                                                   L.n_active, L.offsets, E, L.hq, L.hds, R, d, f,
                                                   L.y, L.ws),
        "combine_topk": lambda: m.moe_combine_topk(L.y, R, L.slot, w, T, K, d, L.out),
    }
    return _time_stage(args, cfg, calls[args.stage], L.ws, int(L.n_active.item()), wl.rec_bytes)


def _time_stage(args, cfg, fn, ws, n_active, rec_bytes):
    import torch

    import quantized_routed_expert_q8_gb300 as m

    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        fn()
    ms = []
    for s in range(args.steps):
        flush.fill_(s & 0xFF)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    bits = m.moe_device_error(ws)
    assert bits == 0, f"device error bits {bits:#x}"
    stages, _, _ = layer_accounting(cfg, n_active, rec_bytes, cfg.T * cfg.K)
    t = float(np.mean(ms)) / 1e3
    peaks, peak_src = load_peaks()
    return {"stage": args.stage, "config": cfg.describe(), "ms": round(t * 1e3, 4),
            "n_active_experts": n_active, "mmq_path": mmq_path(),
            **stage_roofline(*stages[args.stage], t, float(peaks["hbm_gbs"]),
                             float(peaks["bf16_tflops"]), peak_src)}


# ------------------------------------------------------------- CPU oracle --

def oracle_sample(wl, n_tokens: int, seed: int = 1):
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(wl.cfg.T, n_tokens, replace=False))
    return wl.subset(toks)


def time_oracle(wl, n_tokens):
    import oracle
    sub = oracle_sample(wl, n_tokens)
    cfg = wl.cfg
    t = time.perf_counter()
    oracle.layer_forward(cfg.wtype, wl.arena, wl.rec_bytes, wl.arena_stride, sub.x, sub.ids, sub.w,
                         cfg.E, cfg.d, cfg.f)
    return time.perf_counter() - t


def calibrate_tokens(wl, budget_s: float) -> int:
    t4 = time_oracle(wl, 4)
    n = int(4 * budget_s / max(t4, 1e-3))
    return max(4, min(n, wl.cfg.T))


def time_oracle_threads(wl, n_tokens, threads):
    """The oracle's layer on a token sample split into one contiguous slice per
    host thread (tokens are independent; the C calls release the interpreter
    lock), all slices running at once.  Returns the wall time."""
    import concurrent.futures
    import oracle
    sub = oracle_sample(wl, n_tokens)
    cfg = wl.cfg
    parts = [p for p in np.array_split(np.arange(n_tokens), threads) if len(p)]
    subs = [sub.subset(p) for p in parts]

    def run(s):
        oracle.layer_forward(cfg.wtype, wl.arena, wl.rec_bytes, wl.arena_stride, s.x, s.ids, s.w,
                             cfg.E, cfg.d, cfg.f)

    t = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(subs)) as ex:
        list(ex.map(run, subs))
    return time.perf_counter() - t


def host_cpu_model() -> str:
    """The host CPU's name as /proc/cpuinfo gives it (x86 'model name', or the
    Arm implementer / part numbers), else the machine type."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model"):
        for line in info.splitlines():
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    impl = part = None
    for line in info.splitlines():
        if line.startswith("CPU implementer") and impl is None:
            impl = line.split(":", 1)[1].strip()
        if line.startswith("CPU part") and part is None:
            part = line.split(":", 1)[1].strip()
    if impl or part:
        return f"{platform.machine()} implementer {impl} part {part}"
    return platform.machine()


def time_oracle_quantize(wl):
    """The oracle's stage 2 alone on the whole workload (single-threaded C):
    GB/s over the stage's algorithmic bytes."""
    import oracle
    cfg = wl.cfg
    sm = oracle.build_slot_map(wl.ids, cfg.E)
    R = int(sm["offsets"][cfg.E])
    t = time.perf_counter()
    oracle.quantize_scatter_q8_1(wl.x, sm["slot"], cfg.K, R, layout=oracle.layout_of(cfg.wtype))
    sec = time.perf_counter() - t
    q8 = 1.25 if cfg.wtype == mw.Q2_K else 1.125
    nbytes = cfg.T * cfg.d * 4 + R * cfg.d * q8 + cfg.T * cfg.K * 4
    return {"GB/s": round(nbytes / sec / 1e9, 3), "ms": round(sec * 1e3, 2),
            "sample": f"all {cfg.T} tokens, single-threaded C"}


def cpu_baseline(wl, budget_s: float = 15.0):
    n = calibrate_tokens(wl, budget_s)
    sec = time_oracle(wl, n)
    cores = os.cpu_count() or 1
    out = {"value": round(n / sec, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": f"{n} seeded tokens of the {wl.cfg.T}-token workload with their routing "
                     f"(all seven stages, single-threaded C, {sec:.1f} s)",
           "host_cores": cores, "host_cpu": host_cpu_model(),
           "quantize_scatter": time_oracle_quantize(wl)}
    if cores > 1:
        # the same oracle functions, one host thread per core over disjoint tokens
        nm = min(wl.cfg.T, n * cores)
        secm = time_oracle_threads(wl, nm, cores)
        out["all_cores"] = {"value": round(nm / secm, 3), "unit": "tokens/s", "cores": cores,
                            "sample": f"{nm} seeded tokens split over {cores} host threads "
                                      f"({secm:.1f} s)"}
    return out


def run_reference(args, rank):
    if rank != 0:
        return None
    cfg = mw.CONFIGS[args.config]
    wl = mw.make_workload(cfg)
    per_step = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    n = calibrate_tokens(wl, per_step)
    for _ in range(args.warmup):
        time_oracle(wl, n)
    secs = [time_oracle(wl, n) for _ in range(args.steps)]
    ms = 1e3 * float(np.mean(secs))
    value = n / (ms / 1e3)
    sample = (f"{n} seeded tokens of the {cfg.T}-token workload per step (all seven stages, "
              f"single-threaded C oracle)")
    return {
        "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 x int8 block dots, fp32 scales and accumulation", "data": "synthetic",
        "config": dict(cfg.describe(), sample_tokens=n), "impl": "reference",
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": 1,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=list(mw.CONFIGS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-quantize-large", action="store_true",
                    help="skip the stand-alone quantizer measurement on the T=32768 workload")
    ap.add_argument("--streamed", action="store_true",
                    help="also time the layer with the expert records streamed from pinned host memory")
    ap.add_argument("--ring-groups", type=int, default=3)
    ap.add_argument("--no-ab", action="store_true",
                    help="skip the gather-quantization and per-expert gather comparisons")
    ap.add_argument("--stage", default=None,
                    help="time one stage alone (for profiler captures): slot_map, quantize_scatter, "
                         "mmq_gateup, mmq_down, requant_hidden, combine_topk, group_gather")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.stage:
        line = run_stage(args)
    elif args.impl == "reference":
        line = run_reference(args, rank)
    else:
        line = run_gpu(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
