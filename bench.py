#!/usr/bin/env python3
"""Benchmark of libgemm on one GB300 (or N independent replicas).

A step is one pass of the whole hot path: C = A*B at M = K = N = 4096 once in
each precision mode -- exact FP32 on the CUDA cores, TF32 and BF16-input on the
tensor cores -- on seeded synthetic inputs uniform on [0, 1) (the square
sweep's largest size, the size the headline metric is quoted at).  Each GEMM
counts 2*M*N*K floating-point operations, as the first page counts them
("Matrix Multiplication -- Naive to Tiled", section 03).

Timing: W untimed warm-up steps, then K timed steps between a barrier and a
device synchronisation on both sides.  Before every GEMM a 256 MiB buffer is
written to flush the 129 MB L2; each GEMM is bracketed by CUDA events on the
stream it runs on, so the flush is outside the measured time.  ms_per_step is
the mean over steps of the three GEMMs' event times.  The JSON line also
carries the roofline of the dominant kernel, the fp64 oracle's throughput on
the host cores (cpu_baseline), an end-to-end figure with host buffers (every
step copies its inputs in from pinned host memory -- A and B as float32,
shared by the FP32 and TF32 products, and as bfloat16 -- and every product's C
back out; copy-in, compute and copy-out run on three streams so that one
product's copies overlap another's compute), the SM clocks seen during the timed region
and the number of library launches.

``--impl reference`` times the fp64 CPU oracle instead (a bounded sample of
rows of the same workload per step), on the same metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (FP32 and TF32/BF16) at N=4096, % of sm_103a peak"
UNIT = "TFLOP/s"
MODES = ("fp32", "tf32", "bf16")               # the bench line's step
# further modes that --modes can select, to time or profile their kernels:
# binary16 inputs (the BF16 kernel's kind::f16 with f16 operands), FP32
# data rounded to bfloat16 by a conversion launch before the BF16 kernel,
# and FP32 data rounded to TF32 to nearest by a launch before the TF32 kernel
EXTRA_MODES = ("fp16", "fp32_via_bf16", "tf32_rn")
ALL_MODES = MODES + EXTRA_MODES
L2_FLUSH_BYTES = 256 << 20

# GB300 facts used for the roofline denominators.
NUM_SMS = 152
SM_MAX_MHZ = 2070.0
FP32_LANES_PER_SM = 128                      # FFMA lanes per SM (4 sub-partitions x 32)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
TF32_PER_BF16 = 1.1 / 2.25                   # nominal dense TF32 / BF16 tensor rates
NOMINAL_TFLOPS = {"bf16": 2250.0, "tf32": 1100.0, "fp16": 2250.0,
                  "fp32_via_bf16": 2250.0, "tf32_rn": 1100.0}   # stated dense peaks (no sparsity)

# DRAM traffic of one launch of the dominant kernel, from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by the sha256 of the
# kernel source it was taken on; reported as null once the source changes.
TRAFFIC = {
    # profiles/ffma_sgemm_fp32_4096.md: 275.18 MB read + 70.31 MB written
    "ffma_sgemm.cu": ("dbb86d08c9e528c09b5955bfa79c0e51eb370675e9c9fb9f2cfcc92729ff199d", 345.49e6),
}


def flops(M: int, K: int, N: int) -> float:
    """Floating-point operations of one product: M*N outputs, K multiplies and K adds each."""
    return 2.0 * M * N * K


def tflops(M: int, K: int, N: int, seconds: float) -> float:
    return flops(M, K, N) / seconds / 1e12


def _measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)) or None, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, None, "fallback"


def fp32_ffma_peak(mhz: float = SM_MAX_MHZ, sms: int = NUM_SMS) -> float:
    """FP32 FFMA peak in TFLOP/s: SMs x lanes x 2 FLOP x clock."""
    return sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def device_sms(dev) -> int:
    """The device's SM count (152 on GB300)."""
    import torch
    return int(torch.cuda.get_device_properties(dev).multi_processor_count)


def _src_hash(name: str) -> str:
    with open(os.path.join(ROOT, "accelerator_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


# --------------------------------------------------------------------------
# clocks during the timed region
_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """Samples the SM clock and the clock-event reasons every few ms in a
    thread while the timed region runs, through NVML (libnvidia-ml, read-only
    queries).  Falls back to nvidia-smi when NVML cannot be loaded."""

    def __init__(self, torch_device_index: int, period_s: float = 0.004):
        self.index = torch_device_index
        self.period = period_s
        self.samples = []
        self.max_mhz = None
        self._stop = None
        self._thread = None
        self._nvml = None
        self._handle = None
        self._smi = None

    def _open_nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        handle = ctypes.c_void_p()
        ok = False
        try:
            import torch
            uuid = "GPU-" + str(torch.cuda.get_device_properties(self.index).uuid)
            ok = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(handle)) == 0
        except Exception:
            ok = False
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(handle)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:   # 1 = SM clock
            self.max_mhz = float(mx.value)
        self._nvml, self._handle = lib, handle

    def _poll(self):
        import ctypes
        lib, h = self._nvml, self._handle
        clk, why = ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                r = why.value if get_reasons(h, ctypes.byref(why)) == 0 else 0
                self.samples.append((float(clk.value), int(r)))
            self._stop.wait(self.period)

    def __enter__(self):
        import threading
        try:
            self._open_nvml()
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        except Exception:
            self._nvml = None
            try:
                import tempfile
                fd, path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
                os.close(fd)
                self._smi = (path, subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index),
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=open(path, "w"), stderr=subprocess.DEVNULL))
            except Exception:
                self._smi = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self._smi is not None:
            path, proc = self._smi
            proc.terminate()
            try:
                proc.wait(timeout=5)
            except Exception:
                proc.kill()
            with open(path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    try:
                        self.samples.append((float(parts[0]), int(parts[2], 16)))
                        self.max_mhz = float(parts[1])
                    except (ValueError, IndexError):
                        continue
            os.unlink(path)

    def summary(self):
        if not self.samples:
            return None
        reasons = sorted({name for _, r in self.samples for bit, name in _REASONS.items() if r & bit})
        return {"sm_mhz": float(np.median([c for c, _ in self.samples])),
                "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "source": "nvml" if self._nvml else "nvidia-smi"}


# --------------------------------------------------------------------------
def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device="cpu") -> float:
    """The largest x over all ranks (x itself with one rank).  The timed
    figure of a multi-rank run is the slowest rank's."""
    if ws <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(ws: int, products_per_rank: int, flops_per_product: float, ms: float) -> float:
    """Whole-job throughput: the products all ranks completed over the
    slowest rank's time (replicas: every rank does the same work)."""
    return ws * products_per_rank * flops_per_product / (ms / 1e3) / 1e12


def _cpu_sample(A: np.ndarray, B: np.ndarray, fmt: str, rows: int):
    """fp64 oracle on the first `rows` rows of C; returns seconds."""
    import oracle
    t0 = time.perf_counter()
    oracle.gemm(np.ascontiguousarray(A[:rows]), B, fmt=fmt)
    return time.perf_counter() - t0


def cpu_baseline(A: np.ndarray, B: np.ndarray, target_s: float = 15.0):
    """The oracle as it stands, on all host cores, on a bounded sample: the
    first rows of C, as many as take about target_s seconds."""
    import oracle
    n = A.shape[0]
    K, N = B.shape
    cores = oracle.threads()
    t1 = _cpu_sample(A, B, "f32", 16)
    t2 = _cpu_sample(A, B, "f32", 48)
    per_row = max((t2 - t1) / 32, 1e-6)
    fixed = max(t1 - 16 * per_row, 0.0)
    rows = int(max(16, min(n, (target_s - fixed) / per_row)))
    t = _cpu_sample(A, B, "f32", rows)
    return {"value": tflops(rows, K, N, t), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {rows} of {n} rows of C for the {n}x{K}x{N} FP32 input "
                      f"(fp64 triple loop, {t:.1f} s)"}


def run_reference(args):
    """The fp64 CPU oracle as the reference arm."""
    ws, rank, _ = _dist_env()
    if rank != 0:
        return 0
    import oracle
    from accelerator_gb300 import inputs
    n = args.size
    A, B = inputs.matrices(n, n, n, "u01")
    fmt_inputs = {"fp32": (A, B, "f32"), "tf32": (A, B, "tf32"),
                  "bf16": (inputs.bf16_bits(A), inputs.bf16_bits(B), "bf16")}
    cores = oracle.threads()
    # size each step so the whole run stays within a few minutes
    t = _cpu_sample(A, B, "f32", 2)
    per_step = max(1.0, min(8.0, 150.0 / (args.steps + args.warmup)))
    rows = int(max(1, min(n, 2 * per_step / 3 / max(t, 1e-3))))

    def step():
        for m in MODES:
            a, b, fmt = fmt_inputs[m]
            oracle.gemm(np.ascontiguousarray(a[:rows]), b, fmt=fmt)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = 3 * flops(rows, n, n) / dt / 1e12
    sample = f"first {rows} of {n} rows of C per mode, 3 modes per step (fp64 triple loop)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"square GEMM M=K=N={n}, modes fp32+tf32+bf16, U[0,1) seed 42",
                   "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


def run_libgemm(args):
    import torch
    import torch.distributed as dist
    from accelerator_gb300 import binding, build, inputs

    ws, rank, local = _dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    binding.lib()
    dev = torch.device("cuda", local)
    n = args.size
    A, B = inputs.matrices(n, n, n, "u01")
    a32, b32 = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
    a16 = torch.from_numpy(inputs.bf16_bits(A).view(np.int16)).view(torch.bfloat16).to(dev)
    b16 = torch.from_numpy(inputs.bf16_bits(B).view(np.int16)).view(torch.bfloat16).to(dev)
    ops = {"fp32": (a32, b32, binding.FP32), "tf32": (a32, b32, binding.TF32),
           "bf16": (a16, b16, binding.BF16), "fp32_via_bf16": (a32, b32, binding.FP32_VIA_BF16),
           "tf32_rn": (a32, b32, binding.TF32_RN)}
    if "fp16" in args.modes:
        ops["fp16"] = (torch.from_numpy(inputs.fp16_bits(A).view(np.int16)).view(torch.float16).to(dev),
                       torch.from_numpy(inputs.fp16_bits(B).view(np.int16)).view(torch.float16).to(dev),
                       binding.FP16)
    C = torch.zeros((n, n), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    f = flops(n, n, n)

    def step(events=None):
        for m in args.modes:
            a, b, mode = ops[m]
            flush.zero_()
            if events is not None:
                events[m][0].record(stream)
            binding.gemm(a, b, C, mode=mode, stream=stream)
            if events is not None:
                events[m][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if binding.debug_status(stream) != binding.OK:
        raise RuntimeError("a kernel reported a timeout during warm-up")

    evs = [{m: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for m in args.modes} for _ in range(args.steps)]
    launches0 = binding.launch_count()
    with ClockSampler(local) as clocks:
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for s in range(args.steps):
            step(evs[s])
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        if ws > 1:
            dist.barrier()
    launches = binding.launch_count() - launches0
    per_mode = {m: np.array([evs[s][m][0].elapsed_time(evs[s][m][1]) for s in range(args.steps)])
                for m in args.modes}
    ms_step = max_over_ranks(float(np.mean(sum(per_mode[m] for m in args.modes))), ws, dev)
    value = job_tflops(ws, len(args.modes), f, ms_step)
    if binding.debug_status(stream) != binding.OK:
        raise RuntimeError("a kernel reported a timeout during the timed region")
    clk = clocks.summary()

    # e2e: host buffers, copies inside the timed region.  Every step copies
    # its inputs in from pinned host memory (once each, shared by the products
    # that read them) and every product's C back out; three streams overlap
    # one product's copies with another's compute, as a user of the library
    # would.
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, A, B, n, dev, stream, ws, f)

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return 0

    hbm, bf16_peak, bf16_sus, src = _measured_peaks()
    tf32_peak = bf16_peak * TF32_PER_BF16
    sm_mhz = clk["sm_mhz"] if clk else None
    max_mhz = float(clk["sm_max_mhz"]) if clk and clk.get("sm_max_mhz") else SM_MAX_MHZ
    sms = device_sms(dev)
    modes_out = {}
    for m in args.modes:
        ms = float(np.mean(per_mode[m]))
        achieved = f / (ms / 1e3) / 1e12
        if m == "fp32":
            peak, bound = fp32_ffma_peak(max_mhz, sms), "alu"
            note = f"FP32 FFMA: {sms} SMs x 128 lanes x 2 x {max_mhz:.0f} MHz (device SM count, NVML max SM clock)"
        elif m == "tf32":
            peak, bound, note = tf32_peak, "tensor", f"{src} bf16 x nominal tf32/bf16 ratio"
        elif m == "fp32_via_bf16":
            peak, bound, note = bf16_peak, "tensor", f"{src} bf16 burst (conversion launch included in the time)"
        elif m == "tf32_rn":
            peak, bound, note = tf32_peak, "tensor", (f"{src} bf16 x nominal tf32/bf16 ratio "
                                                      "(rounding launch included in the time)")
        else:   # bf16, fp16: one kind::f16 rate
            peak, bound, note = bf16_peak, "tensor", f"{src} bf16 burst"
        modes_out[m] = {"ms_mean": ms, "ms_median": float(np.median(per_mode[m])),
                        "tflops": achieved, "bound": bound, "peak": peak, "frac": achieved / peak,
                        "peak_source": note}
        modes_out[m]["frac_nominal"] = achieved / NOMINAL_TFLOPS.get(m, fp32_ffma_peak(max_mhz, sms))
        if m == "fp32" and sm_mhz:
            modes_out[m]["frac_at_observed_clock"] = achieved / fp32_ffma_peak(sm_mhz, sms)
    dom = max(args.modes, key=lambda m: modes_out[m]["ms_mean"])
    dom_file = "ffma_sgemm.cu" if dom == "fp32" else "tc_gemm.cu"
    traffic = None
    if dom_file in TRAFFIC and TRAFFIC[dom_file][0] == _src_hash(dom_file):
        traffic = TRAFFIC[dom_file][1]
    roofline = {"bound": modes_out[dom]["bound"], "achieved": modes_out[dom]["tflops"],
                "peak": modes_out[dom]["peak"], "unit": "TFLOP/s",
                "frac": modes_out[dom]["frac"], "traffic": traffic,
                "kernel": dom_file, "per_launch_flops": f,
                "peak_source": modes_out[dom]["peak_source"]}

    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(A, B)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "+".join(args.modes), "data": "synthetic",
        "config": {"workload": f"square GEMM M=K=N={n}, one product per mode "
                               f"({', '.join(args.modes)}), U[0,1) seed 42",
                   "l2": "flushed before every GEMM (256 MiB write, outside the events)",
                   "parallelism": f"replicas x{ws}"},
        "modes": modes_out,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


# The input set each mode reads on the end-to-end leg: A and B as float32
# serve FP32, TF32 and FP32_VIA_BF16; bfloat16 and binary16 copies serve the
# others.  Bytes per element of each set.
E2E_GROUP_OF = {"fp32": "f32", "tf32": "f32", "fp32_via_bf16": "f32", "tf32_rn": "f32",
                "bf16": "bf16", "fp16": "fp16"}
E2E_GROUP_BYTES = {"f32": 4, "bf16": 2, "fp16": 2}


# The order of an end-to-end step's products: the longest (FP32) last, so
# that the other products' copies out overlap it and after the last step only
# its C is still to copy; TF32 first, whose inputs are FP32's and so are
# copied first.  Measured at 4096: 161.5 TFLOP/s against 159.5-159.9 with
# FP32 first.
E2E_RANK = {"tf32": 0, "tf32_rn": 1, "fp32_via_bf16": 2, "bf16": 3, "fp16": 4, "fp32": 9}


def e2e_order(modes):
    """The step's products in the order the end-to-end leg runs them."""
    return tuple(sorted(modes, key=lambda m: E2E_RANK[m]))


def e2e_input_groups(modes):
    """The input sets a step copies, once each, in the order its products
    first read them (so the first product waits only for its own inputs)."""
    return list(dict.fromkeys(E2E_GROUP_OF[m] for m in modes))


def e2e_bytes_per_step(modes, n):
    """(host-to-device, device-to-host) bytes of one end-to-end step of
    square n x n products: A and B of every input set in, every C out."""
    h2d = sum(2 * n * n * E2E_GROUP_BYTES[g] for g in e2e_input_groups(modes))
    return h2d, len(modes) * n * n * 4


def run_e2e(args, A, B, n, dev, stream, ws, f):
    """E2E throughput: per step, the H2D copies of the step's inputs from
    pinned host memory, one product per mode, and the D2H copy of every
    product's C, all inside the timed region.  The inputs are copied once per
    step and shared by the products that take them (A and B as float32 serve
    FP32, TF32 and FP32_VIA_BF16, as on the device-timed leg).  The copy-in
    stream, the compute stream and the copy-out stream are ordered by events,
    so a buffer is only overwritten after every earlier use has finished.
    The products run in e2e_order."""
    import torch
    from accelerator_gb300 import binding, inputs
    mode_ids = {"fp32": binding.FP32, "tf32": binding.TF32, "bf16": binding.BF16,
                "fp16": binding.FP16, "fp32_via_bf16": binding.FP32_VIA_BF16,
                "tf32_rn": binding.TF32_RN}
    group_of = E2E_GROUP_OF
    modes = e2e_order(args.modes)
    host = {}
    for g in e2e_input_groups(modes):
        if g == "f32":
            host[g] = (torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory(), None)
        elif g == "bf16":
            host[g] = (torch.from_numpy(inputs.bf16_bits(A).view(np.int16)).pin_memory(),
                       torch.from_numpy(inputs.bf16_bits(B).view(np.int16)).pin_memory(),
                       torch.bfloat16)
        else:
            host[g] = (torch.from_numpy(inputs.fp16_bits(A).view(np.int16)).pin_memory(),
                       torch.from_numpy(inputs.fp16_bits(B).view(np.int16)).pin_memory(),
                       torch.float16)
    # two sets of device buffers, used by alternate steps, so that a step's
    # copies need not wait for the previous step's products
    ins, outs = [{}, {}], [{}, {}]
    for k in range(2):
        for g, (ha, hb, view) in host.items():
            ins[k][g] = dict(ha=ha, hb=hb, view=view,
                             xa=torch.empty(ha.shape, dtype=ha.dtype, device=dev),
                             xb=torch.empty(hb.shape, dtype=hb.dtype, device=dev),
                             loaded=torch.cuda.Event(), readers=[])
        for m in modes:
            outs[k][m] = dict(c=torch.empty((n, n), dtype=torch.float32, device=dev),
                              hc=torch.empty((n, n), dtype=torch.float32).pin_memory(),
                              done=torch.cuda.Event(), out=torch.cuda.Event(), used=False)
    h2d = sum(ha.numel() * ha.element_size() + hb.numel() * hb.element_size()
              for ha, hb, _ in host.values())
    d2h = len(modes) * n * n * 4
    assert (h2d, d2h) == e2e_bytes_per_step(modes, n)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    parity = [0]

    def e2e_step():
        k = parity[0]
        for g, b in ins[k].items():
            with torch.cuda.stream(s_in):
                for ev in b["readers"]:
                    s_in.wait_event(ev)                # the last products have read xa, xb
                b["xa"].copy_(b["ha"], non_blocking=True)
                b["xb"].copy_(b["hb"], non_blocking=True)
                b["loaded"].record(s_in)
            b["readers"] = []
        for m in modes:
            b, o = ins[k][group_of[m]], outs[k][m]
            stream.wait_event(b["loaded"])
            if o["used"]:
                stream.wait_event(o["out"])             # the last copy-out has read c
            xa, xb = b["xa"], b["xb"]
            if b["view"] is not None:
                xa, xb = xa.view(b["view"]), xb.view(b["view"])
            binding.gemm(xa, xb, o["c"], mode=mode_ids[m], stream=stream)
            o["done"].record(stream)
            b["readers"].append(o["done"])
            with torch.cuda.stream(s_out):
                s_out.wait_event(o["done"])
                o["hc"].copy_(o["c"], non_blocking=True)
                o["out"].record(s_out)
            o["used"] = True
        parity[0] ^= 1

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for _ in range(args.steps):
        e2e_step()
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws, dev)   # the slowest rank's
    if binding.debug_status(stream) != binding.OK:
        raise RuntimeError("a kernel reported a timeout during the end-to-end run")
    return {"value": ws * len(modes) * f / (ms / 1e3) / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "overlap": "copy-in, compute and copy-out on three streams; each input copied "
                       "once per step and shared by the modes that read it; products in the "
                       "order " + ",".join(modes) + " (the longest last)"}


def _cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def run_cpu_sweep(args):
    """The fp64 oracle on the host cores, full C: one core for N <= 2048 and
    all cores for N <= 4096, on the sweep's inputs (U[0,1), seed 42).  Prints
    one JSON line; not a bench line."""
    import oracle
    from accelerator_gb300 import inputs
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    rows = []
    for n in (128, 256, 512, 1024, 2048, 4096):
        A, B = inputs.matrices(n, n, n, "u01")
        for threads in ((1, cores) if n <= 2048 else (cores,)):
            used = oracle.threads(threads)
            t0 = time.perf_counter()
            oracle.gemm(A, B, "f32", nthreads=threads)
            dt = time.perf_counter() - t0
            rows.append({"n": n, "threads": used, "seconds": dt, "gflops": flops(n, n, n) / dt / 1e9})
    print(json.dumps({"cpu_sweep": rows, "kind": "oracle", "cpu_model": _cpu_model(),
                      "cores_available": cores, "data": "synthetic U[0,1), seed 42"}), flush=True)
    return 0


def run_sweep(args):
    """The square sweep: N = 128 .. 4096 in every mode (and 8192 on the tensor
    modes), U[0,1) inputs, L2 flushed before each launch, `warmup` untimed
    launches then the median of `steps` CUDA-event-timed launches per (N,
    mode).  Prints one JSON line holding the table; not a bench line."""
    import torch
    from accelerator_gb300 import binding, build, inputs
    torch.cuda.set_device(0)
    build.build()
    dev = torch.device("cuda", 0)
    _, bf16_peak, bf16_sustained, src = _measured_peaks()
    tensor_rate = {"tf32": TF32_PER_BF16, "tf32_rn": TF32_PER_BF16, "bf16": 1.0, "fp16": 1.0,
                   "fp32_via_bf16": 1.0}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    rows = []
    sampler = ClockSampler(0)
    sampler.__enter__()
    for n in (128, 256, 512, 1024, 2048, 4096, 8192):
        A, B = inputs.matrices(n, n, n, "u01")
        a32, b32 = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
        a16 = torch.from_numpy(inputs.bf16_bits(A).view(np.int16)).view(torch.bfloat16).to(dev)
        b16 = torch.from_numpy(inputs.bf16_bits(B).view(np.int16)).view(torch.bfloat16).to(dev)
        h16 = None
        if "fp16" in args.modes:
            h16 = (torch.from_numpy(inputs.fp16_bits(A).view(np.int16)).view(torch.float16).to(dev),
                   torch.from_numpy(inputs.fp16_bits(B).view(np.int16)).view(torch.float16).to(dev))
        C = torch.zeros((n, n), dtype=torch.float32, device=dev)
        for m in args.modes:
            if n > 4096 and m == "fp32":
                continue
            a, b = (a16, b16) if m == "bf16" else h16 if m == "fp16" else (a32, b32)
            mode = binding.MODES[m]
            times = []
            for r in range(args.warmup + args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                binding.gemm(a, b, C, mode=mode, stream=stream)
                e1.record(stream)
                torch.cuda.synchronize()
                if r >= args.warmup:
                    times.append(e0.elapsed_time(e1))
            if binding.debug_status(stream) != binding.OK:
                raise RuntimeError(f"a kernel reported a timeout at N={n} {m}")
            ms = float(np.median(times))
            tf = flops(n, n, n) / (ms / 1e3) / 1e12
            row = {"n": n, "mode": m, "ms_median": ms, "tflops": tf}
            if m == "fp32":
                row.update(bound="alu", peak=fp32_ffma_peak(SM_MAX_MHZ, device_sms(dev)))
            else:
                row.update(bound="tensor", peak=bf16_peak * tensor_rate[m])
                if bf16_sustained:   # the power-capped loop's figure, for context
                    row["frac_sustained"] = tf / (bf16_sustained * tensor_rate[m])
            row["frac"] = tf / row["peak"]
            rows.append(row)
        del a32, b32, a16, b16, h16, C
        torch.cuda.empty_cache()
    sampler.__exit__(None, None, None)
    print(json.dumps({"sweep": rows, "unit": UNIT, "peak_source": src, "warmup": args.warmup,
                      "repeats": args.steps, "l2": "flushed before every launch",
                      "clocks": sampler.summary(),
                      "data": "synthetic U[0,1), seed 42"}), flush=True)
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["libgemm", "reference"], default="libgemm")
    p.add_argument("--size", type=int, default=4096)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--sweep", action="store_true",
                   help="print the square sweep N = 128 .. 8192 instead of the bench line")
    p.add_argument("--cpu-sweep", action="store_true",
                   help="print the fp64 oracle's timings on the host cores, N = 128 .. 4096")
    p.add_argument("--modes", default=",".join(MODES),
                   help="comma-separated subset of " + ",".join(ALL_MODES) + " (default: "
                        + ",".join(MODES) + ", the bench line; other selections time or "
                        "profile single kernels)")
    args = p.parse_args(argv)
    unknown = [m for m in args.modes.split(",") if m not in ALL_MODES]
    if unknown:
        p.error(f"unknown mode(s) {unknown}; choose from {','.join(ALL_MODES)}")
    args.modes = tuple(m for m in ALL_MODES if m in args.modes.split(","))
    if not args.modes:
        p.error("--modes selects no mode")
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.cpu_sweep:
        return run_cpu_sweep(args)
    if args.sweep:
        return run_sweep(args)
    return run_libgemm(args)


if __name__ == "__main__":
    sys.exit(main())
