"""Throughput of the fused SDPA training step on GB300.

One step = the whole hot path over one batch: the forward pass with its per-row LSE,
then the backward pass (dQ, dK, dV), for the bf16 causal d=128 training workload at
s = 8192 (b=2, h=16), through the library's C ABI.  FLOPs follow the pages' counting
convention: 4*b*h*s_q*s_kv*d for the forward pass, halved for causal, backward 2.5x that.

Prints one JSON line (rank 0).  Flags:
  --gpus N --steps K --warmup W   standard contract (N>1: one rank per GPU under torchrun,
                                  independent replicas, max time over ranks, weak scaling)
  --impl reference                time the fp64 CPU oracle instead (bounded row slices of the
                                  same workload) and print the reference line
  --profile-step                  run one untimed fwd+bwd (the command profiled with ncu)
  --profile-workload NAME         one untimed fwd (+bwd) of a --sweep workload, for ncu
  --sweep                         one line per configuration (tables; not the contract line)
  --only A,B                      with --sweep: only the named configurations
  --measure-peaks                 dense GEMM peaks of this GPU through the vendor library:
                                  bf16 (torch.matmul) and E4M3 (torch._scaled_mm), 8192^3
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SDPA fwd & fwd+bwd TFLOP/s (bf16/fp8) and % of GB300 tensor peak"
UNIT = "TFLOP/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(PEAKS_FALLBACK)
    d["source"] = "fallback"
    return d


def bench_workload():
    from sdpa_workloads import training
    return training(8192)


# ---------------------------------------------------------------------------
# distributed plumbing (independent replicas; no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def aggregate(local_units: float, local_seconds: float, dist=None, device=None):
    """Whole-job figures: units summed over ranks, time = max over ranks."""
    import torch
    if dist is None:
        return local_units, local_seconds
    t = torch.tensor([local_units, local_seconds], dtype=torch.float64, device=device)
    u = t[:1].clone()
    s = t[1:].clone()
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    dist.all_reduce(s, op=dist.ReduceOp.MAX)
    return float(u.item()), float(s.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """Samples the GPU's SM clock, power draw and clock-event (throttle) reasons every few
    milliseconds from a background thread, through NVML's read-only queries (ctypes on the
    driver's libnvidia-ml; no setting is changed).  ``mark(True/False)`` brackets the timed
    regions: only samples taken inside them count as "under load"."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str | None, bus_id: str | None, period_s: float = 0.002):
        import threading
        self.period = period_s
        self.samples = []          # (t, in_timed_region, sm_mhz, power_w, reasons_bits)
        self.timed = False
        self.stop_ev = threading.Event()
        self.thread = None
        self.err = None
        self.nvml = self.dev = None
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            dev = ctypes.c_void_p()
            rc = -1
            if uuid:
                rc = nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(dev))
            if rc != 0 and bus_id:
                rc = nv.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(dev))
            if rc != 0:
                raise RuntimeError(f"no NVML handle for {uuid} / {bus_id}")
            self.nvml, self.dev, self.ct = nv, dev, ctypes
            self.reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint(0)
            nv.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx))   # NVML_CLOCK_SM
            self.max_mhz = float(mx.value) or None
        except Exception as e:  # no NVML: the line says so
            self.err = str(e)

    def _poll(self):
        ct, nv, dev = self.ct, self.nvml, self.dev
        clk, pw, rs = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        while not self.stop_ev.is_set():
            nv.nvmlDeviceGetClockInfo(dev, 1, ct.byref(clk))
            nv.nvmlDeviceGetPowerUsage(dev, ct.byref(pw))
            self.reason_fn(dev, ct.byref(rs))
            self.samples.append((time.perf_counter(), self.timed, float(clk.value), pw.value / 1e3,
                                 int(rs.value)))
            self.stop_ev.wait(self.period)

    def start(self):
        if self.nvml is None:
            return
        import threading
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()

    def mark(self, timed: bool):
        self.timed = timed

    def stop(self):
        if self.thread is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"],
                    "how": f"NVML unavailable: {self.err}"}
        self.stop_ev.set()
        self.thread.join(timeout=5)
        try:
            self.nvml.nvmlShutdown()
        except Exception:
            pass
        under = [x for x in self.samples if x[1]]
        if not under:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"],
                    "samples": len(self.samples), "samples_under_load": 0}
        bits = 0
        for x in under:
            bits |= x[4]
        reasons = sorted(name for b, name in self.REASONS.items() if bits & b)
        return {"sm_mhz": statistics.median(x[2] for x in under), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(x[2] for x in under), "reasons": reasons,
                "power_w_median": statistics.median(x[3] for x in under),
                "power_w_max": max(x[3] for x in under),
                "samples": len(self.samples), "samples_under_load": len(under),
                "how": f"NVML read-only queries every {self.period * 1e3:.0f} ms from a thread, over the "
                       "device-timed and end-to-end timed regions"}


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

class Step:
    """Device buffers and one training step (fwd with LSE, then bwd) of a workload."""

    def __init__(self, w, seed: int, device, host=None):
        import torch
        import attention_flashattention_sdpa_gb300 as sdpa
        from sdpa_workloads import make_inputs
        self.sdpa, self.w, self.torch = sdpa, w, torch
        if host is None:
            x = make_inputs(w, seed=seed, with_do=True)
            host = [t.contiguous().pin_memory() for t in (x.q, x.k, x.v, x.do)]
        self.host = host
        q, k, v, do = (t.to(device) for t in self.host)
        self.q, self.k, self.v, self.do = q, k, v, do
        self.o = torch.empty_like(q)
        self.lse = torch.empty(w.b, w.h_q, w.s_q, dtype=torch.float32, device=device)
        self.dq, self.dk, self.dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        p = sdpa.make_problem(q, k, v, self.o, attn_scale=w.scale, causal=w.causal, dout=do,
                              dq=self.dq, dk=self.dk, dv=self.dv)
        self.ws = torch.empty(sdpa.sdpa_workspace_size(p, True), dtype=torch.uint8, device=device)
        self.out_host = [torch.empty_like(t, device="cpu").pin_memory()
                         for t in (self.dq, self.dk, self.dv)]

    def fwd(self):
        w = self.w
        self.sdpa.sdpa_fwd(self.q, self.k, self.v, self.o, self.lse, attn_scale=w.scale,
                           causal=w.causal)

    def bwd(self):
        w = self.w
        self.sdpa.sdpa_bwd(self.q, self.k, self.v, self.o, self.do, self.lse, self.dq, self.dk,
                           self.dv, self.ws, attn_scale=w.scale, causal=w.causal)

    def h2d(self, which=slice(None)):
        for dst, src in list(zip((self.q, self.k, self.v, self.do), self.host))[which]:
            dst.copy_(src, non_blocking=True)

    def d2h(self):
        for dst, src in zip(self.out_host, (self.dq, self.dk, self.dv)):
            dst.copy_(src, non_blocking=True)

    def twin(self, device):
        """A second set of device and output buffers over the same pinned inputs."""
        return Step(self.w, 0, device, host=self.host)

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host)

    def d2h_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.out_host)


def time_device(step: "Step", steps: int, warmup: int, clocks=None):
    """CUDA-event timing on the launching stream: whole steps, and fwd / bwd separately."""
    import torch
    st = torch.cuda.current_stream()
    for _ in range(warmup):
        step.fwd()
        step.bwd()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clocks is not None:
        clocks.mark(True)
    start.record(st)
    for e0, e1, e2 in ev:
        e0.record(st)
        step.fwd()
        e1.record(st)
        step.bwd()
        e2.record(st)
    end.record(st)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark(False)
    total_ms = start.elapsed_time(end)
    fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    bwd_ms = [b.elapsed_time(c) for _, b, c in ev]
    return total_ms, fwd_ms, bwd_ms


def time_e2e(pair, steps: int, warmup: int, clocks=None):
    """Same metric through the public API with host buffers: every step copies its Q, K, V,
    dO in from pinned memory, runs fwd + bwd, and copies dQ, dK, dV out, all inside the
    timed region.  Two buffer sets and three streams (H2D, compute, D2H) let step n+1's
    inputs travel while step n computes and step n-1's gradients travel back, as a training
    loop would overlap them; events order each buffer set's reuse.  dO is copied after Q, K, V
    and only the backward pass waits for it, so it travels while the forward pass runs."""
    import torch
    comp = torch.cuda.current_stream()
    h2d_st, d2h_st = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {"h2d": [None, None], "h2d_do": [None, None], "comp": [None, None], "d2h": [None, None]}

    def event(stream):
        e = torch.cuda.Event()
        e.record(stream)
        return e

    def run(n):
        i = n % 2
        s = pair[i]
        with torch.cuda.stream(h2d_st):
            if ev["comp"][i] is not None:          # this set's inputs are free again
                h2d_st.wait_event(ev["comp"][i])
            s.h2d(slice(0, 3))                     # Q, K, V
            ev["h2d"][i] = event(h2d_st)
            s.h2d(slice(3, 4))                     # dO
            ev["h2d_do"][i] = event(h2d_st)
        comp.wait_event(ev["h2d"][i])
        if ev["d2h"][i] is not None:               # this set's gradients have left
            comp.wait_event(ev["d2h"][i])
        s.fwd()
        comp.wait_event(ev["h2d_do"][i])
        s.bwd()
        ev["comp"][i] = event(comp)
        with torch.cuda.stream(d2h_st):
            d2h_st.wait_event(ev["comp"][i])
            s.d2h()
            ev["d2h"][i] = event(d2h_st)

    def finish():
        for e in ev["d2h"]:
            if e is not None:
                comp.wait_event(e)

    for n in range(warmup):
        run(n)
    finish()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clocks is not None:
        clocks.mark(True)
    a.record(comp)
    h2d_st.wait_stream(comp)
    d2h_st.wait_stream(comp)
    for n in range(steps):
        run(n)
    finish()
    b.record(comp)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark(False)
    return a.elapsed_time(b)


def cpu_oracle_sample(w, seconds: float = 12.0, rows_per_slice: int = 512):
    """Times the fp64 oracle (as it stands) on row slices of one head of the workload until
    `seconds` have passed.  Returns (TFLOP/s by the same counting rule, description)."""
    import numpy as np
    import oracle
    from sdpa_workloads import make_inputs, Workload
    one = Workload(w.name, 1, 1, 1, w.s_q, w.s_kv, w.d, w.dtype, causal=w.causal)
    x = make_inputs(one, seed=0, with_do=True)
    q, k, v, do = (oracle.to_f64(t)[0, 0] for t in (x.q, x.k, x.v, x.do))
    flops, n_slices, t0 = 0.0, 0, time.perf_counter()
    r1 = w.s_q
    while time.perf_counter() - t0 < seconds and r1 > 0:
        r0 = max(0, r1 - rows_per_slice)
        rows = np.arange(r0, r1)
        oracle.forward_rows(q[r0:r1], rows, k, v, w.scale, w.causal)
        oracle.backward_dq_rows(q[r0:r1], do[r0:r1], rows, k, v, w.scale, w.causal)
        oracle.backward_kv_rows(q[r0:r1], do[r0:r1], rows, k, v, w.scale, w.causal)
        pairs = float(np.minimum(rows + 1, w.s_kv).sum()) if w.causal else float(len(rows) * w.s_kv)
        flops += 3.5 * 4.0 * w.d * pairs
        n_slices += 1
        r1 = r0
    dt = time.perf_counter() - t0
    desc = (f"fp64 numpy oracle: forward rows, dQ rows and dK/dV contributions of {n_slices} "
            f"slices of {rows_per_slice} query rows (the last, most-visible rows) of one head "
            f"of {w.name}; counted with the fwd+bwd rule on the visible pairs")
    return flops / dt / 1e12, desc


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = bench_workload()
    import numpy as np
    import oracle
    from sdpa_workloads import make_inputs, Workload
    one = Workload(w.name, 1, 1, 1, w.s_q, w.s_kv, w.d, w.dtype, causal=w.causal)
    x = make_inputs(one, seed=0, with_do=True)
    q, k, v, do = (oracle.to_f64(t)[0, 0] for t in (x.q, x.k, x.v, x.do))
    rows_per_step = 128

    def one_step(i):
        r1 = w.s_q - (i * rows_per_step) % w.s_q
        r0 = max(0, r1 - rows_per_step)
        rows = np.arange(r0, r1)
        oracle.forward_rows(q[r0:r1], rows, k, v, w.scale, w.causal)
        oracle.backward_dq_rows(q[r0:r1], do[r0:r1], rows, k, v, w.scale, w.causal)
        oracle.backward_kv_rows(q[r0:r1], do[r0:r1], rows, k, v, w.scale, w.causal)
        pairs = float(np.minimum(rows + 1, w.s_kv).sum()) if w.causal else float(len(rows) * w.s_kv)
        return 3.5 * 4.0 * w.d * pairs

    for i in range(args.warmup):
        one_step(i)
    flops, t0 = 0.0, time.perf_counter()
    for i in range(args.steps):
        flops += one_step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name} (bf16 causal d=128, b=2, h=16): one 128-row query "
                               f"slice of one head per step", "b": w.b, "h": w.h_q, "s": w.s_q,
                   "d": w.d, "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{rows_per_step} query rows of one head per step "
                                   f"(fwd rows, dQ rows, dK/dV contributions), fp64 numpy"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_profile_workload(args):
    """One untimed forward (and backward, for training workloads) of a named sweep workload:
    the command an ncu capture of that workload's kernels runs."""
    import torch
    from sdpa_workloads import all_workloads
    torch.cuda.set_device(0)
    ws = [w for w in all_workloads() if w.name == args.profile_workload]
    if not ws:
        print("unknown workload; choose one of: " + ", ".join(w.name for w in all_workloads()))
        return 2
    # A short sweep_one (3 warm-up + 3 timed calls each way, no graphs); a capture picks its
    # launches with -k / -s / -c.
    line = sweep_one(ws[0], load_peaks(), args, quick=True)
    print(json.dumps(line))
    return 0


def run_cuda(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init(world, "nccl")
    w = bench_workload()
    step = Step(w, seed=rank, device=device)
    peaks = load_peaks()

    if args.profile_step:
        step.fwd()
        step.bwd()
        torch.cuda.synchronize()
        assert step.sdpa.sdpa_device_error() == 0
        print("profile step done")
        return 0

    props = torch.cuda.get_device_properties(device)
    uuid = bus = None
    try:
        uuid = "GPU-" + str(props.uuid)
        bus = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id, props.pci_device_id)
    except Exception:
        pass
    twin = step.twin(device)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(uuid, bus)
    clocks.start()
    total_ms, fwd_ms, bwd_ms = time_device(step, args.steps, args.warmup, clocks)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    assert step.sdpa.sdpa_device_error() == 0, "device-side error during the timed region"

    step_flops = w.fwd_flops() + w.bwd_flops()
    units, seconds = aggregate(step_flops * args.steps, total_ms / 1e3, dist, device)
    value = units / seconds / 1e12

    # The end-to-end leg times as many steps as the device leg.
    e2e_steps = args.steps
    e2e_ms = time_e2e((step, twin), e2e_steps, max(3, args.warmup), clocks)
    clk = clocks.stop()
    e2e_units, e2e_s = aggregate(step_flops * e2e_steps, e2e_ms / 1e3, dist, device)

    fwd_avg = statistics.mean(fwd_ms)
    bwd_avg = statistics.mean(bwd_ms)
    fwd_tflops = w.fwd_flops() / (fwd_avg / 1e3) / 1e12
    bwd_tflops = w.bwd_flops() / (bwd_avg / 1e3) / 1e12
    peak = peaks["bf16_tflops"]
    traffic = _load_traffic()

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "training bf16 causal d=128 s=8192: b=2, h_q=h_kv=16, fwd (O+LSE) "
                               "+ bwd (dQ,dK,dV) per step",
                   "b": w.b, "h": w.h_q, "s": w.s_q, "d": w.d, "causal": True,
                   "l2": "inputs larger than L2 (Q,K,V,dO,O 67 MB each)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "fwd": {"tflops": fwd_tflops, "ms": fwd_avg, "frac_of_bf16_peak": fwd_tflops / peak},
        "bwd": {"tflops": bwd_tflops, "ms": bwd_avg, "frac_of_bf16_peak": bwd_tflops / peak},
        "roofline": {"bound": "tensor", "kernel": "sdpa_bwd (bwd_main dominant; pre and dQ-convert "
                     "launches included in the timed call)",
                     "achieved": bwd_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": bwd_tflops / peak, "peak_source": f"bf16_tflops ({peaks['source']}, burst)",
                     "traffic": traffic},
        "clocks": clk,
        "e2e": {"value": e2e_units / e2e_s / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": step.h2d_bytes(), "d2h_bytes_per_step": step.d2h_bytes(),
                "overlap": "2 buffer sets; H2D, compute and D2H on separate streams"},
        "gpu_launches": 4 * args.steps,
    }
    if rank == 0 and not args.no_cpu:
        cval, desc = cpu_oracle_sample(w, seconds=args.cpu_seconds)
        line["cpu_baseline"] = {"value": cval, "unit": UNIT, "cores": cpu_cores(),
                                "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def _load_traffic():
    """DRAM bytes per launch of the backward main kernel from the committed ncu capture, or
    None when there is none or the kernel's sources changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        m = hashlib.sha256()
        for rel in d["source_files"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                m.update(f.read())
        if m.hexdigest() != d["source_sha256"]:
            return None
        return d.get("bwd_main_dram_bytes_per_launch")
    except Exception:
        return None


def gemm_peak_tflops(dtype_name: str, n: int = 8192, reps: int = 20) -> float:
    """Best-of-`reps` dense n^3 GEMM throughput through the vendor library (CUDA events).

    bf16: torch.matmul.  e4m3: torch._scaled_mm with unit scales and a bf16 output (the
    FP8 denominator: MEASURED_PEAKS.json holds none)."""
    import torch
    dt = {"bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}[dtype_name]
    g = torch.Generator(device="cuda").manual_seed(0)
    a = torch.randn(n, n, device="cuda", generator=g).to(dt)
    b = torch.randn(n, n, device="cuda", generator=g).to(dt).t()
    one = torch.tensor(1.0, device="cuda")
    if dtype_name == "bf16":
        f = lambda: a @ b
    else:
        f = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    for _ in range(5):
        f()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(); f(); e.record()
        torch.cuda.synchronize()
        best = min(best, s.elapsed_time(e))
    return 2.0 * n ** 3 / best / 1e9


def run_measure_peaks(args):
    import torch
    torch.cuda.set_device(0)
    line = {"bf16_tflops_burst": gemm_peak_tflops("bf16"),
            "e4m3_tflops_burst": gemm_peak_tflops("e4m3"),
            "how": "8192^3 GEMM, best of 20, CUDA events; bf16 torch.matmul, e4m3 torch._scaled_mm"}
    print(json.dumps(line), flush=True)
    return 0


def run_sweep(args):
    """One line per configuration (for tables)."""
    import torch
    from sdpa_workloads import all_workloads
    torch.cuda.set_device(0)
    peaks = load_peaks()
    try:
        peaks["e4m3_tflops"] = gemm_peak_tflops("e4m3")
    except Exception:  # no FP8 GEMM in this torch build: report no FP8 fraction
        peaks["e4m3_tflops"] = None
    only = set(args.only.split(",")) if args.only else None
    for w in all_workloads():
        if w.name.startswith("tiny") or (only is not None and w.name not in only):
            continue
        try:
            line = sweep_one(w, peaks, args)
        except Exception as e:  # report and continue
            line = {"workload": w.name, "error": str(e)}
        print(json.dumps(line), flush=True)
    return 0


def graph_ms(fn, calls: int, reps: int = 10) -> float:
    """Device time of one `fn()` from CUDA-graph replays of `calls` back-to-back calls: no
    host work (argument marshalling, tensor-map encoding) between kernels, so small problems
    show their kernels' time rather than the host's.  Median over `reps` replays."""
    import torch
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        fn()                                  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(st)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            fn()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(); g.replay(); b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / calls)
    return statistics.median(ts)


def fwd_flops(w) -> float:
    """Forward FLOPs of a workload: its own counting rule, except that workloads with
    per-batch lengths or a bottom-right diagonal count 4*d FLOPs for every (row, key) pair
    a row can see."""
    if w.lens_q is None and not w.bottom_right:
        return w.fwd_flops()
    lq_all = w.lens_q or (w.s_q,) * w.b
    lkv_all = w.lens_kv or (w.s_kv,) * w.b
    pairs = 0
    for lq, lkv in zip(lq_all, lkv_all):
        if not w.causal:
            pairs += lq * lkv
            continue
        off = lkv - lq if w.bottom_right else 0
        for i in range(lq):   # row i sees keys j <= i + off
            pairs += min(max(i + off + 1, 0), lkv)
    return 4.0 * w.h_q * w.d * pairs


def sweep_one(w, peaks, args, quick: bool = False):
    import torch
    import attention_flashattention_sdpa_gb300 as sdpa
    from sdpa_workloads import make_inputs
    x = make_inputs(w, seed=0, with_do=w.backward)
    dev = lambda t: torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, device="cuda").copy_(t)
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    kw = {}
    odt = q.dtype if w.dtype != "e4m3" else torch.bfloat16
    if w.dtype == "e4m3":
        kw = dict(descale_q=torch.tensor([x.descale_q], device="cuda"),
                  descale_k=torch.tensor([x.descale_k], device="cuda"),
                  descale_v=torch.tensor([x.descale_v], device="cuda"))
    o = torch.empty_strided(q.shape, q.stride(), dtype=odt, device="cuda")
    lse = torch.empty(w.b, w.h_q, w.s_q, dtype=torch.float32, device="cuda") if (w.stats or w.backward) else None
    st = torch.cuda.current_stream()
    causal = "bottom_right" if w.bottom_right else w.causal
    if w.lens_q is not None:
        kw["seq_lens_q"] = torch.tensor(w.lens_q, dtype=torch.int32, device="cuda")
        kw["seq_lens_kv"] = torch.tensor(w.lens_kv, dtype=torch.int32, device="cuda")
    ff = fwd_flops(w)
    bf = 2.5 * ff
    mask = mask_t = None
    mask_ms = None
    if w.dropout > 0:
        n, n_t = sdpa.sdpa_dropout_mask_size(w.b, w.h_q, w.s_q, w.s_kv)
        mask = torch.empty(n // 4, dtype=torch.int32, device="cuda")
        mask_t = torch.empty(n_t // 4, dtype=torch.int32, device="cuda")
        gen = lambda: sdpa.sdpa_dropout_mask(w.b, w.h_q, w.s_q, w.s_kv, w.dropout, 1234, 0, mask, mask_t,
                                             causal=w.causal)
        for _ in range(3):
            gen()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st); gen(); b_.record(st)
        torch.cuda.synchronize()
        mask_ms = a.elapsed_time(b_)
        kw["dropout_p"], kw["dropout_mask"] = w.dropout, mask
    if w.bias:
        from sdpa_workloads import make_bias
        kw["bias"] = make_bias(w).cuda()
    fwd = lambda: sdpa.sdpa_fwd(q, k, v, o, lse, attn_scale=w.scale, causal=causal, alibi=w.alibi,
                                **kw)
    reps = 3 if quick else max(5, min(200, int(2e13 / max(ff, 1))))
    for _ in range(3):
        fwd()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st); fwd(); b.record(st)
        ts.append((a, b))
    torch.cuda.synchronize()
    fwd_ms = statistics.median(a.elapsed_time(b) for a, b in ts)
    peak = peaks["bf16_tflops"]
    line = {"workload": w.name, "fwd_ms": fwd_ms, "fwd_tflops": ff / fwd_ms / 1e9}
    calls = max(4, min(64, int(2e12 / max(ff, 1))))
    if not quick:
        gms = graph_ms(fwd, calls)
        line["fwd_ms_graph"] = gms
        line["fwd_tflops_graph"] = ff / gms / 1e9
    if mask_ms is not None:
        line["dropout_mask_ms"] = mask_ms
    es = 1 if w.dtype == "e4m3" else 2
    io_bytes = (q.numel() + k.numel() + v.numel()) * es + o.numel() * o.element_size() + \
        (lse.numel() * 4 if lse is not None else 0)
    line["fwd_hbm_gbs"] = io_bytes / fwd_ms / 1e6
    line["fwd_frac_of_bf16_peak"] = line["fwd_tflops"] / peak if w.dtype != "e4m3" else None
    if w.dtype == "e4m3" and peaks.get("e4m3_tflops"):
        line["e4m3_peak_tflops"] = peaks["e4m3_tflops"]
        line["fwd_frac_of_e4m3_peak"] = line["fwd_tflops"] / peaks["e4m3_tflops"]
    if w.backward:
        do = dev(x.do)
        dkw = {} if w.dropout == 0 else {"dropout_p": w.dropout, "dropout_mask_t": mask_t}
        if w.lens_q is not None:
            dkw["seq_lens_q"], dkw["seq_lens_kv"] = kw["seq_lens_q"], kw["seq_lens_kv"]
        if w.bias:
            dkw["bias"] = kw["bias"]
        if w.dtype == "e4m3":   # E4M3 Q, K, V and E5M2 dO; O and the gradients in bf16
            dkw.update(kw)
            dkw["descale_do"] = torch.tensor([x.descale_do], device="cuda")
        dq, dk, dv = (torch.empty(t.shape, dtype=odt, device="cuda") for t in (q, k, v))
        p = sdpa.make_problem(q, k, v, o, attn_scale=w.scale, causal=causal, dout=do, dq=dq, dk=dk, dv=dv,
                              descale_q=dkw.get("descale_q"), descale_k=dkw.get("descale_k"),
                              descale_v=dkw.get("descale_v"), descale_do=dkw.get("descale_do"),
                              bias=dkw.get("bias"), seq_lens_q=dkw.get("seq_lens_q"),
                              seq_lens_kv=dkw.get("seq_lens_kv"))
        ws = torch.empty(sdpa.sdpa_workspace_size(p, True), dtype=torch.uint8, device="cuda")
        bwd = lambda: sdpa.sdpa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, attn_scale=w.scale, causal=causal,
                                    alibi=w.alibi, **dkw)
        for _ in range(3):
            bwd()
        torch.cuda.synchronize()
        ts = []
        for _ in range(max(3, reps // 2)):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st); bwd(); b.record(st)
            ts.append((a, b))
        torch.cuda.synchronize()
        bwd_ms = statistics.median(a.elapsed_time(b) for a, b in ts)
        line["bwd_ms"] = bwd_ms
        if not quick:
            gb = graph_ms(bwd, max(2, calls // 2))
            line["bwd_ms_graph"] = gb
            line["bwd_tflops_graph"] = bf / gb / 1e9
        line["bwd_tflops"] = bf / bwd_ms / 1e9
        line["fwdbwd_tflops"] = (ff + bf) / (fwd_ms + bwd_ms) / 1e9
        line["fwdbwd_frac_of_bf16_peak"] = line["fwdbwd_tflops"] / peak
    assert sdpa.sdpa_device_error() == 0
    return line


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--profile-step", action="store_true")
    ap.add_argument("--profile-workload", default=None)
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--only", default=None, help="--sweep: comma-separated workload names")
    ap.add_argument("--measure-peaks", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args(argv)
    if args.warmup < 3 and not args.profile_step:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.profile_workload:
        return run_profile_workload(args)
    if args.measure_peaks:
        return run_measure_peaks(args)
    return run_cuda(args)


if __name__ == "__main__":
    sys.exit(main())
