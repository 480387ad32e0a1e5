"""Benchmark: Lightning Attention chunkwise prefill, tokens/s and fraction of roofline.

Workload: fixed-length MHA prefill, B=2, T=8192, H=HV=64, D=V=128, BF16 q/k/v/o,
FP32 initial state N(0, 0.02^2) per (sequence, head) read and FP32 final state
written (the seeded synthetic inputs of workloads.config(2)).  One step = one
call of la_prefill_fwd over that batch.  The step's inputs (1.07 GB of Q/K/V/O)
are larger than the 129 MB L2, so no flush is needed between steps.

Prints one JSON line (rank 0).  ``--impl reference`` times the FP64 CPU oracle on
the host cores instead (a bounded sample of the same workload per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LA prefill tokens/s and % of roofline (B=2,T=8192,H=64,D=V=128) on 1 GB300"
UNIT = "tokens/s"
WORKLOAD = "fixed MHA prefill B=2 T=8192 H=HV=64 D=V=128, bf16 q/k/v/o, fp32 h0 in + final state out"
B, T, H, HV, D, V = 2, 8192, 64, 64, 128, 128
TOKENS = B * T
# algorithmic bytes per step: Q + K read once per q/k head, V read, O written, h0 read, h_final written
ALG_BYTES = 2 * TOKENS * H * D * 2 + 2 * TOKENS * HV * V * 2 + 2 * B * HV * V * D * 4
# dense-tile FLOPs per step: 4*C*D*V + 4*C^2*D per 64-token chunk per value head
ALG_FLOPS = (TOKENS // 64) * HV * (4 * 64 * D * V + 4 * 64 * 64 * D)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
KERNEL_NAME = "la_prefill_fwd_kernel"
KERNEL_SOURCES = ["linear_attention_prefill_chunkwise_gb300/csrc/la_prefill_kernel.cuh",
                  "linear_attention_prefill_chunkwise_gb300/csrc/sm103_ptx.cuh",
                  "linear_attention_prefill_chunkwise_gb300/csrc/la_prefill_api.cu",
                  "linear_attention_prefill_chunkwise_gb300/csrc/la_host_common.h"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "la_prefill_fwd_kernel_B2_T8192_H64.dram.txt")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as fh:
                d = json.load(fh)
            hbm = d.get("hbm_gbs")
            if isinstance(hbm, dict):
                hbm = hbm.get("value")
            if hbm:
                return float(hbm), "measured"
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Dense BF16 tensor peak (burst) from MEASURED_PEAKS.json, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as fh:
                d = json.load(fh)
            tf = d.get("bf16_tflops")
            if isinstance(tf, dict):
                tf = tf.get("value")
            if tf:
                return float(tf), "measured"
        except (OSError, ValueError):
            pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def dram_traffic_per_launch():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernel source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    vals = {}
    with open(TRAFFIC_FILE) as fh:
        for line in fh:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return int(float(vals["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons sampled during the timed region.

    A thread polls NVML (read-only queries through ctypes on the driver's libnvidia-ml) about
    once a millisecond, so that even a timed region of a few milliseconds holds samples; only
    samples taken between mark_start() and mark_end() are summarised.  Without NVML it falls
    back to `nvidia-smi -lms`, started before the timed region and given time to print its
    first line."""

    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,temperature.gpu")

    def __init__(self, gpu_uuid: str, period_s: float = 0.001):
        self.uuid = gpu_uuid
        self.period = period_s
        self.samples = []  # (perf_counter, sm_mhz, max_mhz, power_w, reason names[, temperature_c])
        self.source = None
        self.t0 = self.t1 = None
        self._stop = None
        self._thread = None
        self._smi = None

    # ---- NVML through ctypes
    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) != 0:
            raise OSError(f"no NVML device {self.uuid}")
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons_fn

    def _nvml_loop(self, lib, h, reasons_fn):
        import ctypes
        sm, mx, pw, rs, tc = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        while not self._stop.is_set():
            ok = (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0 and
                  lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0)
            if ok:
                power = pw.value / 1000.0 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 else None
                names = [n for bit, n in self.REASON_BITS.items() if reasons_fn(h, ctypes.byref(rs)) == 0
                         and rs.value & bit]
                temp = float(tc.value) if lib.nvmlDeviceGetTemperature(h, 0, ctypes.byref(tc)) == 0 else None
                self.samples.append((time.perf_counter(), float(sm.value), float(mx.value), power, names, temp))
            self._stop.wait(self.period)

    # ---- nvidia-smi fallback
    def _smi_reader(self):
        for line in self._smi.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                names = [n for n, val in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                              "sw_power_cap"], parts[5:9]) if val.lower().startswith("active")]
                temp = float(parts[9]) if len(parts) > 9 and parts[9].replace(".", "", 1).isdigit() else None
                self.samples.append((time.perf_counter(), float(parts[1]), float(parts[2]), float(parts[3]),
                                     names, temp))
            except ValueError:
                continue

    def __enter__(self):
        import threading
        self._stop = threading.Event()
        try:
            lib, h, reasons_fn = self._nvml_open()
            self._thread = threading.Thread(target=self._nvml_loop, args=(lib, h, reasons_fn), daemon=True)
            self.source = "nvml"
        except (OSError, AttributeError):
            try:
                self._smi = subprocess.Popen(
                    ["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self._thread = threading.Thread(target=self._smi_reader, daemon=True)
                self.source = "nvidia-smi"
            except OSError:
                return self
        self._thread.start()
        deadline = time.perf_counter() + 5.0
        while not self.samples and time.perf_counter() < deadline:  # sampling is live before timing starts
            time.sleep(0.005)
        return self

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def __exit__(self, *exc):
        if self._stop is not None:
            self._stop.set()
        if self._smi is not None:
            self._smi.terminate()
            try:
                self._smi.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self._smi.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self):
        inside = [s for s in self.samples if self.t0 is not None and self.t1 is not None and self.t0 <= s[0] <= self.t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0,
                    "source": self.source}
        reasons = sorted({n for s in inside for n in s[4]})
        power = [s[3] for s in inside if s[3] is not None]
        temps = [s[5] for s in inside if len(s) > 5 and s[5] is not None]
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "power_w_median": statistics.median(power) if power else None,
                "temperature_c_max": max(temps) if temps else None, "samples": len(inside), "source": self.source}


def gpu_id_for_smi(device) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except (AttributeError, RuntimeError):
        return str(device.index)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, world, device=None):
    """The largest of every rank's ``x`` (the slowest rank's time); ``x`` itself on one rank.
    Uses the default process group (NCCL with CUDA tensors, gloo with CPU tensors)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, steps, world, slowest_ms):
    """Whole-job throughput of ``world`` replicas, each processing ``units_per_rank`` per step,
    over ``steps`` steps that took ``slowest_ms`` on the slowest rank."""
    return world * units_per_rank * steps / (slowest_ms / 1e3)


def pin_to_gpu_numa_node(device):
    """Run this process on the CPUs next to ``device`` (the PCI device's local_cpulist) so that
    the pinned host buffers allocated next are first touched on the GPU's own NUMA node.
    Returns (CPU list used or None, the previous affinity to restore afterwards)."""
    import subprocess
    before = os.sched_getaffinity(0)
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader",
                              "-i", gpu_id_for_smi(device)], capture_output=True, text=True, timeout=20).stdout
        dom, rest = out.strip().split(":", 1)
        path = f"/sys/bus/pci/devices/{int(dom, 16):04x}:{rest.lower()}/local_cpulist"
        with open(path) as fh:
            spec = fh.read().strip()
        cpus = set()
        for part in spec.split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        cpus &= before
        if not cpus:
            return None, before
        os.sched_setaffinity(0, cpus)
        return spec, before
    except (OSError, ValueError, subprocess.SubprocessError):
        return None, before


def make_inputs(device):
    import numpy as np
    import torch

    import workloads as W
    p = W.config(2)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    host = {"q": bf(p.q_bits), "k": bf(p.k_bits), "v": bf(p.v_bits), "slopes": torch.from_numpy(p.slopes),
            "h0": torch.from_numpy(p.h0)}
    dev = {k_: t.to(device) for k_, t in host.items()}
    dev["o"] = torch.empty((TOKENS, HV, V), dtype=torch.bfloat16, device=device)
    dev["h_final"] = torch.empty((B, HV, V, D), dtype=torch.float32, device=device)
    return p, host, dev


def run_cuda(args):
    import torch
    import torch.distributed as dist

    import linear_attention_prefill_chunkwise_gb300 as lap

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    p, host, dev = make_inputs(device)
    scale = p.scale

    def step(d, s):
        lap.la_prefill_fwd(d["q"], d["k"], d["v"], d["slopes"], scale, h0=d["h0"], o=d["o"],
                           h_final=d["h_final"], seq_len=T, stream=s)

    def barrier():
        if world > 1:
            dist.barrier(device_ids=[device.index])

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(dev, stream)
    torch.cuda.synchronize(device)

    # ---- device-resident timing: K steps, one kernel launch each, back to back between two
    #      events on the launch stream (an event between launches would add its own gap)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    barrier()
    torch.cuda.synchronize(device)
    with ClockSampler(gpu_id_for_smi(device)) as clk:
        clk.mark_start()
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for i in range(args.steps):
                step(dev, stream)
            ev[1].record(stream)
        torch.cuda.synchronize(device)
        clk.mark_end()
    barrier()
    region_ms = ev[0].elapsed_time(ev[1])
    total_ms = max_over_ranks(region_ms, world, device)
    ms_per_step = total_ms / args.steps
    value = job_throughput(TOKENS, args.steps, world, total_ms)

    # ---- end to end through the public API: every step copies its inputs from pinned host
    #      memory and reads its outputs (o and the final states) back.  Steps are pipelined
    #      over two device buffer sets, as a serving loop runs them: the inputs of step i+1
    #      travel (copy stream) while step i computes (launch stream) and the outputs of step
    #      i-1 return (return stream).
    numa, affinity = pin_to_gpu_numa_node(device)
    pinned = {k_: t.pin_memory() for k_, t in host.items()}
    nset = 2
    out_o = [torch.empty((TOKENS, HV, V), dtype=torch.bfloat16).pin_memory() for _ in range(nset)]
    out_h = [torch.empty((B, HV, V, D), dtype=torch.float32).pin_memory() for _ in range(nset)]
    os.sched_setaffinity(0, affinity)  # the buffers are placed; the CPU baseline gets every core back
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = out_o[0].numel() * out_o[0].element_size() + out_h[0].numel() * out_h[0].element_size()
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    sets = []
    for _ in range(nset):
        sb = {k_: torch.empty_like(t, device=device) for k_, t in pinned.items()}
        sb["o"] = torch.empty((TOKENS, HV, V), dtype=torch.bfloat16, device=device)
        sb["h_final"] = torch.empty((B, HV, V, D), dtype=torch.float32, device=device)
        sets.append(sb)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_loaded = [torch.cuda.Event() for _ in range(nset)]
    ev_done = [torch.cuda.Event() for _ in range(nset)]
    ev_back = [torch.cuda.Event() for _ in range(nset)]
    used = [False] * nset

    def e2e_step(i):
        b = i % nset
        sb = sets[b]
        if used[b]:
            s_in.wait_event(ev_done[b])      # the set's previous kernel has read its inputs
            stream.wait_event(ev_back[b])    # and its previous outputs have been copied back
        with torch.cuda.stream(s_in):
            for k_, t in pinned.items():
                sb[k_].copy_(t, non_blocking=True)
            ev_loaded[b].record(s_in)
        stream.wait_event(ev_loaded[b])
        step(sb, stream)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            out_o[b].copy_(sb["o"], non_blocking=True)
            out_h[b].copy_(sb["h_final"], non_blocking=True)
            ev_back[b].record(s_out)
        used[b] = True

    for i in range(2 * nset):
        e2e_step(i)
    torch.cuda.synchronize(device)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)  # after the last step's outputs are back, which follow every earlier copy and launch
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, device)
    e2e_value = job_throughput(TOKENS, e2e_steps, world, e2e_ms)

    if rank == 0:
        peak, peak_kind = measured_peaks()
        tflops, tf_kind = measured_bf16_tflops()
        launch_ms = region_ms / args.steps  # this rank's average launch duration over the timed region
        achieved = ALG_BYTES / (launch_ms / 1e3) / 1e9
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": B * world, "seq_len": T, "heads": H, "value_heads": HV,
                       "head_dim": D, "chunk": 64, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (1.07 GB per step), no flush"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": dram_traffic_per_launch(),
                         "peak_source": f"{peak_kind} hbm_gbs", "alg_bytes_per_launch": ALG_BYTES,
                         "alg_flops_per_launch": ALG_FLOPS, "kernel": KERNEL_NAME,
                         "launch_ms_mean": round(launch_ms, 5),
                         "tensor": {"achieved": round(ALG_FLOPS / (launch_ms / 1e3) / 1e12, 1), "peak": tflops,
                                    "unit": "TFLOP/s",
                                    "frac": round(ALG_FLOPS / (launch_ms / 1e3) / 1e12 / tflops, 4),
                                    "peak_source": f"{tf_kind} bf16_tflops (dense)"}},
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "pipelined": "2 buffer sets: copy-in, launch and copy-out streams",
                    "host_numa": numa},
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(p, args.cpu_heads)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def workload_roofline(p):
    """Algorithmic bytes and dense-tile FLOPs of one call on workload ``p``: per non-padded
    sequence, Q and K once per q/k head, V read and O written per value head, h0 read and the
    final state written per value head when present; 4*C*D*V + 4*C^2*D FLOPs per 64-token
    chunk (C = 64) per value head.  Returns (tokens, bytes, flops)."""
    import numpy as np
    lengths = p.lengths()
    live = np.ones(len(lengths), dtype=bool) if p.state_indices is None else p.state_indices >= 0
    toks = int(lengths[live].sum())
    nseq = int(live.sum())
    d, v = p.D, p.V
    state_bytes = p.HV * v * d * 4
    nbytes = 2 * toks * p.H * d * 2 + 2 * toks * p.HV * v * 2
    if p.h0 is not None:
        nbytes += nseq * state_bytes
    if p.want_final:
        nbytes += nseq * state_bytes
    chunks = int(((lengths[live] + 63) // 64).sum())
    flops = chunks * p.HV * (4 * 64 * d * v + 4 * 64 * 64 * d)
    return toks, nbytes, flops


def run_sweep(args):
    """Every workload of workloads.config(1..5): mean kernel time over ``--sweep-steps``
    launches (CUDA events around each launch, L2 flushed between launches by writing a
    256 MB buffer), tokens/s over non-padded tokens, and the fraction of the roofline
    max(bytes / HBM peak, FLOPs / BF16 tensor peak).  One JSON line per workload."""
    import numpy as np
    import torch

    import linear_attention_prefill_chunkwise_gb300 as lap
    import workloads as W

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    hbm, hbm_kind = measured_peaks()
    tflops, tf_kind = measured_bf16_tflops()

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)

    # (label, problem): the five workloads, then the other head dimensions
    work = [(i, None) for i in range(1, 6)] + [
        ("d64", W.custom(seed=3002, B=2, T=8192, H=64, HV=64, D=64,
                         name="D=V=64 fixed MHA B=2 T=8192 H=HV=64, h0 + final state")),
        ("d64_short", short_d64_problem()),
        ("d256", W.custom(seed=3010, B=2, T=8192, H=16, HV=16, D=256,
                          name="D=V=256 fixed B=2 T=8192 H=HV=16, h0 + final state")),
        ("d256_short", d256_short_problem()),
        ("d256_short_packed", short_d64_problem(D=256, H=16, seed=1106))]
    for label, extra_p in (work if args.sweep_what in ("all", "prefill") else ()):
        p = W.config(label) if extra_p is None else extra_p
        q, k, v = bf(p.q_bits), bf(p.k_bits), bf(p.v_bits)
        sl = torch.from_numpy(p.slopes).to(device)
        h0 = None if p.h0 is None else torch.from_numpy(p.h0).to(device)
        idx = None if p.state_indices is None else torch.from_numpy(p.state_indices).to(device)
        cu = None if p.cu_seqlens is None else torch.from_numpy(p.cu_seqlens).to(device)
        o = torch.empty((p.tokens, p.HV, p.V), dtype=torch.bfloat16, device=device)
        if p.in_place:
            hf = h0
        elif p.want_final:
            hf = torch.empty((p.pool_size, p.HV, p.V, p.D), dtype=torch.float32, device=device)
        else:
            hf = None

        if p.D == 256:
            ws = torch.empty(lap.la_prefill_d256_workspace(p.B, p.T, p.N, p.HV, h0 is not None or hf is not None),
                             dtype=torch.uint8, device=device)

            def call():
                lap.la_prefill_fwd_d256(q, k, v, sl, p.scale, h0=h0, state_indices=idx, cu_seqlens=cu, o=o,
                                        h_final=hf, seq_len=None if cu is not None else p.T, workspace=ws,
                                        stream=stream)
        else:
            def call():
                lap.la_prefill_fwd(q, k, v, sl, p.scale, h0=h0, state_indices=idx, cu_seqlens=cu, o=o, h_final=hf,
                                   seq_len=None if cu is not None else p.T, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(3):
                call()
            times = []
            for _ in range(args.sweep_steps):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call()
                e1.record(stream)
                times.append((e0, e1))
        torch.cuda.synchronize(device)
        ms = statistics.fmean(a.elapsed_time(b) for a, b in times)
        toks, nbytes, flops = workload_roofline(p)
        t_roof = max(nbytes / (hbm * 1e9), flops / (tflops * 1e12))
        line = {"sweep": True, "workload": label, "name": p.name, "ms": round(ms, 5),
                "tokens_per_s": round(toks / (ms / 1e3), 1), "tokens": toks, "alg_bytes": nbytes,
                "alg_flops": flops, "achieved_gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
                "roofline_ms": round(t_roof * 1e3, 5), "frac": round(t_roof * 1e3 / ms, 4),
                "bound": "hbm" if nbytes / (hbm * 1e9) >= flops / (tflops * 1e12) else "tensor",
                "peaks": {"hbm_gbs": hbm, "hbm_source": hbm_kind, "bf16_tflops": tflops, "tflops_source": tf_kind},
                "steps": args.sweep_steps, "l2": "flushed between launches (256 MB write)"}
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = oracle_forward_baseline(p, ms)
        print(json.dumps(line), flush=True)
    if args.sweep_what in ("all", "decode"):
        run_decode_sweep(args, device, stream, flush, hbm, hbm_kind)
    if args.sweep_what in ("all", "segmented"):
        run_segment_sweep(args, device, stream, flush, hbm, hbm_kind, tflops, tf_kind)
    if args.sweep_what in ("all", "backward"):
        run_backward_sweep(args, device, stream, flush, hbm, hbm_kind)


def short_d64_problem(D=64, H=64, seed=1105):
    """The short-continuation workload (128 requests of 8 tokens, 256-slot pool, 16 padded) at
    D = V = 64 (H=HV=64), or another head dimension and head count."""
    import numpy as np
    import workloads as W
    rng = np.random.default_rng(seed)
    idx = rng.permutation(256)[:128].astype(np.int32)
    idx[rng.choice(128, 16, replace=False)] = -1
    return W.custom(seed=seed, lengths=[8] * 128, H=H, HV=H, D=D, pool=256, indices=idx, in_place=True,
                    name=f"D=V={D} short packed N=128 T=8 H=HV={H}, 256-slot pool, 16 padded")


def d256_short_problem():
    """128 fixed-length sequences of 8 tokens at D = V = 256, H=HV=16, 256-slot pool in place
    with 16 padded (the tokenwise path of la_prefill_fwd_d256)."""
    import numpy as np
    import workloads as W
    rng = np.random.default_rng(1107)
    idx = rng.permutation(256)[:128].astype(np.int32)
    idx[rng.choice(128, 16, replace=False)] = -1
    return W.custom(seed=1107, B=128, T=8, H=16, HV=16, D=256, pool=256, indices=idx, in_place=True,
                    name="D=V=256 short fixed B=128 T=8 H=HV=16, 256-slot pool, 16 padded")


def run_decode_sweep(args, device, stream, flush, hbm, hbm_kind):
    """The speculative-decoding ops on the short-continuation workload (workloads.config(5):
    128 requests of 8 draft tokens, H=HV=64, 256-slot pool, 16 padded), and on the same shape
    at D = V = 64, and at D = V = 256 with H=HV=16: MTP decode, verify with the KV-buffer copy, and commit of every accepted
    token.  Bytes: per live (request, value head) the state (64 KB, or 16 KB at D = 64) read
    (and written, decode and commit), the tokens' q, k (once per q/k head), v and o, and the
    KV buffer written (verify) or read (commit)."""
    for p in (__import__("workloads").config(5), short_d64_problem(), short_d64_problem(D=256, H=16, seed=1106)):
        decode_sweep_one(args, p, device, stream, flush, hbm, hbm_kind)


def decode_sweep_one(args, p, device, stream, flush, hbm, hbm_kind):
    import numpy as np
    import torch

    import linear_attention_prefill_chunkwise_gb300 as lap

    D, V = p.D, p.V
    Bq, Tq = p.N, 8
    live = int((p.state_indices >= 0).sum())
    toks = live * Tq
    state_b = live * p.HV * V * D * 4
    tok_b = toks * (2 * p.H * D * 2 + 2 * p.HV * V * 2)
    kv_b = toks * (p.H * D * 2 + p.HV * V * 2)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)

    q, k, v = bf(p.q_bits), bf(p.k_bits), bf(p.v_bits)
    sl = torch.from_numpy(p.slopes).to(device)
    pool = torch.from_numpy(p.h0).to(device)
    idx = torch.from_numpy(p.state_indices).to(device)
    o = torch.empty((p.tokens, p.HV, V), dtype=torch.bfloat16, device=device)
    kbuf = torch.zeros((p.pool_size, Tq, p.H, D), dtype=torch.bfloat16, device=device)
    vbuf = torch.zeros((p.pool_size, Tq, p.HV, V), dtype=torch.bfloat16, device=device)
    acc = torch.full((Bq,), Tq, dtype=torch.int32, device=device)
    ops = {
        "la_decode_mtp": (lambda: lap.la_decode_mtp(q, k, v, sl, p.scale, pool, Tq, state_indices=idx, o=o,
                                                    stream=stream), 2 * state_b + tok_b),
        "la_verify": (lambda: lap.la_verify(q, k, v, sl, p.scale, pool, Tq, state_indices=idx, o=o, kbuf=kbuf,
                                            vbuf=vbuf, stream=stream), state_b + tok_b + kv_b),
        "la_commit": (lambda: lap.la_commit(pool, kbuf, vbuf, acc, sl, state_indices=idx, stream=stream),
                      2 * state_b + kv_b),
    }
    # the oracle's recurrence over the same requests and draft tokens (decode's outputs and states;
    # verify's outputs; commit's states with every token accepted): one CPU time for the three
    if not args.no_cpu_baseline:
        import oracle
        threads = oracle.max_threads()
        t0 = time.perf_counter()
        oracle.tokenwise(p.q(), p.k(), p.v(), p.slopes, p.scale, h0=p.h0.astype(np.float64),
                         state_indices=p.state_indices, cu_seqlens=p.cu_seqlens, nthreads=threads)
        cpu_ms = (time.perf_counter() - t0) * 1e3
    for name, (fn, nbytes) in ops.items():
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            times = []
            for _ in range(args.sweep_steps):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                times.append((e0, e1))
        torch.cuda.synchronize(device)
        ms = statistics.fmean(a.elapsed_time(b) for a, b in times)
        t_roof = nbytes / (hbm * 1e9)
        line = {"sweep": True, "op": name, "workload": f"B=128 requests x T=8 draft tokens, H=HV={p.HV}, D=V={D}, "
                "256-slot pool, 16 padded", "ms": round(ms, 5), "tokens_per_s": round(toks / (ms / 1e3), 1),
                "alg_bytes": nbytes, "achieved_gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
                "roofline_ms": round(t_roof * 1e3, 5), "frac": round(t_roof * 1e3 / ms, 4), "bound": "hbm",
                "peaks": {"hbm_gbs": hbm, "hbm_source": hbm_kind}, "steps": args.sweep_steps,
                "l2": "flushed between launches (256 MB write)"}
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = {"ms": round(cpu_ms, 2), "cores": threads, "kind": "oracle",
                                    "gpu_speedup": round(cpu_ms / ms, 1),
                                    "sample": "every request and head, all 8 tokens (FP64 tokenwise recurrence, "
                                              "OpenMP over (request, head))"}
        print(json.dumps(line), flush=True)


SEGMENT_WORKLOADS = (
    # (seed, B, T, H, HV, name)
    (2001, 1, 8192, 64, 64, "one 8K prompt, H=HV=64"),
    (2002, 1, 32768, 16, 16, "B=1 T=32768 H=HV=16 (a 4-way head shard)"),
    (2003, 1, 65536, 8, 8, "B=1 T=65536 H=HV=8 (an 8-way head shard)"),
    (2004, 2, 8192, 64, 64, "fixed MHA B=2 T=8192 H=64"),
    (2005, 1, 32768, 16, 16, "D=V=64: B=1 T=32768 H=HV=16"),
    (2006, 1, 32768, 4, 4, "D=V=256: B=1 T=32768 H=HV=4"),
)


def run_segment_sweep(args, device, stream, flush, hbm, hbm_kind, tflops, tf_kind):
    """Segmented-sequence prefill against the plain chunkwise prefill on batches with few
    (sequence, value head) chains: fixed length, random h0, final state returned.  Same
    timing as the other sweeps; the roofline is the plain prefill's (the segmented path's
    extra pass over K and V is overhead, not work)."""
    import numpy as np
    import torch

    import linear_attention_prefill_chunkwise_gb300 as lap
    import workloads as W

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            times = []
            for _ in range(args.sweep_steps):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                times.append((e0, e1))
        torch.cuda.synchronize(device)
        return statistics.fmean(a.elapsed_time(b) for a, b in times)

    for seed, B, T, H, HV, name in SEGMENT_WORKLOADS:
        Dw = 64 if name.startswith("D=V=64") else 256 if name.startswith("D=V=256") else 128
        p = W.custom(seed=seed, B=B, T=T, H=H, HV=HV, name=name, D=Dw)
        q, k, v = bf(p.q_bits), bf(p.k_bits), bf(p.v_bits)
        sl = torch.from_numpy(p.slopes).to(device)
        h0 = torch.from_numpy(p.h0).to(device)
        o = torch.empty((p.tokens, HV, p.V), dtype=torch.bfloat16, device=device)
        hf = torch.empty_like(h0)
        if Dw == 256:
            nbytes_ws, seg = lap.la_prefill_d256_segmented_workspace(B, T, B, HV, False, 0, True)
            ws = torch.empty(max(nbytes_ws, 1), dtype=torch.uint8, device=device)
            ws_plain = torch.empty(lap.la_prefill_d256_workspace(B, T, B, HV, True), dtype=torch.uint8, device=device)
            ms_plain = timed(lambda: lap.la_prefill_fwd_d256(q, k, v, sl, p.scale, h0=h0, o=o, h_final=hf, seq_len=T,
                                                             workspace=ws_plain, stream=stream))
            ms_seg = timed(lambda: lap.la_prefill_fwd_d256_segmented(q, k, v, sl, p.scale, h0=h0, o=o, h_final=hf,
                                                                     seq_len=T, segment_len=0, workspace=ws,
                                                                     stream=stream))
        else:
            nbytes_ws, seg = lap.la_prefill_segmented_workspace(B, T, B, HV, False, 0)
            ws = torch.empty(max(nbytes_ws, 1), dtype=torch.uint8, device=device)
            ms_plain = timed(lambda: lap.la_prefill_fwd(q, k, v, sl, p.scale, h0=h0, o=o, h_final=hf, seq_len=T,
                                                        stream=stream))
            ms_seg = timed(lambda: lap.la_prefill_fwd_segmented(q, k, v, sl, p.scale, h0=h0, o=o, h_final=hf,
                                                                seq_len=T, segment_len=0, workspace=ws, stream=stream))
        toks, nbytes, flops = workload_roofline(p)
        t_roof = max(nbytes / (hbm * 1e9), flops / (tflops * 1e12))
        cpu = None if args.no_cpu_baseline else oracle_forward_baseline(p, ms_seg)
        print(json.dumps({"sweep": True, "op": "la_prefill_fwd_segmented", "workload": name, "segment_len": seg,
                          "chains": B * HV, "workspace_bytes": nbytes_ws, "ms": round(ms_seg, 5),
                          "ms_plain": round(ms_plain, 5), "speedup_vs_plain": round(ms_plain / ms_seg, 3),
                          "tokens_per_s": round(toks / (ms_seg / 1e3), 1), "alg_bytes": nbytes,
                          "achieved_gbs": round(nbytes / (ms_seg / 1e3) / 1e9, 1),
                          "roofline_ms": round(t_roof * 1e3, 5), "frac": round(t_roof * 1e3 / ms_seg, 4),
                          "frac_plain": round(t_roof * 1e3 / ms_plain, 4),
                          "peaks": {"hbm_gbs": hbm, "hbm_source": hbm_kind, "bf16_tflops": tflops,
                                    "tflops_source": tf_kind},
                          "steps": args.sweep_steps, "l2": "flushed between launches (256 MB write)",
                          **({} if cpu is None else {"cpu_baseline": cpu})}), flush=True)


def run_backward_sweep(args, device, stream, flush, hbm, hbm_kind):
    """The backward pass (la_prefill_bwd) with dL/do and dL/dh_final given and dh0 returned, on
    the bench shape (B=2, T=8192, H=HV=64, h0 given) and on the GVA shape of workload 4 (B=4,
    T=16384, H=16 q/k heads, HV=64 value heads, no h0).  Algorithmic bytes: q, k, dq, dk once per
    q/k head, v, dout, dv once per value head, h0 (when given), dh_final and dh0 once; the three
    chunkwise runs, the state transposes and (GVA) the FP32 parts of dq and dk move more."""
    import numpy as np
    import torch

    import linear_attention_prefill_chunkwise_gb300 as lap
    import workloads as W

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)

    for cfg, seed in ((2, 4402), (4, 4404)):
        p = W.config(cfg)
        Bp, Tp, Hp, HVp = p.B, p.T, p.H, p.HV
        G = HVp // Hp
        rng = np.random.default_rng(seed)
        q, k, v = bf(p.q_bits), bf(p.k_bits), bf(p.v_bits)
        dout = bf(W.bf16_bits(rng.standard_normal(p.v_bits.shape, dtype=np.float32)))
        sl = torch.from_numpy(p.slopes).to(device)
        h0 = None if p.h0 is None else torch.from_numpy(p.h0).to(device)
        dhf = torch.randn((Bp, HVp, V, D), generator=torch.Generator(device=device).manual_seed(seed + 1),
                          device=device) * 0.1
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dh0 = torch.empty_like(dhf)
        ws = torch.empty(max(lap.la_prefill_bwd_workspace(Bp, Tp, Hp, HVp, D, Bp, h0 is not None, True), 256),
                         dtype=torch.uint8, device=device)

        def call():
            lap.la_prefill_bwd(q, k, v, sl, p.scale, dout, h0=h0, dh_final=dhf, dq=dq, dk=dk, dv=dv, dh0=dh0,
                               seq_len=Tp, workspace=ws, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(3):
                call()
            times = []
            for _ in range(args.sweep_steps):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call()
                e1.record(stream)
                times.append((e0, e1))
        torch.cuda.synchronize(device)
        ms = statistics.fmean(a.elapsed_time(b) for a, b in times)
        toks = Bp * Tp
        nbytes = 4 * toks * Hp * D * 2 + 3 * toks * HVp * V * 2 + (2 + (h0 is not None)) * Bp * HVp * V * D * 4
        t_roof = nbytes / (hbm * 1e9)
        line = {"sweep": True, "op": "la_prefill_bwd",
                "workload": (WORKLOAD if cfg == 2 else p.name) + ", dL/do and dL/dh_final in, dh0 out",
                "ms": round(ms, 5), "tokens_per_s": round(toks / (ms / 1e3), 1), "alg_bytes": nbytes,
                "achieved_gbs": round(nbytes / (ms / 1e3) / 1e9, 1), "roofline_ms": round(t_roof * 1e3, 5),
                "frac": round(t_roof * 1e3 / ms, 4), "bound": "hbm",
                "peaks": {"hbm_gbs": hbm, "hbm_source": hbm_kind}, "steps": args.sweep_steps,
                "l2": "flushed between launches (256 MB write)"}
        if not args.no_cpu_baseline:
            # the oracle's backward over every sequence and the first q/k heads (with their value
            # heads, 8 or so), scaled to all heads
            import oracle
            nq = max(1, 8 // G)
            nv = nq * G
            threads = oracle.max_threads()
            dout_h = W.bf16_to_f32(dout.view(torch.int16).cpu().numpy().view(np.uint16))
            t0 = time.perf_counter()
            oracle.backward(p.q()[:, :nq], p.k()[:, :nq], p.v()[:, :nv], p.slopes[:nv], p.scale, dout_h[:, :nv],
                            h0=None if p.h0 is None else p.h0[:, :nv].astype(np.float64),
                            dh_final=dhf[:, :nv].cpu().numpy().astype(np.float64), T=Tp, nthreads=threads)
            cpu_ms = (time.perf_counter() - t0) * 1e3 * HVp / nv
            line["cpu_baseline"] = {"ms": round(cpu_ms, 2), "cores": threads, "kind": "oracle",
                                    "gpu_speedup": round(cpu_ms / ms, 1),
                                    "sample": f"B={Bp} x T={Tp} tokens x {nv} of {HVp} value heads ({nq} of {Hp} "
                                              "q/k heads), scaled to all heads (FP64 forward and reverse sweeps, "
                                              "OpenMP over (sequence, q/k head))"}
        print(json.dumps(line), flush=True)
        del q, k, v, dout, dq, dk, dv, dh0, dhf, h0, ws
        torch.cuda.empty_cache()


def oracle_forward_baseline(p, gpu_ms, sample="the whole workload"):
    """The FP64 oracle's tokenwise recurrence on the host cores over workload ``p`` (every
    sequence and head, its initial states and pool): the CPU time of the same call beside the
    GPU's."""
    import numpy as np

    import oracle
    threads = oracle.max_threads()
    h0 = None if p.h0 is None else p.h0.astype(np.float64)
    t0 = time.perf_counter()
    oracle.tokenwise(p.q(), p.k(), p.v(), p.slopes, p.scale, h0=h0, state_indices=p.state_indices,
                     cu_seqlens=p.cu_seqlens, T=None if p.cu_seqlens is not None else p.T, want_state=p.want_final,
                     nthreads=threads)
    ms = (time.perf_counter() - t0) * 1e3
    return {"ms": round(ms, 2), "cores": threads, "kind": "oracle", "gpu_speedup": round(ms / gpu_ms, 1),
            "sample": f"{sample} (FP64 tokenwise recurrence, OpenMP over (sequence, head))"}


def cpu_baseline(p, heads):
    """The FP64 oracle on the host cores over a bounded sample: both sequences, all T tokens,
    the first `heads` of the 64 heads.  Reported in full-workload tokens/s (a token = all 64 heads)."""
    import numpy as np

    import oracle
    q = p.q()[:, :heads]
    k = p.k()[:, :heads]
    v = p.v()[:, :heads]
    h0 = p.h0[:, :heads].astype(np.float64)
    threads = oracle.max_threads()
    t0 = time.perf_counter()
    oracle.tokenwise(q, k, v, p.slopes[:heads], p.scale, h0=h0, T=T, nthreads=threads)
    dt = time.perf_counter() - t0
    equiv_tokens = TOKENS * heads / HV
    return {"value": round(equiv_tokens / dt, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"B=2 x T=8192 tokens x {heads} of {HV} heads (FP64 tokenwise recurrence, OpenMP over "
                      f"(sequence, head)); wall {dt:.2f} s"}


def oracle_step(p, ntok, nheads):
    """One reference step: the oracle over sequence 0's first `ntok` tokens and `nheads` heads,
    with its initial states.  Returns (seconds, full-workload-equivalent tokens, threads)."""
    import numpy as np

    import oracle
    q = p.q()[:ntok, :nheads]
    k = p.k()[:ntok, :nheads]
    v = p.v()[:ntok, :nheads]
    h0 = p.h0[:1, :nheads].astype(np.float64)
    threads = oracle.max_threads()
    t0 = time.perf_counter()
    oracle.tokenwise(q, k, v, p.slopes[:nheads], p.scale, h0=h0, T=ntok, nthreads=threads)
    return time.perf_counter() - t0, ntok * nheads / HV, threads


def run_reference(args):
    """The oracle, as it stands, on the host cores.  Each step is a bounded sample of the
    workload (one sequence, one head per host thread, a token count sized so that all
    warm-up and timed steps together take about --ref-budget seconds)."""
    import workloads as W
    rank, world, _ = dist_env()
    if rank != 0:
        return
    p = W.config(2)
    import oracle
    nheads = max(1, min(HV, oracle.max_threads()))
    dt, _, _ = oracle_step(p, 256, nheads)  # calibration
    per_step = args.ref_budget / (args.steps + args.warmup)
    ntok = int(max(64, min(T, 256 * per_step / max(dt, 1e-6))))
    for _ in range(args.warmup):
        oracle_step(p, ntok, nheads)
    secs, toks = 0.0, 0.0
    threads = 1
    for _ in range(args.steps):
        dt, eq, threads = oracle_step(p, ntok, nheads)
        secs += dt
        toks += eq
    value = toks / secs
    sample = (f"sequence 0, first {ntok} of {T} tokens, {nheads} of {HV} heads per step, with h0 "
              f"(FP64 tokenwise recurrence, OpenMP over heads); value in full-workload tokens/s")
    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": WORKLOAD, "global_batch": B, "seq_len": T, "heads": H, "value_heads": HV,
                       "head_dim": D, "chunk": 64, "parallelism": "host cores"},
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-heads", type=int, default=64, help="heads in the oracle CPU-baseline sample")
    ap.add_argument("--ref-budget", type=float, default=60.0, help="seconds for the whole reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="time every workload (1..5) instead, one JSON line each (not the headline line)")
    ap.add_argument("--sweep-steps", type=int, default=50)
    ap.add_argument("--sweep-what", choices=["all", "prefill", "decode", "segmented", "backward"], default="all",
                    help="with --sweep: the five prefill workloads, the speculative-decoding ops, the "
                         "segmented prefill on few-chain batches, or all of them")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
