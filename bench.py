#!/usr/bin/env python3
"""Benchmark of the FlashAttention hot path on one GB300 (or N replicas under torchrun).

One step = one pass of the whole path over one batch of synthetic inputs:
  1. split-KV decode   B=32 H=32 Nq=1 Nk=32768 d=64 bf16, 16 splits, seeded merge order
                       (split kernel + merge kernel)
  2. bf16 prefill      B=4  H=16 N=4096 d=64
  3. bf16 prefill      B=2  H=16 N=8192 d=128, Q and K ~ 3 N(0,1)
`value` is the prefill throughput in TFLOP/s (4*B*H*Nq*Nk*d per call, summed over
both prefill calls, divided by their device time); the decode bandwidth
(algorithmic bytes: K, V, q, o) is reported beside it.  Device time comes from
CUDA events on the launching stream.  The 8.6 GB decode pass streams through
L2 (129 MB) before each prefill, so every timed kernel starts with a cold L2.

Output: one JSON line on rank 0.  `--impl reference` times the float64 CPU
oracle instead (the reference arm), on bounded samples of the same workloads.
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

METRIC = "fwd TFLOP/s & % of BF16 tensor peak; split-KV decode HBM GB/s & % of peak"
WORKLOAD = ("bf16 prefill B=4 H=16 N=4096 d=64 + B=2 H=16 N=8192 d=128 (Q,K x3); "
            "split-KV decode B=32 H=32 Nk=32768 d=64 splits=16 (seeded merge order)")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PREFILL = ("mh_prefill", "peaked_d128")
# fp32-in configurations (products on the tensor cores' tf32 path), timed beside the step but not part
# of `value`; their roofline is the tf32 dense peak: the measured bf16 burst peak scaled by the nominal
# dense tf32 / bf16 ratio of the part (1.1 / 2.25 PFLOP/s).
PREFILL_FP32 = ("tiny_fp32", "long_fp32")
TF32_PER_BF16 = 1.1 / 2.25
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="bounded oracle sample for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the causal / GQA / split-KV measurements")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(values, device=None):
    """Element-wise maximum of a list of floats over all ranks (the list itself when not distributed).

    Timing rule: every rank times the same K steps, and the job's time is the
    slowest rank's.
    """
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def clocks_rejected(clocks) -> bool:
    """True when a timed region's clock record disqualifies it: a hardware or thermal slowdown was
    active, or the SM clock sat well below its maximum with no reason given (a leftover clock lock).
    A power cap alone is kept (and shows in the record)."""
    if not clocks or clocks.get("sm_mhz") is None or clocks.get("sm_max_mhz") is None:
        return False
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(clocks.get("reasons", [])):
        return True
    return not clocks.get("reasons") and clocks["sm_mhz"] < 0.9 * clocks["sm_max_mhz"]


def agree_over_ranks(flag: bool, device=None) -> bool:
    """Rank 0's decision, given to every rank (the flag itself when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return bool(flag)
    t = torch.tensor([1 if flag else 0], dtype=torch.int32, device=device)
    dist.broadcast(t, src=0)
    return bool(t.item())


def job_rate(units_per_rank: float, world: int, steps: int, seconds: float) -> float:
    """Whole-job throughput: units every rank processed per step, over the slowest rank's time."""
    return world * steps * units_per_rank / seconds


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "25"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons, loaded = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                s, m, pw = float(parts[1]), float(parts[2]), float(parts[3])
            except ValueError:
                continue
            sm.append(s)
            mx.append(m)
            if pw > 250:
                loaded.append(s)
            for n, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(n)
        use = loaded if loaded else sm
        return {"sm_mhz": statistics.median(use) if use else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": len(loaded)}


KERNEL_SOURCES = {
    "mh_prefill": ("sm103_ptx.cuh", "fa_fwd_kernel.cuh", "fa_fwd_bf16.cu"),
    "peaked_d128": ("sm103_ptx.cuh", "fa_fwd_kernel.cuh", "fa_fwd_bf16.cu"),
    "decode": ("sm103_ptx.cuh", "fa_decode.cu"),
}


def sources_sha256(names):
    """sha256 over the named kernel sources, in the given order."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_forward_05_gb300", "csrc")
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_record():
    """Per-launch DRAM bytes from the committed ncu summary, for each kernel whose sources are unchanged since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return {}
    out = {}
    for key, ent in rec.get("kernels", {}).items():
        if isinstance(ent, dict) and key in KERNEL_SOURCES and ent.get("sha256") == sources_sha256(KERNEL_SOURCES[key]):
            out[key] = ent.get("bytes")
    return out


# ----------------------------------------------------------------------------- reference arm

def oracle_prefill_sample(oracle, q, k, v, scale, seconds, rows_per_call=64, min_calls=1):
    """Times the oracle on successive 64-row samples of successive heads for about `seconds`."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    flops = 0
    t0 = time.perf_counter()
    calls = 0
    while True:
        bh = calls % (B * H)
        b, h = divmod(bh, H)
        r0 = (calls * rows_per_call) % Nq
        qs = q[b, h, r0:r0 + rows_per_call]
        oracle.attention(qs, k[b, h], v[b, h], scale)
        flops += 4 * qs.shape[0] * Nk * d
        calls += 1
        el = time.perf_counter() - t0
        if calls >= min_calls and el >= seconds:
            return flops, el, calls


def oracle_decode_sample(oracle, q, k, v, splits, scale, order, seconds):
    B, H, Nk, d = k.shape
    nbytes = 0
    t0 = time.perf_counter()
    calls = 0
    while True:
        b, h = divmod(calls % (B * H), H)
        oracle.decode_splitkv(q[b, h], k[b, h][None], v[b, h][None], splits, scale, order)
        nbytes += 2 * Nk * d * 2 + 2 * d * 2
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return nbytes, el, calls


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return "unknown"
    fields = {}
    for line in info.splitlines():
        if ":" in line:
            key, val = (x.strip() for x in line.split(":", 1))
            fields.setdefault(key.lower(), val)
    if "model name" in fields:
        return fields["model name"]
    if "cpu implementer" in fields:  # Arm: implementer / part codes
        return f"Arm implementer {fields['cpu implementer']} part {fields.get('cpu part', '?')}"
    return "unknown"


class OneCore:
    """Pins the calling thread to one allowed core for the oracle timing (process-local; restores the
    previous affinity on exit) and describes the host for the cpu_baseline record."""

    def __enter__(self):
        self.old = None
        self.core = None
        if hasattr(os, "sched_setaffinity"):
            try:
                self.old = os.sched_getaffinity(0)
                self.core = max(self.old)
                os.sched_setaffinity(0, {self.core})
            except OSError:
                self.old = self.core = None
        return self

    def __exit__(self, *exc):
        if self.old is not None:
            os.sched_setaffinity(0, self.old)
        return False

    def record(self) -> dict:
        return {"host_cpus": os.cpu_count(), "cpu_model": cpu_model(),
                "pinned_core": self.core, "threads": 1}


def host_inputs(name):
    """CPU copies of a workload's inputs (heads generated on demand are enough for the oracle samples)."""
    from attention_forward_05_gb300.inputs import WORKLOADS, make_qkv
    w = WORKLOADS[name]
    # a 2-head slice of the same recipe: the oracle samples rows of single heads
    return w, make_qkv(1, 2, w.Nq, w.Nk, w.d, w.dtype, w.seed, w.qk_mult, device="cpu")


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from attention_forward_05_gb300.inputs import merge_order
    oracle.build()
    w, (q, k, v) = host_inputs("mh_prefill")
    total_flops, total_t = 0, 0.0
    per_step = []
    with OneCore() as pin:
        for i in range(args.warmup + args.steps):
            f, t, _ = oracle_prefill_sample(oracle, q, k, v, w.scale, seconds=0.0, rows_per_call=64, min_calls=2)
            if i >= args.warmup:
                total_flops += f
                total_t += t
                per_step.append(t)
    value = total_flops / total_t / 1e12
    cores = 1
    sample = f"{2 * 64} query rows of one mh_prefill head (Nk=4096, d=64) per step, float64 C, 1 thread"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(per_step),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample,
                         **pin.record()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def cpu_baseline(seconds):
    """The oracle as it stands, on bounded samples of the prefill and decode workloads (1 host thread)."""
    import oracle
    from attention_forward_05_gb300.inputs import merge_order
    oracle.build()
    w, (q, k, v) = host_inputs("mh_prefill")
    from attention_forward_05_gb300.inputs import WORKLOADS, make_qkv
    wd = WORKLOADS["decode"]
    qd, kd, vd = make_qkv(1, 2, 1, wd.Nk, wd.d, "bf16", wd.seed, device="cpu")
    order = merge_order(wd.splits, wd.order_seed)
    with OneCore() as pin:
        f, t, calls = oracle_prefill_sample(oracle, q, k, v, w.scale, seconds=seconds * 0.7)
        nb, td, cd = oracle_decode_sample(oracle, qd, kd, vd, wd.splits, wd.scale, order, seconds * 0.3)
    pre = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
           "sample": f"{calls} x 64 query rows of mh_prefill heads (Nk=4096, d=64), float64 C, 1 thread, {t:.1f} s",
           **pin.record()}
    dec = {"value": nb / td / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"{cd} decode heads (Nk=32768, d=64, 16 splits), float64 C, 1 thread, {td:.1f} s",
           **pin.record()}
    return pre, dec


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import attention_forward_05_gb300 as fa
    from attention_forward_05_gb300 import accounting
    from attention_forward_05_gb300.inputs import WORKLOADS, merge_order, workload_inputs

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.lib()  # fails loudly if the CUDA library is missing
    peaks, peak_src = read_peaks()

    # ---- inputs resident in HBM (each rank holds a full replica: weak scaling)
    pre = {}
    for name in PREFILL:
        w = WORKLOADS[name]
        q, k, v = workload_inputs(w, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.Nq), device=dev, dtype=torch.float32)
        pre[name] = (w, q, k, v, o, lse)
    wd = WORKLOADS["decode"]
    qd, kd, vd = workload_inputs(wd, device=dev)
    od = torch.empty((wd.B, wd.H, wd.d), device=dev, dtype=torch.bfloat16)
    ws = torch.empty(fa.fa_decode_workspace_bytes(wd.B, wd.H, wd.d, wd.splits) // 4, device=dev,
                     dtype=torch.float32)
    order = torch.as_tensor(merge_order(wd.splits, wd.order_seed), device=dev)
    stream = torch.cuda.current_stream()

    def decode():
        fa.fa_decode_splitkv_ex(qd, kd, vd, wd.splits, workspace=ws, merge_order=order, o=od, stream=stream)

    def prefill(name):
        w, q, k, v, o, lse = pre[name]
        fa.fa_fwd(q, k, v, scale=w.scale, o=o, lse=lse, stream=stream)

    launches_per_step = 2 + len(PREFILL)
    for _ in range(args.warmup):
        decode()
        for n in PREFILL:
            prefill(n)
    torch.cuda.synchronize()
    if fa.fa_check_device_error() != fa.FA_OK:
        raise RuntimeError("device timeout during warm-up")

    # ---- timed region: events around every kernel launch group on the launching stream
    K = args.steps

    def timed_region():
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 + len(PREFILL))] for _ in range(K)]
        sampler = ClockSampler(local) if rank == 0 else None
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        if sampler:
            sampler.start()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(K):
            e = ev[i]
            e[0].record(stream)
            decode()
            e[1].record(stream)
            for j, n in enumerate(PREFILL):
                prefill(n)
                e[2 + j].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
        clocks = sampler.stop() if sampler else None
        if world > 1:
            dist.barrier()
        if fa.fa_check_device_error() != fa.FA_OK:
            raise RuntimeError("device timeout in the timed region")
        total_ms = start.elapsed_time(end)
        dec_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
        pre_ms = {n: [ev[i][1 + j].elapsed_time(ev[i][2 + j]) for i in range(K)] for j, n in enumerate(PREFILL)}
        return total_ms, dec_ms, pre_ms, clocks

    total_ms, dec_ms, pre_ms, clocks = timed_region()
    # a region whose clock record disqualifies it is measured once more (rank 0 samples and decides)
    if agree_over_ranks(rank == 0 and clocks_rejected(clocks), device=dev):
        first = clocks
        total_ms, dec_ms, pre_ms, clocks = timed_region()
        if clocks is not None:
            clocks = dict(clocks, remeasured_after=first)

    total_ms, dec_tot, pre_tot = max_over_ranks(
        [total_ms, sum(dec_ms), sum(sum(x) for x in pre_ms.values())], device=dev)

    pre_flops = {n: accounting.fwd_flops(w.B, w.H, w.Nq, w.Nk, w.d) for n, (w, *_r) in pre.items()}
    flops_step = sum(pre_flops.values())
    value = job_rate(flops_step, world, K, pre_tot / 1e3) / 1e12
    dec_bytes = accounting.decode_min_bytes(wd.B, wd.H, wd.Nk, wd.d)
    dec_gbs = job_rate(dec_bytes, world, K, dec_tot / 1e3) / 1e9

    # ---- end to end through the public API with host buffers (pinned), copies inside the timed region
    e2e = e2e_dec = None
    if rank == 0 or world > 1:
        e2e, e2e_dec = measure_e2e(fa, torch, pre, (wd, qd, kd, vd, od, ws, order), stream, args.e2e_steps,
                                   flops_step, dec_bytes)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    traffic = traffic_record()
    parts = {}
    for n, (w, *_r) in pre.items():
        ms = statistics.mean(pre_ms[n])
        ach = pre_flops[n] / (ms / 1e3) / 1e12
        parts[n] = {"ms": ms, "tflops": ach, "frac": ach / peaks["bf16_tflops"],
                    "flops_per_launch": pre_flops[n]}
    dom = max(parts, key=lambda n: parts[n]["ms"])
    parts.update(measure_fp32(fa, torch, accounting, dev, stream, peaks["bf16_tflops"] * TF32_PER_BF16, peak_src))
    ms_dec = statistics.mean(dec_ms)
    roof = {"bound": "tensor", "kernel": f"fa_fwd_kernel bf16 ({dom})",
            "achieved": parts[dom]["tflops"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": parts[dom]["frac"], "traffic": traffic.get(dom),
            "peak_source": f"{peak_src} bf16 burst (kernel timed alone per launch)"}
    roof_dec = {"bound": "hbm", "kernel": "fa_decode_split_kernel + fa_decode_merge_kernel",
                "achieved": dec_bytes / (ms_dec / 1e3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": dec_bytes / (ms_dec / 1e3) / 1e9 / peaks["hbm_gbs"], "traffic": traffic.get("decode"),
                "peak_source": f"{peak_src} HBM copy bandwidth"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs > L2, or L2 flushed by the preceding 8.6 GB decode pass",
                   "value_definition": "prefill FLOPs (4*B*H*Nq*Nk*d) / prefill device time"},
        "prefill": parts,
        "decode": {"metric": "split-KV decode HBM GB/s", "value": dec_gbs, "unit": "GB/s", "ms": ms_dec,
                   "bytes_per_step": dec_bytes, "frac": roof_dec["frac"], "e2e": e2e_dec},
        "roofline": roof,
        "roofline_decode": roof_dec,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
    }
    if not args.no_extras:
        line["extras"] = measure_extras(fa, torch, accounting, dev, stream, hbm_gbs=peaks["hbm_gbs"])
    if not args.no_cpu_baseline:
        cb_pre, cb_dec = cpu_baseline(args.cpu_seconds)
        line["cpu_baseline"] = cb_pre
        line["decode"]["cpu_baseline"] = cb_dec
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def measure_fp32(fa, torch, accounting, dev, stream, tf32_peak, peak_src, launches=50):
    """The fp32-in workloads through fa_fwd as a user calls it (automatic key splits): each launch
    group (prep, forward, merge) timed alone with CUDA events on `stream`, after 3 warm-up calls, with
    L2 flushed before every timed launch (the inputs are far smaller than L2)."""
    from attention_forward_05_gb300.inputs import WORKLOADS, workload_inputs
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    out = {}
    for name in PREFILL_FP32:
        w = WORKLOADS[name]
        q, k, v = workload_inputs(w, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.Nq), device=dev, dtype=torch.float32)
        call = lambda: fa.fa_fwd(q, k, v, scale=w.scale, o=o, lse=lse, stream=stream)
        for _ in range(3):
            call()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches)]
        with torch.cuda.stream(stream):
            for a, b in evs:
                flush.fill_(1)
                a.record(stream)
                call()
                b.record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        fl = accounting.fwd_flops(w.B, w.H, w.Nq, w.Nk, w.d)
        ach = fl / (ms / 1e3) / 1e12
        out[name] = {"ms": ms, "tflops": ach, "frac": ach / tf32_peak, "flops_per_launch": fl,
                     "in_value": False, "dtype": "fp32 in, tf32 products", "peak": tf32_peak,
                     "peak_source": f"{peak_src} bf16 burst x 1.1/2.25 (nominal dense tf32/bf16 ratio)",
                     "l2": "flushed before every timed launch", "launches": launches}
        del q, k, v, o, lse
    if fa.fa_check_device_error() != fa.FA_OK:
        raise RuntimeError("device timeout in the fp32 measurements")
    return out


def measure_extras(fa, torch, accounting, dev, stream, launches=20, hbm_gbs=None):
    """Rates of the extensions beyond the headline step, each timed alone with CUDA events on
    `stream` after 3 warm-up launches (not part of `value`):
      causal        the two bf16 prefill workloads with the causal mask (visible-key FLOPs)
      gqa           B=4 H=16 N=4096 d=64 bf16 with 2 key/value heads
      split_kv      B=1 H=1 N=4096 d=64 fp32 (TF32) with automatic key splits vs one split (a call lasts
                    tens of microseconds, less than its host-side submission: each call is timed alone
                    behind an L2 flush, as the fp32 prefill entries are)
      decode_gqa    the decode workload (B=32, H=32 query heads, Nk=32768, d=64, 16 splits) with 8 and 4
                    key/value heads (groups of 4 and 8), GB/s of K/V read once plus q and o
      bwd           fa_bwd on the two bf16 prefill workloads, plain and causal, and on the fp32
                    single-head N=4096 workload (FLOPs of the five backward contractions, 2.5x the
                    forward's)
    """
    from attention_forward_05_gb300.inputs import WORKLOADS, make_dout, make_qkv, workload_inputs

    def timed(fn):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(launches):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / launches

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def timed_each(fn, n=50):
        # one call per event pair, each behind an L2 flush whose run covers the call's host-side submission
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            for a, b in evs:
                flush.fill_(1)
                a.record(stream)
                fn()
                b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    out = {}
    for name in PREFILL:
        w = WORKLOADS[name]
        q, k, v = workload_inputs(w, device=dev)
        ms = timed(lambda: fa.fa_fwd(q, k, v, scale=w.scale, causal=True, stream=stream))
        out[f"causal_{name}"] = {"ms": ms, "tflops": accounting.fwd_flops_causal(w.B, w.H, w.Nq, w.Nk, w.d) / ms / 1e9}
        del q, k, v
    w = WORKLOADS["mh_prefill"]
    q, _, _ = make_qkv(w.B, w.H, w.Nq, 1, w.d, "bf16", seed=w.seed, device=dev)
    _, k, v = make_qkv(w.B, 2, 1, w.Nk, w.d, "bf16", seed=w.seed + 1, device=dev)
    ms = timed(lambda: fa.fa_fwd(q, k, v, scale=w.scale, stream=stream))
    out["gqa_mh_prefill_hkv2"] = {"ms": ms, "tflops": accounting.fwd_flops(w.B, w.H, w.Nq, w.Nk, w.d) / ms / 1e9}
    w = WORKLOADS["long_fp32"]
    q, k, v = workload_inputs(w, device=dev)
    fl = accounting.fwd_flops(w.B, w.H, w.Nq, w.Nk, w.d)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), device=dev, dtype=torch.float32)
    for tag, ks in (("split_kv_auto", 0), ("split_kv_off", 1)):
        ms = timed_each(lambda: fa.fa_fwd(q, k, v, scale=w.scale, o=o, lse=lse, kv_splits=ks, stream=stream))
        out[f"{tag}_long_fp32"] = {"ms": ms, "tflops": fl / ms / 1e9, "l2": "flushed before every timed call"}
    del q, k, v, o, lse, flush
    w = WORKLOADS["decode"]
    qd, _, _ = make_qkv(w.B, w.H, 1, 1, w.d, "bf16", seed=w.seed, device=dev)
    for hkv in (8, 4):
        _, kd, vd = make_qkv(w.B, hkv, 1, w.Nk, w.d, "bf16", seed=w.seed + hkv, device=dev)
        ws = torch.empty(fa.fa_decode_workspace_bytes(w.B, w.H, w.d, w.splits), dtype=torch.uint8, device=dev)
        ms = timed(lambda: fa.fa_decode_splitkv_gqa(qd, kd, vd, w.splits, workspace=ws, stream=stream))
        nbytes = accounting.decode_gqa_min_bytes(w.B, w.H, hkv, w.Nk, w.d)
        out[f"decode_gqa_hkv{hkv}"] = {"ms": ms, "gbs": nbytes / ms / 1e6, "bytes": nbytes,
                                       "frac_of_hbm_peak": nbytes / ms / 1e6 / hbm_gbs if hbm_gbs else None}
        del kd, vd
    del qd
    for name in PREFILL:
        w = WORKLOADS[name]
        q, k, v = workload_inputs(w, device=dev)
        dout = make_dout(w.B, w.H, w.Nq, w.d, "bf16", seed=w.seed + 700, device=dev)
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.Nq, w.d), dtype=torch.uint8, device=dev)
        for causal in (False, True):
            o, lse = fa.fa_fwd(q, k, v, scale=w.scale, causal=causal, stream=stream)
            ms = timed(lambda: fa.fa_bwd(q, k, v, o, dout, lse, scale=w.scale, causal=causal, dq=grads[0],
                                         dk=grads[1], dv=grads[2], workspace=ws, stream=stream))
            fl = (accounting.bwd_flops_causal if causal else accounting.bwd_flops)(w.B, w.H, w.Nq, w.Nk, w.d)
            out[f"bwd_{'causal_' if causal else ''}{name}"] = {"ms": ms, "tflops": fl / ms / 1e9}
        del q, k, v, dout, grads, o, lse
    w = WORKLOADS["long_fp32"]
    q, k, v = workload_inputs(w, device=dev)
    dout = make_dout(w.B, w.H, w.Nq, w.d, "fp32", seed=w.seed + 700, device=dev)
    o, lse = fa.fa_fwd(q, k, v, scale=w.scale, stream=stream)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.Nq, w.d), dtype=torch.uint8, device=dev)
    ms = timed(lambda: fa.fa_bwd(q, k, v, o, dout, lse, scale=w.scale, dq=grads[0], dk=grads[1], dv=grads[2],
                                 workspace=ws, stream=stream))
    out["bwd_long_fp32"] = {"ms": ms, "tflops": accounting.bwd_flops(w.B, w.H, w.Nq, w.Nk, w.d) / ms / 1e9,
                            "arithmetic": "fp32 FMA on the CUDA cores"}
    del q, k, v, dout, grads, o, lse
    if fa.fa_check_device_error() != fa.FA_OK:
        raise RuntimeError("device timeout in the extra measurements")
    return out


def measure_e2e(fa, torch, pre, dec, stream, steps, flops_step, dec_bytes):
    """Same metrics through the public API, with pinned host inputs copied in and results read back
    inside the timed region every step: fa_fwd_host for the prefill workloads (host tensors in and out),
    host-to-device copies, fa_decode_splitkv_ex and a device-to-host copy for decode."""
    host = {}
    h2d = d2h = 0
    for n, (w, q, k, v, o, lse) in pre.items():
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        ho, hl = torch.empty_like(o, device="cpu").pin_memory(), torch.empty_like(lse, device="cpu").pin_memory()
        ws = torch.empty(fa.fa_fwd_host_workspace_bytes(w.B, w.H, w.H, w.Nq, w.Nk, w.d, q.dtype), dtype=torch.uint8,
                         device=q.device)
        host[n] = (hq, hk, hv, ho, hl, ws)
        h2d += sum(x.numel() * x.element_size() for x in (hq, hk, hv))
        d2h += ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    wd, qd, kd, vd, od, ws, order = dec
    hqd, hkd, hvd = (x.cpu().pin_memory() for x in (qd, kd, vd))
    hod = torch.empty_like(od, device="cpu").pin_memory()
    dh2d = sum(x.numel() * x.element_size() for x in (hqd, hkd, hvd))
    dd2h = hod.numel() * hod.element_size()

    # The two prefill problems are independent: each runs on its own stream, so one's copies can
    # overlap the other's compute as well as its own.
    wstreams = {n: torch.cuda.Stream(device=stream.device) for n in pre}
    ev_go, ev_done = torch.cuda.Event(), {n: torch.cuda.Event() for n in pre}

    # The larger problem is enqueued first: its copies go first on the shared host link, and the
    # smaller one's last chunk is then the only compute and copy-out left after the last copy in.
    pre_order = sorted(pre, key=lambda n: -pre[n][1].numel())

    def pre_step():
        # the library's host-buffer entry point: copies in and out overlap the compute, chunk by chunk
        ev_go.record(stream)
        for n in pre_order:
            w, q, k, v, o, lse = pre[n]
            hq, hk, hv, ho, hl, ws = host[n]
            wstreams[n].wait_event(ev_go)
            fa.fa_fwd_host(hq, hk, hv, scale=w.scale, o=ho, lse=hl, workspace=ws, stream=wstreams[n])
            ev_done[n].record(wstreams[n])
        for n in pre:
            stream.wait_event(ev_done[n])

    def dec_step():
        qd.copy_(hqd, non_blocking=True)
        kd.copy_(hkd, non_blocking=True)
        vd.copy_(hvd, non_blocking=True)
        fa.fa_decode_splitkv_ex(qd, kd, vd, wd.splits, workspace=ws, merge_order=order, o=od, stream=stream)
        hod.copy_(od, non_blocking=True)

    res = []
    for fn in (pre_step, dec_step):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        res.append(a.elapsed_time(b) / steps)
    ms_pre, ms_dec = res
    e2e = {"value": flops_step / (ms_pre / 1e3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": ms_pre, "steps": steps}
    e2e_dec = {"value": dec_bytes / (ms_dec / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": dh2d,
               "d2h_bytes_per_step": dd2h, "ms_per_step": ms_dec, "steps": steps}
    return e2e, e2e_dec


def main():
    args = parse_args()
    if args.warmup < 3:
        print("warm-up must be at least 3 steps", file=sys.stderr)
        return 2
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
