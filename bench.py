#!/usr/bin/env python3
"""Throughput of the attention forward on GB300: one JSON line.

A step is one attention forward (every step of the fused path, in one kernel)
over one batch of the workload.  Default workload: the FP8 DiT-block attention
shaped like the one the FP8 CuTe-DSL page times (B=1, H=56, N=30272, d=128,
e4m3 Q/K/V with per-tensor descales, non-causal), the largest single-GPU
workload.  Inputs are resident in HBM before timing; L2 is
flushed (a 512 MiB device write) before every timed step, outside the timed
interval; each step is timed with CUDA events on the stream the kernel runs
on, and the sum over the K steps gives the throughput.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the float64 oracle on the host cores

Multi-GPU (torchrun, one process per GPU): every rank runs its own replica of
the workload (attention heads are independent, no data-path collective), the
slowest rank's time is used, and `value` counts the work of all ranks (weak
scaling).
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from tiled_attention_fa2_gb300 import inputs  # noqa: E402

METRIC = "attention fwd TFLOPS & % of GB300 dense bf16/fp8 tensor peak; ms per call"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "dit_e4m3"
FLUSH_BYTES = 512 << 20
# Published figures for an exact workload (other hardware: context only).
PUBLISHED_TFLOPS = {"dit_e4m3": 26.27e12 / 123.6e-3 / 1e12}  # RTX 5080, final FP8 CuTe-DSL kernel
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 datasheet dense (no 2:4 sparsity) tensor peaks, TFLOP/s: context beside the measured ones.
DATASHEET_DENSE_TFLOPS = {"bf16": 2250.0, "e4m3": 4500.0}


# The sources the tensor-core forward kernel and its launch are built from; a
# change anywhere else (backward, fp32 path, split-KV merge) leaves it as it was.
FWD_SOURCES = ("attn_api.cu", "attn_kernels.h", "attn_tc_bf16.cu", "attn_tc_e4m3.cu", "attn_tc_e4m3_poly.cu",
               "attn_tc_sm103.cuh", "exp2_poly.h", "ptx_sm103.cuh")


def kernel_source_hash(files=FWD_SOURCES) -> str:
    d = os.path.join(ROOT, "tiled_attention_fa2_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(files):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def datasheet_fraction(dtype: str, achieved: float) -> dict:
    """The datasheet dense peak of the contraction dtype and the fraction of it
    reached (reported beside the measured-peak fraction; fp32 runs on the CUDA
    cores and has none)."""
    p = DATASHEET_DENSE_TFLOPS.get(dtype)
    if p is None:
        return {}
    return {"datasheet_peak": p, "frac_of_datasheet": round(achieved / p, 4)}


def dtype_peak(dtype: str, peaks: dict):
    """Dense tensor peak for the contraction dtype: bf16 measured (cuBLAS burst);
    e4m3 = bf16 x 2 (nominal fp8:bf16 ratio); f32 runs on the CUDA cores."""
    if dtype == "e4m3":
        return 2.0 * peaks["bf16_tflops"], "bf16 burst x 2 (nominal fp8/bf16 ratio)"
    return peaks["bf16_tflops"], "bf16 burst"


def profile_traffic(workload: str):
    """DRAM bytes per launch from an ncu capture of the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        t = json.load(f)
    e = t.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval_ms: int = 20):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []  # (host time, csv line)
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, t0: float, t1: float):
        """The host-time interval of the timed region."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        # Only samples printed while the timed region ran count (nvidia-smi prints a
        # sample when it has taken it, so the host time of the line bounds it).
        lines = [ln for t, ln in self.lines if self.window is None or self.window[0] <= t <= self.window[1]]
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples_under_load": len(sm),
                "interval_ms": self.interval_ms}


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The slowest rank's value (the job ends when the last rank ends)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    dev = device if (device is not None and dist.get_backend() == "nccl") else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, world: int, steps: int, max_ms: float) -> float:
    """Whole-job TFLOP/s under weak scaling: every rank processes its own batch
    of the workload, so the work is world * steps * flops_per_step and the
    time is the slowest rank's."""
    return flops_per_step * world * steps / (max_ms * 1e-3) / 1e12


def kv_heads(w: dict) -> int:
    """K/V heads of a workload (fewer than H under grouped-query attention)."""
    return int(w.get("Hkv", w["H"]))


def make_device_inputs(w: dict, device, seed: int):
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    q, k, v = inputs.make_qkv_f32(B, H, N, d, seed=seed, q_mult=w["q_mult"], n_kv_heads=kv_heads(w))
    descales = (1.0, 1.0, 1.0)
    if w["dtype"] == "bf16":
        host = tuple(inputs.to_bf16(t) for t in (q, k, v))
    elif w["dtype"] == "e4m3":
        qs, ks, vs = (inputs.quantize_e4m3(t) for t in (q, k, v))
        host = (qs[0], ks[0], vs[0])
        descales = (qs[1], ks[1], vs[1])
    else:
        host = (q, k, v)
    return host, tuple(t.to(device) for t in host), descales


def run_gpu_arm(args, w):
    from tiled_attention_fa2_gb300 import binding

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    lib = binding.load_library()

    B, H, N, d, causal = w["B"], w["H"], w["N"], w["d"], w["causal"]
    host, (q, k, v), descales = make_device_inputs(w, device, seed=rank)
    code = {"f32": 0, "bf16": 1, "e4m3": 2}[w["dtype"]]
    odt = torch.float32 if code == 0 else torch.bfloat16
    o = torch.empty((B, H, N, d), dtype=odt, device=device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    Hkv = kv_heads(w)

    def launch():
        if Hkv != H:
            st = lib.attn_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hkv,
                                  N, d, scale, *descales, int(causal), code, sh)
        elif code == 2:
            st = lib.attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                                  scale, *descales, int(causal), sh)
        else:
            st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                              scale, int(causal), code, sh)
        if st != 0:
            raise RuntimeError(lib.attn_last_error().decode())

    for _ in range(args.warmup):
        flush.fill_(1)
        launch()
    torch.cuda.synchronize()

    sampler = ClockSampler(device.index)
    sampler.start()
    time.sleep(0.2)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        launch()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    if dist:
        dist.barrier()
    wall = time.perf_counter() - t0
    sampler.mark(t0, t1)
    clocks = sampler.stop()
    st = binding.get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")
    times_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(times_ms), dist, device)
    flops = inputs.attention_flops(B, H, N, d, causal)
    value = job_throughput(flops, world, args.steps, total_ms)
    mean_ms = total_ms / args.steps

    # ---- end to end: pinned host buffers through the C ABI (copies inside the timed region).
    # Steps alternate between two streams, each with its own device staging buffers and
    # host result buffers, so step i+1's host-to-device copies run while step i computes
    # and copies its result back; every step still moves all of its inputs and results.
    e2e_steps = max(1, min(args.steps, 20))
    h_in = [t.pin_memory() for t in host]
    e2e_streams = [stream, torch.cuda.Stream(device)]
    e2e_sets = []
    for _ in e2e_streams:
        e2e_sets.append({
            "d_in": [torch.empty_like(t) for t in (q, k, v)],
            "o": torch.empty_like(o), "lse": torch.empty_like(lse),
            "h_o": torch.empty(o.shape, dtype=o.dtype).pin_memory(),
            "h_l": torch.empty(lse.shape, dtype=torch.float32).pin_memory(),
        })

    def e2e_call(i):
        st_obj, bufs = e2e_streams[i % 2], e2e_sets[i % 2]
        d_in = bufs["d_in"]
        if Hkv != H:
            # Grouped-query attention has no host entry point: the same copies
            # through the stream, then attn_fwd_gqa, then the copies back.
            with torch.cuda.stream(st_obj):
                for dst, src in zip(d_in, h_in):
                    dst.copy_(src, non_blocking=True)
                st = lib.attn_fwd_gqa(d_in[0].data_ptr(), d_in[1].data_ptr(), d_in[2].data_ptr(),
                                      bufs["o"].data_ptr(), bufs["lse"].data_ptr(), B, H, Hkv, N, d, scale,
                                      *descales, int(causal), code, st_obj.cuda_stream)
                if st != 0:
                    raise RuntimeError(lib.attn_last_error().decode())
                bufs["h_o"].copy_(bufs["o"], non_blocking=True)
                bufs["h_l"].copy_(bufs["lse"], non_blocking=True)
            return
        st = lib.attn_fwd_host(h_in[0].data_ptr(), h_in[1].data_ptr(), h_in[2].data_ptr(), bufs["h_o"].data_ptr(),
                               bufs["h_l"].data_ptr(), d_in[0].data_ptr(), d_in[1].data_ptr(), d_in[2].data_ptr(),
                               bufs["o"].data_ptr(), bufs["lse"].data_ptr(), B, H, N, d, scale, *descales,
                               int(causal), code, st_obj.cuda_stream)
        if st != 0:
            raise RuntimeError(lib.attn_last_error().decode())

    e2e_call(0)
    e2e_call(1)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    e0.record(stream)
    e2e_streams[1].wait_event(e0)
    for i in range(e2e_steps):
        e2e_call(i)
    stream.wait_stream(e2e_streams[1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, device)
    in_bytes = sum(t.numel() * t.element_size() for t in host)
    out_bytes = o.numel() * o.element_size() + lse.numel() * 4

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    peaks, peaks_src = load_peaks()
    peak, peak_note = dtype_peak(w["dtype"], peaks)
    achieved = flops / (mean_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(mean_ms, 5),
        "ms_per_step_median": round(statistics.median(times_ms), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(value / PUBLISHED_TFLOPS[args.workload], 3) if args.workload in PUBLISHED_TFLOPS else None,
        "dtype": w["dtype"],
        "data": "synthetic: i.i.d. N(0,1) Q/K/V from a seeded CPU generator (seed = rank)",
        "config": {"workload": args.workload, "B": B, "H": H, "H_kv": Hkv, "N": N, "d": d, "causal": bool(causal),
                   "flops_per_step": flops, "l2": "flushed before every timed step (512 MiB device write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "pct_of_peak": round(100.0 * achieved / peak, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peaks_src}: {peak_note}",
                     "traffic": profile_traffic(args.workload),
                     **datasheet_fraction(w["dtype"], achieved)},
        "clocks": clocks,
        "e2e": {"value": round(job_throughput(flops, world, e2e_steps, e2e_ms), 3), "unit": UNIT,
                "ms_per_step": round(e2e_ms / e2e_steps, 4), "steps": e2e_steps,
                "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
                "streams": len(e2e_streams)},
        "gpu_launches": args.steps,
        "wall_s_timed_region": round(wall, 4),
        "kernel_source_hash": kernel_source_hash(),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, host, descales, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def _oracle_head_inputs(w, host, descales, h):
    """Query head h (over B*H) and the K/V head it reads, decoded by the oracle."""
    import oracle

    fmt = w["dtype"]
    H, Hkv = w["H"], kv_heads(w)
    b, hq = divmod(h, H)
    hk = b * Hkv + oracle.kv_head_of(hq, H, Hkv)
    out = []
    for t, ds, i in zip(host, descales, (h, hk, hk)):
        shape = (-1, w["N"], w["d"])
        if fmt == "bf16":
            c = inputs.bits_u16(t).reshape(shape)[i]
        elif fmt == "e4m3":
            c = inputs.bits_u8(t).reshape(shape)[i]
        else:
            c = t.reshape(shape)[i].numpy()
        out.append(oracle.dequantize(c, fmt, ds))
    return out


def oracle_sample(w, host, descales, heads, rows_per_head):
    """Oracle on a sample: the first `rows_per_head` query rows (in seeded
    sample order) of the given heads.  Returns (seconds, flops of the sample)."""
    import oracle

    N, d, causal = w["N"], w["d"], w["causal"]
    rows = inputs.sample_rows(N, w["B"], w["H"], count=min(N, max(rows_per_head, 2)))
    flops = 0.0
    t0 = time.perf_counter()
    for h in heads:
        q, k, v = _oracle_head_inputs(w, host, descales, h)
        r = rows[h][None]
        oracle.attention_rows(q[None], k[None], v[None], r, 1 / math.sqrt(d), causal)
        keys = (r[0] + 1) if causal else np.full(r.shape[1], N)
        flops += float(4.0 * d * keys.sum())
    return time.perf_counter() - t0, flops


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name on x86, implementer and
    part numbers on Arm)."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return "unknown"
    fields = {}
    for ln in info:
        if ":" in ln:
            k, v = (x.strip() for x in ln.split(":", 1))
            fields.setdefault(k, v)
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return f"Arm implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    return "unknown"


def cpu_baseline(w, host, descales, budget_s=15.0):
    """Time the oracle as it stands on this host's cores, on a bounded sample of
    about `budget_s` seconds: the whole workload (repeated to fill the budget)
    when it is small enough, else as many heads x 512 sampled rows as fit."""
    BH, N = w["B"] * w["H"], w["N"]
    rows = min(N, 512)
    secs, flops = oracle_sample(w, host, descales, [0], rows)  # calibration
    whole_est = secs * BH * N / rows
    if 2 * whole_est <= budget_s:
        secs = flops = 0.0
        reps = 0
        while secs < budget_s and reps < 100000:  # repeat until the budget is used
            s_, f_ = oracle_sample(w, host, descales, list(range(BH)), N)
            secs, flops, reps = secs + s_, flops + f_, reps + 1
        sample = f"the whole workload ({BH} heads x {N} query rows) x {reps}"
    else:
        heads = [0]
        if secs < budget_s:
            heads = list(range(max(1, min(BH, int(budget_s / max(secs, 1e-3))))))
            secs, flops = oracle_sample(w, host, descales, heads, rows)
        sample = f"{len(heads)} of {BH} heads x {rows} sampled query rows"
    out = {"value": round(flops / secs / 1e12, 6), "unit": UNIT, "cores": os.cpu_count(), "cpu": cpu_model(),
           "kind": "oracle",
           "sample": f"{sample} (causal rows see keys <= row); {secs:.1f} s; numpy float64, BLAS threads = all cores",
           "seconds": round(secs, 2)}
    total = inputs.attention_flops(w["B"], w["H"], N, w["d"], w["causal"])
    out["extrapolated_full_call_s"] = round(total / (flops / secs), 3)  # one whole call at the sample's rate
    return out


def run_reference_arm(args, w):
    """The oracle as the reference arm: each step is a bounded sample of the
    workload (one head x 512 sampled rows) timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    host, descales = make_host_inputs(w)
    BH = w["B"] * w["H"]
    rows = min(w["N"], 512)
    for i in range(args.warmup):
        oracle_sample(w, host, descales, [i % BH], rows)
    tot_s, tot_f = 0.0, 0.0
    for i in range(args.steps):
        s, f = oracle_sample(w, host, descales, [i % BH], rows)
        tot_s += s
        tot_f += f
    value = tot_f / tot_s / 1e12
    sample = f"each step: 1 head x {rows} sampled query rows of the workload; numpy float64, BLAS threads = all cores"
    line = {"metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * tot_s / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (same recipe as the GPU arm)",
            "config": {"workload": args.workload, "B": w["B"], "H": w["H"], "H_kv": kv_heads(w), "N": w["N"],
                       "d": w["d"], "causal": bool(w["causal"])},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": os.cpu_count(), "cpu": cpu_model(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def make_host_inputs(w):
    q, k, v = inputs.make_qkv_f32(w["B"], w["H"], w["N"], w["d"], seed=0, q_mult=w["q_mult"],
                                  n_kv_heads=kv_heads(w))
    if w["dtype"] == "bf16":
        return tuple(inputs.to_bf16(t) for t in (q, k, v)), (1.0, 1.0, 1.0)
    if w["dtype"] == "e4m3":
        qs, ks, vs = (inputs.quantize_e4m3(t) for t in (q, k, v))
        return (qs[0], ks[0], vs[0]), (qs[1], ks[1], vs[1])
    return (q, k, v), (1.0, 1.0, 1.0)


def run_gpu_bwd(args, w):
    """The backward pass (bf16 workloads): dQ, dK, dV for a seeded dO, with O and
    L from one forward call made before the timed region.  A step = the three
    backward launches (D and the dQ accumulator, the tensor-core pass, dQ to
    bf16); algorithmic FLOPs = 2.5 x the forward's (five products instead of
    two), halved for causal like the forward's."""
    from tiled_attention_fa2_gb300 import binding

    if w["dtype"] != "bf16":
        raise SystemExit("--pass bwd runs the bf16 workloads only")
    rank = int(os.environ.get("RANK", "0"))
    device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(device)
    lib = binding.load_library()
    B, H, N, d, causal = w["B"], w["H"], w["N"], w["d"], w["causal"]
    host, (q, k, v), _ = make_device_inputs(w, device, seed=rank)
    h_do = inputs.to_bf16(inputs.make_dout_f32(B, H, N, d, seed=rank + 1))
    dout = h_do.to(device)
    o, lse = binding.attn_fwd(q, k, v, causal=causal)
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    nbytes = binding.bwd_workspace_size(B, H, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    def launch():
        st = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(), nbytes, B, H, N, d, scale,
                          int(causal), sh)
        if st != 0:
            raise RuntimeError(lib.attn_last_error().decode())

    for _ in range(args.warmup):
        flush.fill_(1)
        launch()
    torch.cuda.synchronize()
    sampler = ClockSampler(device.index)
    sampler.start()
    time.sleep(0.2)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        launch()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    sampler.mark(t0, t0 + wall)
    clocks = sampler.stop()
    if binding.get_device_status() != 0:
        raise RuntimeError("device status set after the timed region")
    times_ms = [a.elapsed_time(b) for a, b in ev]
    mean_ms = sum(times_ms) / args.steps
    flops = 2.5 * inputs.attention_flops(B, H, N, d, causal)
    achieved = flops / (mean_ms * 1e-3) / 1e12

    # end to end: the step's inputs from pinned host memory, the gradients back to it
    h_in = [t.pin_memory() for t in (*host, o.cpu(), lse.cpu(), h_do)]
    d_in = [q, k, v, o, lse, dout]
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv)]
    e2e_steps = max(1, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        for dst, src in zip(d_in, h_in):
            dst.copy_(src, non_blocking=True)
        launch()
        for dst, src in zip(h_out, (dq, dk, dv)):
            dst.copy_(src, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    peaks, peaks_src = load_peaks()
    peak, peak_note = dtype_peak("bf16", peaks)
    line = {
        "metric": "attention bwd TFLOPS (2.5 x forward FLOPs) & % of GB300 dense bf16 tensor peak",
        "pass": "bwd",
        "value": round(achieved, 3),
        "unit": UNIT,
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(mean_ms, 5),
        "ms_per_step_median": round(statistics.median(times_ms), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: i.i.d. N(0,1) Q/K/V/dO from seeded CPU generators",
        "config": {"workload": args.workload, "B": B, "H": H, "N": N, "d": d, "causal": bool(causal),
                   "flops_per_step": flops, "l2": "flushed before every timed step (512 MiB device write)",
                   "parallelism": "single GPU"},
        "pct_of_peak": round(100.0 * achieved / peak, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peaks_src}: {peak_note}",
                     "note": "whole step (three launches) against the tensor peak", "traffic": None,
                     **datasheet_fraction("bf16", achieved)},
        "clocks": clocks,
        "e2e": {"value": round(flops * e2e_steps / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
                "ms_per_step": round(e2e_ms / e2e_steps, 4), "steps": e2e_steps,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in h_in),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in h_out)},
        "gpu_launches": 3 * args.steps,
        "wall_s_timed_region": round(wall, 4),
        "kernel_source_hash": kernel_source_hash(tuple(sorted(os.listdir(os.path.join(
            ROOT, "tiled_attention_fa2_gb300", "csrc"))))),
    }
    if not args.no_cpu_baseline:
        import oracle

        # one head of the same shape, gradients in float64, scaled to the whole job
        hq, hk, hv, hd = (t[0, 0].double().numpy() for t in (*host, h_do))
        t0 = time.perf_counter()
        oracle.attention_backward(hq, hk, hv, hd, scale, causal)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": round(flops / (B * H) / dt / 1e12, 6), "unit": UNIT,
                                "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"one head ({N}x{d}) of the workload, oracle.attention_backward, "
                                          f"{dt:.2f} s"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="pass_", default="fwd", choices=["fwd", "bwd"],
                    help="bwd: time the backward pass instead (auxiliary line, bf16 workloads)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} needs one process per GPU (torchrun --nproc-per-node {args.gpus}); "
                 f"this launch has WORLD_SIZE={world}")
    w = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference_arm(args, w)
    elif args.pass_ == "bwd":
        if kv_heads(w) != w["H"]:
            ap.error("the backward is implemented for multi-head attention only (H_kv = H)")
        run_gpu_bwd(args, w)
    else:
        run_gpu_arm(args, w)


if __name__ == "__main__":
    main()
