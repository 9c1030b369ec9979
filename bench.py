"""Benchmark: exact attention forward on GB300, through the library's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one attention forward over the bf16 causal workload B=4, H=16, N=2048, d=128
(scale 1/sqrt(128)), O in bf16 and lse in fp32, inputs resident in HBM.  value = algorithmic
TFLOP/s: 2*(dk + dv) FLOPs per visible (query, key) pair, causal pairs only, divided by the
device time of a step.  Timing: CUDA events on the launching stream around K back-to-back
steps, the K-step measurement repeated until about a quarter of a second of device time (so
the clock record holds many samples); consecutive steps read different copies of the inputs,
rotated over a set larger than L2, so no step finds its inputs in L2 and no flush is needed.
The same line carries:
  e2e           the same metric with the step's inputs copied host->device from pinned memory
                and o, lse copied back inside the timed interval;
  roofline      the fused kernel's achieved TFLOP/s against the measured dense-bf16 peak;
  long_causal   the causal B=1, H=32, N=16384, d=128 workload (one key per row raised by +8),
                timed the same way, with its own tensor roofline and CPU-oracle baseline;
  padbias       the padded workload with a bias, B=8, H=8, N=1024, dk=192, dv=128: its
                roofline is max(FLOPs / tensor peak, algorithmic bytes / HBM peak), bytes-bound;
  decode        split-KV decode on B=64, H=32, L=8192 (kv_len ~ U{1..8192}), d=128, 16 splits:
                KV GB/s (visible keys only) against the measured HBM peak, and against a
                read-only pass measured in the same run;
  backward      dQ, dK, dV of the 2k causal workload;
  cpu_baseline  the float64 CPU oracle timed on a bounded sample of the same workload;
  clocks        SM clocks and throttle reasons sampled during the timed regions.
Under torchrun (N > 1) every rank runs its own replica (weak scaling, no collective on the data
path); value = total FLOPs of all ranks / the slowest rank's time.

--impl reference times the float64 CPU oracle (the only reference there is: the pages publish
no GPU kernel) on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (prefill) and KV-read GB/s (decode) on 1 GB300, % of roofline"
WORKLOAD = "bf16_causal_b4_h16_n2048_d128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}  # datasheet: HBM3e 7.9 TB/s, dense bf16 2.25 PFLOP/s


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_sha(*names):
    """First 16 hex digits of the sha256 of the concatenated kernel sources."""
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "online_softmax_fa2_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary, source):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current source."""
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    m = re.search(r"<!--\s*bench:\s*(\{.*?\})\s*-->", open(path).read(), re.S)
    if not m:
        return None
    d = json.loads(m.group(1))
    if d.get("source_sha256") != kernel_sha(*source):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clocks and throttle reasons sampled while running: through NVML (the library
    nvidia-smi reads) every 2 ms where it loads, otherwise nvidia-smi every 20 ms."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.nvml = None
        self.samples = []   # (time, sm MHz, max MHz, set of reasons)
        self.stop_flag = threading.Event()
        self.source = None

    def _nvml_open(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        found = False
        try:  # the CUDA device's own UUID: NVML may number the GPUs differently
            import torch
            uid = "GPU-" + str(torch.cuda.get_device_properties(self.index).uuid)
            found = lib.nvmlDeviceGetHandleByUUID(uid.encode(), ctypes.byref(h)) == 0
        except Exception:
            found = False
        if not found and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            return None
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        if reasons is None:
            return None
        return lib, h, reasons

    def _nvml_loop(self):
        import ctypes
        lib, h, reasons = self.nvml
        mhz, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag.is_set():
            ok = (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and
                  lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and
                  reasons(h, ctypes.byref(rs)) == 0)
            if ok:
                active = {n for n, bit in self.REASON_BITS.items() if rs.value & bit}
                self.samples.append((time.time(), float(mhz.value), float(mx.value), active))
            time.sleep(0.002)

    def start(self):
        self.nvml = self._nvml_open()
        if self.nvml is not None:
            self.source = "nvml, every 2 ms"
            self.t = threading.Thread(target=self._nvml_loop, daemon=True)
            self.t.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, every 20 ms"
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)  # nvidia-smi needs a moment before its first sample
        except OSError:
            self.proc = None

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.proc.stdout:
            parts = [p.strip() for p in ln.strip().split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            active = {nm for nm, val in zip(names, parts[4:8]) if val.lower().startswith("active")}
            self.samples.append((time.time(), sm, mx, active))

    def stop(self, windows):
        """Clock summary over the samples inside the (t0, t1) host-time windows."""
        self.stop_flag.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.nvml is None and self.proc is None:
            return None
        self.t.join(timeout=5)
        sm, mx, reasons = [], [], set()
        for t, f, m, r in list(self.samples):
            if any(t0 - 0.005 <= t <= t1 + 0.005 for t0, t1 in windows):
                sm.append(f)
                mx.append(m)
                reasons |= r
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_min_mhz": sm[0], "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm), "source": self.source}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device):
    """The largest of every rank's x (the job is as slow as its slowest replica)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, ms, scale=1e12):
    """Whole-job throughput: the units all `world` replicas processed over the slowest rank's
    time per step (`scale` 1e12 for TFLOP/s, 1e9 for GB/s)."""
    return world * units_per_rank / (ms / 1e3) / scale


def head_flops(a, b):
    """Algorithmic FLOPs of one (b, h) head of workload `a` (visible pairs of sequence b)."""
    n = a.kv_len_list()[b]
    if a.causal:
        pairs = sum(max(0, min(n, i + n - a.Nq + 1)) for i in range(a.Nq))
    else:
        pairs = a.Nq * n
    return pairs * 2 * (a.dk + a.dv)


def cpu_oracle_sample(a, seconds_target, seed=0):
    """Time the float64 oracle on whole (b, h) heads of workload `a`, taken in a fixed seeded
    order, until about `seconds_target` of CPU work.  Returns (TFLOP/s, seconds, sample
    description, threads, heads done)."""
    import numpy as np
    import oracle

    q = a.q.detach().cpu().float()
    k = a.k.detach().cpu().float()
    v = a.v.detach().cpu().float()
    bias = None if a.bias is None else a.bias.detach().cpu()
    lens = a.kv_len_list()
    rng = np.random.default_rng(seed)
    order = rng.permutation(a.B * a.H)
    done, t_used, threads, flops = 0, 0.0, 0, 0
    while t_used < seconds_target:  # passes over the heads until the time target is reached
        for bh in order:
            b, h = divmod(int(bh), a.H)
            hb = None if bias is None else bias[b:b + 1, h:h + 1].contiguous()
            t0 = time.perf_counter()
            _, _, threads = oracle.attn_fwd(q[b:b + 1, :, h:h + 1], k[b:b + 1, :, h:h + 1],
                                            v[b:b + 1, :, h:h + 1], bias=hb,
                                            kv_lens=None if a.kv_lens is None else [lens[b]],
                                            causal=a.causal, scale=a.scale)
            t_used += time.perf_counter() - t0
            flops += head_flops(a, b)
            done += 1
            if t_used >= seconds_target:
                break
    desc = (f"{done} head evaluations over the {a.B * a.H} (b, h) heads (whole heads, every row, "
            f"float64)")
    return flops / t_used / 1e12, t_used, desc, threads, done


def cpu_oracle_rows(a, rows, what):
    """Time the float64 oracle on the flat rows (b*H + h)*Nq + i of workload `a` (no bias).
    Returns (TFLOP/s over those rows' visible pairs, seconds, sample description, threads)."""
    import numpy as np
    import oracle

    q = a.q.detach().cpu().float()
    k = a.k.detach().cpu().float()
    v = a.v.detach().cpu().float()
    lens = a.kv_len_list()
    rows = np.asarray(rows, np.int64)
    i = rows % a.Nq
    b = rows // (a.H * a.Nq)
    n = np.asarray(lens, np.int64)[b]
    pairs = np.minimum(n, i + n - a.Nq + 1).clip(min=0) if a.causal else n
    flops = int(pairs.sum()) * 2 * (a.dk + a.dv)
    t0 = time.perf_counter()
    _, _, threads = oracle.attn_fwd(q, k, v, kv_lens=None if a.kv_lens is None else lens,
                                    causal=a.causal, scale=a.scale, rows=rows)
    secs = time.perf_counter() - t0
    return flops / secs / 1e12, secs, f"{rows.size} rows ({what}), {int(pairs.sum())} visible pairs, float64", threads


def time_steps(step, steps, stream, min_seconds, est_ms, barrier, clk_windows):
    """Device time per step of `steps` back-to-back steps (step(s) queues step number s),
    bracketed by CUDA events on `stream`; the K-step measurement is repeated until about
    `min_seconds` of device time, the step numbers running on across repeats.  The host-time
    window of the timed region is appended to `clk_windows`.  Returns (ms per step, repeats)."""
    import torch

    repeats = max(1, min(1000, math.ceil(min_seconds * 1e3 / max(est_ms * steps, 1e-3))))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(repeats)]
    barrier()
    t0 = time.time()
    n = 0
    for s_, e_ in evs:
        s_.record(stream)
        for _ in range(steps):
            step(n)
            n += 1
        e_.record(stream)
    barrier()
    clk_windows.append((t0, time.time()))
    total = sum(s_.elapsed_time(e_) for s_, e_ in evs)
    return total / (repeats * steps), repeats


def warm(step, warmup, stream):
    """Run `warmup` untimed steps; returns their mean device time in ms (an estimate)."""
    import torch

    s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step(0)
    s_.record(stream)
    for n in range(warmup):
        step(n)
    e_.record(stream)
    torch.cuda.synchronize()
    return s_.elapsed_time(e_) / max(1, warmup)


def rotated_inputs(a, n_sets):
    """n_sets copies of a workload's inputs with outputs of their own: consecutive steps read
    different copies, so a step never finds its inputs in L2 when the copies together are
    larger than L2."""
    import torch

    sets = []
    for t in range(n_sets):
        cp = (lambda x: None if x is None else (x if t == 0 else x.clone()))
        o = torch.empty((a.B, a.Nq, a.H, a.dv), dtype=a.q.dtype, device=a.q.device)
        lse = torch.empty((a.B, a.H, a.Nq), dtype=torch.float32, device=a.q.device)
        sets.append((cp(a.q), cp(a.k), cp(a.v), cp(a.bias), o, lse))
    return sets


def set_bytes(a):
    """Bytes of one input/output set of a forward workload (q, k, v, bias, o, lse)."""
    t = [a.q, a.k, a.v, a.bias]
    n = sum(x.numel() * x.element_size() for x in t if x is not None)
    return n + a.B * a.Nq * a.H * a.dv * a.q.element_size() + a.B * a.H * a.Nq * 4


def run_reference(args):
    """The oracle as the reference arm, on the same workload: each step evaluates as many whole
    (b, h) heads as keep the run within --ref-seconds (all 64 heads, the whole workload, when
    the steps are few), on the host cores."""
    from online_softmax_fa2_gb300 import workloads as wl
    import oracle

    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    a = wl.causal_2k("cpu")
    q, k, v = a.q.float(), a.k.float(), a.v.float()
    n_heads = a.B * a.H
    flops_head = a.flops() / n_heads
    all_heads = [(i % a.B, (i * 7) % a.H) for i in range(n_heads)]  # every (b, h) once, 7 coprime to H

    def head(i):
        b, h = all_heads[i % n_heads]
        _, _, threads = oracle.attn_fwd(q[b:b + 1, :, h:h + 1], k[b:b + 1, :, h:h + 1],
                                        v[b:b + 1, :, h:h + 1], causal=True, scale=a.scale)
        return threads

    t0 = time.perf_counter()
    threads = head(0)
    t_head = time.perf_counter() - t0
    per_step = args.ref_seconds / max(1, args.steps + args.warmup)
    hps = max(1, min(n_heads, int(per_step / max(t_head, 1e-6))))  # heads per step
    times, nxt = [], 0
    for n in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        for _ in range(hps):
            threads = head(nxt)
            nxt += 1
        dt = time.perf_counter() - t0
        if n >= args.warmup:
            times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    val = hps * flops_head / (ms / 1e3) / 1e12
    sample = ("the whole workload (all 64 heads)" if hps == n_heads else
              f"{hps} of the 64 (b, h) heads per step, whole heads, taken in turn")
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": a.B, "H": a.H, "N": a.Nq, "d": a.dk, "causal": True,
                   "flops_per_step": hps * flops_head, "l2": "n/a (host cores)",
                   "timing": "wall clock per step on the host", "parallelism": "replicas x1"},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample + " per step"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def prefill_object(ofa, a, args, stream, pk, pk_kind, clk_windows, barrier, world, dev, n_sets,
                   roof_kind, traffic, **fwd_kwargs):
    """Time one forward workload (rotated input copies, back-to-back steps) and describe it:
    value, time per step and roofline ("tensor", or "combined": max(FLOPs / tensor peak,
    algorithmic bytes / HBM peak)).  fwd_kwargs go to every attn_fwd call (dropout)."""
    sets = rotated_inputs(a, n_sets)

    def step(n):
        q, k, v, b, o, lse = sets[n % n_sets]
        ofa.attn_fwd(q, k, v, bias=b, kv_lens=a.kv_lens, causal=a.causal, scale=a.scale, out=o, lse=lse,
                     **fwd_kwargs)

    est = warm(step, max(3, args.warmup), stream)
    ofa.device_error_flags()
    ms, reps = time_steps(step, args.steps, stream, args.min_seconds, est, barrier, clk_windows)
    if ofa.device_error_flags() & 1:
        raise RuntimeError(f"a kernel gave up a bounded wait during the timed region of {a.name}")
    ms = max_over_ranks(ms, world, dev)
    flops, nbytes = a.flops(), a.algo_bytes()
    tflops = job_rate(1, flops, ms)
    gbs = job_rate(1, nbytes, ms, 1e9)
    obj = {"workload": a.name, "value": job_rate(world, flops, ms), "unit": "TFLOP/s", "ms_per_step": ms,
           "steps": args.steps, "repeats": reps, "flops_per_step": flops, "algo_bytes_per_step": nbytes,
           "gpu_launches_per_step": 1,
           "l2": f"inputs rotated over {n_sets} copies ({n_sets * set_bytes(a) / 1e6:.0f} MB > 129 MB L2), no flush"}
    if roof_kind == "tensor":
        obj["roofline"] = {"bound": "tensor", "achieved": tflops, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                           "frac": tflops / pk["bf16_tflops"], "peak_kind": f"{pk_kind} dense bf16 (burst)",
                           "frac_sustained": tflops / pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                           "frac_nominal": tflops / NOMINAL["bf16_tflops"], "traffic": traffic}
    else:
        # bytes-bound: the roofline time is max(FLOPs / tensor peak, bytes / HBM peak)
        t_tc = flops / (pk["bf16_tflops"] * 1e12)
        t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
        obj["roofline"] = {"bound": "hbm" if t_hbm >= t_tc else "tensor", "achieved": gbs,
                           "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                           "peak_kind": f"{pk_kind} copy bandwidth",
                           "roofline_ms": 1e3 * max(t_tc, t_hbm), "frac_of_combined": 1e3 * max(t_tc, t_hbm) / ms,
                           "tensor_frac": tflops / pk["bf16_tflops"], "traffic": traffic}
    del sets
    return obj


def run_ours(args):
    import torch
    import online_softmax_fa2_gb300 as ofa
    from online_softmax_fa2_gb300 import workloads as wl

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    ofa.load()
    pk, pk_kind = peaks()
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    clk = ClockSampler(local)
    clk.start()
    windows = []          # host-time windows of the headline's timed region
    other_windows = []    # the other workloads' timed regions

    # ---------------------------------------------------------------- the headline: 2k causal
    a = wl.causal_2k(dev)
    flops = a.flops()
    head_src = ("fwd_bf16_pair_sm103.cu", "fwd_bf16_common.cuh", "sm100_ptx.cuh", "dropout_rng.cuh",
                "attn_internal.h")
    head = prefill_object(ofa, a, args, stream, pk, pk_kind, windows, barrier, world, dev, 4, "tensor",
                          profiled_traffic("fwd_bf16_pair_kernel.causal_b4_h16_n2048_d128.md", head_src))
    ms = head["ms_per_step"]
    value = job_rate(world, flops, ms)
    achieved = job_rate(1, flops, ms)

    # end to end through the public API: pinned host inputs in, o and lse out, every step.  The
    # steps are pipelined the way a serving loop runs them: step k's inputs copy in on one
    # stream while step k-1 computes and step k-2's outputs copy out on another (two sets of
    # device buffers; events order each buffer's reuse)
    hq = a.q.cpu().pin_memory()
    hk = a.k.cpu().pin_memory()
    hv = a.v.cpu().pin_memory()
    o = torch.empty((a.B, a.Nq, a.H, a.dv), dtype=a.q.dtype, device=dev)
    lse = torch.empty((a.B, a.H, a.Nq), dtype=torch.float32, device=dev)
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    hl = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    dqkv = [(torch.empty_like(a.q), torch.empty_like(a.k), torch.empty_like(a.v)) for _ in range(2)]
    dout = [(torch.empty_like(o), torch.empty_like(lse)) for _ in range(2)]
    h2d = hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2
    d2h = ho[0].numel() * 2 + hl[0].numel() * 4
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {(name, i): torch.cuda.Event() for name in ("in", "comp", "out") for i in range(2)}
    started = {(name, i): False for name in ("in", "comp", "out") for i in range(2)}

    def e2e_step(k):
        i = k % 2
        dq, dk, dv = dqkv[i]
        do, dl = dout[i]
        with torch.cuda.stream(s_in):
            if started[("comp", i)]:
                s_in.wait_event(ev[("comp", i)])   # step k-2 has read these inputs
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            ev[("in", i)].record(s_in)
        stream.wait_event(ev[("in", i)])
        if started[("out", i)]:
            stream.wait_event(ev[("out", i)])       # step k-2's outputs have been copied out
        ofa.attn_fwd(dq, dk, dv, causal=True, scale=a.scale, out=do, lse=dl, stream=stream)
        ev[("comp", i)].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev[("comp", i)])
            ho[i].copy_(do, non_blocking=True)
            hl[i].copy_(dl, non_blocking=True)
            ev[("out", i)].record(s_out)
        for name in ("in", "comp", "out"):
            started[(name, i)] = True

    for k in range(4):
        e2e_step(k)
    n_e2e = max(5, min(args.steps, 50))
    barrier()
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    es.record(s_in)
    for k in range(n_e2e):
        e2e_step(k)
    ee.record(s_out)
    barrier()
    ms_e2e = es.elapsed_time(ee) / n_e2e
    ms_e2e = max_over_ranks(ms_e2e, world, dev)
    del dqkv, dout, hq, hk, hv, ho, hl

    # ---------------------------------------------------------------- the other prefill workloads
    extra = {}
    if not args.no_extra:
        lc = wl.long_causal(dev)
        del lc.meta["jstar"]
        long_src = head_src

        def lc_cpu():
            import numpy as np
            # every row of heads 0 and 31, and the last 256 rows of every head
            whole = np.concatenate([np.arange(lc.Nq) + h * lc.Nq for h in (0, lc.H - 1)])
            last = np.concatenate([np.arange(lc.Nq - 256, lc.Nq) + h * lc.Nq for h in range(lc.H)])
            rows = np.unique(np.concatenate([whole, last]))
            val, secs, desc, threads = cpu_oracle_rows(lc, rows, "every row of heads 0 and 31, the last 256 of every head")
            return {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc,
                    "seconds": secs}

        extra["long_causal"] = prefill_object(
            ofa, lc, args, stream, pk, pk_kind, other_windows, barrier, world, dev, 2, "tensor",
            profiled_traffic("fwd_bf16_pair_kernel.causal_b1_h32_n16384_d128.md", long_src))
        if rank == 0 and not args.no_cpu:
            extra["long_causal"]["cpu_baseline"] = lc_cpu()
        del lc
        pb = wl.padded_bias(dev)
        extra["padbias"] = prefill_object(
            ofa, pb, args, stream, pk, pk_kind, other_windows, barrier, world, dev, 3, "combined",
            profiled_traffic("fwd_bf16_kernel.padbias_b8_h8_n1024_dk192_dv128.md",
                             ("fwd_bf16_sm103.cu", "fwd_bf16_common.cuh", "sm100_ptx.cuh",
                              "dropout_rng.cuh", "attn_internal.h")))
        if rank == 0 and not args.no_cpu:
            val, secs, desc, threads, _ = cpu_oracle_sample(pb, args.cpu_seconds / 2, seed=1)
            extra["padbias"]["cpu_baseline"] = {"value": val, "unit": "TFLOP/s", "cores": threads,
                                                "kind": "oracle", "sample": desc, "seconds": secs}
        del pb
        # the headline workload with dropout p = 0.1: keep decisions drawn in-kernel, and read
        # from a bit-packed keep mask (33.5 MB, one per step here)
        dr = wl.causal_2k(dev)
        keep_mask = wl.pack_keep_mask(wl.dropout_keep(dr.B, dr.H, dr.Nq, dr.Nk, 0.1, seed=1, device=dev))
        extra["dropout"] = {
            "in_kernel_draws": prefill_object(ofa, dr, args, stream, pk, pk_kind, other_windows, barrier, world,
                                              dev, 4, "tensor", None, dropout_p=0.1, dropout_seed=1),
            "keep_mask": prefill_object(ofa, dr, args, stream, pk, pk_kind, other_windows, barrier, world, dev,
                                        4, "tensor", None, dropout_mask=keep_mask, dropout_p=0.1),
            "p": 0.1}
        del dr, keep_mask

    # ---------------------------------------------------------------- split-KV decode (HBM)
    dec = None
    if not args.no_decode:
        # a read-only pass over 4 GiB (torch's sum) as the read bandwidth this run reaches
        x = torch.ones(1 << 30, dtype=torch.float32, device=dev)
        x.sum()
        rs, re_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        rs.record(stream)
        for _ in range(5):
            x.sum()
        re_.record(stream)
        torch.cuda.synchronize()
        read_gbs = 5 * x.numel() * 4 / (rs.elapsed_time(re_) / 1e3) / 1e9
        del x
        d = wl.decode(dev)
        ws = torch.empty(ofa.decode_workspace_bytes(d.B, d.H, d.dv, d.num_splits) // 4,
                         dtype=torch.float32, device=dev)
        wsf = torch.empty(ofa.decode_fused_workspace_bytes(d.B, d.H, d.dv, d.num_splits) // 4 + 4,
                          dtype=torch.float32, device=dev)
        od = torch.empty((d.B, 1, d.H, d.dv), dtype=d.q.dtype, device=dev)
        ld = torch.empty((d.B, d.H, 1), dtype=torch.float32, device=dev)

        def dstep(n):  # two launches: split kernel, then merge kernel
            ofa.attn_decode_splitkv(d.q, d.k, d.v, kv_lens=d.kv_lens, num_splits=d.num_splits,
                                    scale=d.scale, workspace=ws, out=od, lse=ld)

        def dstep_fused(n):  # one launch: the split kernel's last CTA of each (b, h) merges
            ofa.attn_decode_splitkv_fused(d.q, d.k, d.v, kv_lens=d.kv_lens, num_splits=d.num_splits,
                                          scale=d.scale, workspace=wsf, out=od, lse=ld)

        # the 8.6 GB cache is far larger than L2: no flush, no copies needed
        est = warm(dstep_fused, max(3, args.warmup), stream)
        ms_f, _ = time_steps(dstep_fused, args.steps, stream, args.min_seconds / 2, est, barrier, other_windows)
        est = warm(dstep, max(3, args.warmup), stream)
        ms_d, reps = time_steps(dstep, args.steps, stream, args.min_seconds, est, barrier, other_windows)
        ms_d = max_over_ranks(ms_d, world, dev)
        ms_f = max_over_ranks(ms_f, world, dev)
        del ws, wsf, od, ld
        # four query rows per sequence (bottom-right causal) against the same cache
        d4 = wl.decode(dev, nq=4, causal=True)
        ws4 = torch.empty(ofa.decode_workspace_bytes(d4.B, d4.H, d4.dv, d4.num_splits, 4) // 4,
                          dtype=torch.float32, device=dev)
        o4 = torch.empty((d4.B, 4, d4.H, d4.dv), dtype=d4.q.dtype, device=dev)
        l4 = torch.empty((d4.B, d4.H, 4), dtype=torch.float32, device=dev)

        def dstep4(n):
            ofa.attn_decode_splitkv(d4.q, d4.k, d4.v, kv_lens=d4.kv_lens, num_splits=d4.num_splits,
                                    scale=d4.scale, workspace=ws4, out=o4, lse=l4, causal=True)

        est = warm(dstep4, max(3, args.warmup), stream)
        ms_4, reps4 = time_steps(dstep4, args.steps, stream, args.min_seconds / 2, est, barrier, other_windows)
        ms_4 = max_over_ranks(ms_4, world, dev)
        del d4, ws4, o4, l4
        gbs = job_rate(1, d.kv_bytes(), ms_d, 1e9)  # one GPU's rate, against one GPU's peak
        dec = {"workload": "bf16_decode_b64_h32_l8192_d128_splits16",
               "value": job_rate(world, d.kv_bytes(), ms_d, 1e9),
               "unit": "GB/s", "ms_per_step": ms_d, "steps": args.steps, "repeats": reps,
               "kv_bytes_per_step": d.kv_bytes(), "gpu_launches_per_step": 2,
               "path": "attn_decode_splitkv (split kernel + merge kernel)",
               "fused": {"ms_per_step": ms_f, "value": job_rate(world, d.kv_bytes(), ms_f, 1e9),
                         "path": "attn_decode_splitkv_fused (the last split CTA of each (b, h) merges; one launch)"},
               "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"],
                            "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                            "peak_kind": f"{pk_kind} copy bandwidth (read + write)",
                            "read_peak_gbs": read_gbs, "frac_read": gbs / read_gbs,
                            "read_peak_kind": "torch sum over 4 GiB, this run (read only)",
                            "frac_nominal": gbs / NOMINAL["hbm_gbs"],
                            "traffic": profiled_traffic("decode_split_kernel.decode_b64_h32_l8192_d128.md",
                                                        ("decode.cu", "sm100_ptx.cuh", "warp_mma.cuh",
                                                         "attn_internal.h"))}}
        g4 = job_rate(1, d.kv_bytes(), ms_4, 1e9)
        dec["rows4"] = {"workload": "bf16_decode_b64_h32_l8192_d128_nq4_causal_splits16",
                        "value": job_rate(world, d.kv_bytes(), ms_4, 1e9), "unit": "GB/s", "ms_per_step": ms_4,
                        "repeats": reps4, "path": "attn_decode_splitkv, 4 query rows per sequence (decode_rows_mma_kernel + merge)",
                        "roofline": {"bound": "hbm", "achieved": g4, "peak": pk["hbm_gbs"], "unit": "GB/s",
                                     "frac": g4 / pk["hbm_gbs"], "peak_kind": f"{pk_kind} copy bandwidth (read + write)"}}
        del d

    # backward of the same workload (dQ, dK, dV from o, lse and a seeded random dO): reported
    # beside the forward's line with its own tensor roofline, taken over the whole backward
    # step (row terms, products, dQ conversion: three launches)
    bwd = None
    if not args.no_backward:
        def backward_ms(wa, **drop):
            """Time the backward of workload wa (dQ, dK, dV from o, lse and a seeded random dO)
            over three input copies with gradients of their own, stepped back to back like the
            forward; drop: the forward's dropout settings, passed again."""
            o_b, l_b = ofa.attn_fwd(wa.q, wa.k, wa.v, bias=wa.bias, causal=wa.causal, scale=wa.scale, **drop)
            gen = torch.Generator(device=dev)
            gen.manual_seed(7)
            dout_b = torch.randn(o_b.shape, generator=gen, device=dev).to(o_b.dtype)
            ws_b = torch.empty(ofa.bwd_workspace_bytes(wa.B, wa.H, wa.Nq, wa.dk) // 4 + 4, dtype=torch.float32,
                               device=dev)
            bsets = []
            for t in range(3):
                cp = (lambda x: x if (t == 0 or x is None) else x.clone())
                bsets.append((cp(wa.q), cp(wa.k), cp(wa.v), cp(wa.bias), cp(o_b), cp(l_b), cp(dout_b),
                              torch.empty_like(wa.q), torch.empty_like(wa.k), torch.empty_like(wa.v)))

            def bstep(n):
                q_, k_, v_, b_, o_, l_, g_, dq_, dk_, dv_ = bsets[n % 3]
                ofa.attn_bwd(q_, k_, v_, o_, l_, g_, bias=b_, causal=wa.causal, scale=wa.scale, dq=dq_, dk=dk_,
                             dv=dv_, workspace=ws_b, **drop)

            est_b = warm(bstep, max(3, args.warmup), stream)
            ofa.device_error_flags()
            ms_b, reps_b = time_steps(bstep, args.steps, stream, args.min_seconds / (1 if not drop and wa is a else 2),
                                      est_b, barrier, other_windows)
            if ofa.device_error_flags() & 1:
                raise RuntimeError("a backward kernel gave up a bounded wait during the timed region")
            return max_over_ranks(ms_b, world, dev), reps_b

        def backward_obj(wa, ms_b, reps_b, name):
            bflops = wa.visible_pairs() * (6 * wa.dk + 4 * wa.dv)   # five products per visible pair
            tb = job_rate(1, bflops, ms_b)
            return {"workload": name, "value": job_rate(world, bflops, ms_b), "unit": "TFLOP/s",
                    "ms_per_step": ms_b, "steps": args.steps, "repeats": reps_b, "flops_per_step": bflops,
                    "gpu_launches_per_step": 3,
                    "l2": "inputs rotated over 3 copies (more than 129 MB L2), no flush",
                    "roofline": {"bound": "tensor", "achieved": tb, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                                 "frac": tb / pk["bf16_tflops"], "peak_kind": f"{pk_kind} dense bf16 (burst)",
                                 "frac_nominal": tb / NOMINAL["bf16_tflops"],
                                 "over": "the whole backward step (bwd_prep_kernel, bwd_tc_kernel, bwd_dq_kernel)"}}

        ms_b, reps_b = backward_ms(a)
        bwd = backward_obj(a, ms_b, reps_b, "bf16_causal_b4_h16_n2048_d128_backward")
        bwd["roofline"]["traffic"] = profiled_traffic("bwd_tc_kernel.causal_b4_h16_n2048_d128.md",
                                                      ("bwd_tc_sm103.cu", "sm100_ptx.cuh", "fwd_bf16_common.cuh",
                                                       "dropout_rng.cuh", "attn_internal.h"))
        bwd["roofline"]["traffic_kernel"] = "bwd_tc_kernel (its DRAM bytes per launch)"
        if not args.no_extra:
            # the same backward with dropout p = 0.1 drawn in-kernel; at d = 64; with an fp32 bias
            ms_x, reps_x = backward_ms(a, dropout_p=0.1, dropout_seed=1)
            bwd["dropout_in_kernel_draws"] = backward_obj(a, ms_x, reps_x, "bf16_causal_b4_h16_n2048_d128_backward_dropout0.1")
            a64 = wl.causal_2k(dev, d=64)
            ms_x, reps_x = backward_ms(a64)
            bwd["d64"] = backward_obj(a64, ms_x, reps_x, a64.name + "_backward")
            del a64
            ab = wl.causal_2k(dev, bias=True, B=2, H=8)
            ms_x, reps_x = backward_ms(ab)
            bwd["bias"] = backward_obj(ab, ms_x, reps_x, ab.name + "_backward")
            del ab

    clocks = clk.stop(windows)
    clk_all = None
    if clocks is not None:
        # the same sampler over every other timed region, for the record
        sm = [f for t, f, m, r in clk.samples if any(t0 - 0.005 <= t <= t1 + 0.005 for t0, t1 in other_windows)]
        rs_ = set().union(*[r for t, f, m, r in clk.samples
                            if any(t0 - 0.005 <= t <= t1 + 0.005 for t0, t1 in other_windows)] or [set()])
        if sm:
            sm.sort()
            clk_all = {"sm_mhz": sm[len(sm) // 2], "sm_min_mhz": sm[0], "reasons": sorted(rs_), "samples": len(sm)}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": a.B, "H": a.H, "N": a.Nq, "d": a.dk,
                   "causal": True, "flops_per_step": flops, "l2": head["l2"],
                   "timing": f"{head['repeats']} repeats of {args.steps} back-to-back steps, CUDA events "
                             f"around each repeat; ms_per_step = their total / ({head['repeats']} x {args.steps})",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": head["repeats"] * args.steps,
        "e2e": {"value": job_rate(world, flops, ms_e2e), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
                "pipelining": "step k copies in while step k-1 computes and step k-2 copies out"},
        "roofline": dict(head["roofline"],
                         frac_sustained=achieved / pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                         kernel="fwd_bf16_pair_kernel<128, 128, false, false>"),
        "clocks": clocks,
    }
    line.update(extra)
    if dec:
        line["decode"] = dec
    if bwd is not None:
        line["backward"] = bwd
    if clk_all:
        line["clocks_other_regions"] = clk_all
    if rank == 0 and not args.no_cpu:
        val, secs, sample, threads, nheads = cpu_oracle_sample(a, args.cpu_seconds)
        line["cpu_baseline"] = {"value": val, "unit": "TFLOP/s", "cores": threads,
                                "kind": "oracle", "sample": sample, "seconds": secs}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


CASES = {
    # name: (workload factory kwargs, kind)
    "prefill": ("causal_2k", {}, "fwd"),
    "prefill_dropout": ("causal_2k", {}, "fwd_dropout"),
    "prefill_dropout_rng": ("causal_2k", {}, "fwd_dropout_rng"),
    "padbias": ("padded_bias", {}, "fwd"),
    "long_causal": ("long_causal", {}, "fwd"),
    "fp32": ("fp32_small", {}, "fwd"),
    "decode": ("decode", {}, "decode"),
    "decode_fused": ("decode", {}, "decode_fused"),
    "decode_b16": ("decode", {"B": 16}, "decode"),
    "decode_nq4": ("decode", {"nq": 4, "causal": True}, "decode"),
    "decode_nq8": ("decode", {"nq": 8, "causal": True}, "decode"),
    "decode_nq4_b16": ("decode", {"B": 16, "nq": 4, "causal": True}, "decode"),
    "bwd": ("causal_2k", {}, "bwd"),
    "bwd_dropout": ("causal_2k", {}, "bwd_dropout"),
    "bwd_dropout_rng": ("causal_2k", {}, "bwd_dropout_rng"),
    "bwd_long": ("long_causal", {"H": 8}, "bwd"),
    "bwd_d64": ("causal_2k", {"d": 64}, "bwd"),
    "bwd_bias": ("causal_2k", {"bias": True, "B": 2, "H": 8}, "bwd"),
}


def run_case(args):
    """Run one workload's kernels `--steps` times after `--warmup` (no extras): per-launch
    device time and throughput.  Used for the other workloads and as the command under ncu."""
    import torch
    import online_softmax_fa2_gb300 as ofa
    from online_softmax_fa2_gb300 import workloads as wl

    fac, kw, kind = CASES[args.case]
    dev = torch.device("cuda", 0)
    a = getattr(wl, fac)(dev, **kw)
    ofa.load()
    if kind in ("fwd", "fwd_dropout", "fwd_dropout_rng"):
        o = torch.empty((a.B, a.Nq, a.H, a.dv), dtype=a.q.dtype, device=dev)
        lse = torch.empty((a.B, a.H, a.Nq), dtype=torch.float32, device=dev)
        mask, p_drop, seed = None, 0.0, None
        if kind == "fwd_dropout":  # a seeded keep mask with p = 0.1, bit-packed (33.5 MB here)
            p_drop = 0.1
            mask = wl.pack_keep_mask(wl.dropout_keep(a.B, a.H, a.Nq, a.Nk, p_drop, seed=1, device=dev))
        if kind == "fwd_dropout_rng":  # p = 0.1, the keep decisions drawn in-kernel
            p_drop, seed = 0.1, 1
        fn = lambda: ofa.attn_fwd(a.q, a.k, a.v, bias=a.bias, kv_lens=a.kv_lens, causal=a.causal,
                                  scale=a.scale, out=o, lse=lse, dropout_mask=mask, dropout_p=p_drop,
                                  dropout_seed=seed)
        work, unit = a.flops() / 1e12, "TFLOP/s"
    elif kind in ("bwd", "bwd_dropout", "bwd_dropout_rng"):
        mask, p_drop, seed = None, 0.0, None
        if kind == "bwd_dropout":  # the forward's seeded keep mask with p = 0.1
            p_drop = 0.1
            mask = wl.pack_keep_mask(wl.dropout_keep(a.B, a.H, a.Nq, a.Nk, p_drop, seed=1, device=dev))
        if kind == "bwd_dropout_rng":  # p = 0.1, the keep decisions drawn in-kernel
            p_drop, seed = 0.1, 1
        o, lse = ofa.attn_fwd(a.q, a.k, a.v, bias=a.bias, kv_lens=a.kv_lens, causal=a.causal,
                              scale=a.scale, dropout_mask=mask, dropout_p=p_drop, dropout_seed=seed)
        gen = torch.Generator(device=dev)
        gen.manual_seed(7)
        dout = torch.randn(o.shape, generator=gen, device=dev).to(o.dtype)
        ws = torch.empty(ofa.bwd_workspace_bytes(a.B, a.H, a.Nq, a.dk) // 4 + 4, dtype=torch.float32,
                         device=dev)
        dq, dk, dv = torch.empty_like(a.q), torch.empty_like(a.k), torch.empty_like(a.v)
        fn = lambda: ofa.attn_bwd(a.q, a.k, a.v, o, lse, dout, bias=a.bias, kv_lens=a.kv_lens,
                                  causal=a.causal, scale=a.scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                                  dropout_mask=mask, dropout_p=p_drop, dropout_seed=seed)
        # 2 (S) + 2 (dP) + 2 (dV) + 2 (dK) + 2 (dQ) products: (6 dk + 4 dv) FLOPs per visible pair
        work, unit = a.visible_pairs() * (6 * a.dk + 4 * a.dv) / 1e12, "TFLOP/s"
    elif kind == "decode_fused":
        ws = torch.empty(ofa.decode_fused_workspace_bytes(a.B, a.H, a.dv, a.num_splits, a.Nq) // 4 + 4,
                         dtype=torch.float32, device=dev)
        o = torch.empty((a.B, a.Nq, a.H, a.dv), dtype=a.q.dtype, device=dev)
        lse = torch.empty((a.B, a.H, a.Nq), dtype=torch.float32, device=dev)
        fn = lambda: ofa.attn_decode_splitkv_fused(a.q, a.k, a.v, kv_lens=a.kv_lens, bias=a.bias,
                                                   num_splits=a.num_splits, scale=a.scale,
                                                   workspace=ws, out=o, lse=lse, causal=a.causal)
        work, unit = a.kv_bytes() / 1e9, "GB/s"
    else:
        ws = torch.empty(ofa.decode_workspace_bytes(a.B, a.H, a.dv, a.num_splits, a.Nq) // 4,
                         dtype=torch.float32, device=dev)
        o = torch.empty((a.B, a.Nq, a.H, a.dv), dtype=a.q.dtype, device=dev)
        lse = torch.empty((a.B, a.H, a.Nq), dtype=torch.float32, device=dev)
        fn = lambda: ofa.attn_decode_splitkv(a.q, a.k, a.v, kv_lens=a.kv_lens, bias=a.bias,
                                             num_splits=a.num_splits, scale=a.scale,
                                             workspace=ws, out=o, lse=lse, causal=a.causal)
        work, unit = a.kv_bytes() / 1e9, "GB/s"
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        ts.append((s, e))
    torch.cuda.synchronize()
    ms = sorted(s.elapsed_time(e) for s, e in ts)
    med = ms[len(ms) // 2]
    print(json.dumps({"case": args.case, "workload": a.name, "ms_median": med, "ms_min": ms[0],
                      "value_median": work / (med / 1e3), "unit": unit, "steps": args.steps,
                      "error_flags": ofa.device_error_flags()}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="leave out the long causal and padded workloads")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="wall-time budget of the reference arm's run (sets the heads per step)")
    ap.add_argument("--min-seconds", type=float, default=0.25,
                    help="device time each timed region is repeated up to (in whole K-step repeats)")
    ap.add_argument("--case", choices=sorted(CASES), default=None,
                    help="time one workload's kernels only (also the command profiled by ncu)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.case:
        return run_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
