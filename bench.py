"""Benchmark: exact attention forward on GB300, through the library's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one attention forward over the bf16 causal workload B=4, H=16, N=2048, d=128
(scale 1/sqrt(128)), O in bf16 and lse in fp32, inputs resident in HBM.  value = algorithmic
TFLOP/s: 2*(dk + dv) FLOPs per visible (query, key) pair, causal pairs only, divided by the
device time of the step (CUDA events on the launching stream; L2 flushed before every timed
step by writing a 256 MiB buffer outside the timed interval).  The same line carries:
  e2e           the same metric with the step's inputs copied host->device from pinned memory
                and o, lse copied back inside the timed interval;
  roofline      the fused kernel's achieved TFLOP/s against the measured dense-bf16 peak;
  decode        split-KV decode on B=64, H=32, L=8192 (kv_len ~ U{1..8192}), d=128, 16 splits:
                KV GB/s (visible keys only) against the measured HBM peak;
  cpu_baseline  the float64 CPU oracle timed on a bounded sample of the same workload;
  clocks        SM clocks sampled with nvidia-smi during the timed region.
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
    """nvidia-smi clocks and throttle reasons sampled every 20 ms while running."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)  # nvidia-smi needs a moment before its first sample
        except OSError:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def mark(self):
        return time.time()

    def stop(self, t0, t1):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            if not (t0 - 0.05 <= t <= t1 + 0.05):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


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


def cpu_oracle_sample(a, seconds_target, seed=0):
    """Time the float64 oracle on whole heads of workload `a` (taken in a fixed seeded order)
    until about `seconds_target` of CPU work; returns (TFLOP/s, sample description, threads)."""
    import numpy as np
    import torch
    import oracle

    q = a.q.detach().cpu().float()
    k = a.k.detach().cpu().float()
    v = a.v.detach().cpu().float()
    rng = np.random.default_rng(seed)
    order = rng.permutation(a.B * a.H)
    flops_head = a.flops() / (a.B * a.H)
    done, t_used, threads = 0, 0.0, 0
    while t_used < seconds_target:  # passes over the heads until the time target is reached
        for bh in order:
            b, h = divmod(int(bh), a.H)
            t0 = time.perf_counter()
            _, _, threads = oracle.attn_fwd(q[b:b + 1, :, h:h + 1], k[b:b + 1, :, h:h + 1],
                                            v[b:b + 1, :, h:h + 1], causal=a.causal, scale=a.scale)
            t_used += time.perf_counter() - t0
            done += 1
            if t_used >= seconds_target:
                break
    return (done * flops_head / t_used / 1e12, t_used,
            f"{done} head evaluations over the {a.B * a.H} (b, h) heads (whole heads, all causal "
            f"rows, float64)", threads, done)


def run_reference(args):
    """The oracle as the reference arm: each step is one (b, h) head of the workload."""
    import torch
    from online_softmax_fa2_gb300 import workloads as wl
    import oracle

    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    a = wl.causal_2k("cpu")
    q, k, v = a.q.float(), a.k.float(), a.v.float()
    flops_head = a.flops() / (a.B * a.H)
    # one head per step keeps --steps K --warmup W within minutes on the host cores
    heads = [(i % a.B, (i * 7) % a.H) for i in range(args.steps + args.warmup)]
    times, threads = [], 0
    for n, (b, h) in enumerate(heads):
        t0 = time.perf_counter()
        _, _, threads = oracle.attn_fwd(q[b:b + 1, :, h:h + 1], k[b:b + 1, :, h:h + 1],
                                        v[b:b + 1, :, h:h + 1], causal=True, scale=a.scale)
        dt = time.perf_counter() - t0
        if n >= args.warmup:
            times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    val = flops_head / (ms / 1e3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "step": "one (b, h) head of the workload per step",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": "one (b, h) head (2048 causal rows) per step"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


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

    a = wl.causal_2k(dev)
    flops = a.flops()
    o = torch.empty((a.B, a.Nq, a.H, a.dv), dtype=a.q.dtype, device=dev)
    lse = torch.empty((a.B, a.H, a.Nq), dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def step():
        ofa.attn_fwd(a.q, a.k, a.v, causal=True, scale=a.scale, out=o, lse=lse)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    ofa.device_error_flags()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clk = ClockSampler(local)
    clk.start()
    barrier()
    t0 = time.time()
    for s, e in ev:
        flush.zero_()            # L2 flush, outside the timed interval
        s.record(stream)
        step()
        e.record(stream)
    barrier()
    t1 = time.time()
    clocks = clk.stop(t0, t1)
    ms_steps = [s.elapsed_time(e) for s, e in ev]
    ms = sum(ms_steps) / len(ms_steps)
    if ofa.device_error_flags() & 1:
        raise RuntimeError("a kernel gave up a bounded wait during the timed region")
    ms = max_over_ranks(ms, world, dev)
    value = job_rate(world, flops, ms)
    achieved = job_rate(1, flops, ms)

    # end to end through the public API: pinned host inputs in, o and lse out, every step.  The
    # steps are pipelined the way a serving loop runs them: step k's inputs copy in on one
    # stream while step k-1 computes and step k-2's outputs copy out on another (two sets of
    # device buffers; events order each buffer's reuse)
    hq = a.q.cpu().pin_memory()
    hk = a.k.cpu().pin_memory()
    hv = a.v.cpu().pin_memory()
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

    # split-KV decode on the long-cache workload (its own roofline: HBM)
    dec = None
    if not args.no_decode:
        d = wl.decode(dev)
        ws = torch.empty(ofa.decode_workspace_bytes(d.B, d.H, d.dv, d.num_splits) // 4,
                         dtype=torch.float32, device=dev)
        od = torch.empty((d.B, 1, d.H, d.dv), dtype=d.q.dtype, device=dev)
        ld = torch.empty((d.B, d.H, 1), dtype=torch.float32, device=dev)

        def dstep():
            ofa.attn_decode_splitkv(d.q, d.k, d.v, kv_lens=d.kv_lens, num_splits=d.num_splits,
                                    scale=d.scale, workspace=ws, out=od, lse=ld)

        for _ in range(max(3, args.warmup)):
            dstep()
        nd = max(5, min(args.steps, 100))
        barrier()
        ds, de = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ds.record(stream)
        for _ in range(nd):       # the 8.6 GB cache is far larger than L2: no flush needed
            dstep()
        de.record(stream)
        barrier()
        ms_d = max_over_ranks(ds.elapsed_time(de) / nd, world, dev)
        gbs = job_rate(1, d.kv_bytes(), ms_d, 1e9)  # one GPU's rate, against one GPU's peak
        dec = {"workload": "bf16_decode_b64_h32_l8192_d128_splits16",
               "value": job_rate(world, d.kv_bytes(), ms_d, 1e9),
               "unit": "GB/s", "ms_per_step": ms_d, "steps": nd,
               "kv_bytes_per_step": d.kv_bytes(), "gpu_launches_per_step": 2,
               "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"],
                            "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                            "peak_kind": f"{pk_kind} copy bandwidth",
                            "frac_nominal": gbs / NOMINAL["hbm_gbs"],
                            "traffic": profiled_traffic("decode_split_kernel.decode_b64_h32_l8192_d128.md",
                                                        ("decode.cu",))}}
        del d, ws

    # backward of the same workload (dQ, dK, dV from o, lse and a seeded random dO): reported
    # beside the forward's line with its own tensor roofline, taken over the whole backward
    # step (row terms, products, dQ conversion: three launches)
    bwd = None
    if not args.no_backward:
        o_b, l_b = ofa.attn_fwd(a.q, a.k, a.v, causal=True, scale=a.scale)
        gen = torch.Generator(device=dev)
        gen.manual_seed(7)
        dout_b = torch.randn(o_b.shape, generator=gen, device=dev).to(o_b.dtype)
        ws_b = torch.empty(ofa.bwd_workspace_bytes(a.B, a.H, a.Nq, a.dk) // 4 + 4, dtype=torch.float32,
                           device=dev)
        gq, gk, gv = torch.empty_like(a.q), torch.empty_like(a.k), torch.empty_like(a.v)

        def bstep():
            ofa.attn_bwd(a.q, a.k, a.v, o_b, l_b, dout_b, causal=True, scale=a.scale, dq=gq, dk=gk, dv=gv,
                         workspace=ws_b)

        for _ in range(max(3, min(args.warmup, 10))):
            flush.zero_()
            bstep()
        nb = max(5, min(args.steps, 50))
        evb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nb)]
        barrier()
        for s_, e_ in evb:
            flush.zero_()            # L2 flush, outside the timed interval
            s_.record(stream)
            bstep()
            e_.record(stream)
        barrier()
        if ofa.device_error_flags() & 1:
            raise RuntimeError("a backward kernel gave up a bounded wait during the timed region")
        ms_b = max_over_ranks(sum(s_.elapsed_time(e_) for s_, e_ in evb) / nb, world, dev)
        bflops = a.visible_pairs() * (6 * a.dk + 4 * a.dv)   # five products per visible pair
        tb = job_rate(1, bflops, ms_b)
        bwd = {"workload": "bf16_causal_b4_h16_n2048_d128_backward", "value": job_rate(world, bflops, ms_b),
               "unit": "TFLOP/s", "ms_per_step": ms_b, "steps": nb, "flops_per_step": bflops,
               "gpu_launches_per_step": 3, "l2": "flushed before every step",
               "roofline": {"bound": "tensor", "achieved": tb, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": tb / pk["bf16_tflops"], "peak_kind": f"{pk_kind} dense bf16 (burst)",
                            "frac_nominal": tb / NOMINAL["bf16_tflops"],
                            "over": "the whole backward step (bwd_prep_kernel, bwd_tc_kernel, bwd_dq_kernel)",
                            "traffic": None}}
        del o_b, l_b, dout_b, ws_b, gq, gk, gv

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": a.B, "H": a.H, "N": a.Nq, "d": a.dk,
                   "causal": True, "flops_per_step": flops, "l2": "flushed before every step",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": args.steps,
        "e2e": {"value": job_rate(world, flops, ms_e2e), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
                "pipelining": "step k copies in while step k-1 computes and step k-2 copies out"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                     "peak_kind": f"{pk_kind} dense bf16 (burst)",
                     "frac_sustained": achieved / pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                     "frac_nominal": achieved / NOMINAL["bf16_tflops"],
                     "kernel": "fwd_bf16_pair_kernel<128, 128, false, false>",
                     "traffic": profiled_traffic("fwd_bf16_pair_kernel.causal_b4_h16_n2048_d128.md",
                                                 ("fwd_bf16_pair_sm103.cu", "fwd_bf16_common.cuh",
                                                  "sm100_ptx.cuh"))},
        "clocks": clocks,
    }
    if dec:
        line["decode"] = dec
    if bwd is not None:
        line["backward"] = bwd
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
    "padbias": ("padded_bias", {}, "fwd"),
    "long_causal": ("long_causal", {}, "fwd"),
    "fp32": ("fp32_small", {}, "fwd"),
    "decode": ("decode", {}, "decode"),
    "decode_b16": ("decode", {"B": 16}, "decode"),
    "decode_nq4": ("decode", {"nq": 4, "causal": True}, "decode"),
    "decode_nq8": ("decode", {"nq": 8, "causal": True}, "decode"),
    "decode_nq4_b16": ("decode", {"B": 16, "nq": 4, "causal": True}, "decode"),
    "bwd": ("causal_2k", {}, "bwd"),
    "bwd_dropout": ("causal_2k", {}, "bwd_dropout"),
    "bwd_long": ("long_causal", {"H": 8}, "bwd"),
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
    if kind in ("fwd", "fwd_dropout"):
        o = torch.empty((a.B, a.Nq, a.H, a.dv), dtype=a.q.dtype, device=dev)
        lse = torch.empty((a.B, a.H, a.Nq), dtype=torch.float32, device=dev)
        mask, p_drop = None, 0.0
        if kind == "fwd_dropout":  # a seeded keep mask with p = 0.1, bit-packed (33.5 MB here)
            p_drop = 0.1
            mask = wl.pack_keep_mask(wl.dropout_keep(a.B, a.H, a.Nq, a.Nk, p_drop, seed=1, device=dev))
        fn = lambda: ofa.attn_fwd(a.q, a.k, a.v, bias=a.bias, kv_lens=a.kv_lens, causal=a.causal,
                                  scale=a.scale, out=o, lse=lse, dropout_mask=mask, dropout_p=p_drop)
        work, unit = a.flops() / 1e12, "TFLOP/s"
    elif kind in ("bwd", "bwd_dropout"):
        mask, p_drop = None, 0.0
        if kind == "bwd_dropout":  # the forward's seeded keep mask with p = 0.1
            p_drop = 0.1
            mask = wl.pack_keep_mask(wl.dropout_keep(a.B, a.H, a.Nq, a.Nk, p_drop, seed=1, device=dev))
        o, lse = ofa.attn_fwd(a.q, a.k, a.v, bias=a.bias, kv_lens=a.kv_lens, causal=a.causal,
                              scale=a.scale, dropout_mask=mask, dropout_p=p_drop)
        gen = torch.Generator(device=dev)
        gen.manual_seed(7)
        dout = torch.randn(o.shape, generator=gen, device=dev).to(o.dtype)
        ws = torch.empty(ofa.bwd_workspace_bytes(a.B, a.H, a.Nq, a.dk) // 4 + 4, dtype=torch.float32,
                         device=dev)
        dq, dk, dv = torch.empty_like(a.q), torch.empty_like(a.k), torch.empty_like(a.v)
        fn = lambda: ofa.attn_bwd(a.q, a.k, a.v, o, lse, dout, bias=a.bias, kv_lens=a.kv_lens,
                                  causal=a.causal, scale=a.scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                                  dropout_mask=mask, dropout_p=p_drop)
        # 2 (S) + 2 (dP) + 2 (dV) + 2 (dK) + 2 (dQ) products: (6 dk + 4 dv) FLOPs per visible pair
        work, unit = a.visible_pairs() * (6 * a.dk + 4 * a.dv) / 1e12, "TFLOP/s"
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
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
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
