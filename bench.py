#!/usr/bin/env python3
"""Benchmark of the paged FP8 latent-KV MLA decode step on GB300.

One step = one mla_decode_paged call (split-KV decode kernel + split combine)
over one whole batch.  The default workload is the long-context and ragged
serving mix: its ragged batch (128 requests x 12 heads x 1 position, contexts
log-uniform in [1024, 142000], ~2.1 GB of FP8 latents per step) gives the
line's value, and its single 393,216-position request is measured the same way
and reported under "serving_mix".  Other shapes: --workload tiny | tp8_batch |
dcp_shard | verify | long | ragged.  Page 64, block tables randomly permuted,
FP8 E4M3FN latents (576 B per position), bf16 queries.

Metric: latent-KV GB/s = (KV bytes the step must read) / (step time), plus
decode steps/s and the fraction of the HBM roofline.  Inputs are resident in
HBM; L2 is defeated by rotating several cache copies whose total exceeds 3x L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the FP64 CPU oracle on host cores

Multi-GPU (torchrun, one rank per GPU): every rank decodes its own batch of
the same shape (independent requests, no collective on the data path);
value = bytes of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HBM_NOMINAL_GBS = 8000.0  # the post's and the spec sheet's 8 TB/s
MLA_LAYERS = 24  # "Kimi K3 on AMD Instinct MI355X" post, the model section: 24 MLA layers
METRIC = "latent-KV GB/s (KV bytes read / decode-step time); decode steps/s; % of 8 TB/s HBM"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--sustain-s", type=float, default=2.0,
                    help="seconds of back-to-back graph replays after the timed steps (clock record); "
                         "0 skips them")
    ap.add_argument("--requests", type=int, default=0,
                    help="profiling only: keep the first N requests of the workload's batch")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="serving_mix",
                    help="serving_mix (config 5: the ragged batch as the value, the 393,216-position "
                         "request beside it) or one of tiny, tp8_batch, dcp_shard, verify, long, ragged")
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "tcgen05"])
    ap.add_argument("--n-splits", type=int, default=0)
    ap.add_argument("--planner", default="lengths", choices=["lengths", "auto"],
                    help="split count when --n-splits is 0: mla_plan_splits on the host-known "
                         "lengths, or mla_auto_splits from max_pages alone")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-ceiling", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-append", action="store_true",
                    help="skip the append, DCP merge and DCP verify side measurements")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(ms, world, device):
    """The job's time: the slowest rank's (every rank passes its own ms)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(bytes_per_rank, world, ms_step):
    """Whole-job throughput: the bytes of all ranks over the job's step time."""
    return world * bytes_per_rank / (ms_step * 1e-3) / 1e9


def workload_description(name):
    from mla_latent_kv_fp8_gb300 import synth
    return synth.WORKLOADS[name][0]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    return 6800.0, "fallback (6.8 TB/s)"


FP8_PER_BF16 = 2.0  # nominal dense tensor rate ratio (4.5 vs 2.25 PFLOP/s per GPU)
FLOP_PER_ROW_POSITION = 2 * 576 + 2 * 512  # q . x over 576 dims, p * x over 512


def algorithmic_flops(lens, T, H):
    """Useful flops of one decode call: 2,176 per (query row, visible position);
    query t of a request of length L sees L - T + 1 + t positions."""
    return FLOP_PER_ROW_POSITION * H * sum(T * (L - T + 1) + T * (T - 1) // 2 for L in lens if L > 0)


def tensor_roofline(flops, kernel_s):
    """The decode kernel against the FP8 tensor peak: the measured bf16 burst peak
    times the nominal fp8/bf16 ratio (the MMAs are e4m3 x e4m3)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            bf16 = float(json.load(f)["bf16_tflops"])
        src = "measured bf16 burst (MEASURED_PEAKS.json bf16_tflops) x 2, the nominal fp8/bf16 ratio"
    else:
        bf16, src = 1900.0, "fallback bf16 1.9 PFLOP/s x 2, the nominal fp8/bf16 ratio"
    peak = bf16 * FP8_PER_BF16
    achieved = flops / kernel_s / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "peak_source": src, "algorithmic_flops_per_launch": flops,
            "note": "algorithmic flops (2,176 per row and visible position); the kernel issues twice "
                    "that on the tensor cores (two-term query and probability splits)"}


def carve(device, specs, pin=False):
    """One byte buffer holding a tensor per (shape, dtype) at 256-byte aligned
    offsets; returns the buffer and the typed views."""
    import torch
    offs, total = [], 0
    for shape, dtype in specs:
        n = 1
        for d in shape:
            n *= int(d)
        offs.append(total)
        total += (n * torch.empty((), dtype=dtype).element_size() + 255) // 256 * 256
    buf = torch.empty(total, dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = []
    for (shape, dtype), o in zip(specs, offs):
        n = 1
        for d in shape:
            n *= int(d)
        es = torch.empty((), dtype=dtype).element_size()
        views.append(buf[o:o + n * es].view(dtype).view(shape))
    return buf, views


def stream_ceiling(L, base, caches, n_copies, grid, stream, launches=200):
    """Time the library's page-streaming probe on the pages one decode step reads:
    every page of every request once, split evenly over the decode's grid, through
    the same TMA ring, with no arithmetic.  Its GB/s is the ceiling of this access
    pattern at this launch size (ramp-up and tail included)."""
    import torch
    n_req = ((base.seq_lens.long() + 63) // 64).cpu()
    ids = torch.cat([base.block_table[b, :int(n_req[b])] for b in range(base.block_table.shape[0])])
    ctas = max(1, min(grid, ids.numel()))
    ppc = ids.numel() // ctas
    ids = ids[:ctas * ppc].contiguous()
    for i in range(3):
        L.mla_bench_stream_pages(caches[i % n_copies], ids, ctas, ppc, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(launches):
        L.mla_bench_stream_pages(caches[i % n_copies], ids, ctas, ppc, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    if L.mla_device_error() != 0:
        raise RuntimeError("page-streaming probe reported a device error")
    us = e0.elapsed_time(e1) * 1e3 / launches
    nbytes = ids.numel() * 64 * 576
    return {"value": round(nbytes / (us * 1e-6) / 1e9, 1), "unit": "GB/s", "us_per_launch": round(us, 2),
            "ctas": ctas, "pages_per_cta": ppc, "bytes_per_launch": nbytes, "launches": launches,
            "note": "mla_bench_stream_pages: the step's pages copied through the decode's TMA ring "
                    "and discarded, back-to-back launches"}


KERNEL_SOURCES = {
    # family: (kernel file, device headers it includes)
    "tcgen05": ("mla_latent_kv_fp8_gb300/csrc/mla_tc.cu", "mla_latent_kv_fp8_gb300/csrc/mla_tc_wide.cu",
                "mla_latent_kv_fp8_gb300/csrc/mla_tc_ptx.cuh", "mla_latent_kv_fp8_gb300/csrc/mla_internal.cuh"),
    "simt": ("mla_latent_kv_fp8_gb300/csrc/mla_simt.cu", "mla_latent_kv_fp8_gb300/csrc/mla_internal.cuh"),
}
HOST_SIDE_MARKER = "// ---------------------------------------------------------------- host side"


def device_code_digest(rel_paths):
    """Digest of the device code of a kernel family: each file's text before its
    host-side marker (the whole file if it has none), with comments and blank
    lines dropped, so that edits to host code or comments keep recorded ncu
    counters valid while any change to the kernels invalidates them."""
    h = hashlib.sha256()
    for rel in rel_paths:
        with open(os.path.join(ROOT, rel)) as fh:
            text = fh.read()
        text = text.split(HOST_SIDE_MARKER)[0]
        for line in text.splitlines():
            line = line.split("//")[0].rstrip()
            if line:
                h.update(line.encode() + b"\n")
    return h.hexdigest()[:16]


def ncu_traffic(kernel_family, workload):
    """DRAM bytes per launch of the decode kernel from a committed ncu summary
    (profiles/ncu_traffic.json), if the family's device code is unchanged since
    the counters were taken; else None.  A record taken on a reduced case is
    scaled to the full launch by the ratio of KV bytes (the record says so)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p) or kernel_family not in KERNEL_SOURCES:
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel_family}/{workload}")
    if not e or e.get("device_code_digest") != device_code_digest(KERNEL_SOURCES[kernel_family]):
        return None
    return {"dram_bytes_per_launch": e["dram_bytes_per_launch"], "source": e.get("note", ""),
            "ncu_command": e.get("command", "")}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running,
    each sample with its host time, so that a window can be summarised."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"mla_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu=timestamp,{self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts[1:])
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = sorted(v for v in (num(r[1]) for r in rows) if v is not None)
        mx = max((v for v in (num(r[2]) for r in rows) if v is not None), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        pw = [v for v in (num(r[3]) for r in rows) if v is not None]
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


def make_inputs(name, device, requests=0):
    """The workload's inputs; requests > 0 keeps the first that many requests of
    its batch (a smaller case of the same shape, for profiler captures)."""
    from mla_latent_kv_fp8_gb300 import synth
    return synth.workload_case(name, device=device, requests=requests)


# Config 5 of the benchmark ("long-context and ragged serving mix"): its ragged
# batch (5b, the larger workload) is the headline value; its single long
# request (5a) is measured the same way and reported beside it.
SERVING_MIX = ("ragged", "long")


class DecodeStep:
    """One workload prepared for timing: inputs resident in HBM, rotating cache
    copies (more bytes than 3x L2, so every step reads HBM), the split count, and
    a CUDA graph of consecutive steps as a serving loop would launch them."""

    def __init__(self, L, name, args, dev, stream):
        import torch
        self.L, self.name, self.dev, self.stream = L, name, dev, stream
        base = make_inputs(name, "cpu" if name in ("tiny",) else dev, getattr(args, "requests", 0)).to(dev)
        self.base = base
        self.kv_bytes = base.kv_bytes()
        B, T, H = base.B, base.T, base.H
        n_splits = args.n_splits if args.n_splits > 0 else (4 if name == "tiny" else 0)
        self.planner = "explicit" if n_splits > 0 else "mla_auto_splits (from max_pages)"
        if n_splits == 0 and args.planner == "lengths":
            # a serving engine knows its batch's lengths on the host: plan once per batch
            t_plan = time.perf_counter()
            n_splits = L.mla_plan_splits(B, T, H, base.lens, base.block_table.shape[1], 0)
            t_plan = time.perf_counter() - t_plan
            self.planner = (f"mla_plan_splits from the host lengths, once per batch outside the timed "
                            f"steps ({t_plan * 1e6:.0f} us on the host)")
        self.n_splits = n_splits
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n_copies = max(2, -(-3 * self.l2 // max(base.kv_cache.numel(), 1)))
        self.n_copies = min(n_copies, 64)
        self.caches = [base.kv_cache] + [base.kv_cache.clone() for _ in range(self.n_copies - 1)]
        self.out = torch.empty((B, T, H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, T, H), dtype=torch.float32, device=dev)
        mp = base.block_table.shape[1]
        resolved = L.mla_auto_splits(B, T, H, mp, 0) if n_splits == 0 else n_splits
        self.chunk = L.mla_split_chunk_pages(mp, resolved)
        self.n_eff = -(-mp // self.chunk)
        # our kernels per step: the decode, the split combine when split, and for a
        # tensor-core launch with more CTAs than SMs the longest-first ordering
        # kernel before the decode
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        row_ctas = 1 if H * T <= 16 else -(-(H * T) // 32)
        lpt = (args.kernel != "simt" and self.n_eff > 1 and B <= 1024 and B * self.n_eff * row_ctas > sms)
        self.launches_per_step = 1 + (1 if self.n_eff > 1 else 0) + (1 if lpt else 0)
        self.graph = None
        self.gsteps = self.n_copies * max(1, -(-16 // self.n_copies))

    def step(self, i):
        b = self.base
        self.L.mla_decode_paged(b.q, self.caches[i % self.n_copies], b.kv_scale, b.block_table, b.seq_lens,
                                self.n_splits, b.sm_scale, self.out, self.lse, self.stream)

    def capture(self):
        """A CUDA graph of gsteps consecutive calls (captured after warm-up calls,
        so that the library's per-stream scratch already exists)."""
        import torch
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            for i in range(self.gsteps):
                self.step(i)
        with torch.cuda.stream(self.stream):
            self.graph.replay()

    def timed(self, steps, barrier):
        """Exactly `steps` steps between barriers, as graph replays plus direct
        calls for the remainder; returns (ms for all steps, mean step us of each
        replay)."""
        import torch
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_rep, n_rem = divmod(steps, self.gsteps)
        rep_evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep)]
        barrier()
        ev0.record(self.stream)
        with torch.cuda.stream(self.stream):
            for e in rep_evs:
                self.graph.replay()
                e.record(self.stream)
        for i in range(n_rem):
            self.step(i)
        ev1.record(self.stream)
        barrier()
        rep_us = sorted(a.elapsed_time(b_) * 1e3 / self.gsteps for a, b_ in zip([ev0] + rep_evs[:-1], rep_evs))
        return ev0.elapsed_time(ev1), rep_us, (n_rep, n_rem)

    def direct(self, k, barrier):
        import torch
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        ev0.record(self.stream)
        for i in range(k):
            self.step(i)
        ev1.record(self.stream)
        barrier()
        return ev0.elapsed_time(ev1) / k

    def kernel_ms(self, k, barrier):
        """The decode kernel alone, CUDA events recorded around it on its stream."""
        import torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        for a, b_ in evs:  # create the underlying CUDA events on this stream
            a.record(self.stream)
            b_.record(self.stream)
        barrier()
        for i, (a, b_) in enumerate(evs):
            self.L.mla_profile_next_decode(a.cuda_event, b_.cuda_event)
            self.step(i)
        barrier()
        return sorted(a.elapsed_time(b_) for a, b_ in evs)

    def sustained(self, seconds, barrier):
        """Graph replays back to back for at least `seconds` (the clocks seen under
        a long run of this step); returns (us per step, steps), or (None, 0)."""
        import torch
        if seconds <= 0:
            return None, 0
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        ev0.record(self.stream)
        t0, reps = time.perf_counter(), 0
        with torch.cuda.stream(self.stream):
            while True:
                for _ in range(8):
                    self.graph.replay()
                reps += 8
                self.stream.synchronize()
                if time.perf_counter() - t0 >= seconds:
                    break
        ev1.record(self.stream)
        barrier()
        n = reps * self.gsteps
        return ev0.elapsed_time(ev1) * 1e3 / n, n


def kernel_roofline(w, kernel_ms, family, workload):
    peak, peak_src = load_peaks()
    k_avg_ms = sum(kernel_ms) / len(kernel_ms)
    achieved = w.kv_bytes / (k_avg_ms * 1e-3) / 1e9
    traffic = ncu_traffic(family, workload)
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic["dram_bytes_per_launch"] if traffic else None,
            "traffic_source": traffic["source"] if traffic else "no ncu record of the current device code",
            "peak_source": peak_src, "kernel": f"{family} split-KV decode",
            "kernel_avg_us": round(k_avg_ms * 1e3, 2),
            "kernel_p10_us": round(kernel_ms[len(kernel_ms) // 10] * 1e3, 2),
            "kernel_p50_us": round(kernel_ms[len(kernel_ms) // 2] * 1e3, 2),
            "kernel_p90_us": round(kernel_ms[(9 * len(kernel_ms)) // 10] * 1e3, 2),
            "frac_of_8TBps": round(achieved / HBM_NOMINAL_GBS, 4),
            "algorithmic_bytes_per_launch": w.kv_bytes}


def run_ours(args):
    import torch
    from mla_latent_kv_fp8_gb300 import _lib, synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)  # before the process group, so NCCL binds this rank's GPU
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    L = _lib
    L.lib()
    impl = {"auto": 0, "simt": 1, "tcgen05": 2}[args.kernel]
    L.mla_set_impl(impl)
    stream = torch.cuda.Stream(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier(device_ids=[local])
        torch.cuda.synchronize(dev)

    names = list(SERVING_MIX) if args.workload == "serving_mix" else [args.workload]
    primary, others = names[0], names[1:]
    w = DecodeStep(L, primary, args, dev, stream)
    base, kv_bytes, B, T, H = w.base, w.kv_bytes, w.base.B, w.base.T, w.base.H
    for i in range(args.warmup):
        w.step(i)
    barrier()
    assert L.mla_device_error() == 0
    w.capture()
    barrier()
    assert L.mla_device_error() == 0

    # ---- main timed region: exactly K steps; then a sustained run of the same
    # step (>= 2 s) under the same clock sampler ----
    with ClockSampler(local) as clk:
        ms_total, rep_us, (n_rep, n_rem) = w.timed(args.steps, barrier)
        sus_us, sus_steps = w.sustained(args.sustain_s, barrier)
    assert L.mla_device_error() == 0
    clocks = clk.summary()
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_step = ms_total / args.steps
    value = job_gbps(kv_bytes, world, ms_step)
    steps_per_s = 1e3 / ms_step

    # ---- the same steps as individual API calls (host launch cost included) ----
    kdirect = min(args.steps, 2000)
    ms_direct = max_over_ranks(w.direct(kdirect, barrier), world, dev)

    # ---- the dominant kernel alone, with events recorded around it on its stream ----
    kernel_ms = w.kernel_ms(min(max(args.steps, 20), 2000), barrier)
    family = {1: "simt", 2: "tcgen05"}.get(L.mla_last_decode_impl(), "unknown")
    roofline = kernel_roofline(w, kernel_ms, family, primary)
    if clocks.get("sm_mhz"):
        roofline["kernel_p50_kcycles"] = round(roofline["kernel_p50_us"] * clocks["sm_mhz"] / 1e3, 1)
    # the many-row shapes are real contractions: their tensor-core side as well
    roofline_tensor = (tensor_roofline(algorithmic_flops(base.lens, T, H), sum(kernel_ms) / len(kernel_ms) * 1e-3)
                       if H * T > 16 and family == "tcgen05" else None)

    # ---- the ceiling of this access pattern: the same pages, no arithmetic ----
    ceiling = None
    if not args.no_ceiling:
        rows_ctas = 1 if H * T <= 16 else -(-(H * T) // 32)  # CTAs per (request, partition)
        ceiling = stream_ceiling(L, base, w.caches, w.n_copies, B * w.n_eff * rows_ctas, stream)

    # ---- the count a caller without host lengths gets (mla_auto_splits), for comparison ----
    split_plan = None
    auto_n = L.mla_auto_splits(B, T, H, base.block_table.shape[1], 0)
    if w.planner.startswith("mla_plan_splits") and auto_n != w.n_eff:
        keep = (w.n_splits, w.graph)
        w.n_splits = auto_n
        for i in range(3):  # grows the stream's scratch outside any capture
            w.step(i)
        barrier()
        w.capture()
        barrier()
        k_auto = max(200, w.gsteps)
        ms_a, _, _ = w.timed(k_auto, barrier)
        ms_a = max_over_ranks(ms_a, world, dev) / k_auto
        assert L.mla_device_error() == 0
        w.n_splits, w.graph = keep
        with torch.cuda.stream(stream):  # w.out holds the planned count's answer again
            w.graph.replay()
        barrier()
        split_plan = {
            "planned": {"n_splits": w.n_eff, "us_per_step": round(ms_step * 1e3, 2)},
            "automatic": {"n_splits": auto_n, "us_per_step": round(ms_a * 1e3, 2),
                          "value": round(job_gbps(kv_bytes, world, ms_a), 1), "unit": "GB/s", "steps": k_auto},
            "note": "the same step at mla_auto_splits' count (from max_pages alone: what a caller without "
                    "host lengths gets), graph-replayed after the timed region"}

    # ---- the other part of the serving mix, measured the same way ----
    side = {}
    for name in others:
        wo = DecodeStep(L, name, args, dev, stream)
        for i in range(max(args.warmup, 3)):
            wo.step(i)
        barrier()
        wo.capture()
        barrier()
        ms_o, rep_o, _ = wo.timed(max(args.steps, wo.gsteps), barrier)
        ms_o = max_over_ranks(ms_o, world, dev) / max(args.steps, wo.gsteps)
        kms_o = wo.kernel_ms(min(max(args.steps, 20), 2000), barrier)
        assert L.mla_device_error() == 0
        fam_o = {1: "simt", 2: "tcgen05"}.get(L.mla_last_decode_impl(), "unknown")
        ceil_o = None
        if not args.no_ceiling:
            rc = 1 if wo.base.H * wo.base.T <= 16 else -(-(wo.base.H * wo.base.T) // 32)
            ceil_o = stream_ceiling(L, wo.base, wo.caches, wo.n_copies, wo.base.B * wo.n_eff * rc, stream)
        side[name] = {
            "workload": f"{name}: {workload_description(name)}",
            "value": round(job_gbps(wo.kv_bytes, world, ms_o), 1), "unit": "GB/s",
            "ms_per_step": round(ms_o, 5), "decode_steps_per_s": round(1e3 / ms_o, 1),
            "kv_bytes_per_step": wo.kv_bytes, "n_splits": wo.n_eff, "chunk_pages": wo.chunk,
            "planner": wo.planner, "frac_of_8TBps": round(job_gbps(wo.kv_bytes, world, ms_o) / HBM_NOMINAL_GBS, 4),
            "roofline": kernel_roofline(wo, kms_o, fam_o, name), "stream_ceiling": ceil_o,
            "step_us_spread": {"p10": round(rep_o[len(rep_o) // 10], 3), "p50": round(rep_o[len(rep_o) // 2], 3),
                               "p90": round(rep_o[(9 * len(rep_o)) // 10], 3)} if rep_o else None}
        del wo
        torch.cuda.empty_cache()

    # ---- end to end through the C ABI with host buffers ----
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(L, w, args, dev, world, barrier)

    # ---- the DCP shard merge (mla_merge_partials over 8 shards' answers) ----
    dcp_merge = None
    if primary == "dcp_shard" and not args.no_append:
        dcp_merge = time_dcp_merge(L, w, barrier)

    # ---- DCP multi-token verify: one rank's share of an 8-way split of this workload ----
    dcp_verify = None
    if primary == "verify" and not args.no_append:
        dcp_verify = time_dcp_verify(L, base, w.caches, stream, barrier, w.l2, dev)

    # ---- the latent append that precedes each decode step (one call) ----
    append = None
    if not args.no_append:
        append = time_append(L, w, synth, barrier)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(base, budget_s=15.0, out=w.out, lse=w.lse)

    if rank == 0:
        desc = workload_description(primary)
        if args.workload == "serving_mix":
            desc += (" -- part (b) of the long-context and ragged serving mix; part (a), one request at "
                     "393,216 positions, under 'serving_mix'")
        if getattr(args, "requests", 0):
            desc += f" [profiling case: first {args.requests} requests only]"
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE, "data": "synthetic",
            "config": {"workload": f"{primary}: {desc}",
                       "page": 64, "kv_bytes_per_step": kv_bytes, "n_splits": w.n_eff, "planner": w.planner,
                       "chunk_pages": w.chunk, "l2": f"{w.n_copies} rotating cache copies "
                       f"({w.n_copies * base.kv_cache.numel() / 1e6:.0f} MB > 3x L2 {w.l2 / 1e6:.0f} MB): "
                       f"inputs larger than L2, no flush",
                       "kernel_family": family,
                       "timing": f"CUDA-graph replays of {w.gsteps} mla_decode_paged calls "
                                 f"({n_rep} replays + {n_rem} direct calls)"},
            "direct_calls": {"value": round(job_gbps(kv_bytes, world, ms_direct), 1),
                             "unit": "GB/s", "ms_per_step": round(ms_direct, 5), "steps": kdirect,
                             "note": "one host API call per step, no graph"},
            "sustained": ({"value": round(job_gbps(kv_bytes, world, sus_us * 1e-3), 1), "unit": "GB/s",
                           "us_per_step": round(sus_us, 3), "steps": sus_steps,
                           "note": f"graph replays back to back for >= {args.sustain_s:g} s right after the "
                                   f"timed steps; the clock record covers both"} if sus_steps else None),
            "decode_steps_per_s": round(steps_per_s, 1),
            "model_steps_per_s_attention_only": {
                "value": round(steps_per_s / MLA_LAYERS, 1), "layers": MLA_LAYERS,
                "note": "decode steps/s over the model's MLA layers: the attention-only bound on "
                        "whole-model decode steps/s (each step emits one token per request)"},
            "step_us_spread": ({"p10": round(rep_us[len(rep_us) // 10], 3),
                                "p50": round(rep_us[len(rep_us) // 2], 3),
                                "p90": round(rep_us[(9 * len(rep_us)) // 10], 3),
                                "per": f"mean step of each replay of {w.gsteps} calls ({len(rep_us)} replays)"}
                               if rep_us else None),
            "frac_of_8TBps": round(value / HBM_NOMINAL_GBS, 4),
            "roofline": roofline,
            "roofline_tensor": roofline_tensor,
            "serving_mix": side or None,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "stream_ceiling": ceiling,
            "split_plan": split_plan,
            "append": append,
            "dcp_merge": dcp_merge,
            "dcp_verify": dcp_verify,
            "gpu_launches": args.steps * w.launches_per_step,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


DTYPE = "e4m3 x e4m3 tensor-core MMA (bf16 q and fp32 probabilities each split into two e4m3 terms), f32 accumulate"


def measure_e2e(L, w, args, dev, world, barrier):
    """The same step end to end through the C ABI: a serving loop stages a step's
    inputs in one pinned host buffer and reads its results back into one, one
    copy each way per step, stream synchronised every step."""
    import torch
    base, stream = w.base, w.stream
    ins = (base.q, base.block_table, base.seq_lens, base.kv_scale)
    dstage, (dq, dbt, dsl, dks) = carve(dev, [(x.shape, x.dtype) for x in ins])
    hstage, hviews = carve("cpu", [(x.shape, x.dtype) for x in ins], pin=True)
    for hv, x in zip(hviews, ins):
        hv.copy_(x.cpu())
    dres, (eout, e_lse) = carve(dev, [(w.out.shape, w.out.dtype), (w.lse.shape, w.lse.dtype)])
    hres = torch.empty(dres.shape, dtype=dres.dtype).pin_memory()
    ksteps = min(args.steps, 1000)

    def e2e_step(i):
        dstage.copy_(hstage, non_blocking=True)
        L.mla_decode_paged(dq, w.caches[i % w.n_copies], dks, dbt, dsl, w.n_splits, base.sm_scale,
                           eout, e_lse, stream)
        hres.copy_(dres, non_blocking=True)
        stream.synchronize()

    with torch.cuda.stream(stream):  # copies and decode in one stream order
        for i in range(3):
            e2e_step(i)
        barrier()
        t0 = time.perf_counter()
        for i in range(ksteps):
            e2e_step(i)
        barrier()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / ksteps
    hout = hres[:eout.numel() * eout.element_size()].view(eout.dtype).view(eout.shape)
    if not torch.equal(hout, w.out.cpu()):
        raise RuntimeError("end-to-end result differs from the device-timed result")
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    # the same step (copy in, decode, copy out) captured once per cache copy and
    # replayed as one CUDA graph per step
    graphs = []
    for c in range(w.n_copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            dstage.copy_(hstage, non_blocking=True)
            L.mla_decode_paged(dq, w.caches[c], dks, dbt, dsl, w.n_splits, base.sm_scale, eout, e_lse, stream)
            hres.copy_(dres, non_blocking=True)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for i in range(3):
            graphs[i % w.n_copies].replay()
            stream.synchronize()
        barrier()
        t0 = time.perf_counter()
        for i in range(ksteps):
            graphs[i % w.n_copies].replay()
            stream.synchronize()
        barrier()
        e2e_graph_ms = (time.perf_counter() - t0) * 1e3 / ksteps
    if not torch.equal(hout, hres[:eout.numel() * eout.element_size()].view(eout.dtype).view(eout.shape)):
        raise RuntimeError("graph-replayed end-to-end result differs")
    e2e_graph_ms = max_over_ranks(e2e_graph_ms, world, dev)
    kv = w.kv_bytes
    return {"value": round(job_gbps(kv, world, e2e_ms), 1), "unit": "GB/s",
            "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": hstage.numel(),
            "d2h_bytes_per_step": hres.numel(), "steps": ksteps,
            "note": "one pinned host buffer holding q/block_table/seq_lens/kv_scale -> device, decode, one copy "
                    "of out+lse -> pinned host, stream synchronised every step, each step issued as host API "
                    "calls; the latent cache is resident decode state",
            "graph": {"value": round(job_gbps(kv, world, e2e_graph_ms), 1), "unit": "GB/s",
                      "ms_per_step": round(e2e_graph_ms, 4),
                      "note": "the same step (copy in, decode, copy out) replayed as one CUDA graph, "
                              "synchronised every step"}}


def time_dcp_merge(L, w, barrier, S_sh=8):
    """mla_merge_partials of S_sh shards' bf16 answers of this workload's shape."""
    import torch
    B, T, H, dev, stream = w.base.B, w.base.T, w.base.H, w.dev, w.stream
    g_m = torch.Generator(device=dev).manual_seed(33)
    po = (0.25 * torch.randn((S_sh, B, T, H, 512), generator=g_m, device=dev)).to(torch.bfloat16)
    pl = torch.randn((S_sh, B, T, H), generator=g_m, device=dev) * 3
    n_rot = max(2, -(-3 * w.l2 // (po.numel() * 2)))  # copies of the answers: each call reads HBM
    pos = [po] + [po.clone() for _ in range(n_rot - 1)]
    mo = torch.empty((B, T, H, 512), dtype=torch.bfloat16, device=dev)
    ml = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    for i in range(5):
        L.mla_merge_partials(pos[i % n_rot], pl, S_sh, mo, ml, stream)
    barrier()
    gm = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gm, stream=stream):
        for i in range(50):
            L.mla_merge_partials(pos[i % n_rot], pl, S_sh, mo, ml, stream)
    with torch.cuda.stream(stream):
        gm.replay()
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(10):
            gm.replay()
    ev1.record(stream)
    barrier()
    m_us = ev0.elapsed_time(ev1) * 1e3 / 500
    m_bytes = po.numel() * 2 + pl.numel() * 4 + mo.numel() * 2 + ml.numel() * 4
    return {"us_per_call": round(m_us, 3), "bytes_per_call": m_bytes,
            "gbps": round(m_bytes / (m_us * 1e-6) / 1e9, 1),
            "frac_of_measured_hbm": round(m_bytes / (m_us * 1e-6) / 1e9 / load_peaks()[0], 4),
            "note": f"mla_merge_partials of {S_sh} shards' bf16 answers and lse "
                    f"([{S_sh}, {B}, {T}, {H}, 512]) into one, CUDA-graph replays of 50 calls "
                    f"over {n_rot} rotating copies of the answers (> 3x L2)"}


def time_append(L, w, synth, barrier):
    """mla_append_latent of one new latent per query position, as CUDA-graph
    replays (launch-bound by size)."""
    import torch
    base, dev, stream = w.base, w.dev, w.stream
    B, T = base.B, base.T
    lat = synth.make_latent(77, B, T, device=dev)
    start = (base.seq_lens - T).to(torch.int32)
    kv_app = w.caches[-1]  # after the timed regions: rewriting the newest positions is harmless now

    def app():
        L.mla_append_latent(lat, base.kv_scale, base.block_table, start, kv_app, stream)

    for _ in range(10):
        app()
    barrier()
    gapp = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gapp, stream=stream):
        for _ in range(100):
            app()
    with torch.cuda.stream(stream):
        gapp.replay()
    barrier()
    napp = 10
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(napp):
            gapp.replay()
    ev1.record(stream)
    barrier()
    assert L.mla_device_error() == 0
    app_us = ev0.elapsed_time(ev1) * 1e3 / (napp * 100)
    app_bytes = B * T * (576 * 2 + 576) + B * (4 + 4)
    return {"us_per_call": round(app_us, 3), "bytes_per_call": app_bytes,
            "gbps": round(app_bytes / (app_us * 1e-6) / 1e9, 2), "positions": B * T,
            "note": "mla_append_latent of one new latent per query position (bf16 in, e4m3 out), "
                    "CUDA-graph replays of 100 calls; launch-bound by size"}


def time_dcp_verify(L, base, caches, stream, barrier, l2, dev, n_sh=8, reps=8):
    """One rank's step of a multi-token verify split over n_sh contiguous shards of
    every history (page-aligned; the T draft positions lie in the last shard).  A
    shard before the last is decoded as T = 1 with T*H rows, the last one with the
    causal rule, then the n_sh bf16 answers are merged.  All shards of all ranks are
    timed here on one GPU, each call reading its own pages from HBM; the exchange of
    answers between GPUs (mla_latent_kv_fp8_gb300.dcp) is not part of it."""
    import torch
    B, T, H = base.B, base.T, base.H
    from mla_latent_kv_fp8_gb300.dcp import shard_plan
    plan = shard_plan([int(x) for x in base.seq_lens.cpu().tolist()], base.block_table.cpu(), n_sh, T)
    shard_bt = [t.to(dev) for t, _ in plan[:-1]]
    sh_lens = plan[0][1].to(dev)
    tail_bt, tail_lens = plan[-1][0].to(dev), plan[-1][1].to(dev)
    tails = plan[-1][1].tolist()
    q1 = base.q.reshape(B, 1, T * H, 576)
    o1 = torch.empty((B, 1, T * H, 512), dtype=torch.bfloat16, device=dev)
    l1 = torch.empty((B, 1, T * H), dtype=torch.float32, device=dev)
    ot = torch.empty((B, T, H, 512), dtype=torch.bfloat16, device=dev)
    lt = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    nc = len(caches)

    # each rank plans its call from the lengths it holds (all shards before the last
    # have the same lengths)
    ns_shard = L.mla_plan_splits(B, 1, T * H, plan[0][1].tolist(), shard_bt[0].shape[1], 0)
    ns_tail = L.mla_plan_splits(B, T, H, tails, tail_bt.shape[1], 0)

    def shard_call(i):  # shard i % (n_sh - 1), cache copy i // (n_sh - 1): new pages every call
        L.mla_decode_paged(q1, caches[(i // (n_sh - 1)) % nc], base.kv_scale, shard_bt[i % (n_sh - 1)],
                           sh_lens, ns_shard, base.sm_scale, o1, l1, stream)

    # the last shard is one region of the cache: enough copies of it to defeat L2
    tail_bytes = sum(tails) * 576
    tail_caches = list(caches) + [caches[0].clone()
                                  for _ in range(max(0, -(-3 * l2 // tail_bytes) - nc))]

    def tail_call(i):
        L.mla_decode_paged(base.q, tail_caches[i % len(tail_caches)], base.kv_scale, tail_bt, tail_lens,
                           ns_tail, base.sm_scale, ot, lt, stream)

    g_m = torch.Generator(device=dev).manual_seed(44)
    po = (0.25 * torch.randn((n_sh, B, T, H, 512), generator=g_m, device=dev)).to(torch.bfloat16)
    pl = torch.randn((n_sh, B, T, H), generator=g_m, device=dev) * 3
    n_rot = max(2, -(-3 * l2 // (po.numel() * 2)))
    pos = [po] + [po.clone() for _ in range(n_rot - 1)]
    mo = torch.empty((B, T, H, 512), dtype=torch.bfloat16, device=dev)
    ml = torch.empty((B, T, H), dtype=torch.float32, device=dev)

    def merge_call(i):
        L.mla_merge_partials(pos[i % n_rot], pl, n_sh, mo, ml, stream)

    def per_call_us(fn, n):
        for i in range(3):
            fn(i)
        barrier()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn(i)
        with torch.cuda.stream(stream):
            g.replay()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                g.replay()
        e1.record(stream)
        barrier()
        return e0.elapsed_time(e1) * 1e3 / (reps * n)

    a = per_call_us(shard_call, (n_sh - 1) * nc * 2)
    b_ = per_call_us(tail_call, len(tail_caches) * 2)
    c = per_call_us(merge_call, 50)
    assert L.mla_device_error() == 0
    step = max(a, b_) + c
    kv = base.kv_bytes()
    return {"shards": n_sh, "n_splits": {"shard": ns_shard, "last_shard": ns_tail,
                                         "planner": "mla_plan_splits on each rank's host lengths"},
            "shard_call_us": round(a, 2), "last_shard_call_us": round(b_, 2),
            "merge_us": round(c, 2), "rank_step_us": round(step, 2),
            "kv_gbps_per_rank": round(kv / n_sh / (step * 1e-6) / 1e9, 1),
            "job_kv_gbps": round(kv / (step * 1e-6) / 1e9, 1),
            "note": f"one rank's step: its shard decoded (a shard before the last as T = 1 with "
                    f"{T * H} rows, the last causal), then mla_merge_partials of the {n_sh} bf16 "
                    f"answers; each part timed as CUDA-graph replays on this GPU, shards and cache "
                    f"copies rotated so every call reads HBM; the exchange of answers between GPUs "
                    f"is not included; job_kv_gbps = all {n_sh} shards' KV bytes / the rank step"}


def cpu_baseline(case, budget_s=15.0, out=None, lse=None):
    """The FP64 oracle as it stands, on this host's cores, over a bounded sample of
    the same workload (whole requests, all heads), reported in the same unit.
    Given the device answer of the timed steps (out, lse), the sampled requests'
    rows are also compared with the oracle's (the parity tolerances)."""
    import numpy as np
    import oracle
    c = case.to("cpu")
    # calibrate on the first request, then take as many requests as fit the budget
    t0 = time.perf_counter()
    oracle.decode(c.q[:1], c.kv_cache, c.kv_scale, c.block_table[:1], c.seq_lens[:1], c.sm_scale)
    t1 = time.perf_counter() - t0
    n_req = int(max(1, min(c.B, budget_s / max(t1, 1e-3) * max(os.cpu_count() or 1, 1) / 2)))
    t0 = time.perf_counter()
    ro, rl, threads = oracle.decode(c.q[:n_req], c.kv_cache, c.kv_scale, c.block_table[:n_req],
                                    c.seq_lens[:n_req], c.sm_scale, return_threads=True)
    dt = time.perf_counter() - t0
    kvb = 576 * int(np.sum(c.lens[:n_req]))
    res = {"value": round(kvb / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": f"{n_req} of {c.B} requests (all heads, full context), {dt:.2f} s",
           "seconds": round(dt, 3)}
    if out is not None and lse is not None:
        res["parity"] = parity_of(out[:n_req].float().cpu().numpy(), lse[:n_req].cpu().numpy(), ro, rl)
    return res


def parity_of(o, l, ro, rl):
    """Errors of a device answer against the oracle's on the same rows, and whether
    they meet the tolerances: per element |dout| <= 1e-2 + half a bf16 ulp of the
    reference (the output's own rounding), max|dout| / max|out| <= 1.6e-2,
    |dlse| <= max(1e-4, 2^-20 |lse|); empty rows must be out = 0, lse = -inf."""
    import numpy as np
    empty = np.isneginf(rl)
    full = ~empty
    res = {"rows": int(rl.size), "empty_rows": int(empty.sum())}
    ok = bool(np.all(o[empty] == 0) and np.all(np.isneginf(l[empty])))
    if full.any():
        d = np.abs(o[full] - ro[full])
        dl = np.abs(l[full] - rl[full])
        _, ex = np.frexp(np.maximum(np.abs(ro[full]), 2.0 ** -126))
        out_bound = 1e-2 + np.ldexp(1.0, ex - 9)
        lse_bound = np.maximum(1e-4, 2.0 ** -20 * np.abs(rl[full]))
        res["max_abs_out"] = float(d.max())
        res["rel_out"] = float(d.max() / max(float(np.abs(ro[full]).max()), 1e-30))
        res["max_abs_lse"] = float(dl.max())
        ok = ok and bool(np.isfinite(o[full]).all() and np.isfinite(l[full]).all())
        ok = ok and bool(np.all(d <= out_bound)) and res["rel_out"] <= 1.6e-2 and bool(np.all(dl <= lse_bound))
    res["pass"] = ok
    return res


def run_reference(args):
    """Reference arm: the FP64 CPU oracle on the host cores, same metric and unit."""
    import torch
    import numpy as np
    import oracle
    from mla_latent_kv_fp8_gb300 import synth

    rank, world, _ = dist_env()
    if rank != 0:
        return
    name = SERVING_MIX[0] if args.workload == "serving_mix" else args.workload
    case = synth.workload_case(name, device="cpu")
    c = case
    # each step is a bounded sample: every request's first n positions, all heads
    # (the oracle runs its (request, position) units on all host cores)
    budget_total = 120.0
    per_step = budget_total / max(args.steps + args.warmup, 1)
    t0 = time.perf_counter()
    L0 = c.lens[0]
    oracle.decode(c.q[:1], c.kv_cache, c.kv_scale, c.block_table[:1], c.seq_lens[:1], c.sm_scale)
    t_full = time.perf_counter() - t0
    n = int(max(64, min(max(c.lens), L0 * per_step / max(t_full, 1e-6))))
    mask = np.zeros(max(c.lens), dtype=np.uint8)
    mask[:n] = 1

    def step():
        return oracle.decode(c.q, c.kv_cache, c.kv_scale, c.block_table, c.seq_lens,
                             c.sm_scale, pos_mask=mask, return_threads=True)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    threads = 1
    for _ in range(args.steps):
        threads = step()[2]
    dt = (time.perf_counter() - t0) / args.steps
    kvb = 576 * int(sum(min(n, x) for x in c.lens))
    value = kvb / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{name}: {workload_description(name)}",
                       "sample_per_step": f"all {c.B} requests, positions [0, {n}), all {c.H * c.T} rows"},
            "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": f"all {c.B} requests, first {n} positions each, per step"},
            "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
