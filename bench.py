#!/usr/bin/env python3
"""Decode-step benchmark of the CLO hot path (decoded tokens/s).

Default workload: Llama3-8B-shaped attention stack, 32 layers, 32/8 heads,
head_dim 128, batch 8, 32K-token context per sequence in pinned host memory,
top-k 10 %, 4 persistent heads per layer, thresholds from 16 profiling steps.

One step = one clo_decode_step over all layers (reuse test, query hashing,
scoring + top-k, zero-copy fetch of missed rows, sparse attention), one decoded
token per sequence.  The method's 16 profiling steps run before the W warm-up
steps and are not timed (CLO profiles offline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama32k]
  python bench.py --impl reference ...   # the CPU oracle on the same workload
Prints one JSON line (rank 0).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decoded tokens/s through offloaded top-k attention"
UNIT = "tokens/s"


def _env_int(name, default):
    v = os.environ.get(name)
    return int(v) if v not in (None, "") else default


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=64)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--workload", default="llama32k")
    p.add_argument("--layers", type=int, default=0, help="override the layer count (profiling runs only)")
    p.add_argument("--batch", type=int, default=0,
                   help="override the batch (for workloads whose host pool exceeds the box's memory)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--adaptive-tau", action="store_true",
                   help="online adaptive thresholds after warm-up (running average of the live cosines)")
    p.add_argument("--kv-bits", type=int, default=16, choices=[16, 4, 2],
                   help="host pool storage: bf16, or 4/2-bit asymmetric codes dequantised on the GPU")
    p.add_argument("--grow", action="store_true",
                   help="streaming growth: every step first appends one token per (layer, sequence)")
    p.add_argument("--layerwise", action="store_true",
                   help="decode each step with one clo_decode_layer call per layer, in order")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--plan", action="store_true",
                   help="print each rank's plan (device, seed, pool bytes, host-memory check) and exit: "
                        "runs without a GPU")
    p.add_argument("--cpu-steps", type=int, default=24,
                   help="oracle steps timed for the CPU baseline (about 10 s of CPU work on llama32k)")
    return p.parse_args()


# ----------------------------------------------------------------------------- helpers
def mem_available_bytes():
    with open("/proc/meminfo") as f:
        for line in f:
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    return 0


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.reader = None

    def start(self, wait_samples: int = 2, timeout_s: float = 10.0):
        """Starts nvidia-smi polling and returns once it has delivered wait_samples
        samples, so that its start-up (driver queries) is over before timing begins."""
        import threading

        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def read():
            for line in self.proc.stdout:
                self.lines.append(line)

        self.reader = threading.Thread(target=read, daemon=True)
        self.reader.start()
        t0 = time.time()
        while len(self.lines) < wait_samples and time.time() - t0 < timeout_s and self.proc.poll() is None:
            time.sleep(0.02)
        self.skip = len(self.lines)   # samples taken before the timed region

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.reader.join(timeout=5)
        out = "".join(self.lines[self.skip:])
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def traffic_from_profiles(kernel: str, workload: str):
    """dram bytes per launch recorded by an ncu capture under profiles/, if the kernel's
    source has not changed since (the summary stores the source digest)."""
    import hashlib

    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    want, traffic = None, None
    for line in txt.splitlines():
        if line.startswith("source_sha256:"):
            want = line.split(":", 1)[1].strip()
        if line.startswith("traffic_bytes_per_launch:"):
            val = line.split(":", 1)[1].strip()
            traffic = None if val in ("", "null") else float(val)
    src = os.path.join(ROOT, "host_offloaded_kv_gb300", "csrc", "clo_fused.cu")
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if want != digest:
        return None
    return traffic


def pinned_h2d_gbs(dev, nbytes: int = 1 << 30, trials: int = 8) -> float:
    """The machine's host-link peak: best of several timed pinned host -> device copies of
    a warmed 1 GiB buffer (CUDA events)."""
    import torch

    hb = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    hb.fill_(1)
    db = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    for _ in range(2):
        db.copy_(hb, non_blocking=True)
    torch.cuda.synchronize()
    best = 0.0
    for _ in range(trials):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        db.copy_(hb, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del hb, db
    return best


def max_over_ranks(x: float, world: int) -> float:
    """Largest value over all ranks (the slowest rank's time); identity for one rank.
    Works with the gloo (CPU tensors) and nccl (CUDA tensors) backends."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, seconds_slowest: float, world: int) -> float:
    """Whole-job throughput: units processed by all ranks / the slowest rank's time."""
    return world * units_per_rank / seconds_slowest


def kernel_roofline(hbm_bytes: float, host_bytes: float, ms: float, hbm_peak_gbs: float, link_peak_gbs: float):
    """Roofline of one launch from its algorithmic bytes: the bound is whichever side
    needs more time at its peak (HBM bytes at the HBM peak, host bytes at the link
    peak); both fractions are reported."""
    sec = ms / 1e3
    hbm_gbs = hbm_bytes / sec / 1e9
    link_gbs = host_bytes / sec / 1e9
    t_hbm = hbm_bytes / (hbm_peak_gbs * 1e9)
    t_link = host_bytes / (link_peak_gbs * 1e9)
    bound = "hbm" if t_hbm >= t_link else "host-link"
    achieved, peak = (hbm_gbs, hbm_peak_gbs) if bound == "hbm" else (link_gbs, link_peak_gbs)
    return {"bound": bound, "achieved": achieved, "peak": peak, "frac": achieved / peak,
            "hbm_gbs": hbm_gbs, "link_gbs": link_gbs, "frac_hbm": hbm_gbs / hbm_peak_gbs,
            "frac_link": link_gbs / link_peak_gbs}


# ----------------------------------------------------------------------------- workload
def step_roofline(step_bytes, hbm_bytes: float, host_bytes: float, step_ms: float, hbm_peak_gbs: float,
                  link_peak_gbs: float) -> dict:
    """Roofline of a run of steps that execute one after another: the ideal time is the
    sum over the steps of each step's max(HBM bytes / HBM peak, host bytes / link peak).
    step_bytes holds (host, HBM) bytes per timed step; hbm_bytes and host_bytes are the
    run's totals, which give the aggregate form max(total HBM / peak, total host / peak)
    (it understates the ideal when link-bound and HBM-bound steps alternate)."""
    steps = len(step_bytes)
    hbm_s, link_s = hbm_peak_gbs * 1e9, link_peak_gbs * 1e9
    ideal_ms = sum(max(m / hbm_s, h / link_s) for h, m in step_bytes) * 1e3 / steps
    aggregate_ms = max(hbm_bytes / hbm_s, host_bytes / link_s) * 1e3 / steps
    return {"bound": "sum over the timed steps of max(HBM alg bytes / HBM peak, host bytes / link peak)",
            "ideal_ms": ideal_ms, "measured_ms": step_ms, "frac": ideal_ms / step_ms,
            "aggregate_ideal_ms": aggregate_ms, "aggregate_frac": aggregate_ms / step_ms,
            "link_bound_steps": sum(1 for h, m in step_bytes if h / link_s >= m / hbm_s),
            "hbm_bytes_per_step": hbm_bytes / steps, "host_bytes_per_step": host_bytes / steps,
            "link_peak_gbs": link_peak_gbs, "hbm_peak_gbs": hbm_peak_gbs}


def workload_from_args(args):
    from host_offloaded_kv_gb300.synth import get_workload

    w = get_workload(args.workload)
    if args.layers:
        w = w.scaled(n_layers=args.layers)
    if args.batch:
        w = w.scaled(batch=args.batch)
    return w


def rank_plan(args, rank, world, local_rank):
    """What one replica runs: its device, its own seed (independent sequences per rank)
    and the bytes of its pinned host pool."""
    w = workload_from_args(args)
    rec_bytes = 4 * w.head_dim if args.kv_bits == 16 else 2 * w.head_dim * args.kv_bits // 8
    n_grow = ((w.warmup_steps if w.tau_fixed is None else 0) + args.warmup + 2 * args.steps + 1) if args.grow else 0
    ncap = w.n_tokens + n_grow
    pool = w.n_layers * w.batch * w.n_kv_heads * ncap * rec_bytes
    return {"rank": rank, "world": world, "local_rank": local_rank, "device": f"cuda:{local_rank}",
            "seed": w.seed + 1000 * rank, "workload": w.name, "batch": w.batch, "max_tokens": ncap,
            "pool_bytes": pool, "host_need_bytes": int(pool * 1.15) + (1 << 30)}


def host_memory_check(plan, world, avail=None):
    """All replicas of one node pin their pools in the same host memory: the sum of their
    needs must fit what was available before any of them allocated.  Returns (ok, total
    need, available)."""
    avail = mem_available_bytes() if avail is None else avail
    need = plan["host_need_bytes"]
    if world > 1:
        import torch
        import torch.distributed as dist

        dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
        t = torch.tensor([float(need)], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        need = int(t.item())
        avail = int(max_over_ranks(-avail, world) * -1)   # the smallest reading
    return need <= avail, need, avail


def spawn_ranks(n: int, argv) -> int:
    """Starts n replicas of this script on this node under torch.distributed.run (one
    process per GPU, rendezvous on 127.0.0.1) and returns their launcher's exit code."""
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def topk_of(w):
    if w.topk > 0:
        return min(w.topk, w.n_tokens)
    return max(1, min(w.n_tokens, int(math.ceil(w.topk_ratio * w.n_tokens))))


def run_gb300(args, rank, world, local_rank):
    import torch

    from host_offloaded_kv_gb300.clo import CLOContext
    from host_offloaded_kv_gb300.synth import Synth

    w = workload_from_args(args)
    L, B, Hq, Hkv, d, N = w.n_layers, w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_tokens
    rec_bytes = 4 * d if args.kv_bits == 16 else 2 * d * args.kv_bits // 8
    K, W = args.steps, args.warmup
    n_grow = (w.warmup_steps if w.tau_fixed is None else 0) + W + 2 * K + 1 if args.grow else 0
    Ncap = N + n_grow                       # growth appends one token per step
    pool_bytes = L * B * Hkv * Ncap * rec_bytes
    ok, need, avail = host_memory_check(rank_plan(args, rank, world, local_rank), world)
    if not ok:
        raise SystemExit(f"not enough host memory for {world} pinned pool(s) of {w.name}: need "
                         f"{need / 2**30:.1f} GiB, {avail / 2**30:.1f} GiB available")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.Stream(device=dev)
    syn = Synth(w.seed + 1000 * rank, w.hh_ratio)
    R = syn.hash_matrices(L, Hkv, d)
    tau = None if w.tau_fixed is None else np.full(L * Hkv, w.tau_fixed, dtype=np.float32)
    t0 = time.time()
    lib = CLOContext(n_layers=L, batch=B, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, max_tokens=Ncap, hash_R=R,
                     topk=w.topk, topk_ratio=w.topk_ratio, tau=tau, warmup_steps=w.warmup_steps,
                     tau_offset=w.tau_offset, n_persist=w.n_persist if tau is None else 0, timing=True,
                     stream=stream.cuda_stream, adaptive_tau=args.adaptive_tau, kv_bits=args.kv_bits)
    if args.layerwise:
        def decode(q, o, io_on_device=None):
            for l in range(L):
                lib.decode_layer(l, q[l], o[l], io_on_device)
    else:
        def decode(q, o, io_on_device=None):
            lib.decode_step(q, o, io_on_device)
    grow_src = {"dev": None, "host": None, "i": 0}

    def step_fn(q, o, io_on_device=None):
        if args.grow:   # one new token per (layer, sequence), then the step over the grown context
            src = grow_src["dev"] if io_on_device is None else grow_src["host"]
            i = grow_src["i"]
            lib.append_step(src[0][i % src[0].shape[0]], src[1][i % src[1].shape[0]],
                            None if io_on_device is None else io_on_device)
            grow_src["i"] = i + 1
        decode(q, o, io_on_device)
    Kbuf = np.empty((N, Hkv, d), dtype=np.uint16)
    Vbuf = np.empty((N, Hkv, d), dtype=np.uint16)
    for l in range(L):
        for b in range(B):
            syn.layer_seq_kv(l, b, Hkv, 0, N, d, Kbuf, Vbuf)
            lib.append_kv(l, b, Kbuf, Vbuf, src_is_device=False)
    t_setup = time.time() - t0
    pool_node = lib.pool_node()
    del Kbuf, Vbuf

    if args.grow:   # the appended tokens' rows, from the generator at positions N, N+1, ...
        kn = np.empty((n_grow, L, B, Hkv, d), dtype=np.uint16)
        vn = np.empty_like(kn)
        for i in range(n_grow):
            for l in range(L):
                for b in range(B):
                    Kt, Vt = syn.layer_seq_kv(l, b, Hkv, N + i, 1, d)
                    kn[i, l, b], vn[i, l, b] = Kt[0], Vt[0]
        grow_src["dev"] = (torch.from_numpy(kn.view(np.int16)).to(dev), torch.from_numpy(vn.view(np.int16)).to(dev))
        grow_src["host"] = (torch.from_numpy(kn.view(np.int16)).pin_memory(), torch.from_numpy(vn.view(np.int16)).pin_memory())
    qs = syn.query_stream(L, B, Hq, d, w.rho_lo, w.rho_hi)
    n_prof = w.warmup_steps if tau is None else 0
    n_dev = n_prof + W + K
    qdev = torch.empty((n_dev, L, B, Hq, d), dtype=torch.int16, device=dev)
    qh = np.empty((L, B, Hq, d), dtype=np.uint16)
    for i in range(n_dev):
        qs.next(qh)
        qdev[i].copy_(torch.from_numpy(qh.view(np.int16)))
    out = torch.empty((L, B, Hq, d), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    # the link peak is measured before the warm-up steps: large pinned copies evict the
    # device's translations of host pages, and the first steps after them refill those
    link_gbs_before = pinned_h2d_gbs(dev)
    with torch.cuda.stream(stream):
        for i in range(n_prof + W):
            step_fn(qdev[i], out)
    lib.sync()
    lib.stats()  # drops the per-phase events of untimed steps
    before = lib.stats()

    sampler = ClockSampler(local_rank)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(K):
            step_fn(qdev[n_prof + W + i], out)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms_total = ev0.elapsed_time(ev1)
    st = lib.stats()
    timeline = lib.timeline()
    step_bytes = lib.step_bytes(n_prof + W, n_prof + W + K)   # [K][2] host, HBM bytes of each timed step
    if timeline is not None:
        timeline["host_bytes"] = st["last_host_bytes"]
    host_bytes = st["host_bytes"] - before["host_bytes"]
    hbm_bytes = st["hbm_bytes_alg"] - before["hbm_bytes_alg"]
    hits = st["units_hit"] - before["units_hit"]
    miss = st["units_miss"] - before["units_miss"]
    pers = st["units_persist"] - before["units_persist"]
    phases = {p: st[f"sum_ms_{p}"] for p in ("decide", "fused")}
    ms_total = max_over_ranks(ms_total, world)
    del qdev

    # end to end through the C ABI with host buffers (pinned): H2D of q, D2H of out per step
    e2e = None
    if not args.no_e2e:
        Ke = K
        qpin = torch.empty((Ke, L, B, Hq, d), dtype=torch.int16, pin_memory=True)
        for i in range(Ke):
            qs.next(qh)
            qpin[i].copy_(torch.from_numpy(qh.view(np.int16)))
        opin = torch.empty((L, B, Hq, d), dtype=torch.float32, pin_memory=True)
        step_fn(qpin[0].numpy(), opin.numpy(), io_on_device=False)
        e_before = lib.stats()
        if world > 1:
            torch.distributed.barrier()
        t1 = time.perf_counter()
        for i in range(1, Ke):
            step_fn(qpin[i].numpy(), opin.numpy(), io_on_device=False)
        t2 = time.perf_counter()
        e_after = lib.stats()
        sec = max_over_ranks(t2 - t1, world)
        e_hit = e_after["units_hit"] - e_before["units_hit"]
        e_miss = e_after["units_miss"] - e_before["units_miss"]
        # the e2e steps continue the query stream after the device-timed ones, so their
        # reuse decisions (and host bytes) differ: both regions report theirs
        e2e = {"value": whole_job_rate(B * (Ke - 1), sec, world), "unit": UNIT,
               "h2d_bytes_per_step": L * B * Hq * d * 2 + (2 * L * B * Hkv * d * 2 if args.grow else 0),
               "d2h_bytes_per_step": L * B * Hq * d * 4, "steps": Ke - 1,
               "host_link_bytes_per_step": (e_after["host_bytes"] - e_before["host_bytes"]) / (Ke - 1),
               "hit_rate_nonpersistent": e_hit / max(1, e_hit + e_miss)}

    link_gbs = max(link_gbs_before, pinned_h2d_gbs(dev))
    lib.close()

    hbm_peak, hbm_src = measured_peaks()
    kmax = topk_of(w)
    steps = K
    tokens = world * B * steps
    value = whole_job_rate(B * steps, ms_total / 1e3, world)
    kern = {p: {"ms_per_launch": phases[p] / steps} for p in phases}
    # the fused kernel's algorithmic bytes per launch: HBM from the library's counter
    # (codes read once per selected unit, index writes and reads, attention rows, bf16
    # slot writes of the fetched rows, queries and outputs; the decide kernel's query and
    # cached-query bytes, under 0.1 %, are included) and the host bytes over the link
    fused_ms = phases["fused"] / steps
    roof = kernel_roofline(hbm_bytes / steps, host_bytes / steps, fused_ms, hbm_peak, link_gbs)
    kern["fused"].update(hbm_gbs=roof["hbm_gbs"], link_gbs=roof["link_gbs"], frac_hbm=roof["frac_hbm"],
                         frac_link=roof["frac_link"], bound=roof["bound"])
    # the capture must match the launch: a pool format or mode without its own capture
    # under profiles/ reports no traffic
    mode = ("" if args.kv_bits == 16 else f"_int{args.kv_bits}") + ("_layerwise" if args.layerwise else "") + \
        ("_grow" if args.grow else "") + ("_adaptive" if args.adaptive_tau else "")
    traffic = traffic_from_profiles("k_step_fused", w.name + mode)
    roofline = {"kernel": "k_step_fused", "bound": roof["bound"], "achieved": roof["achieved"],
                "peak": roof["peak"], "unit": "GB/s", "frac": roof["frac"], "traffic": traffic,
                "frac_hbm": roof["frac_hbm"], "frac_link": roof["frac_link"],
                "hbm_bytes_per_launch": hbm_bytes / steps, "host_bytes_per_launch": host_bytes / steps,
                "peak_source": {"hbm": f"MEASURED_PEAKS.json hbm_gbs ({hbm_src})",
                                "host-link": "pinned H2D copy, best of 16 timed 1 GiB copies in this run"}}
    step_ms = ms_total / steps
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": W,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded generator; N(0,1) bf16 K/V, 1% heavy hitters, AR(1) queries)",
        "config": {"workload": w.name, "layers": L, "batch_per_gpu": B, "q_heads": Hq, "kv_heads": Hkv,
                   "head_dim": d, "context": N, "topk": kmax, "persistent_heads": w.n_persist if tau is None else 0,
                   "tau": (f"s_hat-{w.tau_offset} after {w.warmup_steps} profiling steps" if tau is None
                           else f"{w.tau_fixed} fixed") + (", then adaptive (running average, weight 1/16)"
                                                           if args.adaptive_tau else ""), "kv_dtype": "bf16" if args.kv_bits == 16 else
                   f"int{args.kv_bits} host pool (asymmetric, 64-channel groups; fp32 scale/min in HBM), bf16 on the GPU", "parallelism": f"replicas x{world} (independent sequences)",
                   "l2": "inputs larger than L2 (host pool %.0f GiB, HBM codes+slots+resident per step > 1 GB)" %
                         (pool_bytes / 2**30),
                   "hit_rate_nonpersistent": hits / max(1, hits + miss),
                   "host_link_bytes_per_step": host_bytes / steps, "setup_s": round(t_setup, 1),
                   "pool_numa_node": pool_node,
                   "mode": ("layer by layer (clo_decode_layer per layer)" if args.layerwise else "whole step")
                   + (f", growing context: one token appended per step (clo_append_step), {N} -> {Ncap - 1} tokens"
                      if args.grow else "")},
        "gpu_launches": steps * (2 * (L if args.layerwise else 1) + (3 if args.grow else 0)),
        "roofline": roofline,
        "step_roofline": step_roofline(step_bytes.tolist(), hbm_bytes, host_bytes, step_ms, hbm_peak, link_gbs),
        "kernels": kern,
        "clocks": clocks,
        "timeline_last_step": timeline,
        "e2e": e2e,
        "_rank_setup": {"tokens": tokens},
    }


# ----------------------------------------------------------------------------- oracle (CPU)
def oracle_sample(args, steps, warm, layers_sampled=1):
    """Time the CPU oracle on layer 0 of the workload (all sequences and kv heads),
    scaled to a full step by the layer count."""
    import oracle as orc
    from host_offloaded_kv_gb300.synth import Synth

    w = workload_from_args(args)
    L, B, Hq, Hkv, d, N = w.n_layers, w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_tokens
    Ls = layers_sampled
    syn = Synth(w.seed, w.hh_ratio)
    R = syn.hash_matrices(L, Hkv, d)[:Ls]
    tau = None if w.tau_fixed is None else np.full(Ls * Hkv, w.tau_fixed)
    o = orc.OracleCLO(Ls, B, Hq, Hkv, d, R, topk=w.topk, topk_ratio=w.topk_ratio, tau=tau,
                      warmup_steps=w.warmup_steps, tau_offset=w.tau_offset,
                      n_persist=w.n_persist if tau is None else 0, ntok=[N] * B)
    for l in range(Ls):
        for b in range(B):
            for h in range(Hkv):
                o.set_unit_kv(l, b, h, *syn.unit_kv(l, b, h, 0, N, d))
    qs = syn.query_stream(L, B, Hq, d, w.rho_lo, w.rho_hi)
    n_prof = w.warmup_steps if tau is None else 0
    for _ in range(n_prof + warm):
        o.step(qs.next()[:Ls])
    t0 = time.perf_counter()
    for _ in range(steps):
        o.step(qs.next()[:Ls])
    sec = time.perf_counter() - t0
    per_full_step = sec / steps * (L / Ls)
    cores = orc.load_oracle().orc_num_threads()
    return {"value": B / per_full_step, "unit": UNIT, "cores": int(cores), "kind": "oracle",
            "sample": f"layer 0 of {L} ({Ls * B * Hkv} of {L * B * Hkv} units), {steps} post-profiling steps "
                      f"after {n_prof} profiling + {warm} warm-up steps; time per step scaled x{L // Ls} to all layers",
            "seconds_timed": sec}


def run_reference(args, world=1):
    K, W = args.steps, args.warmup
    # bounded: the oracle takes ~0.3-1 s per sampled layer-step; cap the timed steps
    cb = oracle_sample(args, steps=max(1, min(K, 8)), warm=min(W, 3))
    w = workload_from_args(args)
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": world,
            "steps": max(1, min(K, 8)), "warmup": min(W, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator)",
            "config": {"workload": w.name}, "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return line


def print_plan(args, rank, world, local_rank) -> int:
    """--plan: every replica derives its plan; rank 0 prints all of them (gloo when the
    node has no GPU) with the node's aggregate host-memory check."""
    import torch

    plan = rank_plan(args, rank, world, local_rank)
    plans = [plan]
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        plans = [None] * world
        dist.all_gather_object(plans, plan)
    ok, need, avail = host_memory_check(plan, world)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps({"plan": plans, "host_need_bytes": need, "host_available_bytes": avail, "fits": ok}))
    return 0


def main():
    args = parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # launched directly: start one replica per GPU (the same command under torchrun)
        return spawn_ranks(args.gpus, sys.argv[1:])
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local_rank = _env_int("LOCAL_RANK", 0)
    if world != args.gpus and "WORLD_SIZE" in os.environ:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    if args.plan:
        return print_plan(args, rank, world, local_rank)
    if args.impl == "reference":
        if rank != 0:   # the oracle runs once, on rank 0's host cores
            return 0
        print(json.dumps(run_reference(args, world)))
        return 0
    import torch

    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line = run_gb300(args, rank, world, local_rank)
    line.pop("_rank_setup", None)
    if rank == 0 and not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = oracle_sample(args, steps=args.cpu_steps, warm=0)
        except Exception as e:  # the baseline is reported, never required
            line["cpu_baseline"] = {"error": str(e)}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
