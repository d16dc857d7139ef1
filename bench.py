#!/usr/bin/env python3
"""Benchmark of the decode-attention hot path on B300.

One step = one pass of the whole hot path over one batch: for every model
family in the workload, the new token is appended to its cache with RoPE
(kvdec_append_rope), then single-token split-KV decode attention runs over
the whole cache with its split pieces merged by log-sum-exp inside the same
kernel (kvdec_gqa_decode or kvdec_mla_decode_absorbed).

Default workload: the long-context ragged mix.  One step decodes
  * a Llama-3-70B-shaped GQA layer: B=8, h=64, n_kv=8, d=128, and
  * a DeepSeek-V3-shaped MLA layer (absorbed): B=8, n_h=128, 576-wide latent,
both with seqlens U[16384, 131072] in paged 64-token blocks in shuffled order
(2.4 GB + 0.68 GB of cache read per step, far above the 126 MB L2).  The
other workloads (--config) are single families.

Timing: W untimed warm-up steps, then K steps between two CUDA events on the
launching stream, with a synchronize (and a barrier under torchrun) on both
sides.  Per-kernel launch times come from events around each launch inside
the timed region (the host enqueues far ahead of the GPU on this workload,
so they measure the kernel, not host gaps); the mean gives the roofline
figure, the median is reported beside it, together with the host's enqueue
time per step and a back-to-back check (M launches between one event pair).
Enough independent input sets rotate between steps that each set is evicted
from L2 before it comes back (at least 2x the L2 size per rotation).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config C4]
                       [--kv bf16|fp8] [--impl reference]
For N > 1 (launched by torch.distributed.run) every rank runs an independent
replica (the path has no exchange step); value = the bytes all ranks
processed / the slowest rank's time.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step & KV GB/s vs ~8 TB/s HBM; MLA tensor-pipe util"

WORKLOADS = {
    "C4": "long-context ragged mix: Llama-3-70B-shaped GQA decode (B=8 h=64 n_kv=8 d=128) + "
          "DeepSeek-V3-shaped MLA absorbed decode (B=8 n_h=128, latent [pages,64,576]), "
          "seqlens U[16384,131072], paged 64-token blocks in shuffled order",
    "C0": "tiny GQA decode B=1 h=4 n_kv=2 d=64 L=128",
    "C1": "Llama-3-8B-shaped GQA decode B=32 h=32 n_kv=8 d=128 seqlens U[1024,4096] contiguous",
    "C2-MHA": "Llama-2-7B-shaped MHA decode B=16 h=32 n_kv=32 d=128 L=4096",
    "C2-MQA": "Llama-2-7B-shaped MQA decode B=16 h=32 n_kv=1 d=128 L=4096",
    "C3": "DeepSeek-V3-shaped MLA absorbed decode B=64 n_h=128 seqlens U[512,4096] paged latent [pages,64,576]",
    "C4-MLA": "long ragged MLA absorbed decode B=8 n_h=128 seqlens U[16384,131072] paged",
    "C4-GQA": "long ragged Llama-3-70B-shaped GQA decode B=8 h=64 n_kv=8 d=128 seqlens U[16384,131072] paged",
    "P-MLA": "DeepSeek-V3-shaped MLA prefill chunk, non-absorbed: 4096 tokens, 128 heads, causal (expand + attention)",
    "combine": "stand-alone LSE combine of split partials: 16 pieces of [32768 rows, 128] fp32 (268 MB)",
}
# the parts (single-family workloads) one step of each workload runs
PARTS = {"C4": ["C4-GQA", "C4-MLA"]}
PREFILL_TOKENS = 4096
L2_FALLBACK = 126 * 2 ** 20
MAX_SETS = 16


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="C4", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="kvdec", choices=["kvdec", "reference"])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                    help="cache element: bf16, or E4M3 bytes (GQA: per-KV-head scales; "
                         "MLA: a c_kv and a k_R scale)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="profiling runs: no CPU baseline, no e2e leg, no clock hold")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def is_mla(name):
    return name.startswith("C3") or name.endswith("MLA")


def parts_of(config):
    return PARTS.get(config, [config])


# ---------------------------------------------------------------- byte counts

def gqa_bytes(case, out_elem=4):
    """Algorithmic bytes of one decode call: every cached K and V element of
    the attended tokens once, plus q, out, lse, seqlens and the block table
    once.  Returns (total, KV only)."""
    sl = case.seqlens.double().sum().item()
    kv = sl * case.n_kv * 2 * case.d * case.k.element_size()
    q = case.B * case.h * case.d * 2
    out = case.B * case.h * case.d * out_elem + case.B * case.h * 4
    bt = 0 if case.block_table is None else case.block_table.numel() * 4
    scales = 0 if getattr(case, "k_scale", None) is None else 2 * case.n_kv * 4
    return kv + q + out + case.B * 4 + bt + scales, kv


def gqa_append_bytes(case):
    # k_new, v_new read (bf16); rotated K row and V row written; positions read
    return case.B * case.n_kv * case.d * (2 * 2 + 2 * case.k.element_size()) + case.B * 4


def mla_bytes(case, out_elem=4):
    """Per cached token 576 values (1152 B in bf16, 576 B as E4M3 codes),
    plus q (576 per head), out (512 per head), lse, seqlens, block table
    and the two E4M3 scales once."""
    sl = case.seqlens.double().sum().item()
    kv = sl * 576 * case.cache.element_size()
    q = case.B * case.n_h * 576 * 2
    out = case.B * case.n_h * 512 * out_elem + case.B * case.n_h * 4
    scales = 0 if getattr(case, "kv_scale", None) is None else 8
    return kv + q + out + case.B * 4 + case.block_table.numel() * 4 + scales, kv


def mla_flops(case):
    """2 FLOPs per dimension of a 576-long score dot and a 512-long weighted
    sum, for each of the n_h heads and each cached token."""
    return case.seqlens.double().sum().item() * case.n_h * 2 * (576 + 512)


def mla_append_bytes(case):
    # c_kv and k_rope read (bf16); the row written (bf16 or E4M3); positions read
    return case.B * (512 + 64) * (2 + case.cache.element_size()) + case.B * 4


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU works."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        mx = max(r[1] for r in rows)
        loaded = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in loaded:
            for n, v in zip(names, r[3][1:5]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(loaded)}


# ---------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6400.0), d.get("bf16_tflops", 1800.0), \
            d.get("bf16_tflops_sustained", 1400.0), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "decode_attention_kv_softmax_b300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(key, files):
    """DRAM bytes per launch of kernel@workload from the committed ncu
    summary, only while the kernel's source still hashes to the value
    recorded with the counters (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(key)
    except ValueError:
        return None
    if not d or d.get("source_hash") != kernel_source_hash(files):
        return None
    return d.get("bytes_per_launch")


def dist_setup(n_gpus):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def replica_throughput(units_per_rank, seconds_per_rank, ws):
    """Whole-job throughput of ws independent replicas: the units all ranks
    processed over the slowest rank's time (every rank processes the same
    units per step)."""
    return ws * units_per_rank / max_over_ranks(seconds_per_rank, ws)


def l2_bytes(dev):
    import torch
    try:
        return int(torch.cuda.get_device_properties(dev).L2_cache_size) or L2_FALLBACK
    except (AttributeError, RuntimeError):
        return L2_FALLBACK


def sets_needed(kv_bytes, l2):
    """Input sets to rotate so that a set is read again only after at least
    2x the L2 size of other sets' data (capped; small workloads say so)."""
    return max(2, min(MAX_SETS, math.ceil(2 * l2 / max(kv_bytes, 1)) + 1))


# ---------------------------------------------------------------- oracle timing

def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_units(name, case_cpu, n_seq):
    """Independent oracle calls covering the first n_seq sequences: one per
    (sequence, KV head) for GQA -- its g query heads against that head's
    K/V -- and one per sequence for MLA.  Each unit is (fn, kv_bytes); fn runs
    the oracle as it stands on that slice (widening its own bf16 inputs)."""
    import numpy as np
    import torch
    import oracle
    units = []
    sl = case_cpu.seqlens[:n_seq].numpy()
    if is_mla(name):
        for b in range(n_seq):
            L = int(sl[b])
            npg = (L + 63) // 64
            pages = case_cpu.block_table[b, :max(npg, 1)].long()

            def fn(b=b, L=L, pages=pages):
                cache = oracle.bf16_to_f64(case_cpu.cache[pages])
                oracle.mla_decode_absorbed(oracle.bf16_to_f64(case_cpu.q_abs[b:b + 1]),
                                           oracle.bf16_to_f64(case_cpu.q_rope[b:b + 1]), cache,
                                           np.arange(len(pages))[None], [L], case_cpu.scale)
            units.append((fn, L * 576 * 2))
        return units
    g = case_cpu.h // case_cpu.n_kv
    for b in range(n_seq):
        L = int(sl[b])
        for kv in range(case_cpu.n_kv):
            def fn(b=b, kv=kv, L=L):
                q = oracle.bf16_to_f64(case_cpu.q[b:b + 1, kv * g:(kv + 1) * g])
                if case_cpu.block_table is None:
                    k = oracle.bf16_to_f64(case_cpu.k[b:b + 1, kv:kv + 1, :L])
                    v = oracle.bf16_to_f64(case_cpu.v[b:b + 1, kv:kv + 1, :L])
                    oracle.gqa_decode(q, k, v, [L], case_cpu.scale)
                else:
                    npg = (L + 63) // 64
                    pages = case_cpu.block_table[b, :max(npg, 1)].long()
                    k = oracle.bf16_to_f64(case_cpu.k[pages, kv:kv + 1])
                    v = oracle.bf16_to_f64(case_cpu.v[pages, kv:kv + 1])
                    oracle.gqa_decode(q, k, v, [L], case_cpu.scale, np.arange(len(pages))[None])
            units.append((fn, L * 2 * case_cpu.d * 2))
    return units


def run_units(units, threads):
    """Wall time of running the units on a pool of host threads (numpy's
    matrix products, exponentials and reductions release the interpreter
    lock, so the threads run on separate cores).  BLAS is kept to one
    thread per call so that the pool, not BLAS, spreads the work."""
    import contextlib
    from concurrent.futures import ThreadPoolExecutor
    try:
        from threadpoolctl import threadpool_limits
        one_blas_thread = threadpool_limits(limits=1)
    except ImportError:
        one_blas_thread = contextlib.nullcontext()
    with one_blas_thread:
        t0 = time.perf_counter()
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda u: u[0](), units))
        dt = time.perf_counter() - t0
    return dt, float(sum(u[1] for u in units))


def oracle_sample(cases_cpu, target_s, threads, max_seq=None):
    """The oracle on the first n sequences of every part of the workload,
    n grown until the run takes about target_s/4 or more; returns
    (seconds, KV bytes, n)."""
    B = min(c.B for c in cases_cpu.values())
    if max_seq is not None:
        B = min(B, max_seq)
    n = 1
    while True:
        units = [u for name, c in cases_cpu.items() for u in oracle_units(name, c, n)]
        dt, kvb = run_units(units, threads)
        if dt >= target_s / 4 or n >= B:
            return dt, kvb, n
        n = min(B, n * 2 if dt < target_s / 8 else n + max(1, n // 2))


def cpu_cases(config):
    import kvgen
    return {p: kvgen.config_case(p, device="cpu") for p in parts_of(config)}


def cpu_baseline(config, target_s, kv="bf16"):
    if kv != "bf16":
        return {"value": None, "note": "no oracle timing for the FP8 cache line; the bf16 "
                                       "line of the same workload carries it"}
    threads = host_cores()
    cases = cpu_cases(config)
    dt, kvb, n = oracle_sample(cases, target_s, threads)
    return {"value": kvb / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 numpy oracle over the first {n} sequence(s) of each of "
                      f"{', '.join(cases)} (all heads; one oracle call per (sequence, KV head) "
                      f"for GQA, per sequence for MLA, on {threads} host threads), "
                      f"{kvb / 1e6:.1f} MB of KV, {dt:.2f} s"}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle, as it stands, on the host cores: each step is the same
    bounded sample of the workload."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    threads = host_cores()
    cases = cpu_cases(args.config)
    per_step = min(4.0, 150.0 / max(1, args.steps + args.warmup))
    _, _, n = oracle_sample(cases, 4 * per_step, threads)
    units = [u for name, c in cases.items() for u in oracle_units(name, c, n)]
    for _ in range(args.warmup):
        run_units(units, threads)
    times = []
    kvb = 0.0
    for _ in range(args.steps):
        d, kvb = run_units(units, threads)
        times.append(d)
    t = sum(times) / len(times)
    v = kvb / t / 1e9
    line = {"metric": METRIC, "value": v, "unit": "GB/s", "impl": "reference",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOADS[args.config], "name": args.config,
                       "sample_sequences_per_part": n},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"first {n} sequence(s) of each part per step, "
                                       f"{kvb / 1e6:.1f} MB of KV"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- prefill (P-MLA)

def prefill_flops(s, n_h=128):
    """Up-projection 2 s 512 (2 x 128 n_h) and causal attention
    n_h 2 (192 + 128) s^2 / 2 ([ARG] §四.6)."""
    return 2.0 * s * 512 * 256 * n_h, n_h * 2.0 * 320 * s * s / 2


def oracle_prefill_sample(case_cpu, n_rows):
    """fp64 oracle on the last n_rows queries of the chunk (all heads), the
    expensive end of the causal triangle; returns (seconds, FLOPs done)."""
    import oracle
    s = case_cpu["c_kv"].shape[0]
    to = lambda t: oracle.bf16_to_f64(t)
    t0 = time.perf_counter()
    kn, vv = oracle.mla_prefill_expand(to(case_cpu["c_kv"]), to(case_cpu["W_UK"]), to(case_cpu["W_UV"]))
    oracle.mla_prefill(to(case_cpu["q_nope"][-n_rows:]), to(case_cpu["q_rope"][-n_rows:]), kn,
                       to(case_cpu["k_rope"]), vv, kv_offset=s - n_rows)
    dt = time.perf_counter() - t0
    fe, _ = prefill_flops(s)
    return dt, fe + 128 * 2.0 * 320 * s * n_rows


def bench_prefill(args, reference=False):
    """--config P-MLA: one step = kvdec_mla_prefill_expand + kvdec_mla_prefill
    on a 4096-token chunk; value in TFLOP/s of algorithmic FLOPs."""
    import torch
    import kvgen
    s = PREFILL_TOKENS
    fe, fa = prefill_flops(s)
    if reference:
        case = kvgen.mla_prefill_case(s, s, 128, seed=1005, device="cpu")
        n = 1
        times = [oracle_prefill_sample(case, n)[0] for _ in range(max(1, min(args.steps, 3)))]
        _, fl = oracle_prefill_sample(case, n)
        v = fl / (sum(times) / len(times)) / 1e12
        line = {"metric": METRIC, "value": v, "unit": "TFLOP/s", "impl": "reference", "n_gpus": 1,
                "steps": len(times), "warmup": 0, "ms_per_step": sum(times) / len(times) * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": WORKLOADS["P-MLA"], "sample_rows": n},
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                 "sample": f"up-projection of all {s} tokens + the last {n} query row(s)"},
                "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    from decode_attention_kv_softmax_b300 import kvdec
    kvdec.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    hbm_peak, bf16_peak, bf16_sust, peak_src = measured_peaks()
    c = kvgen.mla_prefill_case(s, s, 128, seed=1005, device=dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        k, v = kvdec.mla_prefill_expand(c["c_kv"], c["W_UK"], c["W_UV"], stream=stream)
        if ev is not None:
            ev[1].record(stream)
        out, lse = kvdec.mla_prefill(c["q_nope"], c["q_rope"], k, c["k_rope"], v, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        return out
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clk = ClockSampler(0)
    clk.start()
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    ms = t0.elapsed_time(t1) / args.steps
    exp_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    att_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    value = (fe + fa) / (ms * 1e-3) / 1e12
    att_tf = fa / (att_ms * 1e-3) / 1e12
    host = {k: t.detach().to("cpu").pin_memory() for k, t in c.items()}
    hout = torch.empty((s, 128, 128), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    n_e2e = 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        for k, t in host.items():
            c[k].copy_(t, non_blocking=True)
        hout.copy_(step(), non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n_e2e
    cpu = None
    if not args.no_cpu_baseline and not args.quick:
        case_cpu = kvgen.mla_prefill_case(s, s, 128, seed=1005, device="cpu")
        n = 1
        dt, fl = oracle_prefill_sample(case_cpu, n)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"up-projection of all {s} tokens + the last {n} query row(s), all heads"}
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "us_per_step": ms * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOADS["P-MLA"], "name": "P-MLA", "tokens": s, "heads": 128,
                       "step": "kvdec_mla_prefill_expand + kvdec_mla_prefill",
                       "l2": "inputs 14 MB (L2-resident by design: compute-bound)"},
            "roofline": {"bound": "tensor", "achieved": att_tf, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": att_tf / bf16_peak,
                         "traffic": ncu_traffic("mla_prefill_tc_kernel@P-MLA",
                                                ["mla_prefill_tc.cu", "common.cuh", "tcgen05.cuh"]),
                         "kernel": "mla_prefill_tc_kernel",
                         "peak_source": f"{peak_src} bf16_tflops (cuBLAS GEMM, burst)",
                         "algorithmic_flops_per_launch": fa, "avg_launch_us": att_ms * 1e3},
            "expand": {"avg_launch_us": exp_ms * 1e3, "tflops": fe / (exp_ms * 1e-3) / 1e12},
            "cpu_baseline": cpu,
            "e2e": {"value": (fe + fa) / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": hout.numel() * 4, "ms_per_step": e2e_ms, "steps": n_e2e},
            "clocks": clocks, "gpu_launches": 3 * args.steps}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- decode parts

class Part:
    """One model family of the workload: its input sets (rotated between
    steps), the prepared C-ABI argument blocks of each set, and its byte and
    FLOP counts."""

    def __init__(self, name, kv, dev, lib, rank, l2):
        import ctypes
        import torch
        import kvgen
        from decode_attention_kv_softmax_b300 import kvdec
        self.name = name
        self.mla = is_mla(name)
        self.fp8 = kv == "fp8"
        self.lib = lib
        self.kernel = "mla_decode_kernel" if self.mla else "gqa_decode_kernel"
        self.files = ["mla_decode.cu", "common.cuh", "schedule.cuh", "tcgen05.cuh"] if self.mla else \
            ["gqa_decode.cu", "common.cuh", "schedule.cuh"]
        if self.mla and self.fp8:
            # the E4M3 latent cache is widened to bf16, then decoded: the
            # decode call launches both kernels and is timed as one
            self.kernel = "mla_widen_kernel + mla_decode_kernel"
            self.files = self.files + ["mla_widen.cu"]
        case0 = kvgen.config_case(name, device=dev, kv_dtype="fp8" if self.fp8 else "bf16")
        kvb0 = (mla_bytes if self.mla else gqa_bytes)(case0)[1]
        self.n_sets = sets_needed(kvb0, l2)
        self.sets = []
        for rep in range(self.n_sets):
            case = case0 if rep == 0 else kvgen.config_case(
                name, device=dev, kv_dtype="fp8" if self.fp8 else "bf16")
            if rep > 0:   # an independent draw of the same workload (new cache values)
                g = torch.Generator(device=dev)
                g.manual_seed(7777 + 101 * rep + rank)
                if self.mla and self.fp8:
                    x = torch.randn(case.cache.shape, generator=g, device=dev).to(torch.bfloat16)
                    case.cache.copy_(kvgen.mla_fp8_codes(x, g, dev)[0])
                elif self.mla:
                    case.cache.copy_(torch.randn(case.cache.shape, generator=g, device=dev).to(torch.bfloat16))
                elif self.fp8:
                    case.k.copy_(kvgen.fp8_codes(torch.randn(case.k.shape, generator=g, device=dev), g, dev)[0])
                    case.v.copy_(kvgen.fp8_codes(torch.randn(case.v.shape, generator=g, device=dev), g, dev)[0])
                else:
                    case.k.copy_(torch.randn(case.k.shape, generator=g, device=dev).to(torch.bfloat16))
                    case.v.copy_(torch.randn(case.v.shape, generator=g, device=dev).to(torch.bfloat16))
            self.sets.append(self._prepare(case, rep, dev, kvdec, ctypes, kvgen, torch))
        self.case0 = case0
        if self.mla:
            self.dec_bytes = [mla_bytes(s["case"]) for s in self.sets]
            self.app_bytes = mla_append_bytes(case0)
            self.flops = mla_flops(case0)
        else:
            self.dec_bytes = [gqa_bytes(s["case"]) for s in self.sets]
            self.app_bytes = gqa_append_bytes(case0)
            self.flops = None

    def _prepare(self, case, rep, dev, kvdec, ctypes, kvgen, torch):
        lib = self.lib
        B = case.B
        if self.mla:
            ckv, kr = kvgen.append_inputs_mla(B, seed=55 + rep, device=dev)
            pos = (case.seqlens - 1).contiguous()
            out = torch.empty((B, case.n_h, 512), dtype=torch.float32, device=dev)
            lse = torch.empty((B, case.n_h), dtype=torch.float32, device=dev)
            p = kvdec.mla_params(case.q_abs, case.q_rope, case.cache, case.block_table,
                                 case.seqlens, case.scale, out, lse, None, 0,
                                 kv_scale=getattr(case, "kv_scale", None))
            need = lib.kvdec_mla_workspace_bytes(ctypes.byref(p))
            wsb = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
            p.workspace, p.workspace_bytes = kvdec._ptr(wsb), wsb.numel()
            ap = kvdec.AppendParams()
            ap.mode, ap.batch = kvdec.APPEND_MLA, B
            ap.seqlens, ap.block_table = kvdec._ptr(pos), kvdec._ptr(case.block_table)
            ap.num_pages, ap.max_blocks = case.cache.shape[0], case.block_table.shape[1]
            ap.rope_theta = 10000.0
            ap.c_kv, ap.k_rope, ap.cache = kvdec._ptr(ckv), kvdec._ptr(kr), kvdec._ptr(case.cache)
            if self.fp8:
                ap.kv_format = kvdec.KV_FP8_E4M3
                ap.k_scale = kvdec._ptr(case.kv_scale)
            return dict(case=case, new=(ckv, kr), q=(case.q_abs, case.q_rope), pos=pos, out=out,
                        lse=lse, ws=wsb, p=p, ap=ap, decode=lib.kvdec_mla_decode_absorbed)
        k_new, v_new = kvgen.append_inputs_gqa(B, case.n_kv, case.d, seed=55 + rep, device=dev)
        pos = (case.seqlens - 1).contiguous()
        out = torch.empty(case.q.shape, dtype=torch.float32, device=dev)
        lse = torch.empty(case.q.shape[:2], dtype=torch.float32, device=dev)
        p = kvdec.gqa_params(case.q, case.k, case.v, case.seqlens, case.block_table,
                             case.scale, out, lse, None, 0, k_scale=getattr(case, "k_scale", None),
                             v_scale=getattr(case, "v_scale", None))
        need = lib.kvdec_gqa_workspace_bytes(ctypes.byref(p))
        wsb = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
        p.workspace, p.workspace_bytes = kvdec._ptr(wsb), wsb.numel()
        ap = kvdec.AppendParams()
        ap.mode, ap.batch = kvdec.APPEND_GQA, B
        ap.seqlens = kvdec._ptr(pos)
        if case.block_table is not None:
            ap.block_table = kvdec._ptr(case.block_table)
            ap.num_pages, ap.max_blocks = case.k.shape[0], case.block_table.shape[1]
        else:
            ap.capacity = case.k.shape[2]
        ap.rope_theta = 10000.0
        ap.k_new, ap.v_new = kvdec._ptr(k_new), kvdec._ptr(v_new)
        ap.k, ap.v = kvdec._ptr(case.k), kvdec._ptr(case.v)
        ap.num_kv_heads, ap.head_dim = case.n_kv, case.d
        if self.fp8:
            ap.kv_format = kvdec.KV_FP8_E4M3
            ap.k_scale, ap.v_scale = kvdec._ptr(case.k_scale), kvdec._ptr(case.v_scale)
        return dict(case=case, new=(k_new, v_new), q=(case.q,), pos=pos, out=out, lse=lse, ws=wsb,
                    p=p, ap=ap, decode=lib.kvdec_gqa_decode)

    def append(self, i, sptr):
        import ctypes
        s = self.sets[i % self.n_sets]
        return self.lib.kvdec_append_rope(ctypes.byref(s["ap"]), sptr)

    def decode(self, i, sptr):
        import ctypes
        s = self.sets[i % self.n_sets]
        return s["decode"](ctypes.byref(s["p"]), sptr)

    def step_bytes(self, i):
        return self.dec_bytes[i % self.n_sets][0] + self.app_bytes

    def l2_note(self, l2):
        kvb = self.dec_bytes[0][1]
        rot = kvb * (self.n_sets - 1)
        if rot >= 2 * l2:
            return (f"{self.n_sets} input sets rotated ({kvb / 1e6:.0f} MB of KV each): "
                    f"{rot / 1e6:.0f} MB of other sets' KV between two reads of one set, > 2x L2")
        return (f"{self.n_sets} input sets rotated ({kvb / 1e6:.2f} MB of KV each): "
                f"L2-resident in part (the workload is smaller than L2)")


def bench_combine(args):
    """--config combine: one step = kvdec_combine_splits over 16 normalised
    partials of 32768 rows x 128 (the merge of [ARG] §五.2 on its own);
    value in GB/s of algorithmic bytes (every partial and lse read once, out
    and lse written once)."""
    import torch
    from decode_attention_kv_softmax_b300 import kvdec
    kvdec.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    hbm_peak, _, _, peak_src = measured_peaks()
    S, R, D = 16, 32768, 128
    g = torch.Generator(device=dev).manual_seed(1009)
    sets = [(torch.randn((S, R, D), generator=g, device=dev), torch.randn((S, R), generator=g, device=dev))
            for _ in range(2)]
    outs = [torch.empty((R, D), device=dev) for _ in range(2)]
    alg = S * R * (D + 1) * 4 + R * (D + 1) * 4

    def step(i):
        po, pl = sets[i & 1]
        kvdec.combine_splits(po, pl, out=outs[i & 1], stream=stream)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    clk = ClockSampler(0)
    clk.start()
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    spin_end = torch.cuda.Event()
    # a single ~55 us kernel per step is shorter than the host's enqueue of
    # a step: hold the stream with a spin kernel (before the timed region)
    # while all steps are enqueued, so the launches run back to back and the
    # per-launch events time the kernel, not host gaps.  If the spin has
    # already ended when the last step is enqueued (a slow host), the
    # launches may have waited for it: time again with a longer spin.
    spin = int(args.steps * 4e5)
    for _attempt in range(4):
        torch.cuda._sleep(spin)
        spin_end.record(stream)
        t0.record(stream)
        for i in range(args.steps):
            evs[i][0].record(stream)
            step(i)
            evs[i][1].record(stream)
        t1.record(stream)
        overran = spin_end.query()
        torch.cuda.synchronize()
        if not overran:
            break
        spin *= 4
    clocks = clk.stop()
    ms = t0.elapsed_time(t1) / args.steps
    per = [e[0].elapsed_time(e[1]) * 1e3 for e in evs]
    avg = sum(per) / len(per)
    ach = alg / (avg * 1e-6) / 1e9
    line = {"metric": METRIC, "value": alg / (ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOADS["combine"], "name": "combine",
                       "l2": "two 277 MB input sets alternated (> 2x L2)"},
            "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                         "frac": ach / hbm_peak,
                         "traffic": ncu_traffic("combine_kernel@combine", ["combine.cu", "common.cuh"]),
                         "kernel": "combine_kernel", "peak_source": f"{peak_src} hbm_gbs (copy, burst)",
                         "algorithmic_bytes_per_launch": alg, "avg_launch_us": avg,
                         "median_launch_us": statistics.median(per),
                         "timing": "launches queued behind a spin kernel, run back to back"},
            "cpu_baseline": None, "e2e": None, "clocks": clocks, "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.config == "combine":
        if args.impl == "reference" or args.gpus != 1 or int(os.environ.get("RANK", "0")) != 0:
            return
        bench_combine(args)
        return
    if args.config == "P-MLA":
        if args.gpus != 1 or int(os.environ.get("RANK", "0")) != 0:
            return
        bench_prefill(args, reference=args.impl == "reference")
        return
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    from decode_attention_kv_softmax_b300 import kvdec

    ws, rank, local = dist_setup(args.gpus)
    lib = kvdec.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    sptr = kvdec._stream(stream)
    hbm_peak, bf16_peak, bf16_sust, peak_src = measured_peaks()
    l2 = l2_bytes(dev)
    parts = [Part(name, args.kv, dev, lib, rank, l2) for name in parts_of(args.config)]

    def step(i, evs=None):
        rc = 0
        for k, part in enumerate(parts):
            if evs is not None:
                evs[k][0].record(stream)
            rc |= part.append(i, sptr)
            if evs is not None:
                evs[k][1].record(stream)
            rc |= part.decode(i, sptr)
            if evs is not None:
                evs[k][2].record(stream)
        if rc:
            raise RuntimeError(lib.kvdec_last_error().decode())

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    clk = ClockSampler(local)
    clk.start()
    # keep the GPU busy while the sampler starts (an idle GPU lowers its
    # clocks, and a short timed region would start below them)
    t_busy, i = time.time(), 0
    while time.time() - t_busy < 0.3:
        step(i)
        i += 1
        if i % 4 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in parts]
           for _ in range(args.steps)]
    host_us = []
    barrier(ws)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        h0 = time.perf_counter()
        step(i, evs[i])
        host_us.append((time.perf_counter() - h0) * 1e6)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    total_ms = t_start.elapsed_time(t_end)
    # keep the GPU busy a moment longer so that the clock sampler sees load
    t_keep = time.time()
    while not args.quick and time.time() - t_keep < 1.0:
        for i in range(50):
            step(i)
        torch.cuda.synchronize()
    clocks = clk.stop()

    # host cost of enqueueing one step, on short bursts that cannot fill the
    # launch queue (inside the timed region the enqueue loop also waits for
    # queue space whenever the GPU is the slower side)
    burst_us = []
    for r in range(10):
        torch.cuda.synchronize()
        step(0)                       # the first call after a synchronize is not timed
        h0 = time.perf_counter()
        for i in range(16):
            step(i)
        burst_us.append((time.perf_counter() - h0) / 16 * 1e6)
    torch.cuda.synchronize()

    # back-to-back cross-check: M decode launches of a part between one event pair
    b2b = {}
    M = max(20, min(100, args.steps))
    for part in parts:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(M):
            part.decode(i, sptr)
        e1.record(stream)
        torch.cuda.synchronize()
        b2b[part.name] = e0.elapsed_time(e1) / M * 1e3

    step_bytes = sum(p.step_bytes(i) for p in parts for i in range(args.steps)) / args.steps
    value = replica_throughput(step_bytes * args.steps, total_ms * 1e-3, ws) / 1e9
    total_ms = max_over_ranks(total_ms, ws)
    ms_per_step = total_ms / args.steps

    kernels = {}
    for k, part in enumerate(parts):
        dec_us = [evs[i][k][1].elapsed_time(evs[i][k][2]) * 1e3 for i in range(args.steps)]
        app_us = [evs[i][k][0].elapsed_time(evs[i][k][1]) * 1e3 for i in range(args.steps)]
        mean_us = sum(dec_us) / len(dec_us)
        dec_alg = sum(part.dec_bytes[i % part.n_sets][0] for i in range(args.steps)) / args.steps
        achieved = dec_alg / (mean_us * 1e-6) / 1e9
        tkey = part.kernel + ("[fp8]" if part.fp8 else "") + "@" + part.name
        r = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
             "frac": achieved / hbm_peak, "traffic": ncu_traffic(tkey, part.files),
             "kernel": part.kernel, "workload": part.name,
             "peak_source": f"{peak_src} hbm_gbs (copy, burst)",
             "algorithmic_bytes_per_launch": dec_alg, "avg_launch_us": mean_us,
             "median_launch_us": statistics.median(dec_us), "b2b_launch_us": b2b[part.name],
             "append_avg_us": sum(app_us) / len(app_us), "time_share": None}
        if part.mla:
            tf = part.flops / (mean_us * 1e-6) / 1e12
            t_hbm = dec_alg / (hbm_peak * 1e9)
            t_tc = part.flops / (bf16_peak * 1e12)
            r["tensor"] = {"achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s", "frac": tf / bf16_peak,
                           "peak_source": f"{peak_src} bf16_tflops (cuBLAS GEMM, burst)" +
                           ("; the E4M3 cache's MMAs run in f16, whose nominal dense rate equals "
                            "bf16's (ratio 1)" if part.fp8 else ""),
                           "algorithmic_flops_per_launch": part.flops}
            r["binding"] = "hbm" if t_hbm >= t_tc else "tensor"
            r["frac_of_binding"] = max(t_hbm, t_tc) / (mean_us * 1e-6)
            if r["binding"] == "tensor":
                r.update(bound="tensor", achieved=tf, peak=bf16_peak, unit="TFLOP/s", frac=tf / bf16_peak)
        kernels[part.name] = r
    tot = sum(r["avg_launch_us"] for r in kernels.values())
    for r in kernels.values():
        r["time_share"] = r["avg_launch_us"] / tot
    dominant = max(kernels.values(), key=lambda r: r["avg_launch_us"])
    roof = {k: dominant[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic",
                                     "kernel", "workload", "peak_source",
                                     "algorithmic_bytes_per_launch", "avg_launch_us",
                                     "median_launch_us")}
    roof["kernels"] = kernels

    # ---- end to end through the public API with host buffers
    if args.quick:
        args.no_cpu_baseline = True
    pin = lambda t: t.detach().to("cpu").pin_memory()
    legs = []
    for part in parts:
        s = part.sets[0]
        c = s["case"]
        dev_in = list(s["q"]) + list(s["new"]) + [s["pos"], c.seqlens]
        legs.append(dict(part=part, dev_in=dev_in, host_in=[pin(t) for t in dev_in],
                         out=s["out"], lse=s["lse"],
                         host_out=torch.empty(s["out"].shape, dtype=s["out"].dtype).pin_memory(),
                         host_lse=torch.empty(s["lse"].shape, dtype=s["lse"].dtype).pin_memory()))
    h2d = sum(t.numel() * t.element_size() for lg in legs for t in lg["host_in"])
    d2h = sum(lg["host_out"].numel() * lg["host_out"].element_size() + lg["host_lse"].numel() * 4
              for lg in legs)
    n_e2e = 0 if args.quick else max(10, min(args.steps, 200))

    # Uploads and read-backs run on two copy streams (one per direction),
    # ordered by events against the kernels of the same part: a part's inputs
    # go up once the previous step's kernels have read them, its kernels wait
    # for them and for the previous read-back of its outputs, and its outputs
    # come down once its decode is done.  So one part's copies overlap the
    # other part's kernels, as in a serving loop; every step still moves all
    # its bytes inside the timed region.
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    for lg in legs:
        lg.update(in_ready=torch.cuda.Event(), done=torch.cuda.Event(), out_read=torch.cuda.Event(), first=True)

    def e2e_step():
        rc = 0
        for lg in legs:
            with torch.cuda.stream(up):
                if not lg["first"]:
                    up.wait_event(lg["done"])
                for hsrc, ddst in zip(lg["host_in"], lg["dev_in"]):
                    ddst.copy_(hsrc, non_blocking=True)
                lg["in_ready"].record(up)
        for lg in legs:
            stream.wait_event(lg["in_ready"])
            if not lg["first"]:
                stream.wait_event(lg["out_read"])
            rc |= lg["part"].append(0, sptr)
            rc |= lg["part"].decode(0, sptr)
            lg["done"].record(stream)
        for lg in legs:
            with torch.cuda.stream(down):
                down.wait_event(lg["done"])
                lg["host_out"].copy_(lg["out"], non_blocking=True)
                lg["host_lse"].copy_(lg["lse"], non_blocking=True)
                lg["out_read"].record(down)
            lg["first"] = False
        if rc:
            raise RuntimeError(lib.kvdec_last_error().decode())

    for _ in range(3 if n_e2e else 0):
        e2e_step()
    torch.cuda.synchronize()
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_event(e0)
    down.wait_event(e0)
    for _ in range(n_e2e):
        e2e_step()
    for lg in legs:
        stream.wait_event(lg["out_read"])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_bytes = sum(p.step_bytes(0) for p in parts)
    e2e_rank_ms = e0.elapsed_time(e1) / max(n_e2e, 1)
    e2e_value = replica_throughput(e2e_bytes, e2e_rank_ms * 1e-3, ws) / 1e9
    e2e_ms = max_over_ranks(e2e_rank_ms, ws)
    e2e = None if not n_e2e else {
        "value": e2e_value, "unit": "GB/s",
        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
        "steps": n_e2e, "note": "per-step inputs (queries, the new token's cache entries, positions, "
                                "seqlens) copied from pinned host memory, outputs and lse read back, "
                                "on copy streams overlapping the other part's kernels; the KV caches "
                                "stay resident"}

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(args.config, args.cpu_seconds, args.kv)
    cfg = {"workload": WORKLOADS[args.config], "name": args.config,
           "parts": {p.name: WORKLOADS[p.name] for p in parts},
           "l2": "; ".join(f"{p.name}: {p.l2_note(l2)}" for p in parts),
           "kv_bytes_per_step": sum(p.dec_bytes[0][1] for p in parts),
           "step": " + ".join(f"{p.name}: append_rope + decode (fused split merge)" for p in parts),
           "kv_cache": ("E4M3 bytes (GQA: per-KV-head fp32 scales; MLA: c_kv and k_R fp32 scales)"
                        if args.kv == "fp8" else "bf16"),
           "parallelism": f"replicas x{ws}"}
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "us_per_step": ms_per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8-e4m3 cache, f16 MMA" if args.kv == "fp8" else "bf16",
            "data": "synthetic", "config": cfg,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": sum(3 if (p.mla and p.fp8) else 2 for p in parts) * args.steps,
            "host_enqueue_us_per_step": {"median": statistics.median(burst_us),
                                         "note": "host time to enqueue one step (all parts' append "
                                                 "and decode calls), bursts of 16 steps",
                                         "timed_region_median": statistics.median(host_us)}}
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
