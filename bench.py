#!/usr/bin/env python3
"""Benchmark of the decode-attention hot path on B300.

One step = one pass of the whole hot path over one batch: the new token's K/V
are appended to the cache with RoPE (kvdec_append_rope), then single-token
split-KV decode attention runs over the whole cache, its split pieces merged
by log-sum-exp inside the same kernel (kvdec_gqa_decode or
kvdec_mla_decode_absorbed).

Default workload (the one the headline metric is quoted on): Llama-3-8B-shaped
GQA decode, one layer: B=32, h=32, n_kv=8, d=128, seqlens U[1024, 4096],
contiguous bf16 K/V [32, 8, 4096, 128].  Two independent copies of the inputs
alternate between steps, and each copy's KV (335 MB read per step) is larger
than L2 (126 MB), so KV reads come from HBM.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config C1]
                       [--impl reference]
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
    "C0": "tiny GQA decode B=1 h=4 n_kv=2 d=64 L=128",
    "C1": "Llama-3-8B-shaped GQA decode B=32 h=32 n_kv=8 d=128 seqlens U[1024,4096] contiguous",
    "C2-MHA": "Llama-2-7B-shaped MHA decode B=16 h=32 n_kv=32 d=128 L=4096",
    "C2-MQA": "Llama-2-7B-shaped MQA decode B=16 h=32 n_kv=1 d=128 L=4096",
    "C3": "DeepSeek-V3-shaped MLA absorbed decode B=64 n_h=128 seqlens U[512,4096] paged latent [pages,64,576]",
    "C4-MLA": "long ragged MLA absorbed decode B=8 n_h=128 seqlens U[16384,131072] paged",
    "C4-GQA": "long ragged Llama-3-70B-shaped GQA decode B=8 h=64 n_kv=8 d=128 seqlens U[16384,131072] paged",
    "P-MLA": "DeepSeek-V3-shaped MLA prefill chunk, non-absorbed: 4096 tokens, 128 heads, causal (expand + attention)",
}
PREFILL_TOKENS = 4096


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--config", default="C1", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="kvdec", choices=["kvdec", "reference"])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                    help="GQA cache element: bf16, or E4M3 bytes with per-KV-head scales")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="profiling runs: no CPU baseline, no e2e leg, no clock hold")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


# ---------------------------------------------------------------- byte counts

def gqa_bytes(case, out_elem=4):
    """Algorithmic bytes of one decode call: every cached K and V element of
    the attended tokens once, plus q, out, lse and seqlens once."""
    sl = case.seqlens.double().sum().item()
    kv = sl * case.n_kv * 2 * case.d * case.k.element_size()
    q = case.B * case.h * case.d * 2
    out = case.B * case.h * case.d * out_elem + case.B * case.h * 4
    bt = 0 if case.block_table is None else case.block_table.numel() * 4
    return kv + q + out + case.B * 4 + bt, kv


def gqa_append_bytes(case):
    # k_new, v_new read (bf16); rotated K row and V row written; positions read
    return case.B * case.n_kv * case.d * (2 * 2 + 2 * case.k.element_size()) + case.B * 4


def mla_bytes(case, out_elem=4):
    sl = case.seqlens.double().sum().item()
    kv = sl * 576 * 2
    q = case.B * case.n_h * 576 * 2
    out = case.B * case.n_h * 512 * out_elem + case.B * case.n_h * 4
    return kv + q + out + case.B * 4 + case.block_table.numel() * 4, kv


def mla_flops(case):
    return case.seqlens.double().sum().item() * case.n_h * 2 * (576 + 512)


def mla_append_bytes(case):
    return case.B * (512 + 64) * 2 * 2 + case.B * 4


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


def ncu_traffic(kernel, files):
    """DRAM bytes per launch from a committed ncu summary, only while the
    kernel source still hashes to the value recorded with the counters."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(kernel)
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
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


# ---------------------------------------------------------------- oracle timing

def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return 1


def oracle_gqa_sample(case_cpu, n_seq):
    """Run the oracle on the first n_seq sequences (all heads); returns
    (seconds, KV bytes)."""
    import numpy as np
    import oracle
    q = oracle.bf16_to_f64(case_cpu.q[:n_seq])
    k = oracle.bf16_to_f64(case_cpu.k[:n_seq]) if case_cpu.block_table is None else oracle.bf16_to_f64(case_cpu.k)
    v = oracle.bf16_to_f64(case_cpu.v[:n_seq]) if case_cpu.block_table is None else oracle.bf16_to_f64(case_cpu.v)
    sl = case_cpu.seqlens[:n_seq].numpy()
    bt = None if case_cpu.block_table is None else case_cpu.block_table[:n_seq].numpy()
    t0 = time.perf_counter()
    oracle.gqa_decode(q, k, v, sl, case_cpu.scale, bt)
    dt = time.perf_counter() - t0
    kvb = float(np.sum(sl)) * case_cpu.n_kv * 2 * case_cpu.d * 2
    return dt, kvb


def oracle_mla_sample(case_cpu, n_seq):
    import numpy as np
    import oracle
    sl = case_cpu.seqlens[:n_seq].numpy()
    bt = case_cpu.block_table[:n_seq].numpy()
    qa = oracle.bf16_to_f64(case_cpu.q_abs[:n_seq])
    qr = oracle.bf16_to_f64(case_cpu.q_rope[:n_seq])
    used = np.unique(bt[bt >= 0])
    cache = np.zeros((case_cpu.cache.shape[0], 64, 576))
    cache[used] = oracle.bf16_to_f64(case_cpu.cache[used])
    t0 = time.perf_counter()
    oracle.mla_decode_absorbed(qa, qr, cache, bt, sl, case_cpu.scale)
    dt = time.perf_counter() - t0
    return dt, float(np.sum(sl)) * 576 * 2


def cpu_case(config):
    import kvgen
    return kvgen.config_case(config, device="cpu")


def cpu_baseline(config, target_s, max_seq=None):
    """The oracle as it stands, on the host cores, on a bounded sample of the
    workload (the first n sequences, all heads), grown until it runs about
    target_s seconds.  Returns the cpu_baseline object."""
    case = cpu_case(config)
    mla = config.startswith("C3") or config.endswith("MLA")
    fn = oracle_mla_sample if mla else oracle_gqa_sample
    B = case.B
    n = 1
    dt, kvb = fn(case, n)
    while dt < target_s / 4 and n < B and (max_seq is None or n < max_seq):
        n = min(B, n * 2 if dt < target_s / 8 else n + max(1, n // 2))
        dt, kvb = fn(case, n)
    return {"value": kvb / dt / 1e9, "unit": "GB/s", "cores": oracle_threads(),
            "kind": "oracle",
            "sample": f"fp64 numpy oracle over the first {n} of {B} sequences (all heads) of "
                      f"the {config} workload, {kvb / 1e6:.1f} MB of KV, {dt:.2f} s"}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    case = cpu_case(args.config)
    mla = args.config.startswith("C3") or args.config.endswith("MLA")
    fn = oracle_mla_sample if mla else oracle_gqa_sample
    # size one step so that warmup + steps end within a few minutes
    per_step_budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    n = 1
    dt, kvb = fn(case, n)
    while dt < per_step_budget / 2 and n < case.B:
        n = min(case.B, n * 2)
        dt, kvb = fn(case, n)
    for _ in range(args.warmup):
        fn(case, n)
    times = []
    for _ in range(args.steps):
        d, kvb = fn(case, n)
        times.append(d)
    t = sum(times) / len(times)
    v = kvb / t / 1e9
    line = {"metric": METRIC, "value": v, "unit": "GB/s", "impl": "reference",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOADS[args.config], "sample_sequences": n},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": oracle_threads(),
                             "kind": "oracle",
                             "sample": f"first {n} of {case.B} sequences per step"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- main arm

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
        dt, fl = oracle_prefill_sample(case, n)
        times = [oracle_prefill_sample(case, n)[0] for _ in range(max(1, min(args.steps, 3)))]
        v = fl / (sum(times) / len(times)) / 1e12
        line = {"metric": METRIC, "value": v, "unit": "TFLOP/s", "impl": "reference", "n_gpus": 1,
                "steps": len(times), "warmup": 0, "ms_per_step": sum(times) / len(times) * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": WORKLOADS["P-MLA"], "sample_rows": n},
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
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
    # end to end: the chunk's inputs from pinned host memory, the output back
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
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
               "sample": f"up-projection of all {s} tokens + the last {n} query row(s), all heads"}
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "us_per_step": ms * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOADS["P-MLA"], "name": "P-MLA", "tokens": s, "heads": 128,
                       "step": "kvdec_mla_prefill_expand + kvdec_mla_prefill",
                       "l2": "inputs 14 MB (L2-resident by design: compute-bound)"},
            "roofline": {"bound": "tensor", "achieved": att_tf, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": att_tf / bf16_peak,
                         "traffic": ncu_traffic("mla_prefill_tc_kernel",
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


def main():
    args = parse()
    if args.config == "P-MLA":
        if args.gpus != 1 or int(os.environ.get("RANK", "0")) != 0:
            return
        bench_prefill(args, reference=args.impl == "reference")
        return
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    import kvgen
    from decode_attention_kv_softmax_b300 import kvdec

    ws, rank, local = dist_setup(args.gpus)
    lib = kvdec.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    sptr = kvdec._stream(stream)
    mla = args.config.startswith("C3") or args.config.endswith("MLA")
    if mla and args.kv != "bf16":
        raise SystemExit("--kv fp8 applies to the GQA workloads")
    fp8 = args.kv == "fp8"
    hbm_peak, bf16_peak, bf16_sust, peak_src = measured_peaks()

    # two independent input sets, alternated step by step
    import ctypes
    sets = []
    for rep in range(2):
        case = kvgen.config_case(args.config, device=dev, kv_dtype=args.kv)
        if rep == 1:   # a second, independent draw of the same workload
            g = torch.Generator(device=dev)
            g.manual_seed(7777 + rank)
            if mla:
                case.cache.copy_(torch.randn(case.cache.shape, generator=g, device=dev).to(torch.bfloat16))
            elif fp8:
                case.k.copy_(kvgen.fp8_codes(torch.randn(case.k.shape, generator=g, device=dev), g, dev)[0])
                case.v.copy_(kvgen.fp8_codes(torch.randn(case.v.shape, generator=g, device=dev), g, dev)[0])
            else:
                case.k.copy_(torch.randn(case.k.shape, generator=g, device=dev).to(torch.bfloat16))
                case.v.copy_(torch.randn(case.v.shape, generator=g, device=dev).to(torch.bfloat16))
        st = {"case": case}
        if mla:
            B = case.B
            ckv, kr = kvgen.append_inputs_mla(B, seed=55 + rep, device=dev)
            pos = (case.seqlens - 1).contiguous()
            out = torch.empty((B, case.n_h, 512), dtype=torch.float32, device=dev)
            lse = torch.empty((B, case.n_h), dtype=torch.float32, device=dev)
            p = kvdec.mla_params(case.q_abs, case.q_rope, case.cache, case.block_table,
                                 case.seqlens, case.scale, out, lse, None, 0)
            need = lib.kvdec_mla_workspace_bytes(ctypes.byref(p))
            wsb = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
            p.workspace, p.workspace_bytes = kvdec._ptr(wsb), wsb.numel()
            ap = kvdec.AppendParams()
            ap.mode, ap.batch = kvdec.APPEND_MLA, B
            ap.seqlens, ap.block_table = kvdec._ptr(pos), kvdec._ptr(case.block_table)
            ap.num_pages, ap.max_blocks = case.cache.shape[0], case.block_table.shape[1]
            ap.rope_theta = 10000.0
            ap.c_kv, ap.k_rope, ap.cache = kvdec._ptr(ckv), kvdec._ptr(kr), kvdec._ptr(case.cache)
            st.update(new=(ckv, kr), pos=pos, out=out, lse=lse, ws=wsb, p=p, ap=ap,
                      decode=lib.kvdec_mla_decode_absorbed)
        else:
            B = case.B
            k_new, v_new = kvgen.append_inputs_gqa(B, case.n_kv, case.d, seed=55 + rep, device=dev)
            pos = (case.seqlens - 1).contiguous()
            out = torch.empty(case.q.shape, dtype=torch.float32, device=dev)
            lse = torch.empty(case.q.shape[:2], dtype=torch.float32, device=dev)
            p = kvdec.gqa_params(case.q, case.k, case.v, case.seqlens, case.block_table,
                                 case.scale, out, lse, None, 0, k_scale=case.k_scale,
                                 v_scale=case.v_scale)
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
            if fp8:
                ap.kv_format = kvdec.KV_FP8_E4M3
                ap.k_scale, ap.v_scale = kvdec._ptr(case.k_scale), kvdec._ptr(case.v_scale)
            st.update(new=(k_new, v_new), pos=pos, out=out, lse=lse, ws=wsb, p=p, ap=ap,
                      decode=lib.kvdec_gqa_decode)
        sets.append(st)

    case0 = sets[0]["case"]
    if mla:
        dec_bytes = [mla_bytes(s["case"])[0] for s in sets]
        kv_bytes = [mla_bytes(s["case"])[1] for s in sets]
        app_bytes = mla_append_bytes(case0)
    else:
        dec_bytes = [gqa_bytes(s["case"])[0] for s in sets]
        kv_bytes = [gqa_bytes(s["case"])[1] for s in sets]
        app_bytes = gqa_append_bytes(case0)

    def step(i, ev=None):
        s = sets[i & 1]
        if ev is not None:
            ev[0].record(stream)
        rc = lib.kvdec_append_rope(ctypes.byref(s["ap"]), sptr)
        if ev is not None:
            ev[1].record(stream)
        rc |= s["decode"](ctypes.byref(s["p"]), sptr)
        if ev is not None:
            ev[2].record(stream)
        if rc:
            raise RuntimeError(lib.kvdec_last_error().decode())

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(i, evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    total_ms = t_start.elapsed_time(t_end)
    # keep the GPU busy a moment longer so that the clock sampler sees load
    t_keep = time.time()
    while not args.quick and time.time() - t_keep < 1.0:
        for i in range(200):
            step(i)
        torch.cuda.synchronize()
    clocks = clk.stop()

    dec_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(args.steps)]
    app_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(args.steps)]
    total_ms = max_over_ranks(total_ms, ws)
    ms_per_step = total_ms / args.steps
    step_bytes = sum(dec_bytes[i & 1] + app_bytes for i in range(args.steps)) / args.steps
    value = ws * step_bytes / (ms_per_step * 1e-3) / 1e9
    dec_avg_ms = sum(dec_ms) / len(dec_ms)
    dec_alg = sum(dec_bytes[i & 1] for i in range(args.steps)) / args.steps
    achieved = dec_alg / (dec_avg_ms * 1e-3) / 1e9

    kfile = ["mla_decode.cu", "common.cuh", "schedule.cuh", "tcgen05.cuh"] if mla else \
        ["gqa_decode.cu", "common.cuh", "schedule.cuh"]
    kname = "mla_decode_kernel" if mla else "gqa_decode_kernel"
    tkey = kname + ("[fp8]" if fp8 else "")     # the FP8 instantiation has its own counters
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "traffic": ncu_traffic(tkey, kfile),
            "kernel": kname, "peak_source": f"{peak_src} hbm_gbs (copy, burst)",
            "algorithmic_bytes_per_launch": dec_alg, "avg_launch_us": dec_avg_ms * 1e3}
    extra = {}
    if mla:
        fl = mla_flops(case0)
        tf = fl / (dec_avg_ms * 1e-3) / 1e12
        t_hbm = dec_alg / (hbm_peak * 1e9)
        t_tc = fl / (bf16_peak * 1e12)
        extra["mla"] = {"tflops": tf, "tensor_frac_of_measured_bf16": tf / bf16_peak,
                        "binding": "hbm" if t_hbm >= t_tc else "tensor",
                        "frac_of_binding": max(t_hbm, t_tc) / (dec_avg_ms * 1e-3)}

    # ---- end to end through the public API with host buffers
    e2e = None
    if args.quick:
        args.no_cpu_baseline = True
    s = sets[0]
    c = s["case"]
    pin = lambda t: t.detach().to("cpu").pin_memory()
    host_in = [pin(t) for t in ((c.q_abs, c.q_rope) if mla else (c.q,))] + \
        [pin(t) for t in s["new"]] + [pin(s["pos"]), pin(c.seqlens)]
    dev_in = [t for t in ((c.q_abs, c.q_rope) if mla else (c.q,))] + list(s["new"]) + \
        [s["pos"], c.seqlens]
    host_out = torch.empty(s["out"].shape, dtype=s["out"].dtype).pin_memory()
    host_lse = torch.empty(s["lse"].shape, dtype=s["lse"].dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size() + host_lse.numel() * 4
    n_e2e = 0 if args.quick else max(10, min(args.steps, 500))

    def e2e_step():
        for hsrc, ddst in zip(host_in, dev_in):
            ddst.copy_(hsrc, non_blocking=True)
        rc = lib.kvdec_append_rope(ctypes.byref(s["ap"]), sptr)
        rc |= s["decode"](ctypes.byref(s["p"]), sptr)
        if rc:
            raise RuntimeError(lib.kvdec_last_error().decode())
        host_out.copy_(s["out"], non_blocking=True)
        host_lse.copy_(s["lse"], non_blocking=True)

    for _ in range(3 if n_e2e else 0):
        e2e_step()
    torch.cuda.synchronize()
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / max(n_e2e, 1), ws)
    e2e = None if not n_e2e else {"value": ws * (dec_bytes[0] + app_bytes) / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "steps": n_e2e, "note": "per-step inputs (q, new k/v, positions, seqlens) "
                                   "copied from pinned host memory, output read back; "
                                   "the KV cache stays resident"}

    if rank != 0:
        return
    cpu = None
    if fp8:
        cpu = {"value": None, "note": "no oracle timing for the FP8 cache line; the bf16 "
                                      "line of the same workload carries it"}
    elif not args.no_cpu_baseline:
        cpu = cpu_baseline(args.config, args.cpu_seconds)
    cfg = {"workload": WORKLOADS[args.config], "name": args.config,
           "l2": "inputs larger than L2 (KV bytes per step %.0f MB > 126 MB), two input sets "
                 "alternated" % (kv_bytes[0] / 1e6) if kv_bytes[0] > 2 * 126e6 else
                 "KV smaller than 2x L2: two input sets alternated, partly L2-resident",
           "kv_bytes_per_step": kv_bytes[0], "step": "append_rope + decode (fused split merge)",
           "kv_cache": "E4M3 bytes, per-KV-head fp32 scales" if fp8 else "bf16",
           "parallelism": f"replicas x{ws}"}
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "us_per_step": ms_per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8-e4m3 cache, f16 MMA" if fp8 else "bf16",
            "data": "synthetic", "config": cfg,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": 2 * args.steps,
            "append_us": 1e3 * sum(app_ms) / len(app_ms)}
    line.update(extra)
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
