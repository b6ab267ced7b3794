#!/usr/bin/env python
"""Benchmark: one decode step of the Gemma-4 global-layer workload over a packed
q8_0-K / TBQ3-V cache on one GB300, printed as one JSON line.

A step is the whole hot path for one new token: quantise and append the token's
K and V rows into the cache (kv_pack), then attention of the 16 query heads over
all 32768 cached tokens (attn_decode: split-K decode kernel + split merge with
the inverse transform). Inputs are resident in HBM when the timed region starts.
The packed cache (48.4 MB) is smaller than L2, so steps rotate over enough
copies of it to exceed 4x the L2 size; every step reads its cache from HBM.

--impl reference times the float64 oracle (dequantise to dense, then softmax
attention) on the host cores, on a bounded sample of the same workload.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "compressed-KV decode attn: tokens/s and effective HBM GB/s (% of GB300 peak)"
WORKLOAD = "gemma4_decode"
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic of one attn_decode_kernel<512> launch on this workload, from the
# ncu capture summarised in profiles/attn_decode_gemma4.md, valid for the source
# hash below (null once the kernel source changes).
NCU_TRAFFIC = {"bytes": None, "source_sha": None}


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _decode_source_sha():
    h = hashlib.sha256()
    for name in ("attn_decode.cu", "decode_common.cuh", "ckv_device.cuh"):
        with open(os.path.join(ROOT, "compressed_kv_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while work runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def mark(self):
        return time.time()

    def stop(self, t_begin, t_end):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        # nvidia-smi lines carry no timestamps: keep the samples taken while the
        # GPU was under load (clocks above idle), else all of them.
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        loaded = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows)}


# --------------------------------------------------------------------- ours --

def run_ours(args):
    import torch
    import compressed_kv_attention_gb300 as ckv
    from compressed_kv_attention_gb300 import inputs

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(dev)

    w = inputs.WORKLOADS[WORKLOAD]
    D, Hkv, Hq, T = w.head_dim, w.n_kv_heads, w.n_q_heads, w.seq_len
    outl = inputs.outlier_channels(D, w.n_outliers, w.seed)
    signs = inputs.tbq_signs(D)
    scale = 1.0 / math.sqrt(D)
    with torch.cuda.stream(stream):
        k = inputs.normal_tensor((1, T, Hkv, D), w.seed, "k", outl, device=str(dev))
        v = inputs.normal_tensor((1, T, Hkv, D), w.seed, "v", outl, device=str(dev))
        q = inputs.normal_tensor((1, 1, Hq, D), w.seed, "q", outl, device=str(dev))
        cache_b = ckv.cache_bytes(D, Hkv, 1, T)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n_rot = max(2, math.ceil(4 * l2 / cache_b))
        caches = [ckv.PackedCache(D, Hkv, 1, T, signs, device=dev) for _ in range(n_rot)]
        for c in caches:
            ckv.kv_pack(c, 0, k, v, stream=stream)
        k_new, v_new = k[:, T - 1:T].clone(), v[:, T - 1:T].clone()
        out = torch.empty((1, 1, Hq, D), dtype=torch.float32, device=dev)
        lse = torch.empty((1, 1, Hq), dtype=torch.float32, device=dev)
        ws = torch.empty(ckv.attn_decode_workspace(caches[0], T, 1, Hq), dtype=torch.uint8, device=dev)
        seq = torch.full((1,), T, dtype=torch.int32, device=dev)
    stream.synchronize()

    def step(c):
        ckv.kv_pack(c, T - 1, k_new, v_new, stream=stream)
        ckv.attn_decode(c, seq, T, q, scale, out, lse, ws, stream=stream)

    def decode_only(c):
        ckv.attn_decode(c, seq, T, q, scale, out, lse, ws, stream=stream)

    # Eager warm-up (configures kernel attributes before capture), then graphs.
    for c in caches:
        step(c)
    stream.synchronize()
    assert ckv.read_device_flag(ws, stream=stream) == 0
    reps = max(1, 128 // n_rot)
    big, single, dec_graph = torch.cuda.CUDAGraph(), [], torch.cuda.CUDAGraph()
    with torch.cuda.graph(big, stream=stream):
        for _ in range(reps):
            for c in caches:
                step(c)
    for c in caches:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(c)
        single.append(g)
    with torch.cuda.graph(dec_graph, stream=stream):
        for _ in range(reps):
            for c in caches:
                decode_only(c)
    per_big = reps * n_rot

    def run_steps(n):
        with torch.cuda.stream(stream):
            for _ in range(n // per_big):
                big.replay()
            for i in range(n % per_big):
                single[i % n_rot].replay()

    run_steps(max(args.warmup, 3))
    stream.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_begin = time.time()
    ev0.record(stream)
    run_steps(args.steps)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    ms = ev0.elapsed_time(ev1)
    if dist:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
        dist.barrier()

    # Dominant kernel alone: decode calls back to back (header reset + decode kernel).
    n_dec = max(1, (2000 // per_big)) * per_big
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(n_dec // per_big):
            dec_graph.replay()
    e1.record(stream)
    stream.synchronize()
    dec_ms = e0.elapsed_time(e1) / n_dec
    clocks = sampler.stop(t_begin, t_end)
    assert ckv.read_device_flag(ws, stream=stream) == 0

    # End to end through the public API with host buffers (pinned), eager calls.
    q_h = q.cpu().pin_memory()
    kn_h, vn_h = k_new.cpu().pin_memory(), v_new.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    q_d, kn_d, vn_d = torch.empty_like(q), torch.empty_like(k_new), torch.empty_like(v_new)
    n_e2e = min(args.steps, 2000)

    def e2e_step(i):
        c = caches[i % n_rot]
        q_d.copy_(q_h, non_blocking=True)
        kn_d.copy_(kn_h, non_blocking=True)
        vn_d.copy_(vn_h, non_blocking=True)
        ckv.kv_pack(c, T - 1, kn_d, vn_d, stream=stream)
        ckv.attn_decode(c, seq, T, q_d, scale, out, lse, ws, stream=stream)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(min(50, n_e2e)):
            e2e_step(i)
        stream.synchronize()
        t0 = time.perf_counter()
        for i in range(n_e2e):
            e2e_step(i)
        stream.synchronize()
        e2e_s = time.perf_counter() - t0
    h2d = (q.numel() * 2 + k_new.numel() * 2 + v_new.numel() * 2)
    d2h = out.numel() * 4 + lse.numel() * 4

    tokens_per_step = 1  # one new token per sequence per step (batch 1)
    value = world * tokens_per_step * args.steps / (ms / 1e3)
    kv_bytes = Hkv * T * inputs.compressed_bytes_per_token(D)
    peak, peak_kind = _peaks()
    achieved = kv_bytes / (dec_ms / 1e3) / 1e9
    traffic = NCU_TRAFFIC["bytes"] if NCU_TRAFFIC["source_sha"] == _decode_source_sha() else None
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 mma, f32 accumulate (int8 / 3-bit storage)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "head_dim": D, "n_kv_heads": Hkv, "n_q_heads": Hq, "batch": 1,
                   "cached_tokens": T, "n_q": 1, "step": "kv_pack(1 token) + attn_decode",
                   "l2": f"rotating {n_rot} cache copies ({n_rot * cache_b / 1e6:.0f} MB > 4x L2 "
                         f"{l2 / 1e6:.0f} MB)", "parallelism": f"replicas x{world}",
                   "timing": "CUDA graphs, events on the launching stream"},
        "effective_gbs": round(kv_bytes * world * args.steps / (ms / 1e3) / 1e9, 1),
        "roofline": {"bound": "hbm", "kernel": "attn_decode_kernel<512> (split-K decode with in-kernel split merge)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": traffic, "algorithmic_bytes": kv_bytes,
                     "launch_ms": round(dec_ms, 6)},
        "e2e": {"value": round(n_e2e / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": n_e2e, "api": "kv_pack + attn_decode, eager"},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(min_seconds=10.0)
    if dist:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ oracle --

def _oracle_setup(sample_tokens=None):
    import numpy as np
    from compressed_kv_attention_gb300 import inputs
    from tests import helpers as H
    w = inputs.WORKLOADS[WORKLOAD]
    D, Hkv, Hq, T = w.head_dim, w.n_kv_heads, w.n_q_heads, w.seq_len
    Ts = T if sample_tokens is None else sample_tokens
    outl = inputs.outlier_channels(D, w.n_outliers, w.seed)
    k = inputs.normal_tensor((Ts, Hkv, D), w.seed, "bench-oracle/k", outl)
    v = inputs.normal_tensor((Ts, Hkv, D), w.seed, "bench-oracle/v", outl)
    q = inputs.normal_tensor((1, Hq, D), w.seed, "bench-oracle/q", outl)
    signs = inputs.tbq_signs(D)
    qs, d16, codes, n16, _ = H.oracle_quantize(np.swapaxes(k, 0, 1), np.swapaxes(v, 0, 1), signs)
    return dict(D=D, Hkv=Hkv, Hq=Hq, T=T, Ts=Ts, q=q, k_new=k[-1:], v_new=v[-1:], signs=signs,
                qs=qs, d16=d16, codes=codes, n16=n16)


def _oracle_step(s):
    """Oracle decode step: quantise the new token, dequantise the cache to dense
    float64, softmax attention for every query head (decompress-then-attend)."""
    from oracle import ckv_oracle as O
    O.q8_0_quantize(s["k_new"])
    O.tbq3_quantize(s["v_new"], s["signs"])
    kh = O.q8_0_dequantize(s["qs"], s["d16"])
    vh = O.tbq3_dequantize(s["codes"], s["n16"], s["signs"])
    return O.decode_reference(s["q"], kh, vh, s["Ts"], 1.0 / math.sqrt(s["D"]))


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def cpu_baseline(min_seconds=10.0, max_seconds=30.0):
    s = _oracle_setup()
    n, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(s)
        n += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or el * (n + 1) / n > max_seconds:
            break
    return {"value": round(n / el, 4), "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
            "sample": f"{n} full decode steps of {WORKLOAD} (dequantise {s['T']} tokens x {s['Hkv']} kv "
                      f"heads to float64, attend 16 heads), numpy float64"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # Size each step's sample so that warm-up + timed steps take about 2 minutes:
    # a step attends over the first Ts tokens of the cache and its time is
    # scaled by T / Ts to a full step.
    cal = _oracle_setup(sample_tokens=1024)
    t0 = time.perf_counter()
    _oracle_step(cal)
    full_est = (time.perf_counter() - t0) * cal["T"] / cal["Ts"]
    per_step = 120.0 / max(1, args.steps + args.warmup)
    Ts = int(min(cal["T"], max(16, (cal["T"] * per_step / full_est) // 16 * 16)))
    s = _oracle_setup(sample_tokens=Ts)
    frac = s["Ts"] / s["T"]
    for _ in range(max(args.warmup, 0)):
        _oracle_step(s)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(s)
    el = (time.perf_counter() - t0) / frac
    value = args.steps / el
    sample = (f"each step: oracle decode (dequantise to float64 + attend 16 heads) over {s['Ts']} of "
              f"{s['T']} tokens of {WORKLOAD}, time scaled by {1 / frac:.2f}")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / max(args.steps, 1) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = _args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
