#!/usr/bin/env python
"""Benchmark of the compressed-KV attention hot path on one GB300: one JSON line.

Default workload (`gemma4_decode`): one decode step of a Gemma-4 global layer
over a packed q8_0-K / TBQ3-V cache, one call of attn_decode_append: the decode
kernel quantises the new token's K and V rows into the cache, then attends with
the 16 query heads over all 32768 cached tokens (split-K decode, in-kernel split
merge and inverse transform). Inputs are resident in HBM when the timed
region starts. Caches smaller than L2 are rotated over enough copies to exceed
4x the L2 size, so every step reads its cache from HBM.

Other workloads (`--workload`), one line each:
  long_decode      4 sequences x 262144 tokens, one decode step per sequence
  fanout_decode    one 4096-token compressed prefix read by 15 agents (a
                   120-row pass per kv head), a private 512-token fp16 tail per
                   agent, the two partials merged by log-sum-exp
  tiny_decode      1 kv head, 4 query heads, head_dim 128, 256 tokens
  verify_decode    a verify batch of 4 drafted tokens over 32768 tokens
  dca_decode       dual chunk attention decode, 32768 tokens, chunk 8192
  long_decode_tbq2, long_decode_tbq4, long_decode_rot
                   long_decode with 2- or 4-bit V codes, or with the
                   block-diagonal rotation (128-dim groups, two sign diagonals)
  chunked_prefill  2048 new query tokens over 32768 cached ones (pack the new
                   rows, causal attention on tcgen05); tensor roofline
  chunked_prefill_rot  the same over a cache with the block-diagonal rotation
  shared_prefill   15 agents prefill 128 tokens each over one 4096-token
                   compressed prefix plus their private 512-token fp16 tails
  kv_pack          packing 2048 tokens x 2 kv heads of fp16 K/V

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
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM traffic (read + write, bytes) of one step's kernels per workload, from
# one ncu capture of the bench's own workload; each figure holds only for the
# kernel sources whose hash is recorded beside it (null once they change).
# Fan-out and prefill: the sum over the step's kernels (their rooflines time the whole step).
NCU_TRAFFIC = {
    "gemma4_decode": {"bytes": 48518912, "source_sha": "13626d8ac99541f9"},
    "tiny_decode": {"bytes": 116736, "source_sha": "13626d8ac99541f9"},
    "long_decode": {"bytes": 1547972096 + 3602432, "source_sha": "13626d8ac99541f9"},
    "fanout_decode": {"bytes": 6405120 + 33743616, "source_sha": "c19b11ad11052ba4"},
    "chunked_prefill": {"bytes": 8451328 + (121211392 + 61330688) + (106605824 + 23828736),
                        "source_sha": "ae568074c9611238"},
}

_DECODE_SOURCES = ("attn_decode.cu", "attn_decode_kernel.cuh", "decode_common.cuh", "ckv_device.cuh",
                   "ckv_kernels.cuh", "pack_common.cuh")
_SOURCES = {
    "decode": _DECODE_SOURCES,
    "fanout": _DECODE_SOURCES + ("attn_decode_f16.cu", "lse_merge.cu", "attn_prefill.cu", "ckv_api.cu"),
    "prefill": ("attn_prefill.cu", "kv_pack.cu", "pack_common.cuh", "ckv_device.cuh", "ckv_kernels.cuh",
                "ckv_api.cu"),
}


def _source_sha(kind):
    h = hashlib.sha256()
    for name in _SOURCES[kind]:
        with open(os.path.join(ROOT, "compressed_kv_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kind):
    """The recorded ncu DRAM traffic of one step of `workload`, or None when
    none is recorded for the current sources."""
    rec = NCU_TRAFFIC.get(workload)
    if rec and rec["source_sha"] == _source_sha(kind):
        return rec["bytes"]
    return None


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=None,
                   help="ranks (one GPU each); without WORLD_SIZE in the environment, N > 1 starts N ranks")
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="gemma4_decode",
                   choices=["gemma4_decode", "long_decode", "fanout_decode", "tiny_decode", "chunked_prefill",
                            "kv_pack", "verify_decode", "dca_decode", "long_decode_tbq2", "long_decode_tbq4",
                            "long_decode_rot", "shared_prefill", "chunked_prefill_rot"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-config", action="store_true", help="skip the other workloads' figures")
    return p.parse_args()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while work runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu, self.proc, self.path = gpu_index, None, None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
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
        # Lines carry no timestamps: keep the samples taken under load (clocks
        # above half of the highest seen).
        loaded = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def _timed(stream, fn, n):
    """Run fn() n times on `stream`; elapsed ms from CUDA events recorded on that stream."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1)


# -------------------------------------------------------------- workloads --

class DecodeWork:
    """Decode workloads: a step is attn_decode_append of one new token per sequence, or (n_q > 1)
    attn_decode_verify of a batch of n_q drafted tokens already in the cache."""

    graph = True

    def __init__(self, name, dev, stream):
        import torch
        import compressed_kv_attention_gb300 as ckv
        from compressed_kv_attention_gb300 import inputs
        self.ckv, self.torch, self.stream = ckv, torch, stream
        w = inputs.WORKLOADS[name]
        self.w = w
        D, Hkv, Hq, T, B = w.head_dim, w.n_kv_heads, w.n_q_heads, w.seq_len, w.batch
        self.D, self.T, self.B, self.Hq, self.Hkv = D, T, B, Hq, Hkv
        self.n_q = w.n_q
        self.dca = w.dca_chunk  # dual chunk attention: three regime queries, one output token
        self.v_bits = w.v_bits
        self.dtype = f"f16 mma, f32 accumulate (int8 / {w.v_bits}-bit storage)"
        self.rot = w.rot_group
        outl = inputs.outlier_channels(D, w.n_outliers, w.seed)
        signs = inputs.tbq_signs(D)
        self.scale = 1.0 / math.sqrt(D)
        with torch.cuda.stream(stream):
            k = inputs.normal_tensor((B, T, Hkv, D), w.seed, "k", outl, device=str(dev))
            v = inputs.normal_tensor((B, T, Hkv, D), w.seed, "v", outl, device=str(dev))
            self.q = inputs.normal_tensor((B, 3 if self.dca else self.n_q, Hq, D), w.seed, "q", outl,
                                          device=str(dev))
            self.cache_bytes = ckv.cache_bytes(D, Hkv, B, T, w.v_bits, w.rot_group)
            signs2 = inputs.tbq_signs(D, seed=43) if w.rot_group else None
            self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
            self.n_rot = max(2, math.ceil(4 * self.l2 / self.cache_bytes))
            self.caches = [ckv.PackedCache(D, Hkv, B, T, signs, device=dev, v_bits=w.v_bits, signs2=signs2)
                           for _ in range(self.n_rot)]
            for c in self.caches:
                ckv.kv_pack(c, 0, k, v, stream=stream)
            self.k_new, self.v_new = k[:, T - 1:T].clone(), v[:, T - 1:T].clone()
            del k, v
            # out and lse live in one allocation, so that a step's result comes back in one copy
            n_out = B * self.n_q * Hq * D
            self.out_lse = torch.empty(n_out + B * self.n_q * Hq, dtype=torch.float32, device=dev)
            self.out = self.out_lse[:n_out].view(B, self.n_q, Hq, D)
            self.lse = self.out_lse[n_out:].view(B, self.n_q, Hq)
            ws_bytes = (ckv.attn_decode_dca_workspace(self.caches[0], T, Hq) if self.dca else
                        ckv.attn_decode_workspace(self.caches[0], T, self.n_q, Hq))
            self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
            self.seq = torch.full((B,), T, dtype=torch.int32, device=dev)
        stream.synchronize()
        self.tokens_per_step = B * self.n_q
        # the decode kernel (packs the new token or runs the batch, merges splits); DCA with 8 query heads
        # per kv head merges its regimes inside the same launch (co-resident grid), otherwise in a second
        self.launches_per_step = 2 if (self.dca and Hq != 8 * Hkv) else 1
        self.algo_bytes = B * Hkv * T * inputs.compressed_bytes_per_token(D, w.v_bits, w.rot_group)

    def step(self, i):
        c = self.caches[i % self.n_rot]
        if self.dca:
            self.ckv.attn_decode_dca(c, self.seq, self.T, self.dca, self.q, self.scale, self.out, self.lse, self.ws,
                                     stream=self.stream)
        elif self.n_q > 1:
            self.ckv.attn_decode_verify(c, self.seq, self.T, self.q, self.scale, self.out, self.lse, self.ws,
                                        stream=self.stream)
        else:
            self.ckv.attn_decode_append(c, self.seq, self.T, self.k_new, self.v_new, self.q, self.scale, self.out,
                                        self.lse, self.ws, stream=self.stream)


    def check(self):
        assert self.ckv.read_device_flag(self.ws, stream=self.stream) == 0

    def e2e_setup(self):
        t = self.torch
        if not (self.n_q > 1 or self.dca):
            # An append step through the C ABI entry that takes host buffers: Q and the new K/V rows
            # (pinned) in, out and lse back, the copies on the stream inside the call.
            self.h_q = self.q.cpu().pin_memory()
            self.h_k, self.h_v = self.k_new.cpu().pin_memory(), self.v_new.cpu().pin_memory()
            self.h_o = t.empty(self.out.shape, dtype=t.float32).pin_memory()
            self.h_l = t.empty(self.lse.shape, dtype=t.float32).pin_memory()
            self.e2e_api = ("C ABI ckv_attn_decode_append_host: pinned host buffers read and written by the "
                            "kernel across NVLink-C2C, no staging copies")
            return (sum(x.numel() * 2 for x in (self.h_q, self.h_k, self.h_v)),
                    self.h_o.numel() * 4 + self.h_l.numel() * 4)
        self.e2e_api = "public Python API, eager (torch copies)"
        # A verify batch or a DCA step sends only Q; an append sends Q and the new K/V row. The step's
        # inputs sit in one pinned buffer and one device buffer (views), so they go over in one copy,
        # and the result (out, lse) comes back in one.
        ins = (self.q,) if (self.n_q > 1 or self.dca) else (self.q, self.k_new, self.v_new)
        n_in = sum(x.numel() for x in ins)
        self.h_in = t.empty(n_in, dtype=t.float16).pin_memory()
        self.d_in_flat = t.empty(n_in, dtype=t.float16, device=self.q.device)
        self.d_in, o = [], 0
        for x in ins:
            self.h_in[o:o + x.numel()].copy_(x.reshape(-1).cpu())
            self.d_in.append(self.d_in_flat[o:o + x.numel()].view(x.shape))
            o += x.numel()
        self.h_out = t.empty(self.out_lse.shape, dtype=t.float32).pin_memory()
        return n_in * 2, self.out_lse.numel() * 4

    def e2e_step(self, i):
        c = self.caches[i % self.n_rot]
        if not (self.n_q > 1 or self.dca):
            self.ckv.attn_decode_append_host(c, self.seq, self.T, self.h_k, self.h_v, self.h_q, self.scale, self.h_o,
                                             self.h_l, self.ws, stream=self.stream)
            return
        self.d_in_flat.copy_(self.h_in, non_blocking=True)
        if self.dca:
            self.ckv.attn_decode_dca(c, self.seq, self.T, self.dca, self.d_in[0], self.scale, self.out, self.lse,
                                     self.ws, stream=self.stream)
        elif self.n_q > 1:
            self.ckv.attn_decode_verify(c, self.seq, self.T, self.d_in[0], self.scale, self.out, self.lse, self.ws,
                                        stream=self.stream)
        else:
            self.ckv.attn_decode_append(c, self.seq, self.T, self.d_in[1], self.d_in[2], self.d_in[0], self.scale,
                                        self.out, self.lse, self.ws, stream=self.stream)
        self.h_out.copy_(self.out_lse, non_blocking=True)

    def describe(self):
        return {"workload": self.w.name, "head_dim": self.D, "n_kv_heads": self.Hkv, "n_q_heads": self.Hq,
                "batch": self.B, "cached_tokens": self.T, "n_q": self.n_q, "v_bits": self.v_bits,
                "rotation": "128-dim groups, two sign diagonals" if self.rot else "full D-point, one sign diagonal",
                "step": (f"attn_decode_dca (chunk {self.dca}: intra, successive and inter regimes + merge)"
                         if self.dca else
                         "attn_decode_verify (a batch of n_q drafted tokens, causal among them)" if self.n_q > 1
                         else "attn_decode_append (pack 1 new token per sequence in-kernel, then attend)"),
                "l2": f"rotating {self.n_rot} cache copies ({self.n_rot * self.cache_bytes / 1e6:.0f} MB > 4x L2 "
                      f"{self.l2 / 1e6:.0f} MB)"}

    def roofline(self, kernel_ms, peaks):
        hbm, _, kind = peaks
        achieved = self.algo_bytes / (kernel_ms / 1e3) / 1e9
        traffic = ncu_traffic(self.w.name, "decode")
        what = ("DCA regimes as three query rows" if self.dca else
                "verify batch, per-row causal limits" if self.n_q > 1 else "append")
        return {"bound": "hbm",
                "kernel": f"attn_decode_kernel<{self.D}, {self.v_bits}> ({what} + split-K decode + in-kernel merge)",
                "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "peak_kind": kind, "traffic": traffic, "algorithmic_bytes": self.algo_bytes,
                "launch_ms": round(kernel_ms, 6)}


class FanoutWork:
    """Shared-prefix fan-out: attn_decode_fanout, the prefix decode (15 agents as 15 query tokens) writing its
    split partials and the fp16 tails' decode, beside it, whose split merge takes them in."""

    graph = True

    def __init__(self, dev, stream):
        import torch
        import compressed_kv_attention_gb300 as ckv
        from compressed_kv_attention_gb300 import inputs
        self.ckv, self.torch, self.stream = ckv, torch, stream
        w = inputs.WORKLOADS["fanout_decode"]
        self.w = w
        D, Hkv, Hq, P, A, TL = w.head_dim, w.n_kv_heads, w.n_q_heads, w.seq_len, w.n_agents, w.tail_len
        self.D, self.Hkv, self.Hq, self.P, self.A, self.TL = D, Hkv, Hq, P, A, TL
        outl = inputs.outlier_channels(D, w.n_outliers, w.seed)
        signs = inputs.tbq_signs(D)
        self.scale = 1.0 / math.sqrt(D)
        with torch.cuda.stream(stream):
            k = inputs.normal_tensor((1, P, Hkv, D), w.seed, "prefix/k", outl, device=str(dev))
            v = inputs.normal_tensor((1, P, Hkv, D), w.seed, "prefix/v", outl, device=str(dev))
            self.qa = inputs.normal_tensor((A, Hq, D), w.seed, "agents/q", outl, device=str(dev))
            self.per_copy = ckv.cache_bytes(D, Hkv, 1, P) + 2 * A * Hkv * TL * D * 2
            self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
            self.n_rot = max(2, math.ceil(4 * self.l2 / self.per_copy))
            self.caches, self.tails = [], []
            for _ in range(self.n_rot):
                c = ckv.PackedCache(D, Hkv, 1, P, signs, device=dev)
                ckv.kv_pack(c, 0, k, v, stream=stream)
                self.caches.append(c)
                kt = inputs.normal_tensor((A, Hkv, TL, D), w.seed, "tail/k", outl, device=str(dev))
                vt = inputs.normal_tensor((A, Hkv, TL, D), w.seed, "tail/v", outl, device=str(dev))
                self.tails.append((kt, vt))
            self.out = torch.empty((A, Hq, D), dtype=torch.float32, device=dev)
            self.lse = torch.empty((A, Hq), dtype=torch.float32, device=dev)
            # The split counts the step uses: the tail pass runs beside the prefix pass and merges its partials.
            self.ps, self.ts = ckv.fanout_plan(A, Hkv, Hq)
            self.ws = torch.zeros(ckv.attn_decode_fanout_workspace(self.caches[0], P, A, TL, Hq), dtype=torch.uint8,
                                  device=dev)
            self.seq_p = torch.full((1,), P, dtype=torch.int32, device=dev)
            self.seq_t = torch.full((A,), TL, dtype=torch.int32, device=dev)
        stream.synchronize()
        self.tokens_per_step = A
        self.launches_per_step = 2  # prefix decode (split partials), tail decode merging them
        self.algo_bytes = Hkv * P * inputs.compressed_bytes_per_token(D) + 2 * A * Hkv * TL * D * 2

    def _run(self, i, qa):
        ckv, s = self.ckv, self.stream
        c, (kt, vt) = self.caches[i % self.n_rot], self.tails[i % self.n_rot]
        ckv.attn_decode_fanout(c, self.seq_p, self.P, kt, vt, self.seq_t, self.TL, qa, self.scale, self.out, self.lse,
                               self.ws, stream=s)

    def step(self, i):
        self._run(i, self.qa)


    def check(self):
        assert self.ckv.read_device_flag(self.ws, stream=self.stream) == 0

    def e2e_setup(self):
        t = self.torch
        self.h_q = self.qa.cpu().pin_memory()
        self.d_q = t.empty_like(self.qa)
        self.h_out = [t.empty(x.shape, dtype=x.dtype).pin_memory() for x in (self.out, self.lse)]
        return self.h_q.numel() * 2, sum(x.numel() * 4 for x in self.h_out)

    def e2e_step(self, i):
        self.d_q.copy_(self.h_q, non_blocking=True)
        self._run(i, self.d_q)
        self.h_out[0].copy_(self.out, non_blocking=True)
        self.h_out[1].copy_(self.lse, non_blocking=True)

    def describe(self):
        return {"workload": "fanout_decode", "head_dim": self.D, "n_kv_heads": self.Hkv, "n_q_heads": self.Hq,
                "agents": self.A, "prefix_tokens": self.P, "tail_tokens": self.TL,
                "step": "attn_decode_fanout (prefix decode of the 15 agents writing split partials; fp16 tail "
                        "decode beside it, merging them)",
                "splits": {"prefix": self.ps, "tails": self.ts, "from": "ckv_fanout_plan"},
                "l2": f"rotating {self.n_rot} copies ({self.n_rot * self.per_copy / 1e6:.0f} MB > 4x L2)"}

    def roofline(self, kernel_ms, peaks):
        hbm, _, kind = peaks
        achieved = self.algo_bytes / (kernel_ms / 1e3) / 1e9
        return {"bound": "hbm", "kernel": "attn_decode_fanout: prefix decode (split partials) + fp16 tail decode "
                "merging them (whole step)",
                "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "peak_kind": kind, "traffic": ncu_traffic("fanout_decode", "fanout"), "algorithmic_bytes": self.algo_bytes,
                "launch_ms": round(kernel_ms, 6)}


class PrefillWork:
    """Chunked prefill: attn_prefill packs 2048 new rows and attends causally (tcgen05)."""

    graph = False  # long steps: launched eagerly, L2 flushed before each timed step

    def __init__(self, name, dev, stream):
        import torch
        import compressed_kv_attention_gb300 as ckv
        from compressed_kv_attention_gb300 import inputs
        self.ckv, self.torch, self.stream = ckv, torch, stream
        w = inputs.WORKLOADS[name]
        self.w, self.name = w, name
        D, Hkv, Hq, nc, nn = w.head_dim, w.n_kv_heads, w.n_q_heads, w.seq_len, w.n_new
        self.D, self.Hkv, self.Hq, self.nc, self.nn = D, Hkv, Hq, nc, nn
        outl = inputs.outlier_channels(D, w.n_outliers, w.seed)
        self.scale = 1.0 / math.sqrt(D)
        with torch.cuda.stream(stream):
            k = inputs.normal_tensor((1, nc + nn, Hkv, D), w.seed, "k", outl, device=str(dev))
            v = inputs.normal_tensor((1, nc + nn, Hkv, D), w.seed, "v", outl, device=str(dev))
            self.q = inputs.normal_tensor((1, nn, Hq, D), w.seed, "q", outl, device=str(dev), dtype="bfloat16")
            signs2 = inputs.tbq_signs(D, seed=43) if w.rot_group else None
            self.cache = ckv.PackedCache(D, Hkv, 1, nc + nn, inputs.tbq_signs(D), device=dev, v_bits=w.v_bits,
                                         signs2=signs2)
            ckv.kv_pack(self.cache, 0, k[:, :nc].contiguous(), v[:, :nc].contiguous(), stream=stream)
            self.kn, self.vn = k[:, nc:].contiguous(), v[:, nc:].contiguous()
            del k, v
            self.out = torch.empty((1, nn, Hq, D), dtype=torch.float32, device=dev)
            self.lse = torch.empty((1, nn, Hq), dtype=torch.float32, device=dev)
            self.ws = torch.zeros(ckv.attn_prefill_workspace(self.cache, nn, Hq), dtype=torch.uint8, device=dev)
            self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
            self.flush = torch.empty(2 * self.l2, dtype=torch.uint8, device=dev)
        stream.synchronize()
        self.tokens_per_step = nn
        self.launches_per_step = 3  # pack, prefill, de-rotation
        # QK^T and PV over the causal key range: query i sees nc + i + 1 keys.
        self.flops = 2 * 2 * Hq * D * (nn * nc + nn * (nn + 1) // 2)

    def step(self, i):
        self.ckv.attn_prefill(self.cache, self.nc, self.q, self.kn, self.vn, self.scale, self.out, self.lse,
                              self.ws, stream=self.stream)


    def between(self):
        with self.torch.cuda.stream(self.stream):
            self.flush.fill_(1)

    def check(self):
        assert self.ckv.read_device_flag(self.ws, stream=self.stream) == 0

    def e2e_setup(self):
        t = self.torch
        self.h_in = [x.cpu().pin_memory() for x in (self.q, self.kn, self.vn)]
        self.d_in = [t.empty_like(x) for x in (self.q, self.kn, self.vn)]
        self.h_out = [t.empty(x.shape, dtype=x.dtype).pin_memory() for x in (self.out, self.lse)]
        return (sum(x.numel() * x.element_size() for x in self.h_in),
                sum(x.numel() * x.element_size() for x in self.h_out))

    def e2e_step(self, i):
        for h, d in zip(self.h_in, self.d_in):
            d.copy_(h, non_blocking=True)
        self.ckv.attn_prefill(self.cache, self.nc, self.d_in[0], self.d_in[1], self.d_in[2], self.scale,
                              self.out, self.lse, self.ws, stream=self.stream)
        self.h_out[0].copy_(self.out, non_blocking=True)
        self.h_out[1].copy_(self.lse, non_blocking=True)

    def describe(self):
        return {"workload": self.name, "head_dim": self.D, "n_kv_heads": self.Hkv, "n_q_heads": self.Hq,
                "cached_tokens": self.nc, "new_tokens": self.nn, "q_dtype": "bf16", "v_bits": self.w.v_bits,
                "rotation": "128-dim groups, two sign diagonals" if self.w.rot_group else "full D-point",
                "step": "attn_prefill (pack 2048 rows + causal attention + de-rotation)",
                "l2": f"flushed before each step ({2 * self.l2 / 1e6:.0f} MB write)"}

    def roofline(self, kernel_ms, peaks):
        _, tf, kind = peaks
        achieved = self.flops / (kernel_ms / 1e3) / 1e12
        kern = f"attn_prefill_kernel<{self.D}, {self.w.v_bits}, {bool(self.w.rot_group)}>"
        return {"bound": "tensor", "kernel": kern + " (+ pack, de-rotation) on tcgen05",
                "achieved": round(achieved, 1), "peak": tf, "unit": "TFLOP/s", "frac": round(achieved / tf, 4),
                "peak_kind": kind + " bf16 dense (fp16 operands run at the same rate)", "traffic": ncu_traffic(self.name, "prefill"),
                "algorithmic_flops": self.flops, "launch_ms": round(kernel_ms, 6)}


class SharedPrefillWork:
    """Multi-tenant prefill: 15 agents prefill 128 tokens each over one shared compressed prefix
    (tcgen05, prefix-only) and their private fp16 tails (causal), merged exactly."""

    graph = False  # ~1 ms steps: launched eagerly, L2 flushed before each timed step

    def __init__(self, dev, stream):
        import torch
        import compressed_kv_attention_gb300 as ckv
        from compressed_kv_attention_gb300 import inputs
        self.ckv, self.torch, self.stream = ckv, torch, stream
        w = inputs.WORKLOADS["shared_prefill"]
        self.w = w
        D, Hkv, Hq, P, A, TL, n = w.head_dim, w.n_kv_heads, w.n_q_heads, w.seq_len, w.n_agents, w.tail_len, w.n_new
        self.D, self.Hkv, self.Hq, self.P, self.A, self.TL, self.n = D, Hkv, Hq, P, A, TL, n
        outl = inputs.outlier_channels(D, w.n_outliers, w.seed)
        self.scale = 1.0 / math.sqrt(D)
        cap = TL + n
        with torch.cuda.stream(stream):
            k = inputs.normal_tensor((1, P, Hkv, D), w.seed, "prefix/k", outl, device=str(dev))
            v = inputs.normal_tensor((1, P, Hkv, D), w.seed, "prefix/v", outl, device=str(dev))
            self.cache = ckv.PackedCache(D, Hkv, 1, P, inputs.tbq_signs(D), device=dev)
            ckv.kv_pack(self.cache, 0, k, v, stream=stream)
            del k, v
            self.kt = inputs.normal_tensor((A, Hkv, cap, D), w.seed, "tail/k", outl, device=str(dev))
            self.vt = inputs.normal_tensor((A, Hkv, cap, D), w.seed, "tail/v", outl, device=str(dev))
            self.kn = inputs.normal_tensor((A, n, Hkv, D), w.seed, "new/k", outl, device=str(dev))
            self.vn = inputs.normal_tensor((A, n, Hkv, D), w.seed, "new/v", outl, device=str(dev))
            self.q = inputs.normal_tensor((A, n, Hq, D), w.seed, "new/q", outl, device=str(dev), dtype="bfloat16")
            self.tail_len = torch.full((A,), cap, dtype=torch.int32, device=dev)
            self.out = torch.empty((A, n, Hq, D), dtype=torch.float32, device=dev)
            self.lse = torch.empty((A, n, Hq), dtype=torch.float32, device=dev)
            self.ws = torch.zeros(ckv.attn_prefill_shared_workspace(self.cache, A, cap, n, Hq), dtype=torch.uint8,
                                  device=dev)
            self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
            self.flush = torch.empty(2 * self.l2, dtype=torch.uint8, device=dev)
        stream.synchronize()
        self.tokens_per_step = A * n
        self.launches_per_step = 4  # tail append, prefix prefill, de-rotation, tail prefill with the merge
        # QK^T and PV: every query row sees the P prefix keys and TL + i + 1 tail keys.
        self.flops = 2 * 2 * Hq * D * A * (n * P + n * TL + n * (n + 1) // 2)

    def step(self, i):
        self.ckv.attn_prefill_shared(self.cache, self.P, self.kt, self.vt, self.tail_len, self.q, self.kn, self.vn,
                                     self.scale, self.out, self.lse, self.ws, stream=self.stream)


    def between(self):
        with self.torch.cuda.stream(self.stream):
            self.flush.fill_(1)

    def check(self):
        assert self.ckv.read_device_flag(self.ws, stream=self.stream) == 0

    def e2e_setup(self):
        t = self.torch
        self.h_in = [x.cpu().pin_memory() for x in (self.q, self.kn, self.vn)]
        self.d_in = [t.empty_like(x) for x in (self.q, self.kn, self.vn)]
        self.h_out = [t.empty(x.shape, dtype=x.dtype).pin_memory() for x in (self.out, self.lse)]
        return (sum(x.numel() * x.element_size() for x in self.h_in),
                sum(x.numel() * x.element_size() for x in self.h_out))

    def e2e_step(self, i):
        for h, d in zip(self.h_in, self.d_in):
            d.copy_(h, non_blocking=True)
        self.ckv.attn_prefill_shared(self.cache, self.P, self.kt, self.vt, self.tail_len, self.d_in[0],
                                     self.d_in[1], self.d_in[2], self.scale, self.out, self.lse, self.ws,
                                     stream=self.stream)
        self.h_out[0].copy_(self.out, non_blocking=True)
        self.h_out[1].copy_(self.lse, non_blocking=True)

    def describe(self):
        return {"workload": "shared_prefill", "head_dim": self.D, "n_kv_heads": self.Hkv, "n_q_heads": self.Hq,
                "agents": self.A, "prefix_tokens": self.P, "tail_tokens": self.TL, "new_tokens_per_agent": self.n,
                "q_dtype": "bf16",
                "step": "attn_prefill_shared (tail append + prefix-only tcgen05 prefill + causal fp16 tail "
                        "prefill with the prefix partial merged in)",
                "l2": f"flushed before each step ({2 * self.l2 / 1e6:.0f} MB write)"}

    def roofline(self, kernel_ms, peaks):
        _, tf, kind = peaks
        achieved = self.flops / (kernel_ms / 1e3) / 1e12
        return {"bound": "tensor", "kernel": "attn_prefill_shared (whole step; tcgen05 prefix prefill + mma.sync "
                "fp16 tail prefill)", "achieved": round(achieved, 1), "peak": tf, "unit": "TFLOP/s",
                "frac": round(achieved / tf, 4),
                "peak_kind": kind + " bf16 dense (fp16 operands run at the same rate)", "traffic": None,
                "algorithmic_flops": self.flops, "launch_ms": round(kernel_ms, 6)}


class PackWork:
    """kv_pack of 2048 tokens x 2 kv heads (the size of one prefill chunk)."""

    graph = True

    def __init__(self, dev, stream):
        import torch
        import compressed_kv_attention_gb300 as ckv
        from compressed_kv_attention_gb300 import inputs
        self.ckv, self.torch, self.stream = ckv, torch, stream
        w = inputs.WORKLOADS["chunked_prefill"]
        D, Hkv, n = w.head_dim, w.n_kv_heads, w.n_new
        self.D, self.Hkv, self.n = D, Hkv, n
        outl = inputs.outlier_channels(D, w.n_outliers, w.seed)
        with torch.cuda.stream(stream):
            self.k = inputs.normal_tensor((1, n, Hkv, D), w.seed, "k", outl, device=str(dev))
            self.v = inputs.normal_tensor((1, n, Hkv, D), w.seed, "v", outl, device=str(dev))
            self.per = ckv.cache_bytes(D, Hkv, 1, n) + 2 * self.k.numel() * 2
            self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
            self.n_rot = max(2, math.ceil(4 * self.l2 / self.per))
            self.caches = [ckv.PackedCache(D, Hkv, 1, n, inputs.tbq_signs(D), device=dev) for _ in range(self.n_rot)]
            self.ins = [(self.k.clone(), self.v.clone()) for _ in range(self.n_rot)]
        stream.synchronize()
        self.tokens_per_step = n
        self.launches_per_step = 1
        self.algo_bytes = 2 * n * Hkv * D * 2 + n * Hkv * inputs.compressed_bytes_per_token(D)

    def step(self, i):
        k, v = self.ins[i % self.n_rot]
        self.ckv.kv_pack(self.caches[i % self.n_rot], 0, k, v, stream=self.stream)


    def check(self):
        pass

    def e2e_setup(self):
        t = self.torch
        self.h_in = [x.cpu().pin_memory() for x in (self.k, self.v)]
        self.d_in = [t.empty_like(x) for x in (self.k, self.v)]
        return sum(x.numel() * 2 for x in self.h_in), 0

    def e2e_step(self, i):
        for h, d in zip(self.h_in, self.d_in):
            d.copy_(h, non_blocking=True)
        self.ckv.kv_pack(self.caches[i % self.n_rot], 0, self.d_in[0], self.d_in[1], stream=self.stream)

    def describe(self):
        return {"workload": "kv_pack", "head_dim": self.D, "n_kv_heads": self.Hkv, "tokens": self.n,
                "step": "kv_pack of 2048 tokens (q8_0 K + TBQ3 V)",
                "l2": f"rotating {self.n_rot} input/cache copies ({self.n_rot * self.per / 1e6:.0f} MB > 4x L2)"}

    def roofline(self, kernel_ms, peaks):
        hbm, _, kind = peaks
        achieved = self.algo_bytes / (kernel_ms / 1e3) / 1e9
        return {"bound": "hbm", "kernel": f"kv_pack_kernel<{self.D}>", "achieved": round(achieved, 1),
                "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4), "peak_kind": kind,
                "traffic": None, "algorithmic_bytes": self.algo_bytes, "launch_ms": round(kernel_ms, 6)}


def _make_work(name, dev, stream):
    if name in ("gemma4_decode", "long_decode", "tiny_decode", "verify_decode", "dca_decode", "long_decode_tbq2",
                "long_decode_tbq4", "long_decode_rot"):
        return DecodeWork(name, dev, stream)
    if name == "fanout_decode":
        return FanoutWork(dev, stream)
    if name in ("chunked_prefill", "chunked_prefill_rot"):
        return PrefillWork(name, dev, stream)
    if name == "shared_prefill":
        return SharedPrefillWork(dev, stream)
    return PackWork(dev, stream)


# --------------------------------------------------------------------- ours --

def max_over_ranks(values, dist=None, device="cpu"):
    """Each timing's largest value over all ranks: the replica that finishes
    last sets the whole job's time. Without a process group, the values."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def _graph_runner(work, stream, steps):
    """CUDA graphs for `steps` back-to-back steps: one graph of per_big steps
    replayed steps // per_big times, and one graph of the remaining steps, so
    that a timed run of `steps` steps has at most a few graph-launch gaps."""
    import torch
    n_rot = getattr(work, "n_rot", 1)
    reps = max(1, 128 // n_rot)
    per_big = reps * n_rot
    big = None
    if steps >= per_big:
        big = torch.cuda.CUDAGraph()
        with torch.cuda.graph(big, stream=stream):
            for i in range(per_big):
                work.step(i)
    rem, tail = steps % per_big, None
    if rem:
        tail = torch.cuda.CUDAGraph()
        with torch.cuda.graph(tail, stream=stream):
            for i in range(rem):
                work.step(i)

    def run():
        with torch.cuda.stream(stream):
            for _ in range(steps // per_big):
                big.replay()
            if tail is not None:
                tail.replay()
    return run


def measure(work, stream, dev, steps, warmup, dist=None):
    """Time `steps` steps of `work` (after `warmup`), on the device with CUDA
    events on the launching stream, bracketed by a barrier and a synchronize on
    both sides; returns the whole timed region in ms (max over ranks)."""
    import torch
    n_rot = getattr(work, "n_rot", 1)
    # Eager warm-up (configures kernel attributes before any capture).
    with torch.cuda.stream(stream):
        for i in range(max(n_rot, 2)):
            work.step(i)
    stream.synchronize()
    work.check()
    if work.graph:
        # Warm-up replays the timed graph itself (at least max(warmup, 3) steps), so that
        # the timed replay is not the graph's first (its upload would land in the timing).
        run = _graph_runner(work, stream, steps)
        for _ in range(-(-max(warmup, 3) // steps)):
            run()
        stream.synchronize()
    else:
        with torch.cuda.stream(stream):
            for i in range(max(warmup, 3)):
                work.between()
                work.step(i)
        stream.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if work.graph:
        ms = _timed(stream, run, 1)
    else:
        ms = 0.0
        for i in range(steps):
            work.between()
            ms += _timed(stream, lambda: work.step(i), 1)
    torch.cuda.synchronize(dev)
    if dist:
        (ms,) = max_over_ranks([ms], dist, dev)
        dist.barrier()
    work.check()
    return ms


def _graph_time_ms(fn, stream, n):
    """ms per call of fn(i), n calls back to back in one CUDA graph (after 3 eager calls)."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(3):
            fn(i)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn(i)
        g.replay()
        stream.synchronize()
    return _timed(stream, g.replay, 1) / n


def stream_floor(work, stream, dev, n=2000):
    """The decode's data movement alone on the same cache copies (ckv_calibrate_stream):
    the same split grid and staging, no compute; then with the split rendezvous."""
    import torch
    ckv = work.ckv
    n_tiles = work.T // 16
    streams = work.B * work.Hkv
    rec = work.cache_bytes // (streams * n_tiles)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    n_split = max(1, min(sms // streams, n_tiles // 4))
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    res = {"n_split": n_split, "record_bytes": rec}
    for key, rv in (("stream_us", 0), ("stream_rendezvous_us", 1)):
        ms = _graph_time_ms(lambda i: ckv.calibrate_stream(work.caches[i % work.n_rot].data, n_tiles, rec, streams,
                                                           n_split, rv, ws, stream=stream), stream, n)
        res[key] = round(ms * 1e3, 3)
    assert ckv.read_device_flag(ws, stream=stream) == 0
    return res


# Other single-GPU workloads measured in the same run as the headline (steps, warm-up).
PER_CONFIG = (("tiny_decode", 2000, 100), ("fanout_decode", 1000, 50), ("long_decode", 200, 10),
              ("chunked_prefill", 5, 3))


def per_config_lines(dev, stream, peaks):
    """ms per step, roofline fraction and ncu traffic of each other workload."""
    import torch
    res = {}
    for name, steps, warm in PER_CONFIG:
        work = _make_work(name, dev, stream)
        ms = measure(work, stream, dev, steps, warm)
        rl = work.roofline(ms / steps, peaks)
        res[name] = {"ms_per_step": round(ms / steps, 6), "steps": steps,
                     "tokens_per_s": round(work.tokens_per_step * steps / (ms / 1e3), 1),
                     "bound": rl["bound"], "achieved": rl["achieved"], "unit": rl["unit"], "frac": rl["frac"],
                     "traffic": rl["traffic"], "kernel": rl["kernel"]}
        del work
        torch.cuda.empty_cache()
    return res


def run_ours(args):
    import torch

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        sys.stderr.write(f"bench.py: rank {rank} of {world}: no CUDA device\n")
        sys.exit(3)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(dev)
    work = _make_work(args.workload, dev, stream)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ms = measure(work, stream, dev, args.steps, args.warmup, dist)
    clocks = sampler.stop()

    # End to end through the public API with pinned host buffers, eager calls.
    h2d, d2h = work.e2e_setup()
    n_e2e = min(args.steps, 2000 if work.graph else 20)
    with torch.cuda.stream(stream):
        for i in range(min(3, n_e2e)):
            work.e2e_step(i)
        stream.synchronize()
        t0 = time.perf_counter()
        for i in range(n_e2e):
            work.e2e_step(i)
        stream.synchronize()
        e2e_s = time.perf_counter() - t0
    if dist:
        (e2e_s,) = max_over_ranks([e2e_s], dist, dev)

    peaks = _peaks()
    value = world * work.tokens_per_step * args.steps / (ms / 1e3)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": getattr(work, "dtype", "f16 mma, f32 accumulate (int8 / 3-bit storage)"),
        "data": "synthetic",
        "config": dict(work.describe(), parallelism=f"replicas x{world}",
                       timing=("CUDA graphs of exactly `steps` back-to-back steps, events on the launching stream; "
                               "warm-up replays the same graphs (max(warmup, 3) steps rounded up to whole replays)"
                               if work.graph else "events around each step on the launching stream")),
        # the step is one launch of the dominant kernel (decode) or its whole
        # call (prefill, fan-out): the roofline uses the timed region itself
        "roofline": work.roofline(ms / args.steps, peaks),
        "e2e": {"value": round(world * work.tokens_per_step * n_e2e / e2e_s, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
                "api": getattr(work, "e2e_api", "public Python API, eager")},
        "gpu_launches": work.launches_per_step * args.steps,
        "clocks": clocks,
    }
    if hasattr(work, "algo_bytes"):
        line["effective_gbs"] = round(work.algo_bytes * world * args.steps / (ms / 1e3) / 1e9, 1)
    if hasattr(work, "flops"):
        line["effective_tflops"] = round(work.flops * world * args.steps / (ms / 1e3) / 1e12, 1)
    if args.workload == "gemma4_decode" and not args.no_per_config:
        fl = stream_floor(work, stream, dev)
        fl["decode_us"] = round(ms / args.steps * 1e3, 3)
        fl["floor_frac"] = round(work.algo_bytes / (fl["stream_us"] / 1e6) / 1e9 / peaks[0], 4)
        fl["what"] = ("ckv_calibrate_stream on the same cache copies: the decode's grid, staging and programmatic "
                      "launch with no compute (then with the split rendezvous), back to back in a graph")
        line["floor"] = fl
    del work
    torch.cuda.empty_cache()
    if args.workload == "gemma4_decode" and not args.no_per_config:
        line["per_config"] = per_config_lines(dev, stream, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload in ("gemma4_decode",
                                                                                   "chunked_prefill"):
        line["cpu_baseline"] = cpu_baseline(args.workload)
    if dist:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ oracle --

ORACLE_CHUNK = 2048  # tokens per oracle work unit


def _oracle_setup(sample_tokens=None, workload="gemma4_decode"):
    """Seeded inputs of one step and the oracle's quantised cache fields."""
    import numpy as np
    from compressed_kv_attention_gb300 import inputs
    from tests import helpers as H
    w = inputs.WORKLOADS[workload]
    D, Hkv, Hq = w.head_dim, w.n_kv_heads, w.n_q_heads
    T = w.seq_len + w.n_new
    Ts = T if sample_tokens is None else min(T, sample_tokens)
    outl = inputs.outlier_channels(D, w.n_outliers, w.seed)
    k = inputs.normal_tensor((Ts, Hkv, D), w.seed, "bench-oracle/k", outl)
    v = inputs.normal_tensor((Ts, Hkv, D), w.seed, "bench-oracle/v", outl)
    q = inputs.normal_tensor((1, Hq, D), w.seed, "bench-oracle/q", outl)
    signs = inputs.tbq_signs(D)
    qs, d16, codes, n16, _ = H.oracle_quantize(np.swapaxes(k, 0, 1), np.swapaxes(v, 0, 1), signs)
    return dict(D=D, Hkv=Hkv, Hq=Hq, T=T, Ts=Ts, q=q, k_new=k[-1:], v_new=v[-1:], signs=signs,
                qs=qs, d16=d16, codes=codes, n16=n16)


# Worker side of the oracle pool: the step's arrays, memory-mapped from files
# the parent wrote (spawned processes, one BLAS thread each).
_OW = {}


def _oracle_worker_init(paths):
    import numpy as np
    for k, pth in paths.items():
        _OW[k] = np.load(pth, mmap_mode="r")


def _oracle_unit(unit):
    """Oracle work of one (kv head, token chunk): dequantise the chunk to dense
    float64 and attend with the kv head's query heads. Returns the partial
    (output, lse) of those heads over the chunk."""
    import numpy as np
    from oracle import ckv_oracle as O
    h, a, b, G, scale = unit
    kh = O.q8_0_dequantize(np.asarray(_OW["qs"][h, a:b]), np.asarray(_OW["d16"][h, a:b]))
    vh = O.tbq3_dequantize(np.asarray(_OW["codes"][h, a:b]), np.asarray(_OW["n16"][h, a:b]),
                           np.asarray(_OW["signs"]))
    q = np.asarray(_OW["q"][0, h * G:(h + 1) * G], dtype=np.float64)
    o, lse = O.attention(q, kh, vh, scale)
    return h, o, lse


class OraclePool:
    """The oracle's decode step over a pool of spawned processes: independent
    (kv head, 2048-token chunk) units, each dequantise-then-attend, combined
    per query head with the oracle's exact log-sum-exp merge."""

    def __init__(self, s, procs):
        import multiprocessing as mp
        import numpy as np
        self.s = s
        self.dir = tempfile.mkdtemp(prefix="ckv_oracle_")
        paths = {}
        for k in ("qs", "d16", "codes", "n16", "signs", "q"):
            paths[k] = os.path.join(self.dir, k + ".npy")
            np.save(paths[k], s[k])
        G = s["Hq"] // s["Hkv"]
        scale = 1.0 / math.sqrt(s["D"])
        self.units = [(h, a, min(a + ORACLE_CHUNK, s["Ts"]), G, scale)
                      for h in range(s["Hkv"]) for a in range(0, s["Ts"], ORACLE_CHUNK)]
        # One BLAS thread per process: children take the environment at spawn time.
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(procs, initializer=_oracle_worker_init, initargs=(paths,))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.procs = procs

    def step(self):
        from oracle import ckv_oracle as O
        s = self.s
        O.q8_0_quantize(s["k_new"])
        O.tbq3_quantize(s["v_new"], s["signs"])
        parts = {}
        for h, o, lse in self.pool.map(self._unit, self.units, chunksize=1):
            parts.setdefault(h, []).append((o, lse))
        return {h: O.lse_merge([p[0] for p in ps], [p[1] for p in ps]) for h, ps in parts.items()}

    _unit = staticmethod(_oracle_unit)

    def close(self):
        import shutil
        self.pool.close()
        self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def _time_pool(pool, min_seconds, max_seconds):
    pool.step()  # warm: workers loaded, pages mapped
    n, t0 = 0, time.perf_counter()
    while True:
        pool.step()
        n += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or el * (n + 1) / n > max_seconds:
            return n, el


def cpu_baseline(workload="gemma4_decode", min_seconds=8.0, max_seconds=20.0):
    """The oracle timed on the host cores, single-threaded and over every core.
    Decode: whole decode steps. Prefill: one query token's work over the full key
    range (the last query's), in query tokens per second."""
    s = _oracle_setup(workload=workload)
    cores = _cores()
    res = {}
    for label, procs in (("single_thread", 1), ("all_cores", cores)):
        pool = OraclePool(s, procs)
        try:
            n, el = _time_pool(pool, min_seconds, max_seconds)
        finally:
            pool.close()
        res[label] = {"value": round(n / el, 4), "processes": procs, "steps": n, "seconds": round(el, 2)}
    what = ("query tokens of chunked_prefill, each attending over the last query's "
            f"{s['Ts']} dequantised tokens" if workload == "chunked_prefill" else
            f"full decode steps of {workload} (dequantise {s['T']} tokens x {s['Hkv']} kv heads to float64, "
            f"attend {s['Hq']} heads)")
    sample = (f"{res['all_cores']['steps']} {what}, numpy float64, as (kv head, {ORACLE_CHUNK}-token chunk) units "
              f"over {cores} spawned processes of one BLAS thread, merged by the oracle's lse_merge; single-thread: "
              f"{res['single_thread']['steps']} steps in one such process")
    return {"value": res["all_cores"]["value"], "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": sample, "single_thread": res["single_thread"], "all_cores": res["all_cores"],
            "cpu_model": _cpu_model(), "nproc": os.cpu_count()}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    workload = args.workload if args.workload in ("gemma4_decode", "chunked_prefill") else "gemma4_decode"
    cores = _cores()
    # Size each step's sample so that warm-up + timed steps take about 2
    # minutes: a step attends over the first Ts tokens of the cache and its
    # time is scaled by T / Ts to a full step.
    cal = OraclePool(_oracle_setup(sample_tokens=cores * ORACLE_CHUNK // 2, workload=workload), cores)
    try:
        cal.step()
        t0 = time.perf_counter()
        cal.step()
        full_est = (time.perf_counter() - t0) * cal.s["T"] / cal.s["Ts"]
    finally:
        cal.close()
    per_step = 120.0 / max(1, args.steps + args.warmup)
    Ts = int(min(cal.s["T"], max(16, (cal.s["T"] * per_step / full_est) // 16 * 16)))
    pool = OraclePool(_oracle_setup(sample_tokens=Ts, workload=workload), cores)
    try:
        s = pool.s
        frac = s["Ts"] / s["T"]
        for _ in range(max(args.warmup, 1)):
            pool.step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            pool.step()
        el = (time.perf_counter() - t0) / frac
    finally:
        pool.close()
    value = args.steps / el
    sample = (f"each step: oracle work for one query token (dequantise to float64 + attend {s['Hq']} heads) over "
              f"{s['Ts']} of {s['T']} tokens of {workload}, as (kv head, {ORACLE_CHUNK}-token chunk) units over "
              f"{cores} spawned processes, time scaled by {1 / frac:.2f}")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / max(args.steps, 1) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu_model": _cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def _free_port():
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_ranks(n, argv):
    """Start `n` ranks of this script (one per GPU of this node) with
    torch.distributed.run on 127.0.0.1; returns the launcher's exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", f"--master-port={_free_port()}", os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main():
    args = _args()
    env_world = os.environ.get("WORLD_SIZE")
    if env_world is None and args.gpus is not None and args.gpus > 1:
        sys.exit(launch_ranks(args.gpus, sys.argv[1:]))
    if env_world is not None and args.gpus is not None and int(env_world) != args.gpus:
        sys.stderr.write(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={env_world}\n")
        sys.exit(2)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
