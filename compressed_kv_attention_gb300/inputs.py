"""Seeded synthetic inputs for the compressed-KV attention workloads.

This module holds random-number generation and workload shapes only. It does
none of the method's arithmetic (no quantisation, no transform, no attention),
so the CUDA library's tests and the float64 oracle can both draw their inputs
from it without sharing any of the computation they are compared on.

Workloads. The shapes are those of the Gemma-4 global attention layers that the
DCA page ("Feature — Gemma-4 A4B Dual Chunk Attention (DCA), training-free 1M
context", section "Why llamafile is sufficient") describes: head_dim 512, 2 KV
heads, 16 query heads (grouped-query factor 8). The pages measure on RULER and
on agent documents, which are not available here; these tensors stand in for
them. Values are N(0,1) with a seed-chosen set of "outlier" head-dim channels
scaled by 10 (shared by Q, K and V, every head and every token), then rounded
to fp16 (bf16 for the prefill queries).

Sign diagonal. TurboQuant's value rotation draws a +/-1 diagonal from a seed
(the PolyKV page, "F5 M6 — PolyKV (shared compressed KV pool)", section
"Phase-0 fork recon": seeded rotation, TURBO_SEED_ROTATION=42). The page gives
only the seed, so the generator is SplitMix64 (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014) seeded with 42: sign i
is +1 when bit 63 of output number i is clear, else -1. The vector is data: it
is passed to the packer and the attention kernels, and to the oracle.
"""
from __future__ import annotations

import dataclasses
import hashlib

import numpy as np

_MASK64 = (1 << 64) - 1


def splitmix64_stream(seed: int, n: int) -> list[int]:
    """First ``n`` outputs of SplitMix64 started from state ``seed``."""
    out = []
    state = seed & _MASK64
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & _MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        out.append(z ^ (z >> 31))
    return out


def tbq_signs(head_dim: int, seed: int = 42) -> np.ndarray:
    """The +/-1 sign diagonal (int8, length ``head_dim``) shared by every head and
    token; the block-diagonal rotation's second diagonal uses seed 43."""
    words = splitmix64_stream(seed, head_dim)
    return np.array([-1 if (w >> 63) & 1 else 1 for w in words], dtype=np.int8)


def _seed_words(*key) -> list[int]:
    """Stable 32-bit words derived from an arbitrary key (seed, tensor name, indices)."""
    h = hashlib.sha256(repr(key).encode()).digest()
    return [int.from_bytes(h[i:i + 4], "little") for i in range(0, 16, 4)]


def outlier_channels(head_dim: int, n_outliers: int, seed: int) -> np.ndarray:
    """Sorted head-dim indices of the channels scaled by 10 (drawn from ``seed``)."""
    if n_outliers == 0:
        return np.zeros(0, dtype=np.int64)
    rng = np.random.Generator(np.random.PCG64(_seed_words(seed, "outliers")))
    return np.sort(rng.choice(head_dim, size=n_outliers, replace=False))


def normal_tensor(shape, seed: int, name: str, outliers: np.ndarray, *,
                  dtype: str = "float16", device: str = "cpu", torch_out: bool = False):
    """N(0,1) values with the outlier channels (last axis) scaled by 10, rounded to ``dtype``.

    CPU: numpy PCG64 seeded from (seed, name). CUDA: a torch generator seeded
    the same way (a different stream, used only where a whole workload is too
    large to draw on the host; both arms of a comparison then read the same
    device tensor). ``dtype`` is "float16" or "bfloat16" (the latter only with
    torch). Rounding is round-to-nearest-even in both cases.
    """
    shape = tuple(int(s) for s in shape)
    if device == "cpu" and not torch_out and dtype == "float16":
        rng = np.random.Generator(np.random.PCG64(_seed_words(seed, name)))
        x = rng.standard_normal(shape, dtype=np.float32)
        if len(outliers):
            x[..., outliers] *= 10.0
        return x.astype(np.float16)
    import torch
    tdtype = {"float16": torch.float16, "bfloat16": torch.bfloat16}[dtype]
    if device == "cpu":
        rng = np.random.Generator(np.random.PCG64(_seed_words(seed, name)))
        x = torch.from_numpy(rng.standard_normal(shape, dtype=np.float32))
    else:
        g = torch.Generator(device=device)
        w = _seed_words(seed, name)
        g.manual_seed((w[0] << 32 | w[1]) & ((1 << 63) - 1))
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if len(outliers):
        idx = torch.as_tensor(outliers, device=x.device)
        x[..., idx] *= 10.0
    return x.to(tdtype)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, seed and outlier count."""
    name: str
    head_dim: int
    n_kv_heads: int
    n_q_heads: int
    batch: int
    seq_len: int          # cached tokens per sequence (decode) / already cached (prefill)
    seed: int = 0
    n_outliers: int = 0
    n_agents: int = 0     # shared-prefix fan-out: agents reading one prefix
    tail_len: int = 0     # shared-prefix fan-out: private fp16 tail per agent
    n_new: int = 0        # prefill: new tokens appended and attended causally
    n_q: int = 1          # decode: query tokens per sequence (a verify batch when > 1)
    dca_chunk: int = 0    # decode: dual chunk attention with this chunk (three regime queries)
    q_dtype: str = "float16"
    v_bits: int = 3       # bits per V code (3: TBQ3; 2 and 4: the neighbouring tiers)
    rot_group: int = 0    # 0: full D-point transform; 128: block-diagonal rotation with two sign diagonals

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


def _one_percent(d: int) -> int:
    return int(round(0.01 * d))


# The five workloads: a tiny decode that the oracle finishes in well under a
# second, the Gemma-4 global-layer decode, the shared-prefix fan-out decode, the
# long-context decode and the chunked prefill; and a verify batch of 4 drafted
# tokens over the Gemma-4 global-layer cache (multi-query decode), dual chunk
# attention of one token over it with 8192-token chunks, and the long-context
# decode over caches whose V codes have 2 or 4 bits or use the block-diagonal
# rotation; and the multi-tenant prefill of 15 agents, 128 new tokens each,
# over the shared 4096-token compressed prefix and their 512-token fp16 tails.
WORKLOADS = {
    "tiny_decode": Workload("tiny_decode", head_dim=128, n_kv_heads=1, n_q_heads=4, batch=1,
                            seq_len=256, seed=0, n_outliers=2),
    "gemma4_decode": Workload("gemma4_decode", head_dim=512, n_kv_heads=2, n_q_heads=16, batch=1,
                              seq_len=32768, seed=1, n_outliers=_one_percent(512)),
    "fanout_decode": Workload("fanout_decode", head_dim=512, n_kv_heads=2, n_q_heads=16, batch=1,
                              seq_len=4096, seed=2, n_outliers=_one_percent(512),
                              n_agents=15, tail_len=512),
    "long_decode": Workload("long_decode", head_dim=512, n_kv_heads=2, n_q_heads=16, batch=4,
                            seq_len=262144, seed=3, n_outliers=_one_percent(512)),
    "verify_decode": Workload("verify_decode", head_dim=512, n_kv_heads=2, n_q_heads=16, batch=1,
                              seq_len=32768, seed=5, n_outliers=_one_percent(512), n_q=4),
    "dca_decode": Workload("dca_decode", head_dim=512, n_kv_heads=2, n_q_heads=16, batch=1,
                           seq_len=32768, seed=6, n_outliers=_one_percent(512), dca_chunk=8192),
    "long_decode_tbq2": Workload("long_decode_tbq2", head_dim=512, n_kv_heads=2, n_q_heads=16, batch=4,
                                 seq_len=262144, seed=7, n_outliers=_one_percent(512), v_bits=2),
    "long_decode_tbq4": Workload("long_decode_tbq4", head_dim=512, n_kv_heads=2, n_q_heads=16, batch=4,
                                 seq_len=262144, seed=8, n_outliers=_one_percent(512), v_bits=4),
    "long_decode_rot": Workload("long_decode_rot", head_dim=512, n_kv_heads=2, n_q_heads=16, batch=4,
                                seq_len=262144, seed=9, n_outliers=_one_percent(512), rot_group=128),
    "shared_prefill": Workload("shared_prefill", head_dim=512, n_kv_heads=2, n_q_heads=16, batch=1,
                               seq_len=4096, seed=10, n_outliers=_one_percent(512), n_agents=15, tail_len=512,
                               n_new=128, q_dtype="bfloat16"),
    "chunked_prefill": Workload("chunked_prefill", head_dim=512, n_kv_heads=2, n_q_heads=16,
                                batch=1, seq_len=32768, seed=4, n_outliers=_one_percent(512),
                                n_new=2048, q_dtype="bfloat16"),
    "chunked_prefill_rot": Workload("chunked_prefill_rot", head_dim=512, n_kv_heads=2, n_q_heads=16,
                                    batch=1, seq_len=32768, seed=11, n_outliers=_one_percent(512),
                                    n_new=2048, q_dtype="bfloat16", rot_group=128),
}


def compressed_bytes_per_token(head_dim: int, v_bits: int = 3, rot_group: int = 0) -> int:
    """Packed bytes per (token, kv-head): q8_0 K (D int8 + D/32 fp16 scales) and TBQ V
    (v_bits bits per value + one fp16 norm per vector, or per rot_group dims)."""
    n_norms = head_dim // rot_group if rot_group else 1
    return head_dim + 2 * (head_dim // 32) + v_bits * head_dim // 8 + 2 * n_norms
