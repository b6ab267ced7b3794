"""Shared test machinery: oracle runs over whole workloads (chunked so memory
stays bounded), bit-level comparison of packed caches, and the attention
tolerance. Used by the GPU parity tests, the smoke check and the benchmark's
CPU-baseline leg. Nothing here computes the method itself: the arithmetic is
the oracle's (oracle/), the bytes under test are the CUDA library's.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import ckv_oracle as O
from oracle import layout as LY

#: Attention acceptance: max |o_gpu - o_ref| <= ATOL_REL * max |o_ref| per query row.
ATOL_REL = 2e-3
#: lse acceptance (natural log units): |lse_gpu - lse_ref| <= LSE_ATOL + LSE_RTOL * |lse_ref|.
LSE_ATOL, LSE_RTOL = 2e-3, 1e-5
#: A TBQ code may differ from the oracle's only when the oracle's normalised
#: coordinate lies within this distance of a centroid midpoint.
TIE_WINDOW = 1e-6
MIDPOINTS = (O.LLOYD_MAX_3BIT[1:] + O.LLOYD_MAX_3BIT[:-1]) / 2


def midpoints(bits: int = 3):
    c = O.tbq_centroids(bits)
    return (c[1:] + c[:-1]) / 2

CHUNK = 4096  # tokens per oracle chunk


def oracle_quantize(k, v, signs, bits: int = 3, signs2=None):
    """Oracle q8_0 / TBQ (``bits`` per V code) of fp16 K, V [..., T, D] (leading
    dims kept), chunked over T; ``signs2`` given: the block-diagonal rotation
    (norms then [..., T, D/128])."""
    k = np.asarray(k, np.float16)
    v = np.asarray(v, np.float16)
    T = k.shape[-2]
    qs, d16, codes, n16, u = [], [], [], [], []
    for a in range(0, T, CHUNK):
        q_, d_ = O.q8_0_quantize(k[..., a:a + CHUNK, :])
        if signs2 is None:
            c_, n_, u_ = O.tbq_quantize(v[..., a:a + CHUNK, :], signs, bits)
        else:
            c_, n_, u_ = O.tbq_quantize_blocked(v[..., a:a + CHUNK, :], signs, signs2, bits)
        qs.append(q_); d16.append(d_); codes.append(c_); n16.append(n_); u.append(u_.astype(np.float32))
    return (np.concatenate(qs, -2), np.concatenate(d16, -2), np.concatenate(codes, -2),
            np.concatenate(n16, -1 if signs2 is None else -2), np.concatenate(u, -2))


def oracle_attention_chunked(q, k_of, v_of, T, scale, visible_of=None):
    """Softmax attention of q [R, D] over T keys produced chunk by chunk.

    k_of(a, b) / v_of(a, b) return dense float64 keys / values for positions
    [a, b); the per-chunk results are combined with the oracle's exact
    log-sum-exp merge (pinned against single-pass attention).
    """
    outs, lses = [], []
    for a in range(0, max(T, 1), CHUNK):
        b = min(T, a + CHUNK)
        if b <= a:
            break
        vis = None if visible_of is None else visible_of(a, b)
        o, l = O.attention(q, k_of(a, b), v_of(a, b), scale, visible=vis)
        outs.append(o)
        lses.append(l)
    if not outs:
        return np.zeros((q.shape[0], q.shape[1])), np.full(q.shape[0], -np.inf)
    return O.lse_merge(outs, lses)


def oracle_decode(qh, k_hat, v_hat, seq_len, scale):
    """qh [n_q, Hq, D]; k_hat, v_hat [Hkv, T, D] float64 -> (o [n_q, Hq, D], lse [n_q, Hq])."""
    return O.decode_reference(qh, k_hat, v_hat, seq_len, scale)


def check_attention(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """Assert the attention acceptance row by row; returns the worst normalised error."""
    o_gpu = np.asarray(o_gpu, np.float64).reshape(-1, o_ref.shape[-1])
    o_ref = np.asarray(o_ref, np.float64).reshape(-1, o_ref.shape[-1])
    lse_gpu = np.asarray(lse_gpu, np.float64).ravel()
    lse_ref = np.asarray(lse_ref, np.float64).ravel()
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), empty), f"{what}: empty-row pattern differs"
    assert np.all(o_gpu[empty] == 0.0), f"{what}: empty rows must be 0"
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    full = ~empty
    err = np.abs(o_gpu[full] - o_ref[full]).max(axis=1)
    scale = np.abs(o_ref[full]).max(axis=1)
    worst = float((err / np.maximum(scale, 1e-30)).max()) if full.any() else 0.0
    assert np.all(err <= ATOL_REL * scale), f"{what}: worst row error {worst:.3e} of |o|_inf"
    lerr = np.abs(lse_gpu[full] - lse_ref[full])
    assert np.all(lerr <= LSE_ATOL + LSE_RTOL * np.abs(lse_ref[full])), f"{what}: lse max err {lerr.max():.3e}"
    return worst


# ------------------------------------------------------------- packed bytes --

def oracle_records(qs, d16, codes, n16, capacity, bits: int = 3, groups: int = 1):
    """Oracle byte layout of a whole cache: qs etc. shaped [B, Hkv, T, ...] -> uint8
    [B, Hkv, capacity/16, record]."""
    B, H = qs.shape[:2]
    D = qs.shape[-1]
    out = np.zeros((B, H, capacity // 16, LY.record_bytes(D, bits, groups)), np.uint8)
    for b in range(B):
        for h in range(H):
            out[b, h] = LY.pack_records(qs[b, h], d16[b, h], codes[b, h], n16[b, h], capacity, bits, groups)
    return out


def read_fields(records, D, T, bits: int = 3, groups: int = 1):
    """Read the fields of the first T positions out of one stream's records
    (uint8 [n_tiles, record]) using the layout's index maps. Returns
    (qs int8 [T, D], d16 uint16 [T, D/32], codes uint8 [T, D], n16 uint16 [T])."""
    kofs, sofs = LY.k_code_offsets(D), LY.k_scale_offsets(D)
    nofs = LY.v_norm_offsets(D, bits, groups).reshape(16, groups)
    vbits = LY.v_code_bits(D, bits)
    n_tiles = (T + 15) // 16
    rec = records[:n_tiles]
    qs = (rec[:, kofs] ^ np.uint8(0x80)).view(np.int8).reshape(n_tiles * 16, D)[:T]
    sc = (rec[:, sofs].astype(np.uint16) | (rec[:, sofs + 1].astype(np.uint16) << 8)).reshape(-1, D // 32)[:T]
    nm = (rec[:, nofs].astype(np.uint16) | (rec[:, nofs + 1].astype(np.uint16) << 8)).reshape(-1, groups)[:T]
    if groups == 1:
        nm = nm[:, 0]
    codes = np.zeros((n_tiles, 16, D), np.uint8)
    for k in range(bits):
        bit = vbits[..., k]
        codes |= (((rec[:, bit // 8] >> (bit % 8)) & 1) << k).astype(np.uint8)
    return qs, sc, codes.reshape(-1, D)[:T], nm


def compare_pack(gpu_records, qs, d16, codes, n16, u, T, bits: int = 3, groups: int = 1):
    """Compare one stream's GPU records with the oracle's fields. q8_0 bytes and
    scales must match bit for bit; V codes may differ only at centroid-midpoint
    ties (|u - t| < TIE_WINDOW), fp16 norms by at most one ulp. Returns counts."""
    D = qs.shape[-1]
    gq, gs, gc, gn = read_fields(gpu_records, D, T, bits, groups)
    assert np.array_equal(gq, qs[:T]), "q8_0 codes differ"
    assert np.array_equal(gs, d16[:T].view(np.uint16)), "q8_0 scales differ"
    mism = gc != codes[:T]
    n_mism = int(mism.sum())
    if n_mism:
        uu = u[:T][mism].astype(np.float64)
        dist = np.abs(uu[:, None] - midpoints(bits)[None, :]).min(axis=1)
        assert np.all(dist < TIE_WINDOW), f"{n_mism} code mismatches, worst distance to a midpoint {dist.max():.3e}"
        assert np.all(np.abs(gc[mism].astype(int) - codes[:T][mism].astype(int)) == 1)
    on = np.asarray(n16)[:T].view(np.uint16).astype(np.int64).reshape(gn.shape)
    dn = np.abs(gn.astype(np.int64) - on)
    assert np.all(dn <= 1), f"norms differ by up to {dn.max()} ulp"
    return {"code_ties": n_mism, "norm_ulp": int((dn == 1).sum())}
