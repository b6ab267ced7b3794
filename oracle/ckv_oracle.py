"""Float64 CPU oracle for attention over a q8_0-K / TBQ3-V compressed KV cache.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg may import or run this module. The CUDA library never calls it and
shares no code, table or constant with it; the two meet only in the seeded
input generators, which hold none of the method's arithmetic.

What it computes, in the pages' order, with every step in float64 (fp16 only
where the method stores fp16):

  1. q8_0 keys: blocks of 32 values, one fp16 scale per block, int8 codes.
  2. TBQ3 values: sign diagonal, orthonormal fast Walsh-Hadamard transform,
     one fp16 norm per vector, each normalised coordinate snapped to the nearest
     of the 8 Lloyd-Max centroids for N(0,1).
  3. Dequantise both to dense float64 and run softmax attention by its plain
     definition (max-subtracted exponentials, sum, divide), returning the
     output and the log-sum-exp of every query row.
  4. The exact merge of (output, lse) partials over disjoint key sets.

Sources (page titles as published):
  [PolyKV] "F5 M6 — PolyKV (shared compressed KV pool)"
  [DCA]    "Feature — Gemma-4 A4B Dual Chunk Attention (DCA), training-free 1M context"
  [SYNC]   "Protocol — Upstream Sync"

Readings taken where the pages are silent (each is listed with its reason in
the design notes): a full d-point transform with one sign diagonal; the norm
is the plain Euclidean norm of the fp16 input, normalisation uses the unrounded
norm and only the stored copy is rounded to fp16; q8_0 divides by the stored
fp16 scale and rounds half away from zero; an exact centroid-midpoint tie goes
to the centroid of smaller magnitude and u == 0 maps to +0.2451; a zero vector
stores code 4 everywhere and norm 0; a query row with no visible key returns
output 0 and lse -inf.

Parity status: every function here is pinned by the CPU tests against values
the pages print, closed forms or library routines (see tests/test_oracle_pins.py;
the dequantisers by hand-derived worked records, per-block scale indexing and
the relative reconstruction error against the quantiser's distortion),
except end-to-end quality against the pages' models (perplexity, RULER), which
needs trained weights and datasets: parity unpinned for that, and it is not
computed here.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Constants of the method
# ---------------------------------------------------------------------------

#: q8_0 block length. [PolyKV] section "What PolyKV is (reference)": keys go to
#: int8 (q8_0); [SYNC] entry 0130 describes q8_0 blocks of 32 values.
QK8_0 = 32

#: The 8-level Lloyd-Max (minimum-MSE) quantiser for a unit Gaussian, ascending.
#: [PolyKV] section "What PolyKV is (reference)" fixes "Lloyd-Max (MSE-optimal)
#: quantization" for V after the FWHT; section "Phase-0 fork recon" (Gate-1)
#: names the 3-bit table CENTROIDS_3BIT and nearest_centroid_3bit. The values
#: are the classic 4-decimal table for N(0,1).
LLOYD_MAX_3BIT = np.array([-2.1520, -1.3439, -0.7560, -0.2451,
                           0.2451, 0.7560, 1.3439, 2.1520], dtype=np.float64)


def to_fp16(x) -> np.ndarray:
    """Round float64 values to fp16, round-to-nearest-even (numpy's conversion)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16)


# ---------------------------------------------------------------------------
# q8_0 keys
# ---------------------------------------------------------------------------

def q8_0_quantize(x):
    """q8_0-quantise fp16 rows ``x[..., D]`` (D a multiple of 32).

    [PolyKV] section "What PolyKV is (reference)": K is stored as int8 (q8_0),
    the higher-precision half of the asymmetric scheme. Per block of 32 values:
    amax = max |x_i|; d16 = fp16(amax / 127); q_i = x_i / d16 rounded half away
    from zero and clamped to [-127, 127]; a block with d16 == 0 stores q = 0.

    Returns ``(qs int8 [..., D], d16 float16 [..., D/32])``.
    """
    x = np.asarray(x, dtype=np.float16).astype(np.float64)
    D = x.shape[-1]
    if D % QK8_0:
        raise ValueError("head_dim must be a multiple of 32")
    blocks = x.reshape(x.shape[:-1] + (D // QK8_0, QK8_0))
    amax = np.abs(blocks).max(axis=-1)
    d16 = to_fp16(amax / 127.0)
    d = d16.astype(np.float64)[..., None]
    safe_d = np.where(d == 0.0, 1.0, d)
    r = blocks / safe_d
    # x and d16 are both fp16, so x/d16 is either exactly a half-integer or at
    # least 2^-12 away from one; float64 division then decides the rounding
    # exactly as exact arithmetic would.
    q = np.sign(r) * np.floor(np.abs(r) + 0.5)
    q = np.clip(q, -127, 127)
    q = np.where(d == 0.0, 0.0, q)
    return q.astype(np.int8).reshape(x.shape), d16


def q8_0_dequantize(qs, d16) -> np.ndarray:
    """Dense float64 keys: K_hat_i = q_i * d16 of the block holding i."""
    qs = np.asarray(qs).astype(np.float64)
    D = qs.shape[-1]
    d = np.asarray(d16, dtype=np.float16).astype(np.float64)
    blocks = qs.reshape(qs.shape[:-1] + (D // QK8_0, QK8_0)) * d[..., None]
    return blocks.reshape(qs.shape)


# ---------------------------------------------------------------------------
# TBQ3 values (TurboQuant-MSE, 3 bits)
# ---------------------------------------------------------------------------

def fwht(y) -> np.ndarray:
    """Unnormalised fast Walsh-Hadamard transform along the last axis: H_d @ y.

    H_d is the Sylvester Hadamard matrix in natural order, H_1 = [1],
    H_2n = [[H_n, H_n], [H_n, -H_n]]. The transform runs the log2(d) butterfly
    stages of that recursion: at stage h, every pair (a, b) of entries h apart
    inside a block of 2h becomes (a + b, a - b).
    """
    y = np.array(y, dtype=np.float64, copy=True)
    d = y.shape[-1]
    if d & (d - 1):
        raise ValueError("transform length must be a power of two")
    lead = y.shape[:-1]
    h = 1
    while h < d:
        z = y.reshape(lead + (d // (2 * h), 2, h))
        a = z[..., 0, :].copy()
        b = z[..., 1, :].copy()
        z[..., 0, :] = a + b
        z[..., 1, :] = a - b
        y = z.reshape(lead + (d,))
        h *= 2
    return y


def fwht_orthonormal(y) -> np.ndarray:
    """Orthonormal transform H_d y / sqrt(d). It is symmetric, so it is its own inverse."""
    d = np.asarray(y).shape[-1]
    return fwht(y) / np.sqrt(d)


def lloyd_max_gaussian(levels: int) -> np.ndarray:
    """Centroids of the minimum-MSE quantiser of N(0,1) with ``levels`` levels, by
    Lloyd's iteration: thresholds are the midpoints of neighbouring centroids and
    each centroid is the conditional mean of its cell,
    c_k = (phi(t_k) - phi(t_{k+1})) / (Phi(t_{k+1}) - Phi(t_k)), with phi and Phi
    the normal density and distribution function (closed forms via erf). Starts
    from the equal-probability cell centres and stops when no centroid moves by
    1e-15. [PolyKV] section "S2 perf-path Level B" runs the same scheme at 2, 3
    and 4 bits (turbo2 / turbo3 / turbo4).
    """
    import math
    from scipy.special import erfinv

    def pdf(x):
        return 0.0 if not np.isfinite(x) else math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)

    def cdf(x):
        if not np.isfinite(x):
            return 1.0 if x > 0 else 0.0
        return 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))

    c = np.array([math.sqrt(2.0) * erfinv(2.0 * (k + 0.5) / levels - 1.0) for k in range(levels)])
    for _ in range(100000):
        t = np.concatenate([[-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]])
        new = np.array([(pdf(t[k]) - pdf(t[k + 1])) / (cdf(t[k + 1]) - cdf(t[k])) for k in range(levels)])
        moved = np.abs(new - c).max()
        c = new
        if moved < 1e-15:
            break
    return c


#: Value bit widths the cache supports: 2, 3 or 4 bits per coordinate.
TBQ_BITS = (2, 3, 4)


def tbq_centroids(bits: int) -> np.ndarray:
    """Ascending centroid table of the ``bits``-bit quantiser: the printed 3-bit
    table (north of the method), and at 2 and 4 bits the Lloyd-Max centroids of
    N(0,1) rounded to 4 decimals like the printed one."""
    if bits == 3:
        return LLOYD_MAX_3BIT
    if bits not in TBQ_BITS:
        raise ValueError("bits must be 2, 3 or 4")
    return np.round(lloyd_max_gaussian(1 << bits), 4)


def nearest_centroid_bits(u, bits: int) -> np.ndarray:
    """Index (ascending centroids) of the nearest ``bits``-bit centroid; an exact
    tie goes to the neighbour of smaller magnitude and u == 0 to the smallest
    positive centroid (index 2^(bits-1)), as at 3 bits."""
    table = tbq_centroids(bits)
    u = np.asarray(u, dtype=np.float64)
    dist = np.abs(u[..., None] - table)
    best = dist.min(axis=-1, keepdims=True)
    tied = dist == best
    rank = np.abs(table) * 4.0 - (table > 0)
    score = np.where(tied, rank, np.inf)
    return score.argmin(axis=-1).astype(np.uint8)


def nearest_centroid(u) -> np.ndarray:
    """Index (0..7, ascending centroids) of the Lloyd-Max centroid nearest to each u.

    [PolyKV] section "Phase-0 fork recon" (Gate-1) names nearest_centroid_3bit.
    An exact tie between two neighbours goes to the one of smaller magnitude;
    u == 0 (equidistant from -0.2451 and +0.2451) maps to +0.2451 (index 4).
    """
    u = np.asarray(u, dtype=np.float64)
    dist = np.abs(u[..., None] - LLOYD_MAX_3BIT)
    best = dist.min(axis=-1, keepdims=True)
    tied = dist == best
    # Among the nearest centroids prefer the smallest |c|, and +c over -c.
    rank = np.abs(LLOYD_MAX_3BIT) * 4.0 - (LLOYD_MAX_3BIT > 0)
    score = np.where(tied, rank, np.inf)
    return score.argmin(axis=-1).astype(np.uint8)


def tbq3_quantize(x, signs):
    """TBQ3-quantise fp16 vectors ``x[..., D]`` with the +/-1 diagonal ``signs[D]``.

    [PolyKV] section "What PolyKV is (reference)": V goes to 3-bit TurboQuant
    MSE, an FWHT rotation that spreads outlier energy across dims followed by
    Lloyd-Max quantisation; section "S2 perf-path Level B" (the forward
    rotation) applies the sign diagonal, then the butterfly. Steps per vector:
      y = s * x;  z = H_d y / sqrt(d);  r = ||x||_2;  u = z * sqrt(d) / r;
      code_i = nearest centroid of u_i;  n16 = fp16(r).
    A zero vector (r == 0) stores u = 0, hence code 4 everywhere, and n16 = 0.

    Returns ``(codes uint8 [..., D] in 0..7, n16 float16 [...], u float64 [..., D])``;
    u is returned so that tests can see how close each coordinate was to a
    centroid midpoint.
    """
    x = np.asarray(x, dtype=np.float16).astype(np.float64)
    s = np.asarray(signs).astype(np.float64)
    d = x.shape[-1]
    y = s * x
    z = fwht_orthonormal(y)
    r = np.sqrt(np.sum(x * x, axis=-1))
    safe_r = np.where(r == 0.0, 1.0, r)
    u = np.where(r[..., None] == 0.0, 0.0, z * np.sqrt(d) / safe_r[..., None])
    codes = nearest_centroid(u)
    return codes, to_fp16(r), u


def tbq3_dequantize(codes, n16, signs) -> np.ndarray:
    """Dense float64 values: V_hat = s * H_d^T ((n16 / sqrt(d)) * c[code]) / sqrt(d)."""
    return tbq_dequantize(codes, n16, signs, 3)


def tbq_quantize(x, signs, bits: int = 3):
    """TBQ quantisation at ``bits`` bits per coordinate: the steps of
    :func:`tbq3_quantize` with the ``bits``-bit centroid table (a zero vector
    stores the smallest positive centroid's index everywhere and norm 0)."""
    if bits == 3:
        return tbq3_quantize(x, signs)
    x = np.asarray(x, dtype=np.float16).astype(np.float64)
    s = np.asarray(signs).astype(np.float64)
    d = x.shape[-1]
    z = fwht_orthonormal(s * x)
    r = np.sqrt(np.sum(x * x, axis=-1))
    safe_r = np.where(r == 0.0, 1.0, r)
    u = np.where(r[..., None] == 0.0, 0.0, z * np.sqrt(d) / safe_r[..., None])
    return nearest_centroid_bits(u, bits), to_fp16(r), u


def tbq_dequantize(codes, n16, signs, bits: int = 3) -> np.ndarray:
    """Dense float64 values: V_hat = s * H_d^T ((n16 / sqrt(d)) * c_bits[code]) / sqrt(d)."""
    codes = np.asarray(codes)
    d = codes.shape[-1]
    n = np.asarray(n16, dtype=np.float16).astype(np.float64)
    w = (n / np.sqrt(d))[..., None] * tbq_centroids(bits)[codes]
    return np.asarray(signs).astype(np.float64) * fwht_orthonormal(w)


#: Dims per rotation group of the block-diagonal variant.
ROT_GROUP = 128


def tbq_quantize_blocked(x, signs1, signs2, bits: int = 3, group: int = ROT_GROUP):
    """The block-diagonal, two-sign rotation variant of the TBQ quantiser.

    [PolyKV] section "S2 perf-path Level B" (the GGML_OP_TURBO_WHT forward
    direction: first sign diagonal, the WHT, then 1/sqrt(G) times the second
    sign diagonal); section "S2 perf-path D=512 fused turbo-vec" (the transform
    is block-diagonal over 128-dim groups, so D = 512 is four independent
    groups); section "S2 tier-family overview" (one norm per 128 values).
    Steps for every group g of G consecutive dims:
      y_g = s2_g * H_G (s1_g * x_g) / sqrt(G);  r_g = ||x_g||_2;
      u_g = y_g * sqrt(G) / r_g;  codes = nearest centroid;  n16_g = fp16(r_g).
    A zero group stores u = 0 (code 2^(bits-1)) and norm 0.

    Returns ``(codes uint8 [..., D], n16 float16 [..., D / G], u float64 [..., D])``.
    """
    x = np.asarray(x, dtype=np.float16).astype(np.float64)
    d = x.shape[-1]
    if d % group:
        raise ValueError("head dim must be a multiple of the rotation group")
    s1 = np.asarray(signs1).astype(np.float64)
    s2 = np.asarray(signs2).astype(np.float64)
    xg = x.reshape(x.shape[:-1] + (d // group, group))
    yg = s2.reshape(d // group, group) * fwht_orthonormal(s1.reshape(d // group, group) * xg)
    r = np.sqrt(np.sum(xg * xg, axis=-1))
    safe_r = np.where(r == 0.0, 1.0, r)
    u = np.where(r[..., None] == 0.0, 0.0, yg * np.sqrt(group) / safe_r[..., None])
    u = u.reshape(x.shape)
    return nearest_centroid_bits(u, bits), to_fp16(r), u


def tbq_dequantize_blocked(codes, n16, signs1, signs2, bits: int = 3, group: int = ROT_GROUP) -> np.ndarray:
    """Dense float64 values of the block-diagonal variant. [PolyKV] section "S2
    perf-path Level A" gives the inverse order per 128-dim group: the second
    sign diagonal, the butterfly, then 1/sqrt(G) and the first diagonal:
      V_hat_g = s1_g * H_G (s2_g * (n16_g / sqrt(G)) * c[code_g]) / sqrt(G)."""
    codes = np.asarray(codes)
    d = codes.shape[-1]
    ng = d // group
    n = np.asarray(n16, dtype=np.float16).astype(np.float64)
    c = tbq_centroids(bits)[codes].reshape(codes.shape[:-1] + (ng, group))
    w = (n / np.sqrt(group))[..., None] * c
    s1 = np.asarray(signs1).astype(np.float64).reshape(ng, group)
    s2 = np.asarray(signs2).astype(np.float64).reshape(ng, group)
    return (s1 * fwht_orthonormal(s2 * w)).reshape(codes.shape)


# ---------------------------------------------------------------------------
# Attention and the (output, lse) merge
# ---------------------------------------------------------------------------

def attention(q, k, v, scale: float, visible=None):
    """Softmax attention by definition, float64.

    ``q [R, D]``, ``k [T, D]``, ``v [T, DV]``; ``visible`` is an optional boolean
    ``[R, T]`` mask (True = the key is attended). For every row:
      l_j = scale * q . k_j over the visible keys;  m = max_j l_j;
      p_j = exp(l_j - m);  o = sum_j p_j v_j / sum_j p_j;  lse = m + ln sum_j p_j.
    A row with no visible key returns o = 0 and lse = -inf: [DCA] section
    "Section C2b" (empty-regime safety) and [SYNC] entry 0110 (the fully-masked
    row yields the identity 0, not 0/0).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    R, T = q.shape[0], k.shape[0]
    o = np.zeros((R, v.shape[1]), dtype=np.float64)
    lse = np.full(R, -np.inf, dtype=np.float64)
    if T == 0 or R == 0:
        return o, lse
    logits = scale * (q @ k.T)
    if visible is None:
        visible = np.ones((R, T), dtype=bool)
    visible = np.asarray(visible, dtype=bool)
    masked = np.where(visible, logits, -np.inf)
    has_key = visible.any(axis=1)
    m = np.where(has_key, masked.max(axis=1), 0.0)
    p = np.where(visible, np.exp(masked - m[:, None]), 0.0)
    l = p.sum(axis=1)
    o[has_key] = (p[has_key] @ v) / l[has_key, None]
    lse[has_key] = m[has_key] + np.log(l[has_key])
    return o, lse


def lse_merge(outputs, lses):
    """Exact merge of normalised partials over disjoint key sets.

    [DCA] section "Implementation progress + Section-D simplification": with
    partials (O_r, lse_r), M = max_r lse_r, w_r = exp(lse_r - M),
    O = sum_r w_r O_r / sum_r w_r, and the merged lse = M + ln sum_r w_r.
    A partial with lse = -inf (empty key set) gets weight 0; if every partial
    is empty the result is O = 0, lse = -inf ([DCA] section "Section C2b").

    ``outputs``: list of ``[R, DV]``; ``lses``: list of ``[R]``.
    """
    O = np.stack([np.asarray(o, dtype=np.float64) for o in outputs])
    L = np.stack([np.asarray(s, dtype=np.float64) for s in lses])
    M = L.max(axis=0)
    finite = np.isfinite(M)
    Msafe = np.where(finite, M, 0.0)
    w = np.where(np.isfinite(L), np.exp(L - Msafe[None, :]), 0.0)
    wsum = w.sum(axis=0)
    out = np.zeros(O.shape[1:], dtype=np.float64)
    out[finite] = (np.einsum("rn,rnd->nd", w, O)[finite]) / wsum[finite, None]
    lse = np.where(finite, Msafe + np.log(np.where(finite, wsum, 1.0)), -np.inf)
    return out, lse


# ---------------------------------------------------------------------------
# Whole-workload helpers (grouped-query layout, decode and prefill)
# ---------------------------------------------------------------------------

def kv_head_of(q_head: int, n_q_heads: int, n_kv_heads: int) -> int:
    """Grouped-query map: query head h reads kv head floor(h / G), G = Hq / Hkv
    ([SYNC] entry 0080: Gemma-4 head16/kv2 is GQA 8)."""
    return q_head // (n_q_heads // n_kv_heads)


def decode_reference(q, k_hat, v_hat, seq_len, scale: float):
    """Decode attention for one sequence.

    ``q [n_q, Hq, D]``; ``k_hat, v_hat [Hkv, T, D]`` dense float64 (already
    dequantised); every query token sees cached tokens [0, seq_len).
    Returns ``o [n_q, Hq, D]`` and ``lse [n_q, Hq]``.
    """
    q = np.asarray(q, dtype=np.float64)
    n_q, Hq, D = q.shape
    Hkv = k_hat.shape[0]
    o = np.zeros((n_q, Hq, v_hat.shape[-1]))
    lse = np.zeros((n_q, Hq))
    for h in range(Hq):
        kh = kv_head_of(h, Hq, Hkv)
        oh, lh = attention(q[:, h, :], k_hat[kh, :seq_len], v_hat[kh, :seq_len], scale)
        o[:, h, :] = oh
        lse[:, h] = lh
    return o, lse


def verify_decode_reference(q, k_hat, v_hat, seq_len, scale: float):
    """Attention of a verify batch for one sequence.

    ``q [n_q, Hq, D]`` are the last n_q positions of the sequence (the drafted
    tokens, whose K/V rows are the last n_q cached rows); query token i sees
    cached tokens [0, seq_len - n_q + i] (causal among the batch, as the PolyKV
    page's "turbo-MMA verify (n_q>1)" batches check drafted tokens; section
    "WorkStream-1"). A token whose range is empty returns o = 0, lse = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    n_q, Hq, D = q.shape
    Hkv = k_hat.shape[0]
    vis = np.arange(seq_len)[None, :] <= (seq_len - n_q + np.arange(n_q))[:, None]
    o = np.zeros((n_q, Hq, v_hat.shape[-1]))
    lse = np.zeros((n_q, Hq))
    for h in range(Hq):
        kh = kv_head_of(h, Hq, Hkv)
        oh, lh = attention(q[:, h, :], k_hat[kh, :seq_len], v_hat[kh, :seq_len], scale, visible=vis)
        o[:, h, :] = oh
        lse[:, h] = lh
    return o, lse


def dca_ranges(seq_len: int, chunk: int):
    """Key ranges [lo, hi) of the three DCA regimes for the query at position
    i = seq_len - 1 with chunk size c: the [DCA] page's "Section C design"
    keep-masks (chunk of a position = floor(pos / c), causal j <= i) are
    intra: chunk(j) == chunk(i); successive: chunk(j) == chunk(i) - 1;
    inter: chunk(j) < chunk(i) - 1. With k = chunk(i) they are the ranges
    [k c, i + 1), [(k - 1) c, k c) and [0, (k - 1) c), clipped at 0.
    """
    if seq_len <= 0:
        return [(0, 0)] * 3
    k = (seq_len - 1) // chunk
    intra = (k * chunk, seq_len)
    succ = ((k - 1) * chunk, k * chunk) if k >= 1 else (0, 0)
    inter = (0, (k - 1) * chunk) if k >= 2 else (0, 0)
    return [intra, succ, inter]


def dca_decode_reference(q, k_hat, v_hat, seq_len: int, chunk: int, scale: float):
    """Dual chunk attention of the token at position seq_len - 1 for one sequence.

    ``q [3, Hq, D]`` holds the query of each regime (intra, successive, inter;
    roped for its regime by the caller, [DCA] "rope-K-once, rope-Q-thrice");
    every regime attends over its key range (``dca_ranges``) and the three
    softmaxes are merged by ``lse_merge`` (step 4 of the page's graph body).
    Returns ``o [Hq, D]`` and ``lse [Hq]``.
    """
    q = np.asarray(q, dtype=np.float64)
    _, Hq, D = q.shape
    Hkv = k_hat.shape[0]
    o = np.zeros((Hq, v_hat.shape[-1]))
    lse = np.zeros(Hq)
    for h in range(Hq):
        kh = kv_head_of(h, Hq, Hkv)
        parts = [attention(q[r:r + 1, h, :], k_hat[kh, lo:hi], v_hat[kh, lo:hi], scale)
                 for r, (lo, hi) in enumerate(dca_ranges(seq_len, chunk))]
        oh, lh = lse_merge([p[0] for p in parts], [p[1] for p in parts])
        o[h], lse[h] = oh[0], lh[0]
    return o, lse


def shared_prefill_reference(q, k_prefix, v_prefix, k_tail, v_tail, tail_len: int, scale: float):
    """Multi-tenant prefill of one agent: [PolyKV] section "S1 — SharedKVPool"
    (shared prefix cells are attended by every agent, private suffix cells only
    by their own; the per-agent cost is just the suffix).

    ``q [n_new, Hq, D]`` are the agent's new query tokens, the last n_new
    positions of its private tail; ``k_prefix, v_prefix [Hkv, P, D]`` the shared
    prefix (dequantised); ``k_tail, v_tail [Hkv, >= tail_len, D]`` the agent's
    tail, whose first tail_len rows include the n_new new ones. Query i attends,
    in one softmax, to the P prefix keys followed by tail keys [0, tail_len -
    n_new + i].
    """
    q = np.asarray(q, dtype=np.float64)
    n_new, Hq, D = q.shape
    Hkv = k_prefix.shape[0]
    P = k_prefix.shape[1]
    L = tail_len
    vis = np.ones((n_new, P + L), dtype=bool)
    vis[:, P:] = np.arange(L)[None, :] <= (L - n_new + np.arange(n_new))[:, None]
    o = np.zeros((n_new, Hq, v_prefix.shape[-1]))
    lse = np.zeros((n_new, Hq))
    for h in range(Hq):
        kh = kv_head_of(h, Hq, Hkv)
        keys = np.concatenate([k_prefix[kh], k_tail[kh, :L]], axis=0)
        vals = np.concatenate([v_prefix[kh], v_tail[kh, :L]], axis=0)
        oh, lh = attention(q[:, h, :], keys, vals, scale, visible=vis)
        o[:, h, :] = oh
        lse[:, h] = lh
    return o, lse


def prefill_reference(q, k_hat, v_hat, n_cached: int, scale: float):
    """Causal chunked prefill for one sequence.

    ``q [n_new, Hq, D]`` are the new query tokens at positions n_cached + i;
    ``k_hat, v_hat [Hkv, n_cached + n_new, D]`` hold the cached tokens followed by
    the new tokens in packed-then-dequantised form (the cache stores what the
    packer is handed and attention reads it back). Query i sees keys
    [0, n_cached + i] (causal, [DCA] section "Section C design": keep j <= i).
    """
    q = np.asarray(q, dtype=np.float64)
    n_new, Hq, D = q.shape
    Hkv = k_hat.shape[0]
    T = n_cached + n_new
    vis = np.arange(T)[None, :] <= (n_cached + np.arange(n_new))[:, None]
    o = np.zeros((n_new, Hq, v_hat.shape[-1]))
    lse = np.zeros((n_new, Hq))
    for h in range(Hq):
        kh = kv_head_of(h, Hq, Hkv)
        oh, lh = attention(q[:, h, :], k_hat[kh, :T], v_hat[kh, :T], scale, visible=vis)
        o[:, h, :] = oh
        lse[:, h] = lh
    return o, lse
