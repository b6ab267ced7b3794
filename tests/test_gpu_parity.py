"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle on
the same seeded inputs.

* Packing: q8_0 bytes and scales bit-exact; TBQ3 codes identical except at
  centroid-midpoint ties (|u - t| < 1e-6, counted); fp16 norms within one ulp.
* Attention: max |o_gpu - o_ref| <= 2e-3 * max |o_ref| per query row, lse within
  2e-3, both (i) on the oracle's own packed bytes and (ii) end to end from the
  fp16 inputs.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import compressed_kv_attention_gb300 as ckv  # noqa: E402
from compressed_kv_attention_gb300 import inputs  # noqa: E402
from oracle import ckv_oracle as O  # noqa: E402
from tests import helpers as H  # noqa: E402

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def make_kv(D, Hkv, B, T, seed, n_out, name="kv"):
    outl = inputs.outlier_channels(D, n_out, seed)
    k = inputs.normal_tensor((B, T, Hkv, D), seed, name + "/k", outl)
    v = inputs.normal_tensor((B, T, Hkv, D), seed, name + "/v", outl)
    return k, v, outl


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def oracle_cache(k, v, signs):
    """Oracle fields with streams first: [B, Hkv, T, ...]."""
    kt = np.ascontiguousarray(np.swapaxes(k, 1, 2))
    vt = np.ascontiguousarray(np.swapaxes(v, 1, 2))
    return H.oracle_quantize(kt, vt, signs)


def gpu_pack(k, v, signs, capacity, offsets=None):
    B, T, Hkv, D = k.shape
    cache = ckv.PackedCache(D, Hkv, B, capacity, signs)
    kd, vd = to_dev(k), to_dev(v)
    if offsets is None:
        offsets = [(0, T)]
    for a, b in offsets:
        ckv.kv_pack(cache, a, kd[:, a:b], vd[:, a:b])
    torch.cuda.synchronize()
    return cache


def records_np(cache):
    D = cache.head_dim
    return cache.data.view(cache.batch, cache.n_kv_heads, cache.capacity // 16,
                           23 * D + 32).cpu().numpy()


def run_decode(cache, q, seq_lens, max_seq_len, n_split=0):
    B, n_q, Hq, D = q.shape
    qd = to_dev(q)
    out = torch.empty((B, n_q, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((B, n_q, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_decode_workspace(cache, max_seq_len, n_q, Hq, n_split), dtype=torch.uint8,
                     device=DEV)
    sl = torch.tensor(seq_lens, dtype=torch.int32, device=DEV)
    ckv.attn_decode(cache, sl, max_seq_len, qd, 1.0 / math.sqrt(D), out, lse, ws, n_split=n_split)
    assert ckv.read_device_flag(ws) == 0
    return out.cpu().numpy(), lse.cpu().numpy()


def oracle_decode_all(q, qs, d16, codes, n16, signs, seq_lens):
    B, n_q, Hq, D = q.shape
    o = np.zeros((B, n_q, Hq, D))
    lse = np.zeros((B, n_q, Hq))
    for b in range(B):
        T = seq_lens[b]
        kh = O.q8_0_dequantize(qs[b, :, :T], d16[b, :, :T])
        vh = O.tbq3_dequantize(codes[b, :, :T], n16[b, :, :T], signs)
        o[b], lse[b] = O.decode_reference(q[b], kh, vh, T, 1.0 / math.sqrt(D))
    return o, lse


# ------------------------------------------------------------------ pack ----

@pytest.mark.parametrize("D", [64, 128, 256, 512])
def test_pack_matches_oracle(D):
    _need_gpu()
    B, Hkv, T, cap = 2, 2, 77, 96
    k, v, _ = make_kv(D, Hkv, B, T, seed=100 + D, n_out=max(1, D // 100))
    k[0, 5, 1] = 0.0  # a zero K row (d16 = 0) and a zero V vector
    v[1, 9, 0] = 0.0
    signs = inputs.tbq_signs(D)
    # Two packs: a ragged first range, then the rest from an odd offset (partial tiles).
    cache = gpu_pack(k, v, signs, cap, offsets=[(0, 21), (21, T)])
    qs, d16, codes, n16, u = oracle_cache(k, v, signs)
    recs = records_np(cache)
    for b in range(B):
        for h in range(Hkv):
            H.compare_pack(recs[b, h], qs[b, h], d16[b, h], codes[b, h], n16[b, h], u[b, h], T)


def test_pack_tiny_values_and_ties():
    _need_gpu()
    D = 128
    rng = np.random.default_rng(5)
    k = (rng.standard_normal((1, 32, 1, D)) * 1e-3).astype(np.float16)   # subnormal scales
    k[0, 3, 0, :32] = np.array([127, 2.5, -2.5, 0.5] * 8, dtype=np.float16)  # exact half ties
    v = rng.standard_normal((1, 32, 1, D)).astype(np.float16)
    signs = inputs.tbq_signs(D)
    cache = gpu_pack(k, v, signs, 32)
    qs, d16, codes, n16, u = oracle_cache(k, v, signs)
    H.compare_pack(records_np(cache)[0, 0], qs[0, 0], d16[0, 0], codes[0, 0], n16[0, 0], u[0, 0], 32)


# ---------------------------------------------------------------- decode ----

def test_tiny_decode_workload():
    """The tiny workload: 1 kv head, 4 query heads, head_dim 128, 256 tokens."""
    _need_gpu()
    w = inputs.WORKLOADS["tiny_decode"]
    k, v, outl = make_kv(w.head_dim, w.n_kv_heads, 1, w.seq_len, w.seed, w.n_outliers)
    q = inputs.normal_tensor((1, 1, w.n_q_heads, w.head_dim), w.seed, "q", outl)
    signs = inputs.tbq_signs(w.head_dim)
    qs, d16, codes, n16, u = oracle_cache(k, v, signs)
    o_ref, lse_ref = oracle_decode_all(q, qs, d16, codes, n16, signs, [w.seq_len])
    # (i) the same packed bytes: the oracle's records uploaded as the cache
    cache_i = ckv.PackedCache(w.head_dim, 1, 1, w.seq_len, signs,
                              data=to_dev(H.oracle_records(qs, d16, codes, n16, w.seq_len).ravel()))
    o, l = run_decode(cache_i, q, [w.seq_len], w.seq_len)
    H.check_attention(o, l, o_ref, lse_ref, "tiny (i)")
    # (ii) end to end from fp16 inputs
    cache = gpu_pack(k, v, signs, w.seq_len)
    o, l = run_decode(cache, q, [w.seq_len], w.seq_len)
    H.check_attention(o, l, o_ref, lse_ref, "tiny (ii)")


@pytest.mark.parametrize("D,Hkv,Hq,n_q", [(64, 2, 4, 1), (128, 1, 4, 2), (128, 2, 16, 1), (256, 2, 8, 3),
                                          (512, 2, 16, 1), (512, 1, 8, 2), (512, 2, 4, 1)])
# 40 and 300 splits exceed the 13-14 tiles (empty partials) and give merge
# trees of 7 and 18-slot leaves (several bulk-copy chunks per merge).
@pytest.mark.parametrize("n_split", [0, 1, 5, 40, 300])
def test_decode_shapes_ragged(D, Hkv, Hq, n_q, n_split):
    _need_gpu()
    B, T, cap = 3, 203, 224
    seq_lens = [203, 0, 150]   # ragged, one empty sequence
    k, v, outl = make_kv(D, Hkv, B, T, seed=7 + D + Hq + n_q, n_out=max(1, round(0.01 * D)))
    q = inputs.normal_tensor((B, n_q, Hq, D), 7 + D, "q", outl)
    signs = inputs.tbq_signs(D)
    qs, d16, codes, n16, u = oracle_cache(k, v, signs)
    o_ref, lse_ref = oracle_decode_all(q, qs, d16, codes, n16, signs, seq_lens)
    cache = gpu_pack(k, v, signs, cap)
    o, l = run_decode(cache, q, seq_lens, T, n_split=n_split)
    H.check_attention(o, l, o_ref, lse_ref, f"D={D} Hq={Hq} n_q={n_q} split={n_split}")


def test_decode_at_the_split_limit():
    """The largest split count (1024): one 16-token tile per CTA, the merge
    tree over 1024 slots (32 leaves of 32), a grid that does not fit at once;
    and one more split than that is refused."""
    _need_gpu()
    D, Hkv, Hq, B, T = 128, 1, 4, 2, 1024 * 16
    seq_lens = [T, 1000]
    k, v, outl = make_kv(D, Hkv, B, T, seed=77, n_out=2)
    q = inputs.normal_tensor((B, 1, Hq, D), 77, "q", outl)
    signs = inputs.tbq_signs(D)
    qs, d16, codes, n16, _ = oracle_cache(k, v, signs)
    o_ref, lse_ref = oracle_decode_all(q, qs, d16, codes, n16, signs, seq_lens)
    cache = gpu_pack(k, v, signs, T)
    o, l = run_decode(cache, q, seq_lens, T, n_split=1024)
    H.check_attention(o, l, o_ref, lse_ref, "n_split 1024")
    assert ckv.attn_decode_workspace(cache, T, 1, Hq, 1025) == 0


@pytest.mark.parametrize("D,Hkv,Hq,n_q,n_split", [(128, 2, 16, 4, 0), (512, 2, 16, 2, 0), (512, 2, 16, 8, 0),
                                                  (512, 1, 4, 5, 3), (128, 2, 2, 16, 0), (64, 1, 1, 3, 200)])
def test_verify_decode_is_causal_among_the_batch(D, Hkv, Hq, n_q, n_split):
    """Verify batch: query token i of n_q sees [0, seq_len - n_q + i]; rows of
    a group of 8 mix tokens when the head ratio is below 8; a sequence shorter
    than the batch leaves its first tokens with nothing to see."""
    _need_gpu()
    B, T, cap = 3, 203, 224
    seq_lens = [203, 3, 150]
    k, v, outl = make_kv(D, Hkv, B, T, seed=31 + D + Hq + n_q, n_out=max(1, round(0.01 * D)))
    q = inputs.normal_tensor((B, n_q, Hq, D), 31 + D, "qv", outl)
    signs = inputs.tbq_signs(D)
    qs, d16, codes, n16, u = oracle_cache(k, v, signs)
    o_ref = np.zeros((B, n_q, Hq, D))
    lse_ref = np.zeros((B, n_q, Hq))
    for b in range(B):
        T_b = seq_lens[b]
        kh = O.q8_0_dequantize(qs[b, :, :T_b], d16[b, :, :T_b])
        vh = O.tbq3_dequantize(codes[b, :, :T_b], n16[b, :, :T_b], signs)
        o_ref[b], lse_ref[b] = O.verify_decode_reference(q[b], kh, vh, T_b, 1.0 / math.sqrt(D))
    cache = gpu_pack(k, v, signs, cap)
    out = torch.empty((B, n_q, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((B, n_q, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_decode_workspace(cache, T, n_q, Hq, n_split), dtype=torch.uint8, device=DEV)
    sl = torch.tensor(seq_lens, dtype=torch.int32, device=DEV)
    ckv.attn_decode_verify(cache, sl, T, to_dev(q), 1.0 / math.sqrt(D), out, lse, ws, n_split=n_split)
    assert ckv.read_device_flag(ws) == 0
    H.check_attention(out.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"verify D={D} Hq={Hq} n_q={n_q}")


@pytest.mark.parametrize("D,Hkv,Hq,chunk,n_split", [(128, 2, 16, 64, 0), (512, 2, 16, 50, 0), (512, 1, 4, 16, 7),
                                                    (64, 1, 2, 300, 0), (128, 2, 8, 1, 0), (512, 2, 16, 32, 400)])
def test_dca_decode_matches_oracle(D, Hkv, Hq, chunk, n_split):
    """Dual chunk attention: three regime queries over the intra, successive and
    inter key ranges of the last position, merged by log-sum-exp. Head ratios
    below 8 put several regimes in one group of 8 rows; chunk 1 and a chunk
    longer than the sequence are the degenerate cases."""
    _need_gpu()
    B, T, cap = 3, 203, 224
    seq_lens = [203, 0, 150]
    k, v, outl = make_kv(D, Hkv, B, T, seed=41 + D + Hq + chunk, n_out=max(1, round(0.01 * D)))
    q = inputs.normal_tensor((B, 3, Hq, D), 41 + D, "qdca", outl)
    signs = inputs.tbq_signs(D)
    qs, d16, codes, n16, u = oracle_cache(k, v, signs)
    o_ref = np.zeros((B, Hq, D))
    lse_ref = np.zeros((B, Hq))
    for b in range(B):
        T_b = seq_lens[b]
        kh = O.q8_0_dequantize(qs[b, :, :T_b], d16[b, :, :T_b])
        vh = O.tbq3_dequantize(codes[b, :, :T_b], n16[b, :, :T_b], signs)
        o_ref[b], lse_ref[b] = O.dca_decode_reference(q[b], kh, vh, T_b, chunk, 1.0 / math.sqrt(D))
    cache = gpu_pack(k, v, signs, cap)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_decode_dca_workspace(cache, T, Hq, n_split), dtype=torch.uint8, device=DEV)
    sl = torch.tensor(seq_lens, dtype=torch.int32, device=DEV)
    ckv.attn_decode_dca(cache, sl, T, chunk, to_dev(q), 1.0 / math.sqrt(D), out, lse, ws, n_split=n_split)
    assert ckv.read_device_flag(ws) == 0
    H.check_attention(out.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"dca D={D} Hq={Hq} chunk={chunk}")


def test_decode_seq_len_out_of_range_sets_flag():
    _need_gpu()
    D, T = 128, 64
    k, v, outl = make_kv(D, 1, 1, T, seed=3, n_out=1)
    q = inputs.normal_tensor((1, 1, 4, D), 3, "q", outl)
    cache = gpu_pack(k, v, inputs.tbq_signs(D), T)
    ws = torch.zeros(ckv.attn_decode_workspace(cache, T, 1, 4), dtype=torch.uint8, device=DEV)
    out = torch.empty((1, 1, 4, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((1, 1, 4), dtype=torch.float32, device=DEV)
    sl = torch.tensor([T + 16], dtype=torch.int32, device=DEV)   # beyond max_seq_len
    ckv.attn_decode(cache, sl, T, to_dev(q), 0.1, out, lse, ws)
    assert ckv.read_device_flag(ws) == 2                             # reading clears it
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))   # treated as empty, no read past the end
    assert ckv.read_device_flag(ws) == 0
    sl.fill_(T)
    ckv.attn_decode(cache, sl, T, to_dev(q), 0.1, out, lse, ws)
    assert ckv.read_device_flag(ws) == 0
    ckv.attn_decode(cache, sl, T, to_dev(q), 0.1, out, lse, ws)    # the workspace is reused as is
    assert ckv.read_device_flag(ws) == 0


# ----------------------------------------------------------- fp16 decode ----

def run_decode_f16(k16, v16, q, seq_lens, max_seq_len, n_split=0):
    B, n_q, Hq, D = q.shape
    out = torch.empty((B, n_q, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((B, n_q, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_decode_f16_workspace(D, k16.shape[1], B, max_seq_len, n_q, Hq, n_split),
                     dtype=torch.uint8, device=DEV)
    sl = torch.tensor(seq_lens, dtype=torch.int32, device=DEV)
    ckv.attn_decode_f16(k16, v16, sl, max_seq_len, to_dev(q), 1.0 / math.sqrt(D), out, lse, ws,
                        n_split=n_split)
    assert ckv.read_device_flag(ws) == 0
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("D,Hkv,Hq,n_q", [(64, 1, 2, 1), (128, 2, 8, 2), (256, 1, 8, 1), (512, 2, 16, 1)])
@pytest.mark.parametrize("n_split", [0, 37])
def test_decode_f16_matches_oracle(D, Hkv, Hq, n_q, n_split):
    _need_gpu()
    B, cap = 3, 144
    seq_lens = [144, 77, 0]
    outl = inputs.outlier_channels(D, max(1, D // 100), 11)
    k = inputs.normal_tensor((B, Hkv, cap, D), 11 + D, "k16", outl)
    v = inputs.normal_tensor((B, Hkv, cap, D), 11 + D, "v16", outl)
    q = inputs.normal_tensor((B, n_q, Hq, D), 11 + D, "q16", outl)
    o_ref = np.zeros((B, n_q, Hq, D))
    lse_ref = np.zeros((B, n_q, Hq))
    for b in range(B):
        o_ref[b], lse_ref[b] = O.decode_reference(q[b], k[b].astype(np.float64), v[b].astype(np.float64),
                                                  seq_lens[b], 1.0 / math.sqrt(D))
    o, l = run_decode_f16(to_dev(k), to_dev(v), q, seq_lens, cap, n_split=n_split)
    H.check_attention(o, l, o_ref, lse_ref, f"f16 D={D} n_split={n_split}")


# -------------------------------------------------------------- lse_merge ---

def test_lse_merge_matches_oracle():
    _need_gpu()
    rng = np.random.default_rng(21)
    n_parts, rows, d = 3, 40, 512
    os_ = [rng.standard_normal((rows, d)).astype(np.float32) for _ in range(n_parts)]
    ls = [(rng.standard_normal(rows) * 5).astype(np.float32) for _ in range(n_parts)]
    ls[1][:7] = -np.inf            # some empty partials
    for p in range(n_parts):
        ls[p][10] = -np.inf        # a row where every partial is empty
        os_[p][10] = 0.0
    o_ref, l_ref = O.lse_merge([x.astype(np.float64) for x in os_], [x.astype(np.float64) for x in ls])
    out = torch.empty((rows, d), dtype=torch.float32, device=DEV)
    lse = torch.empty(rows, dtype=torch.float32, device=DEV)
    ckv.lse_merge([to_dev(x) for x in os_], [to_dev(x) for x in ls], out, lse)
    torch.cuda.synchronize()
    assert np.abs(out.cpu().numpy() - o_ref).max() <= 1e-5 * np.abs(o_ref).max()
    lg = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.abs(lg[fin] - l_ref[fin]).max() < 1e-5
