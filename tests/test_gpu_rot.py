"""GPU parity of the block-diagonal two-sign rotation (128-dim groups, a sign
diagonal before and after each group's Walsh-Hadamard transform, one norm per
group) against the float64 oracle, at 2, 3 and 4 bits: packing (q8_0 bytes
bit-exact, V codes equal except at centroid-midpoint ties, group norms within
one ulp) and the decode family (plain on the oracle's bytes and end to end,
verify batch, dual chunk attention, append)."""
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


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def signs_of(D):
    return inputs.tbq_signs(D), inputs.tbq_signs(D, seed=43)


def make_kv(D, Hkv, B, T, seed):
    outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), seed)
    k = inputs.normal_tensor((B, T, Hkv, D), seed, "rot/k", outl)
    v = inputs.normal_tensor((B, T, Hkv, D), seed, "rot/v", outl)
    return k, v, outl


def oracle_fields(k, v, D, bits):
    s1, s2 = signs_of(D)
    kt = np.ascontiguousarray(np.swapaxes(k, 1, 2))
    vt = np.ascontiguousarray(np.swapaxes(v, 1, 2))
    return H.oracle_quantize(kt, vt, s1, bits, signs2=s2)


def gpu_cache(k, v, cap, bits, offsets=None):
    B, T, Hkv, D = k.shape
    s1, s2 = signs_of(D)
    cache = ckv.PackedCache(D, Hkv, B, cap, s1, v_bits=bits, signs2=s2)
    kd, vd = to_dev(k), to_dev(v)
    for a, b in (offsets or [(0, T)]):
        ckv.kv_pack(cache, a, kd[:, a:b], vd[:, a:b])
    torch.cuda.synchronize()
    return cache


def dense(qs, d16, codes, n16, D, bits, b, T):
    s1, s2 = signs_of(D)
    return (O.q8_0_dequantize(qs[b, :, :T], d16[b, :, :T]),
            O.tbq_dequantize_blocked(codes[b, :, :T], n16[b, :, :T], s1, s2, bits))


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("D", [128, 256, 512])
def test_pack_matches_oracle(D, bits):
    _need_gpu()
    B, Hkv, T, cap = 2, 2, 77, 96
    k, v, _ = make_kv(D, Hkv, B, T, seed=500 + D + bits)
    v[1, 9, 0, 128 * (D // 256):128 * (D // 256) + 128] = 0.0   # one zero group
    cache = gpu_cache(k, v, cap, bits, offsets=[(0, 21), (21, T)])
    qs, d16, codes, n16, u = oracle_fields(k, v, D, bits)
    g = D // 128
    rec = 17 * D + 2 * bits * D + 32 * g
    recs = cache.data.view(B, Hkv, cap // 16, rec).cpu().numpy()
    for b in range(B):
        for h in range(Hkv):
            H.compare_pack(recs[b, h], qs[b, h], d16[b, h], codes[b, h], n16[b, h], u[b, h], T, bits, g)


def _run(cache, q, seq_lens, maxs, kind="decode", chunk=0, n_split=0):
    B, n_q, Hq, D = q.shape
    scale = 1.0 / math.sqrt(D)
    sl = torch.tensor(seq_lens, dtype=torch.int32, device=DEV)
    if kind == "dca":
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=DEV)
        lse = torch.empty((B, Hq), dtype=torch.float32, device=DEV)
        ws = torch.zeros(ckv.attn_decode_dca_workspace(cache, maxs, Hq, n_split), dtype=torch.uint8, device=DEV)
        ckv.attn_decode_dca(cache, sl, maxs, chunk, to_dev(q), scale, out, lse, ws, n_split=n_split)
    else:
        out = torch.empty((B, n_q, Hq, D), dtype=torch.float32, device=DEV)
        lse = torch.empty((B, n_q, Hq), dtype=torch.float32, device=DEV)
        ws = torch.zeros(ckv.attn_decode_workspace(cache, maxs, n_q, Hq, n_split), dtype=torch.uint8, device=DEV)
        fn = ckv.attn_decode_verify if kind == "verify" else ckv.attn_decode
        fn(cache, sl, maxs, to_dev(q), scale, out, lse, ws, n_split=n_split)
    assert ckv.read_device_flag(ws) == 0
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("D,Hkv,Hq,n_q,n_split", [(128, 2, 16, 1, 0), (256, 2, 8, 3, 5), (512, 2, 16, 1, 0),
                                                  (512, 1, 8, 2, 300)])
def test_decode_matches_oracle(D, Hkv, Hq, n_q, n_split, bits):
    _need_gpu()
    B, T, cap = 3, 203, 224
    seq_lens = [203, 0, 150]
    k, v, outl = make_kv(D, Hkv, B, T, seed=600 + D + Hq + bits)
    q = inputs.normal_tensor((B, n_q, Hq, D), 600 + D, "rq", outl)
    qs, d16, codes, n16, _ = oracle_fields(k, v, D, bits)
    o_ref = np.zeros((B, n_q, Hq, D))
    lse_ref = np.zeros((B, n_q, Hq))
    for b in range(B):
        kh, vh = dense(qs, d16, codes, n16, D, bits, b, seq_lens[b])
        o_ref[b], lse_ref[b] = O.decode_reference(q[b], kh, vh, seq_lens[b], 1.0 / math.sqrt(D))
    what = f"rot b={bits} D={D} Hq={Hq} n_q={n_q} split={n_split}"
    s1, s2 = signs_of(D)
    recs = H.oracle_records(qs, d16, codes, n16, cap, bits, D // 128)
    cache_i = ckv.PackedCache(D, Hkv, B, cap, s1, data=to_dev(recs.ravel()), v_bits=bits, signs2=s2)
    o, l = _run(cache_i, q, seq_lens, T, n_split=n_split)
    H.check_attention(o, l, o_ref, lse_ref, what + " (i)")
    o, l = _run(gpu_cache(k, v, cap, bits), q, seq_lens, T, n_split=n_split)
    H.check_attention(o, l, o_ref, lse_ref, what + " (ii)")


@pytest.mark.parametrize("bits", [2, 3])
@pytest.mark.parametrize("D", [256, 512])
def test_verify_and_dca_match_oracle(D, bits):
    _need_gpu()
    B, Hkv, Hq, T, cap = 3, 2, 16, 203, 224
    seq_lens = [203, 3, 150]
    k, v, outl = make_kv(D, Hkv, B, T, seed=700 + D + bits)
    qs, d16, codes, n16, _ = oracle_fields(k, v, D, bits)
    cache = gpu_cache(k, v, cap, bits)
    qv = inputs.normal_tensor((B, 4, Hq, D), 700 + D, "rqv", outl)
    qd = inputs.normal_tensor((B, 3, Hq, D), 700 + D, "rqd", outl)
    ov_ref, lv_ref = np.zeros((B, 4, Hq, D)), np.zeros((B, 4, Hq))
    od_ref, ld_ref = np.zeros((B, Hq, D)), np.zeros((B, Hq))
    for b in range(B):
        kh, vh = dense(qs, d16, codes, n16, D, bits, b, seq_lens[b])
        ov_ref[b], lv_ref[b] = O.verify_decode_reference(qv[b], kh, vh, seq_lens[b], 1.0 / math.sqrt(D))
        od_ref[b], ld_ref[b] = O.dca_decode_reference(qd[b], kh, vh, seq_lens[b], 64, 1.0 / math.sqrt(D))
    o, l = _run(cache, qv, seq_lens, T, kind="verify")
    H.check_attention(o, l, ov_ref, lv_ref, f"rot verify b={bits} D={D}")
    o, l = _run(cache, qd, seq_lens, T, kind="dca", chunk=64)
    H.check_attention(o, l, od_ref, ld_ref, f"rot dca b={bits} D={D}")


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("D,lens,n_new,cap", [(128, [37, 256], 1, 256), (512, [64, 33], 16, 64)])
def test_append_writes_kv_pack_bytes(D, lens, n_new, cap, bits):
    _need_gpu()
    B, Hkv, Hq = len(lens), 2, 8
    k, v, outl = make_kv(D, Hkv, B, cap, seed=800 + D + bits)
    q = inputs.normal_tensor((B, 1, Hq, D), 800 + D, "rqa", outl)
    s1, s2 = signs_of(D)
    kd, vd = to_dev(k), to_dev(v)
    fused = ckv.PackedCache(D, Hkv, B, cap, s1, v_bits=bits, signs2=s2)
    ckv.kv_pack(fused, 0, kd, vd)
    per = ckv.cache_bytes(D, Hkv, 1, cap, bits, 128)
    k_new = torch.zeros((B, n_new, Hkv, D), dtype=torch.float16, device=DEV)
    v_new = torch.zeros_like(k_new)
    for b, L in enumerate(lens):
        k_new[b] = kd[b, L - n_new:L]
        v_new[b] = vd[b, L - n_new:L]
        view = ckv.PackedCache(D, Hkv, 1, cap, s1, data=fused.data[b * per:(b + 1) * per], v_bits=bits, signs2=s2)
        ckv.kv_pack(view, L - n_new, torch.flip(k_new[b:b + 1], [1]).contiguous(),
                    (v_new[b:b + 1] * -0.5).contiguous())
    ref = gpu_cache(k, v, cap, bits)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = torch.empty((B, 1, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((B, 1, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_decode_workspace(fused, max(lens), 1, Hq), dtype=torch.uint8, device=DEV)
    ckv.attn_decode_append(fused, sl, max(lens), k_new, v_new, to_dev(q), 1.0 / math.sqrt(D), out, lse, ws)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    assert torch.equal(fused.data, ref.data), "append wrote different cache bytes than kv_pack"
    qs, d16, codes, n16, _ = oracle_fields(k, v, D, bits)
    o_ref, lse_ref = np.zeros((B, 1, Hq, D)), np.zeros((B, 1, Hq))
    for b in range(B):
        kh, vh = dense(qs, d16, codes, n16, D, bits, b, lens[b])
        o_ref[b], lse_ref[b] = O.decode_reference(q[b], kh, vh, lens[b], 1.0 / math.sqrt(D))
    H.check_attention(out.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"rot append b={bits} D={D}")
