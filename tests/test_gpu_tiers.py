"""GPU parity of the other TurboQuant tiers, 2 and 4 bits per V code (4 and 16
Lloyd-Max levels), against the float64 oracle: packing (q8_0 bytes bit-exact,
V codes equal except at centroid-midpoint ties, norms within one ulp) and the
decode family (plain, on the oracle's own bytes and end to end; verify batch;
dual chunk attention; append), with the same attention acceptance as 3 bits."""
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
BITS = [2, 4]


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def make_kv(D, Hkv, B, T, seed, name="tier"):
    outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), seed)
    k = inputs.normal_tensor((B, T, Hkv, D), seed, name + "/k", outl)
    v = inputs.normal_tensor((B, T, Hkv, D), seed, name + "/v", outl)
    return k, v, outl


def oracle_fields(k, v, signs, bits):
    kt = np.ascontiguousarray(np.swapaxes(k, 1, 2))
    vt = np.ascontiguousarray(np.swapaxes(v, 1, 2))
    return H.oracle_quantize(kt, vt, signs, bits)


def gpu_pack(k, v, signs, cap, bits, offsets=None):
    B, T, Hkv, D = k.shape
    cache = ckv.PackedCache(D, Hkv, B, cap, signs, v_bits=bits)
    kd, vd = to_dev(k), to_dev(v)
    for a, b in (offsets or [(0, T)]):
        ckv.kv_pack(cache, a, kd[:, a:b], vd[:, a:b])
    torch.cuda.synchronize()
    return cache


def dense(qs, d16, codes, n16, signs, bits, b, T):
    return (O.q8_0_dequantize(qs[b, :, :T], d16[b, :, :T]),
            O.tbq_dequantize(codes[b, :, :T], n16[b, :, :T], signs, bits))


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("D", [64, 128, 256, 512])
def test_pack_matches_oracle(D, bits):
    _need_gpu()
    B, Hkv, T, cap = 2, 2, 77, 96
    k, v, _ = make_kv(D, Hkv, B, T, seed=300 + D + bits)
    k[0, 5, 1] = 0.0
    v[1, 9, 0] = 0.0   # zero vector: norm 0, code 2^(bits-1) everywhere
    signs = inputs.tbq_signs(D)
    cache = gpu_pack(k, v, signs, cap, bits, offsets=[(0, 21), (21, T)])
    qs, d16, codes, n16, u = oracle_fields(k, v, signs, bits)
    recs = cache.data.view(B, Hkv, cap // 16, 17 * D + 2 * bits * D + 32).cpu().numpy()
    for b in range(B):
        for h in range(Hkv):
            H.compare_pack(recs[b, h], qs[b, h], d16[b, h], codes[b, h], n16[b, h], u[b, h], T, bits)
    assert codes.max() == (1 << bits) - 1


def _decode(cache, q, seq_lens, maxs, n_split=0, kind="decode", chunk=0):
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


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("D,Hkv,Hq,n_q", [(64, 2, 4, 1), (128, 2, 16, 1), (256, 2, 8, 3), (512, 2, 16, 1),
                                          (512, 1, 8, 2)])
@pytest.mark.parametrize("n_split", [0, 5, 300])
def test_decode_matches_oracle(D, Hkv, Hq, n_q, n_split, bits):
    _need_gpu()
    B, T, cap = 3, 203, 224
    seq_lens = [203, 0, 150]
    k, v, outl = make_kv(D, Hkv, B, T, seed=17 + D + Hq + n_q + bits)
    q = inputs.normal_tensor((B, n_q, Hq, D), 17 + D + bits, "tq", outl)
    signs = inputs.tbq_signs(D)
    qs, d16, codes, n16, _ = oracle_fields(k, v, signs, bits)
    o_ref = np.zeros((B, n_q, Hq, D))
    lse_ref = np.zeros((B, n_q, Hq))
    for b in range(B):
        kh, vh = dense(qs, d16, codes, n16, signs, bits, b, seq_lens[b])
        o_ref[b], lse_ref[b] = O.decode_reference(q[b], kh, vh, seq_lens[b], 1.0 / math.sqrt(D))
    what = f"b={bits} D={D} Hq={Hq} n_q={n_q} split={n_split}"
    # (i) the oracle's own bytes
    recs = H.oracle_records(qs, d16, codes, n16, cap, bits)
    cache_i = ckv.PackedCache(D, Hkv, B, cap, signs, data=to_dev(recs.ravel()), v_bits=bits)
    o, l = _decode(cache_i, q, seq_lens, T, n_split)
    H.check_attention(o, l, o_ref, lse_ref, what + " (i)")
    # (ii) end to end
    o, l = _decode(gpu_pack(k, v, signs, cap, bits), q, seq_lens, T, n_split)
    H.check_attention(o, l, o_ref, lse_ref, what + " (ii)")


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("D,Hkv,Hq,n_q", [(128, 2, 16, 4), (512, 2, 16, 2)])
def test_verify_decode_matches_oracle(D, Hkv, Hq, n_q, bits):
    _need_gpu()
    B, T, cap = 3, 203, 224
    seq_lens = [203, 3, 150]
    k, v, outl = make_kv(D, Hkv, B, T, seed=51 + D + bits)
    q = inputs.normal_tensor((B, n_q, Hq, D), 51 + D, "tqv", outl)
    signs = inputs.tbq_signs(D)
    qs, d16, codes, n16, _ = oracle_fields(k, v, signs, bits)
    o_ref = np.zeros((B, n_q, Hq, D))
    lse_ref = np.zeros((B, n_q, Hq))
    for b in range(B):
        kh, vh = dense(qs, d16, codes, n16, signs, bits, b, seq_lens[b])
        o_ref[b], lse_ref[b] = O.verify_decode_reference(q[b], kh, vh, seq_lens[b], 1.0 / math.sqrt(D))
    o, l = _decode(gpu_pack(k, v, signs, cap, bits), q, seq_lens, T, kind="verify")
    H.check_attention(o, l, o_ref, lse_ref, f"verify b={bits} D={D}")


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("D,Hkv,Hq,chunk,n_split", [(128, 2, 16, 64, 0), (512, 2, 16, 50, 7)])
def test_dca_decode_matches_oracle(D, Hkv, Hq, chunk, n_split, bits):
    _need_gpu()
    B, T, cap = 3, 203, 224
    seq_lens = [203, 0, 150]
    k, v, outl = make_kv(D, Hkv, B, T, seed=61 + D + bits)
    q = inputs.normal_tensor((B, 3, Hq, D), 61 + D, "tqd", outl)
    signs = inputs.tbq_signs(D)
    qs, d16, codes, n16, _ = oracle_fields(k, v, signs, bits)
    o_ref = np.zeros((B, Hq, D))
    lse_ref = np.zeros((B, Hq))
    for b in range(B):
        kh, vh = dense(qs, d16, codes, n16, signs, bits, b, seq_lens[b])
        o_ref[b], lse_ref[b] = O.dca_decode_reference(q[b], kh, vh, seq_lens[b], chunk, 1.0 / math.sqrt(D))
    o, l = _decode(gpu_pack(k, v, signs, cap, bits), q, seq_lens, T, n_split, kind="dca", chunk=chunk)
    H.check_attention(o, l, o_ref, lse_ref, f"dca b={bits} D={D} chunk={chunk}")


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("D,lens,n_new,cap", [(128, [37, 256], 1, 256), (512, [64, 33], 16, 64)])
def test_append_writes_kv_pack_bytes_and_matches_oracle(D, lens, n_new, cap, bits):
    """The decode's own append leaves the bytes kv_pack writes and attends over them."""
    _need_gpu()
    B, Hkv, Hq = len(lens), 2, 8
    k, v, outl = make_kv(D, Hkv, B, cap, seed=71 + D + bits)
    q = inputs.normal_tensor((B, 1, Hq, D), 71 + D, "tqa", outl)
    signs = inputs.tbq_signs(D)
    kd, vd = to_dev(k), to_dev(v)
    fused = ckv.PackedCache(D, Hkv, B, cap, signs, v_bits=bits)
    ckv.kv_pack(fused, 0, kd, vd)
    per = ckv.cache_bytes(D, Hkv, 1, cap, bits)
    k_new = torch.zeros((B, n_new, Hkv, D), dtype=torch.float16, device=DEV)
    v_new = torch.zeros_like(k_new)
    for b, L in enumerate(lens):
        k_new[b] = kd[b, L - n_new:L]
        v_new[b] = vd[b, L - n_new:L]
        # stale contents at the new positions: the append must overwrite them
        view = ckv.PackedCache(D, Hkv, 1, cap, signs, data=fused.data[b * per:(b + 1) * per], v_bits=bits)
        ckv.kv_pack(view, L - n_new, torch.flip(k_new[b:b + 1], [1]).contiguous(),
                    (v_new[b:b + 1] * -0.5).contiguous())
    ref = gpu_pack(k, v, signs, cap, bits)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = torch.empty((B, 1, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((B, 1, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_decode_workspace(fused, max(lens), 1, Hq), dtype=torch.uint8, device=DEV)
    ckv.attn_decode_append(fused, sl, max(lens), k_new, v_new, to_dev(q), 1.0 / math.sqrt(D), out, lse, ws)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    assert torch.equal(fused.data, ref.data), "append wrote different cache bytes than kv_pack"
    qs, d16, codes, n16, _ = oracle_fields(k, v, signs, bits)
    o_ref = np.zeros((B, 1, Hq, D))
    lse_ref = np.zeros((B, 1, Hq))
    for b in range(B):
        kh, vh = dense(qs, d16, codes, n16, signs, bits, b, lens[b])
        o_ref[b], lse_ref[b] = O.decode_reference(q[b], kh, vh, lens[b], 1.0 / math.sqrt(D))
    H.check_attention(out.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"append b={bits} D={D}")
