"""Positions that were never written may hold any bytes. Every path that reads
a whole 16-position tile (or a whole 64-key prefill step) past seq_len must
keep those bytes out of the result: a NaN there (fp16 0xFFFF) would otherwise
reach O through a probability of exactly zero. Each case fills the cache (or
the fp16 tails) with 0xFF bytes before packing, leaves the last tile partly
unwritten, and compares with the float64 oracle, which sees only the written
positions."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import compressed_kv_attention_gb300 as ckv  # noqa: E402
from compressed_kv_attention_gb300 import inputs  # noqa: E402
from oracle import ckv_oracle as O  # noqa: E402
from tests import helpers as H  # noqa: E402
from tests import test_gpu_prefill_tiers as PT  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _decode(cache, q, seq_lens, maxs, kind):
    B, n_q, Hq, D = q.shape
    scale = 1.0 / math.sqrt(D)
    sl = torch.tensor(seq_lens, dtype=torch.int32, device=DEV)
    qd = torch.from_numpy(np.ascontiguousarray(q)).to(DEV)
    if kind == "dca":
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=DEV)
        lse = torch.empty((B, Hq), dtype=torch.float32, device=DEV)
        ws = torch.zeros(ckv.attn_decode_dca_workspace(cache, maxs, Hq), dtype=torch.uint8, device=DEV)
        ckv.attn_decode_dca(cache, sl, maxs, 64, qd, scale, out, lse, ws)
    else:
        out = torch.empty((B, n_q, Hq, D), dtype=torch.float32, device=DEV)
        lse = torch.empty((B, n_q, Hq), dtype=torch.float32, device=DEV)
        ws = torch.zeros(ckv.attn_decode_workspace(cache, maxs, n_q, Hq), dtype=torch.uint8, device=DEV)
        fn = ckv.attn_decode_verify if kind == "verify" else ckv.attn_decode
        fn(cache, sl, maxs, qd, scale, out, lse, ws)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("bits,rot", [(3, False), (3, True), (4, True), (2, False)])
@pytest.mark.parametrize("T", [203, 77])
def test_decode_family_ignores_unwritten_bytes(bits, rot, T):
    _need_gpu()
    D, Hkv, Hq, B, cap = 512, 2, 16, 1, 256
    k, v, _ = PT._inputs(D, Hkv, Hq, B, T, 1, seed=1100 + T + bits)
    outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), 1100 + T)
    cache = PT._cache(D, Hkv, B, cap, bits, rot, fill=0xFF)
    ckv.kv_pack(cache, 0, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    kh, vh = PT.dequantised(k, v, 0, bits, rot)
    scale = 1.0 / math.sqrt(D)
    what = f"b={bits} rot={rot} T={T}"
    # The packer clears a position's V bits before setting them: the written
    # positions' fields match the oracle whatever the record held before.
    s1, s2 = PT._signs(D, rot)
    qs, d16, codes, n16, u = H.oracle_quantize(np.ascontiguousarray(np.swapaxes(k[0], 0, 1)),
                                               np.ascontiguousarray(np.swapaxes(v[0], 0, 1)), s1, bits, signs2=s2)
    recs = cache.data.view(B, Hkv, cap // 16, -1).cpu().numpy()
    for h in range(Hkv):
        H.compare_pack(recs[0, h], qs[h], d16[h], codes[h], n16[h], u[h], T, bits, D // 128 if rot else 1)
    q = inputs.normal_tensor((B, 1, Hq, D), 1100 + T, "uw/q", outl)
    o, l = _decode(cache, q, [T], cap, "decode")
    o_ref, l_ref = O.decode_reference(q[0], kh, vh, T, scale)
    H.check_attention(o[0], l[0], o_ref, l_ref, "decode " + what)
    qv = inputs.normal_tensor((B, 4, Hq, D), 1100 + T, "uw/qv", outl)
    o, l = _decode(cache, qv, [T], cap, "verify")
    o_ref, l_ref = O.verify_decode_reference(qv[0], kh, vh, T, scale)
    H.check_attention(o[0], l[0], o_ref, l_ref, "verify " + what)
    qd = inputs.normal_tensor((B, 3, Hq, D), 1100 + T, "uw/qd", outl)
    o, l = _decode(cache, qd, [T], cap, "dca")
    o_ref, l_ref = O.dca_decode_reference(qd[0], kh, vh, T, 64, scale)
    H.check_attention(o[0], l[0], o_ref, l_ref, "dca " + what)


@pytest.mark.parametrize("rows", [False, True])
def test_decode_f16_ignores_unwritten_rows(rows):
    """fp16 tails holding NaN past seq_len; `rows`: many query rows per kv head
    (the row-parallel form)."""
    _need_gpu()
    D, Hkv, B, cap = 512, 2, 3, 144
    Hq, n_q = (16, 8) if rows else (16, 1)
    seq_lens = [141, 77, 0]
    outl = inputs.outlier_channels(D, max(1, D // 100), 12)
    k = inputs.normal_tensor((B, Hkv, cap, D), 12, "uw/k16", outl)
    v = inputs.normal_tensor((B, Hkv, cap, D), 12, "uw/v16", outl)
    q = inputs.normal_tensor((B, n_q, Hq, D), 12, "uw/q16", outl)
    for b, L in enumerate(seq_lens):
        k[b, :, L:] = np.nan
        v[b, :, L:] = np.nan
    out = torch.empty((B, n_q, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((B, n_q, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_decode_f16_workspace(D, Hkv, B, cap, n_q, Hq, 1 if rows else 0), dtype=torch.uint8,
                     device=DEV)
    sl = torch.tensor(seq_lens, dtype=torch.int32, device=DEV)
    to = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(DEV)  # noqa: E731
    ckv.attn_decode_f16(to(k), to(v), sl, cap, to(q), 1.0 / math.sqrt(D), out, lse, ws, n_split=1 if rows else 0)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    for b, L in enumerate(seq_lens):
        kb = np.nan_to_num(k[b].astype(np.float64))
        vb = np.nan_to_num(v[b].astype(np.float64))
        o_ref, l_ref = O.decode_reference(q[b], kb, vb, L, 1.0 / math.sqrt(D))
        H.check_attention(o[b], l[b], o_ref, l_ref, f"f16 rows={rows} b={b}")


@pytest.mark.parametrize("bits,rot", [(3, False), (3, True), (2, True)])
def test_prefill_ignores_unwritten_bytes(bits, rot):
    """The last 64-key step runs past n_cached + n_new into never-written bytes."""
    _need_gpu()
    D, Hkv, Hq, nc, nn = 512, 2, 16, 100, 37
    PT.check_prefill(D, Hkv, Hq, 2, nc, nn, 256, bits, rot, seed=1200 + bits, fill=0xFF)


@pytest.mark.parametrize("rot", [False, True])
def test_prefill_prefix_ignores_unwritten_bytes(rot):
    _need_gpu()
    D, Hkv, Hq, B, P, n_tok = 256, 1, 8, 1, 137, 24
    k, v, q = PT._inputs(D, Hkv, Hq, B, P, n_tok, seed=1250)
    cache = PT._cache(D, Hkv, B, 256, 3, rot, fill=0xFF)
    ckv.kv_pack(cache, 0, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    out = torch.empty((B, n_tok, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((B, n_tok, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_prefill_workspace(cache, n_tok, Hq), dtype=torch.uint8, device=DEV)
    ckv.attn_prefill_prefix(cache, P, q.to(DEV), 1.0 / math.sqrt(D), out, lse, ws)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    kh, vh = PT.dequantised(k, v, 0, 3, rot)
    qf = q.float().numpy().astype(np.float64)[0]
    o_ref, l_ref = np.zeros((n_tok, Hq, D)), np.zeros((n_tok, Hq))
    for h in range(Hq):
        o_ref[:, h], l_ref[:, h] = O.attention(qf[:, h], kh[0, :P], vh[0, :P], 1.0 / math.sqrt(D))
    H.check_attention(out.cpu().numpy()[0], lse.cpu().numpy()[0], o_ref, l_ref, f"prefix rot={rot}")
