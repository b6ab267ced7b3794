"""GPU checks of attn_decode_append (pack the new rows inside the decode kernel,
then attend): the cache bytes it leaves equal those of kv_pack of the same rows,
and its outputs equal attn_decode's over that cache bit for bit; one case is
also checked against the oracle."""
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


def _cache_view(cache, b):
    """batch-1 view of sequence b of a packed cache (its records are contiguous)."""
    per = ckv.cache_bytes(cache.head_dim, cache.n_kv_heads, 1, cache.capacity)
    return ckv.PackedCache(cache.head_dim, cache.n_kv_heads, 1, cache.capacity, cache.signs.cpu().numpy(),
                           data=cache.data[b * per:(b + 1) * per])


def _run(D, Hkv, Hq, lens, n_new, cap, n_split, seed):
    B = len(lens)
    outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), seed)
    signs = inputs.tbq_signs(D)
    k = torch.from_numpy(inputs.normal_tensor((B, cap, Hkv, D), seed, "ap/k", outl)).to(DEV)
    v = torch.from_numpy(inputs.normal_tensor((B, cap, Hkv, D), seed, "ap/v", outl)).to(DEV)
    # Old contents at the new positions differ from the new rows: the append must clear them.
    k_old = torch.from_numpy(inputs.normal_tensor((B, cap, Hkv, D), seed, "ap/k_old", outl)).to(DEV)
    v_old = torch.from_numpy(inputs.normal_tensor((B, cap, Hkv, D), seed, "ap/v_old", outl)).to(DEV)
    q = torch.from_numpy(inputs.normal_tensor((B, 1, Hq, D), seed, "ap/q", outl)).to(DEV)
    k_new = torch.zeros((B, n_new, Hkv, D), dtype=torch.float16, device=DEV)
    v_new = torch.zeros_like(k_new)
    for b, L in enumerate(lens):
        k_new[b] = k[b, L - n_new:L]
        v_new[b] = v[b, L - n_new:L]

    base = ckv.PackedCache(D, Hkv, B, cap, signs)
    ckv.kv_pack(base, 0, k, v)
    for b, L in enumerate(lens):  # stale rows where the new ones go
        view = _cache_view(base, b)
        ckv.kv_pack(view, L - n_new, k_old[b:b + 1, L - n_new:L].contiguous(),
                    v_old[b:b + 1, L - n_new:L].contiguous())
    fused = ckv.PackedCache(D, Hkv, B, cap, signs, data=base.data.clone())
    ref = ckv.PackedCache(D, Hkv, B, cap, signs, data=base.data.clone())
    for b, L in enumerate(lens):
        ckv.kv_pack(_cache_view(ref, b), L - n_new, k_new[b:b + 1].contiguous(), v_new[b:b + 1].contiguous())

    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    maxs = max(lens)
    scale = 1.0 / math.sqrt(D)
    outs = []
    for kind, cache in (("append", fused), ("decode", ref)):
        out = torch.full((B, 1, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
        lse = torch.full((B, 1, Hq), float("nan"), dtype=torch.float32, device=DEV)
        ws = torch.zeros(ckv.attn_decode_workspace(cache, maxs, 1, Hq, n_split), dtype=torch.uint8, device=DEV)
        if kind == "append":
            ckv.attn_decode_append(cache, seq, maxs, k_new, v_new, q, scale, out, lse, ws, n_split=n_split)
        else:
            ckv.attn_decode(cache, seq, maxs, q, scale, out, lse, ws, n_split=n_split)
        torch.cuda.synchronize()
        assert ckv.read_device_flag(ws) == 0
        outs.append((out.cpu(), lse.cpu()))
    assert torch.equal(fused.data, ref.data), "append wrote different cache bytes than kv_pack"
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    return k, v, q, signs, outs[0]


@pytest.mark.parametrize("D,lens,n_new,cap,n_split", [
    (128, [37, 256], 1, 256, 0),      # ragged lengths, auto split
    (256, [17, 100], 3, 128, 0),      # new rows straddle a tile boundary (14..16)
    (512, [64, 33], 16, 64, 0),       # a whole tile of new rows; 33 - 16 straddles
    (512, [32768, 20000], 1, 32768, 0),  # Gemma-4 decode shape
    (128, [48, 17], 2, 64, 3),        # one split per tile: the new rows of one sequence span two CTAs
    (256, [200, 1], 1, 256, 1),       # a single split, a one-token sequence
])
def test_append_matches_pack_then_decode(D, lens, n_new, cap, n_split):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _run(D, 2, 16, lens, n_new, cap, n_split, seed=70 + D + n_new)


def test_append_against_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    D, Hkv, Hq, lens = 128, 2, 16, [45, 160]
    k, v, q, signs, (out, lse) = _run(D, Hkv, Hq, lens, 2, 160, 0, seed=91)
    kn, vn, qn = k.cpu().numpy(), v.cpu().numpy(), q.cpu().numpy().astype(np.float64)
    for b, L in enumerate(lens):
        qs, d16, codes, n16, _ = H.oracle_quantize(np.swapaxes(kn[b, :L], 0, 1), np.swapaxes(vn[b, :L], 0, 1),
                                                   signs)
        kh = O.q8_0_dequantize(qs, d16)
        vh = O.tbq3_dequantize(codes, n16, signs)
        o_ref, l_ref = O.decode_reference(qn[b], kh, vh, L, 1.0 / math.sqrt(D))
        H.check_attention(out[b].numpy(), lse[b].numpy(), o_ref, l_ref, f"append b={b}")


@pytest.mark.parametrize("D,Hkv,Hq,lens,n_new", [(512, 2, 16, [4096], 1), (128, 1, 4, [200, 64, 131], 2)])
def test_append_host_matches_device_append(D, Hkv, Hq, lens, n_new):
    """ckv_attn_decode_append_host (pinned host buffers read and written by the
    kernel, no staging copies) leaves the same cache bytes and returns the
    same outputs, bit for bit, as attn_decode_append on device buffers; host
    memory that is not page-locked is refused before any launch."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, cap, seed = len(lens), (max(lens) + 15) // 16 * 16 + 16, 90 + D
    outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), seed)
    signs = inputs.tbq_signs(D)
    k = torch.from_numpy(inputs.normal_tensor((B, cap, Hkv, D), seed, "ah/k", outl)).to(DEV)
    v = torch.from_numpy(inputs.normal_tensor((B, cap, Hkv, D), seed, "ah/v", outl)).to(DEV)
    q = inputs.normal_tensor((B, 1, Hq, D), seed, "ah/q", outl)
    kn = np.stack([inputs.normal_tensor((n_new, Hkv, D), seed + b, "ah/kn", outl) for b in range(B)])
    vn = np.stack([inputs.normal_tensor((n_new, Hkv, D), seed + b, "ah/vn", outl) for b in range(B)])
    base = ckv.PackedCache(D, Hkv, B, cap, signs)
    ckv.kv_pack(base, 0, k, v)
    dev_c = ckv.PackedCache(D, Hkv, B, cap, signs, data=base.data.clone())
    host_c = ckv.PackedCache(D, Hkv, B, cap, signs, data=base.data.clone())
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(D)
    ws = torch.zeros(ckv.attn_decode_workspace(dev_c, max(lens), 1, Hq), dtype=torch.uint8, device=DEV)
    out_d = torch.empty((B, 1, Hq, D), dtype=torch.float32, device=DEV)
    lse_d = torch.empty((B, 1, Hq), dtype=torch.float32, device=DEV)
    ckv.attn_decode_append(dev_c, seq, max(lens), torch.from_numpy(kn).to(DEV), torch.from_numpy(vn).to(DEV),
                           torch.from_numpy(q).to(DEV), scale, out_d, lse_d, ws)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()  # noqa: E731
    q_h, k_h, v_h = pin(q), pin(kn), pin(vn)
    out_h = torch.full((B, 1, Hq, D), float("nan"), dtype=torch.float32).pin_memory()
    lse_h = torch.full((B, 1, Hq), float("nan"), dtype=torch.float32).pin_memory()
    ws2 = torch.zeros_like(ws)
    ckv.attn_decode_append_host(host_c, seq, max(lens), k_h, v_h, q_h, scale, out_h, lse_h, ws2)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws2) == 0
    assert torch.equal(host_c.data, dev_c.data)
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu())
    unpinned = torch.zeros_like(out_h, device="cpu").clone()
    assert not unpinned.is_pinned()
    with pytest.raises(ckv.CkvError) as err:
        ckv.attn_decode_append_host(host_c, seq, max(lens), k_h, v_h, q_h, scale, unpinned, lse_h, ws2)
    assert err.value.status == -1 and "page-locked" in str(err.value)
