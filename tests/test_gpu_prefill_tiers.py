"""GPU parity of the tcgen05 prefill over the other V tiers (2 and 4 bits per
code) and over the block-diagonal rotation (128-dim groups, a sign diagonal
before and after each group's Walsh-Hadamard transform, one norm per group)
against the float64 oracle: the new rows are packed at the cache's tier, then
query i of the chunk attends causally to positions [0, n_cached + i]. Also a
stream-K schedule (tiles cut between two CTAs) and the prefix-only form."""
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


def _signs(D, rot):
    return inputs.tbq_signs(D), (inputs.tbq_signs(D, seed=43) if rot else None)


def _inputs(D, Hkv, Hq, B, T, n_q, seed):
    outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), seed)
    k = inputs.normal_tensor((B, T, Hkv, D), seed, "pft/k", outl)
    v = inputs.normal_tensor((B, T, Hkv, D), seed, "pft/v", outl)
    q = inputs.normal_tensor((B, n_q, Hq, D), seed, "pft/q", outl, dtype="bfloat16", torch_out=True)
    return k, v, q


def _cache(D, Hkv, B, cap, bits, rot, fill=0):
    s1, s2 = _signs(D, rot)
    data = torch.full((ckv.cache_bytes(D, Hkv, B, cap, bits, 128 if rot else 0),), fill, dtype=torch.uint8,
                      device=DEV)
    return ckv.PackedCache(D, Hkv, B, cap, s1, data=data, v_bits=bits, signs2=s2)


def run_prefill(D, Hkv, Hq, B, n_cached, n_new, cap, bits, rot, seed, fill=0):
    """Pack n_cached rows, then prefill n_new more; `fill` is the byte the cache
    held before any packing."""
    k, v, q = _inputs(D, Hkv, Hq, B, n_cached + n_new, n_new, seed)
    cache = _cache(D, Hkv, B, cap, bits, rot, fill)
    kd, vd = torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV)
    if n_cached:
        ckv.kv_pack(cache, 0, kd[:, :n_cached].contiguous(), vd[:, :n_cached].contiguous())
    out = torch.full((B, n_new, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((B, n_new, Hq), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_prefill_workspace(cache, n_new, Hq), dtype=torch.uint8, device=DEV)
    ckv.attn_prefill(cache, n_cached, q.to(DEV), kd[:, n_cached:].contiguous(), vd[:, n_cached:].contiguous(),
                     1.0 / math.sqrt(D), out, lse, ws)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    return k, v, q.float().numpy().astype(np.float64), out.cpu().numpy(), lse.cpu().numpy()


def dequantised(k, v, b, bits, rot):
    """Oracle K_hat, V_hat [Hkv, T, D] of sequence b at the cache's tier and rotation."""
    D = k.shape[-1]
    s1, s2 = _signs(D, rot)
    kt = np.ascontiguousarray(np.swapaxes(k[b], 0, 1))
    vt = np.ascontiguousarray(np.swapaxes(v[b], 0, 1))
    qs, d16, codes, n16, _ = H.oracle_quantize(kt, vt, s1, bits, signs2=s2)
    kh = O.q8_0_dequantize(qs, d16)
    vh = O.tbq_dequantize_blocked(codes, n16, s1, s2, bits) if rot else O.tbq_dequantize(codes, n16, s1, bits)
    return kh, vh


def check_prefill(D, Hkv, Hq, B, n_cached, n_new, cap, bits, rot, seed, fill=0):
    k, v, qf, out, lse = run_prefill(D, Hkv, Hq, B, n_cached, n_new, cap, bits, rot, seed, fill)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    for b in range(B):
        kh, vh = dequantised(k, v, b, bits, rot)
        o_ref, l_ref = O.prefill_reference(qf[b], kh, vh, n_cached, 1.0 / math.sqrt(D))
        H.check_attention(out[b], lse[b], o_ref, l_ref, f"prefill b={bits} rot={rot} D={D} seq={b}")


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("D,Hkv,Hq,n_cached,n_new", [(64, 1, 4, 50, 33), (128, 2, 16, 100, 37),
                                                     (512, 2, 16, 131, 45)])
def test_prefill_tiers(D, Hkv, Hq, n_cached, n_new, bits):
    _need_gpu()
    cap = ((n_cached + n_new + 15) // 16) * 16 + 16
    check_prefill(D, Hkv, Hq, 2, n_cached, n_new, cap, bits, False, seed=900 + D + bits)


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("D,Hkv,Hq,n_cached,n_new", [(128, 2, 16, 100, 37), (256, 1, 4, 64, 80),
                                                     (512, 2, 16, 131, 45), (512, 1, 8, 0, 20)])
def test_prefill_rotation(D, Hkv, Hq, n_cached, n_new, bits):
    _need_gpu()
    cap = ((n_cached + n_new + 15) // 16) * 16 + 16
    check_prefill(D, Hkv, Hq, 2, n_cached, n_new, cap, bits, True, seed=950 + D + bits)


def test_prefill_rotation_stream_k():
    """320 tiles of 16 tokens x 8 heads (more than the SMs): the stream-K
    schedule with tiles cut between CTAs, at 4 bits with the rotation; every
    row checked."""
    _need_gpu()
    D, Hkv, Hq, nc, nn = 128, 2, 16, 64, 2560
    check_prefill(D, Hkv, Hq, 1, nc, nn, nc + nn + 16, 4, True, seed=977)


@pytest.mark.parametrize("bits,rot", [(2, False), (4, True)])
def test_prefill_prefix_tiers(bits, rot):
    """Prefix-only form over a cache of another tier: every query sees the
    packed prefix [0, P) and nothing else."""
    _need_gpu()
    D, Hkv, Hq, B, P, n_tok = 512, 2, 16, 1, 203, 40
    k, v, q = _inputs(D, Hkv, Hq, B, P, n_tok, seed=990 + bits)
    cache = _cache(D, Hkv, B, P + 21, bits, rot)   # capacity 224
    ckv.kv_pack(cache, 0, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    out = torch.empty((B, n_tok, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((B, n_tok, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_prefill_workspace(cache, n_tok, Hq), dtype=torch.uint8, device=DEV)
    ckv.attn_prefill_prefix(cache, P, q.to(DEV), 1.0 / math.sqrt(D), out, lse, ws)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    kh, vh = dequantised(k, v, 0, bits, rot)
    qf = q.float().numpy().astype(np.float64)[0]
    o_ref, l_ref = np.zeros((n_tok, Hq, D)), np.zeros((n_tok, Hq))
    for h in range(Hq):
        kv = O.kv_head_of(h, Hq, Hkv)
        o_ref[:, h], l_ref[:, h] = O.attention(qf[:, h], kh[kv, :P], vh[kv, :P], 1.0 / math.sqrt(D))
    H.check_attention(out.cpu().numpy()[0], lse.cpu().numpy()[0], o_ref, l_ref, f"prefix b={bits} rot={rot}")
