"""GPU parity of the multi-tenant prefill pieces against the float64 oracle:
queries of several agents over one shared compressed prefix (tcgen05 prefill in
prefix-only mode), causal prefill over private fp16 tails, the fp16 tail
append, and the composite (tails + prefix + exact merge)."""
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


def _prefix(D, Hkv, P, seed, cap=None):
    """A packed one-sequence prefix cache and its oracle dequantisation [Hkv, P, D]."""
    outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), seed)
    k = inputs.normal_tensor((1, P, Hkv, D), seed, "sp/k", outl)
    v = inputs.normal_tensor((1, P, Hkv, D), seed, "sp/v", outl)
    signs = inputs.tbq_signs(D)
    cap = cap or ((P + 15) // 16 * 16 + 16)
    cache = ckv.PackedCache(D, Hkv, 1, cap, signs)
    if P:
        ckv.kv_pack(cache, 0, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    if P == 0:
        return cache, np.zeros((Hkv, 0, D)), np.zeros((Hkv, 0, D)), outl
    qs, d16, codes, n16, _ = H.oracle_quantize(np.swapaxes(k[0], 0, 1), np.swapaxes(v[0], 0, 1), signs)
    return cache, O.q8_0_dequantize(qs, d16), O.tbq3_dequantize(codes, n16, signs), outl


@pytest.mark.parametrize("D,Hkv,Hq,P,n_tok", [(128, 2, 16, 200, 300), (512, 2, 16, 131, 45), (256, 1, 4, 64, 80),
                                              (64, 1, 4, 50, 33), (512, 2, 16, 70, 3000)])
def test_prefill_prefix_matches_oracle(D, Hkv, Hq, P, n_tok):
    """Every query sees exactly the prefix; 3000 tokens x 8 heads per kv head
    makes 376 tiles: the stream-K schedule with cut tiles."""
    _need_gpu()
    cache, kh, vh, outl = _prefix(D, Hkv, P, seed=90 + D)
    q = inputs.normal_tensor((1, n_tok, Hq, D), 91 + D, "sp/q", outl, dtype="bfloat16", torch_out=True)
    out = torch.full((1, n_tok, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((1, n_tok, Hq), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_prefill_workspace(cache, n_tok, Hq), dtype=torch.uint8, device=DEV)
    ckv.attn_prefill_prefix(cache, P, q.to(DEV), 1.0 / math.sqrt(D), out, lse, ws)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    qf = q.float().numpy().astype(np.float64)[0]
    rows = np.arange(n_tok) if n_tok <= 300 else np.r_[0:40, n_tok // 2:n_tok // 2 + 40, n_tok - 40:n_tok]
    o_ref, l_ref = O.decode_reference(qf[rows], kh, vh, P, 1.0 / math.sqrt(D))
    H.check_attention(out.cpu().numpy()[0][rows], lse.cpu().numpy()[0][rows], o_ref, l_ref, f"prefix D={D} P={P}")


def _tails(D, Hkv, A, cap, lens, seed):
    outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), seed)
    k = inputs.normal_tensor((A, Hkv, cap, D), seed, "tl/k", outl)
    v = inputs.normal_tensor((A, Hkv, cap, D), seed, "tl/v", outl)
    return k, v, outl


@pytest.mark.parametrize("D,Hkv,Hq,n_new", [(128, 2, 16, 20), (512, 2, 16, 7), (64, 1, 2, 33), (256, 1, 8, 3)])
# n_split 0 runs row-parallel CTAs (several row groups per CTA, no split);
# 3 forces the split-K form with its merge.
@pytest.mark.parametrize("n_split", [0, 3])
def test_prefill_f16_is_causal_over_the_tail(D, Hkv, Hq, n_new, n_split):
    _need_gpu()
    A, cap = 3, 96
    lens = [90, n_new, 5]                       # the last tail is shorter than the new batch
    k, v, outl = _tails(D, Hkv, A, cap, lens, seed=95 + D)
    q = inputs.normal_tensor((A, n_new, Hq, D), 96 + D, "tl/q", outl, dtype="bfloat16", torch_out=True)
    out = torch.empty((A, n_new, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((A, n_new, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_decode_f16_workspace(D, Hkv, A, cap, n_new, Hq, n_split), dtype=torch.uint8,
                     device=DEV)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    ckv.attn_prefill_f16(torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV), sl, cap, q.to(DEV),
                         1.0 / math.sqrt(D), out, lse, ws, n_split=n_split)
    assert ckv.read_device_flag(ws) == 0
    qf = q.float().numpy().astype(np.float64)
    for a in range(A):
        o_ref, l_ref = O.verify_decode_reference(qf[a], k[a].astype(np.float64), v[a].astype(np.float64),
                                                 lens[a], 1.0 / math.sqrt(D))
        H.check_attention(out.cpu().numpy()[a], lse.cpu().numpy()[a], o_ref, l_ref, f"f16 prefill D={D} a={a}")


@pytest.mark.parametrize("D,Hkv,Hq,P,n_new", [(128, 2, 16, 200, 20), (512, 2, 16, 131, 16), (512, 2, 16, 0, 9),
                                              (256, 1, 8, 64, 40)])
def test_shared_prefill_matches_oracle(D, Hkv, Hq, P, n_new):
    """Three agents over one compressed prefix, each with its own fp16 tail
    (lengths count the new rows; one tail holds only the new rows)."""
    _need_gpu()
    A, cap = 3, 96
    lens = [77, n_new, 50]
    cache, kh, vh, outl = _prefix(D, Hkv, P, seed=100 + D)
    kt, vt, _ = _tails(D, Hkv, A, cap, lens, seed=101 + D)
    kn = inputs.normal_tensor((A, n_new, Hkv, D), 102 + D, "sh/kn", outl)
    vn = inputs.normal_tensor((A, n_new, Hkv, D), 102 + D, "sh/vn", outl)
    q = inputs.normal_tensor((A, n_new, Hq, D), 103 + D, "sh/q", outl, dtype="bfloat16", torch_out=True)
    kt_d, vt_d = torch.from_numpy(kt).to(DEV), torch.from_numpy(vt).to(DEV)
    out = torch.full((A, n_new, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((A, n_new, Hq), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_prefill_shared_workspace(cache, A, cap, n_new, Hq), dtype=torch.uint8, device=DEV)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    ckv.attn_prefill_shared(cache, P, kt_d, vt_d, sl, q.to(DEV), torch.from_numpy(kn).to(DEV),
                            torch.from_numpy(vn).to(DEV), 1.0 / math.sqrt(D), out, lse, ws)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    # The tails now hold the new rows at [len - n_new, len), bit for bit, and nothing else changed.
    kt2, vt2 = kt.copy(), vt.copy()
    for a, L in enumerate(lens):
        kt2[a, :, L - n_new:L] = np.swapaxes(kn[a], 0, 1)
        vt2[a, :, L - n_new:L] = np.swapaxes(vn[a], 0, 1)
    assert np.array_equal(kt_d.cpu().numpy().view(np.uint16), kt2.view(np.uint16))
    assert np.array_equal(vt_d.cpu().numpy().view(np.uint16), vt2.view(np.uint16))
    qf = q.float().numpy().astype(np.float64)
    for a in range(A):
        o_ref, l_ref = O.shared_prefill_reference(qf[a], kh, vh, kt2[a].astype(np.float64),
                                                  vt2[a].astype(np.float64), lens[a], 1.0 / math.sqrt(D))
        H.check_attention(out.cpu().numpy()[a], lse.cpu().numpy()[a], o_ref, l_ref, f"shared D={D} P={P} a={a}")
