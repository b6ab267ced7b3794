"""GPU parity of the chunked prefill (pack the new rows, then causal attention
of the new queries over the packed cache on tcgen05) against the oracle:
query i of the new chunk sees cached positions [0, n_cached + i], the new rows
read back in packed form."""
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


def _case(D, Hkv, Hq, B, n_cached, n_new, cap, seed):
    outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), seed)
    T = n_cached + n_new
    k = inputs.normal_tensor((B, T, Hkv, D), seed, "pf/k", outl)
    v = inputs.normal_tensor((B, T, Hkv, D), seed, "pf/v", outl)
    q = inputs.normal_tensor((B, n_new, Hq, D), seed, "pf/q", outl, dtype="bfloat16", torch_out=True)
    signs = inputs.tbq_signs(D)
    cache = ckv.PackedCache(D, Hkv, B, cap, signs)
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
    return k, v, q.float().numpy().astype(np.float64), signs, out.cpu().numpy(), lse.cpu().numpy()


def _oracle(k, v, qf, signs, n_cached, b, rows=None):
    D = k.shape[-1]
    kt = np.ascontiguousarray(np.swapaxes(k[b], 0, 1))
    vt = np.ascontiguousarray(np.swapaxes(v[b], 0, 1))
    qs, d16, codes, n16, _ = H.oracle_quantize(kt, vt, signs)
    kh = O.q8_0_dequantize(qs, d16)
    vh = O.tbq3_dequantize(codes, n16, signs)
    q = qf[b] if rows is None else qf[b][rows]
    if rows is None:
        return O.prefill_reference(q, kh, vh, n_cached, 1.0 / math.sqrt(D))
    # Selected query tokens only: query index rows[i] sees [0, n_cached + rows[i]].
    Hq, Hkv = q.shape[1], kh.shape[0]
    o = np.zeros(q.shape)
    lse = np.zeros(q.shape[:2])
    for i, qi in enumerate(rows):
        for h in range(Hq):
            kv = O.kv_head_of(h, Hq, Hkv)
            oo, ll = O.attention(q[i:i + 1, h], kh[kv, :n_cached + qi + 1], vh[kv, :n_cached + qi + 1],
                                 1.0 / math.sqrt(D))
            o[i, h], lse[i, h] = oo[0], ll[0]
    return o, lse


@pytest.mark.parametrize("D,Hkv,Hq,n_cached,n_new", [(128, 2, 16, 100, 37), (256, 1, 4, 64, 80),
                                                     (512, 2, 16, 131, 45), (512, 1, 8, 0, 20),
                                                     (64, 1, 4, 50, 33)])
def test_prefill_small(D, Hkv, Hq, n_cached, n_new):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B = 2
    cap = ((n_cached + n_new + 15) // 16) * 16 + 16
    k, v, qf, signs, out, lse = _case(D, Hkv, Hq, B, n_cached, n_new, cap, seed=40 + D + n_new)
    for b in range(B):
        o_ref, l_ref = _oracle(k, v, qf, signs, n_cached, b)
        H.check_attention(out[b], lse[b], o_ref, l_ref, f"prefill D={D} b={b}")


def test_chunked_prefill_workload():
    """2048 new queries over 32768 cached tokens (Gemma-4 global-layer shapes),
    in the benchmark's launch configuration: every query row of kv head 0 (all
    2048 tokens x its 8 query heads, each over its causal key range) checked in
    full, and query tokens sampled across every 128-row tile position for both
    kv heads."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = inputs.WORKLOADS["chunked_prefill"]
    D, Hkv, Hq, nc, nn = w.head_dim, w.n_kv_heads, w.n_q_heads, w.seq_len, w.n_new
    k, v, qf, signs, out, lse = _case(D, Hkv, Hq, 1, nc, nn, nc + nn, seed=w.seed)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    rows = [0, 1, 15, 16, 17, 500, 1023, 1024, 1777, 2046, 2047]
    o_ref, l_ref = _oracle(k, v, qf, signs, nc, 0, rows=rows)
    H.check_attention(out[0][rows], lse[0][rows], o_ref, l_ref, "chunked prefill (sampled)")
    # Kv head 0 in full, chunked over the keys: query i sees [0, nc + i].
    kt = np.ascontiguousarray(k[0, :, 0])
    vt = np.ascontiguousarray(v[0, :, 0])
    qs, d16, codes, n16, _ = H.oracle_quantize(kt, vt, signs)
    kh, vh = O.q8_0_dequantize(qs, d16), O.tbq3_dequantize(codes, n16, signs)
    qpos = np.arange(nn)
    for h in [hq for hq in range(Hq) if O.kv_head_of(hq, Hq, Hkv) == 0]:
        o_ref, l_ref = H.oracle_attention_chunked(
            qf[0, :, h], lambda a, b: kh[a:b], lambda a, b: vh[a:b], nc + nn, 1.0 / math.sqrt(D),
            visible_of=lambda a, b: np.arange(a, b)[None, :] <= nc + qpos[:, None])
        H.check_attention(out[0, :, h], lse[0, :, h], o_ref, l_ref, f"chunked prefill kv head 0, q head {h}")


def test_prefill_stream_k_schedule():
    """More 128-row tiles than SMs, each CTA taking an equal run of 64-key steps:
    tiles cut between two CTAs are merged from two partials. Every row of both
    sequences is checked (head_dim 64 keeps the oracle quick)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    D, Hkv, Hq, B, nc, nn = 64, 2, 16, 2, 64, 2560   # 2 x 2 x 160 tiles of 16 tokens x 8 heads
    cap = nc + nn + 16
    k, v, qf, signs, out, lse = _case(D, Hkv, Hq, B, nc, nn, cap, seed=77)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    for b in range(B):
        o_ref, l_ref = _oracle(k, v, qf, signs, nc, b)
        H.check_attention(out[b], lse[b], o_ref, l_ref, f"stream-K prefill b={b}")


def _stream_k_applies(B, Hkv, Hq, nc, nn, sms):
    """The prefill's schedule rule, restated: more 128-row tiles than SMs, and
    every CTA's share of the 64-key steps at least as long as any tile."""
    qt = 128 // (Hq // Hkv)
    n_qt = -(-nn // qt)
    steps = [-(-(nc + min((t + 1) * qt, nn)) // 64) for t in range(n_qt)]
    return B * Hkv * n_qt > sms and B * Hkv * sum(steps) // sms >= max(steps)


def test_prefill_stream_k_schedule_d512():
    """The stream-K schedule at head_dim 512 (Gemma-4 shapes, 2 sequences of
    2048 cached + 1024 new tokens: 256 tiles of 16 tokens x 8 heads): every
    row of both sequences checked, including the rows of tiles cut between two
    CTAs at the full head dim."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    D, Hkv, Hq, B, nc, nn = 512, 2, 16, 2, 2048, 1024
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert _stream_k_applies(B, Hkv, Hq, nc, nn, sms)
    cap = nc + nn + 16
    k, v, qf, signs, out, lse = _case(D, Hkv, Hq, B, nc, nn, cap, seed=78)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    for b in range(B):
        o_ref, l_ref = _oracle(k, v, qf, signs, nc, b)
        H.check_attention(out[b], lse[b], o_ref, l_ref, f"stream-K prefill D=512 b={b}")
