"""Full-size workloads against the oracle, in the launch configuration the
benchmark times (automatic split count).

* Gemma-4 global-layer decode (head_dim 512, 2 kv heads, 16 query heads,
  32768 tokens): every packed byte and every output row checked.
* Shared-prefix fan-out: one compressed 4096-token prefix read by 15 agents
  (one 120-row pass per kv head), a private 512-token fp16 tail per agent, the
  two partials merged by log-sum-exp: every output row checked.
* Long-context decode (4 x 262144 tokens): the packed bytes and outputs of one
  kv head of every sequence checked in full (one sequence for the other V
  tiers and the block-diagonal rotation); every output must be finite.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import compressed_kv_attention_gb300 as ckv  # noqa: E402
from compressed_kv_attention_gb300 import inputs  # noqa: E402
from oracle import ckv_oracle as O  # noqa: E402
from tests import helpers as H  # noqa: E402
from tests.test_gpu_parity import (DEV, _need_gpu, oracle_cache, records_np, run_decode,  # noqa: E402
                                   to_dev)

pytestmark = pytest.mark.gpu


def test_gemma4_decode_full():
    _need_gpu()
    w = inputs.WORKLOADS["gemma4_decode"]
    D, Hkv, T = w.head_dim, w.n_kv_heads, w.seq_len
    outl = inputs.outlier_channels(D, w.n_outliers, w.seed)
    k = inputs.normal_tensor((1, T, Hkv, D), w.seed, "k", outl)
    v = inputs.normal_tensor((1, T, Hkv, D), w.seed, "v", outl)
    q = inputs.normal_tensor((1, 1, w.n_q_heads, D), w.seed, "q", outl)
    signs = inputs.tbq_signs(D)
    cache = ckv.PackedCache(D, Hkv, 1, T, signs)
    ckv.kv_pack(cache, 0, to_dev(k), to_dev(v))
    torch.cuda.synchronize()
    qs, d16, codes, n16, u = oracle_cache(k, v, signs)
    recs = records_np(cache)
    stats = [H.compare_pack(recs[0, h], qs[0, h], d16[0, h], codes[0, h], n16[0, h], u[0, h], T)
             for h in range(Hkv)]
    o_gpu, l_gpu = run_decode(cache, q, [T], T)
    kh = O.q8_0_dequantize(qs[0], d16[0])
    vh = O.tbq3_dequantize(codes[0], n16[0], signs)
    o_ref, lse_ref = O.decode_reference(q[0], kh, vh, T, 1.0 / math.sqrt(D))
    H.check_attention(o_gpu[0], l_gpu[0], o_ref, lse_ref, "gemma4 decode")
    # (i) the oracle's bytes as the cache
    cache_i = ckv.PackedCache(D, Hkv, 1, T, signs,
                              data=to_dev(H.oracle_records(qs, d16, codes, n16, T).ravel()))
    o_i, l_i = run_decode(cache_i, q, [T], T)
    H.check_attention(o_i[0], l_i[0], o_ref, lse_ref, "gemma4 decode (i)")
    print("pack ties/norm-ulps:", stats)


def test_fanout_decode_full():
    _need_gpu()
    w = inputs.WORKLOADS["fanout_decode"]
    D, Hkv, Hq, P, A, TL = w.head_dim, w.n_kv_heads, w.n_q_heads, w.seq_len, w.n_agents, w.tail_len
    outl = inputs.outlier_channels(D, w.n_outliers, w.seed)
    k = inputs.normal_tensor((1, P, Hkv, D), w.seed, "prefix/k", outl)
    v = inputs.normal_tensor((1, P, Hkv, D), w.seed, "prefix/v", outl)
    kt = inputs.normal_tensor((A, Hkv, TL, D), w.seed, "tail/k", outl)
    vt = inputs.normal_tensor((A, Hkv, TL, D), w.seed, "tail/v", outl)
    qa = inputs.normal_tensor((A, Hq, D), w.seed, "agents/q", outl)
    signs = inputs.tbq_signs(D)
    scale = 1.0 / math.sqrt(D)
    # GPU: prefix pass with the 15 agents as 15 query tokens, tails, merge.
    cache = ckv.PackedCache(D, Hkv, 1, P, signs)
    ckv.kv_pack(cache, 0, to_dev(k), to_dev(v))
    o_pre, l_pre = run_decode(cache, qa[None], [P], P)
    qd = to_dev(qa[:, None])
    o_t = torch.empty((A, 1, Hq, D), dtype=torch.float32, device=DEV)
    l_t = torch.empty((A, 1, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_decode_f16_workspace(D, Hkv, A, TL, 1, Hq), dtype=torch.uint8, device=DEV)
    ckv.attn_decode_f16(to_dev(kt), to_dev(vt), torch.full((A,), TL, dtype=torch.int32, device=DEV), TL,
                        qd, scale, o_t, l_t, ws)
    out = torch.empty((A * Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty(A * Hq, dtype=torch.float32, device=DEV)
    ckv.lse_merge([to_dev(o_pre.reshape(A * Hq, D)), o_t.view(A * Hq, D)],
                  [to_dev(l_pre.reshape(A * Hq)), l_t.view(A * Hq)], out, lse)
    # The benchmark's path: the fan-out step (prefix decode writing split partials, fp16 tail decode
    # beside it merging them).
    ws_f = torch.zeros(ckv.attn_decode_fanout_workspace(cache, P, A, TL, Hq), dtype=torch.uint8, device=DEV)
    out2 = torch.empty((A, Hq, D), dtype=torch.float32, device=DEV)
    lse2 = torch.empty((A, Hq), dtype=torch.float32, device=DEV)
    ckv.attn_decode_fanout(cache, torch.full((1,), P, dtype=torch.int32, device=DEV), P, to_dev(kt), to_dev(vt),
                           torch.full((A,), TL, dtype=torch.int32, device=DEV), TL, to_dev(qa), scale, out2, lse2,
                           ws_f)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws_f) == 0
    # Oracle: per agent, merge(prefix attention over the dequantised pool, tail attention).
    qs, d16, codes, n16, _ = oracle_cache(k, v, signs)
    kh = O.q8_0_dequantize(qs[0], d16[0])
    vh = O.tbq3_dequantize(codes[0], n16[0], signs)
    o_ref = np.zeros((A, Hq, D))
    l_ref = np.zeros((A, Hq))
    for a in range(A):
        op, lp = O.decode_reference(qa[a][None], kh, vh, P, scale)
        ot, lt = O.decode_reference(qa[a][None], kt[a].astype(np.float64), vt[a].astype(np.float64), TL,
                                    scale)
        o_ref[a], l_ref[a] = O.lse_merge([op[0], ot[0]], [lp[0], lt[0]])
    H.check_attention(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "fan-out")
    H.check_attention(out2.cpu().numpy(), lse2.cpu().numpy(), o_ref, l_ref, "fan-out step")


@pytest.mark.parametrize("name,checks", [("long_decode", ((0, 0), (1, 1), (2, 0), (2, 1), (3, 1))),
                                         ("long_decode_tbq2", ((2, 1),)), ("long_decode_tbq4", ((2, 0),)),
                                         ("long_decode_rot", ((2, 1),))])
def test_long_decode_full_size(name, checks):
    """The long-context decode at full size (4 x 262144 tokens), in the
    benchmark's launch configuration: packed bytes and attention of the listed
    (sequence, kv head) pairs checked against the oracle in full — one head of
    every sequence at 3 bits — and every output finite."""
    _need_gpu()
    w = inputs.WORKLOADS[name]
    D, Hkv, Hq, T, B, bits = w.head_dim, w.n_kv_heads, w.n_q_heads, w.seq_len, w.batch, w.v_bits
    groups = D // w.rot_group if w.rot_group else 1
    signs2 = inputs.tbq_signs(D, seed=43) if w.rot_group else None
    outl = inputs.outlier_channels(D, w.n_outliers, w.seed)
    k = inputs.normal_tensor((B, T, Hkv, D), w.seed, "k", outl, device=DEV)
    v = inputs.normal_tensor((B, T, Hkv, D), w.seed, "v", outl, device=DEV)
    q = inputs.normal_tensor((B, 1, Hq, D), w.seed, "q", outl, device=DEV)
    signs = inputs.tbq_signs(D)
    cache = ckv.PackedCache(D, Hkv, B, T, signs, v_bits=bits, signs2=signs2)
    ckv.kv_pack(cache, 0, k, v)
    out = torch.empty((B, 1, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((B, 1, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_decode_workspace(cache, T, 1, Hq), dtype=torch.uint8, device=DEV)
    sl = torch.full((B,), T, dtype=torch.int32, device=DEV)
    ckv.attn_decode(cache, sl, T, q, 1.0 / math.sqrt(D), out, lse, ws)
    assert ckv.read_device_flag(ws) == 0
    o_gpu, l_gpu = out.cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(o_gpu).all() and np.isfinite(l_gpu).all()
    scale = 1.0 / math.sqrt(D)
    recs_all = cache.data.view(B, Hkv, T // 16, 17 * D + 2 * bits * D + 32 * groups)
    for bs, h in checks:
        ks = k[bs, :, h].contiguous().cpu().numpy()   # [T, D]
        vs = v[bs, :, h].contiguous().cpu().numpy()
        recs = recs_all[bs, h].cpu().numpy()
        qn = q[bs, 0].cpu().numpy().astype(np.float64)
        qs, d16, codes, n16, u = H.oracle_quantize(ks, vs, signs, bits, signs2=signs2)
        del ks, vs
        H.compare_pack(recs, qs, d16, codes, n16, u, T, bits, groups)
        if signs2 is None:
            v_of = lambda a, b: O.tbq_dequantize(codes[a:b], n16[a:b], signs, bits)  # noqa: E731
        else:
            v_of = lambda a, b: O.tbq_dequantize_blocked(codes[a:b], n16[a:b], signs, signs2, bits)  # noqa: E731
        rows = [hq for hq in range(Hq) if O.kv_head_of(hq, Hq, Hkv) == h]
        o_ref, l_ref = H.oracle_attention_chunked(
            qn[rows], lambda a, b: O.q8_0_dequantize(qs[a:b], d16[a:b]), v_of, T, scale)
        H.check_attention(o_gpu[bs, 0, rows], l_gpu[bs, 0, rows], o_ref, l_ref, f"{name} b={bs} h={h}")


def test_shared_prefill_full_sampled():
    """The multi-tenant prefill workload at full size (15 agents x 128 new tokens,
    4096-token compressed prefix, 512-token fp16 tails), as the benchmark runs it;
    sampled agents and tokens checked against the oracle."""
    _need_gpu()
    w = inputs.WORKLOADS["shared_prefill"]
    D, Hkv, Hq, P, A, TL, n = w.head_dim, w.n_kv_heads, w.n_q_heads, w.seq_len, w.n_agents, w.tail_len, w.n_new
    cap = TL + n
    outl = inputs.outlier_channels(D, w.n_outliers, w.seed)
    signs = inputs.tbq_signs(D)
    kp = inputs.normal_tensor((1, P, Hkv, D), w.seed, "fp/k", outl)
    vp = inputs.normal_tensor((1, P, Hkv, D), w.seed, "fp/v", outl)
    kt = inputs.normal_tensor((A, Hkv, cap, D), w.seed, "ft/k", outl)
    vt = inputs.normal_tensor((A, Hkv, cap, D), w.seed, "ft/v", outl)
    kn = inputs.normal_tensor((A, n, Hkv, D), w.seed, "fn/k", outl)
    vn = inputs.normal_tensor((A, n, Hkv, D), w.seed, "fn/v", outl)
    q = inputs.normal_tensor((A, n, Hq, D), w.seed, "fn/q", outl, dtype="bfloat16", torch_out=True)
    cache = ckv.PackedCache(D, Hkv, 1, P, signs)
    ckv.kv_pack(cache, 0, torch.from_numpy(kp).to(DEV), torch.from_numpy(vp).to(DEV))
    kt_d, vt_d = torch.from_numpy(kt).to(DEV), torch.from_numpy(vt).to(DEV)
    out = torch.empty((A, n, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((A, n, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_prefill_shared_workspace(cache, A, cap, n, Hq), dtype=torch.uint8, device=DEV)
    sl = torch.full((A,), cap, dtype=torch.int32, device=DEV)
    ckv.attn_prefill_shared(cache, P, kt_d, vt_d, sl, q.to(DEV), torch.from_numpy(kn).to(DEV),
                            torch.from_numpy(vn).to(DEV), 1.0 / math.sqrt(D), out, lse, ws)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    qs, d16, codes, n16, _ = H.oracle_quantize(np.swapaxes(kp[0], 0, 1), np.swapaxes(vp[0], 0, 1), signs)
    kh, vh = O.q8_0_dequantize(qs, d16), O.tbq3_dequantize(codes, n16, signs)
    qf = q.float().numpy().astype(np.float64)
    o_gpu, l_gpu = out.cpu().numpy(), lse.cpu().numpy()
    for a in (0, 7, A - 1):
        ka, va = kt[a].astype(np.float64), vt[a].astype(np.float64)
        ka[:, TL:] = np.swapaxes(kn[a], 0, 1)
        va[:, TL:] = np.swapaxes(vn[a], 0, 1)
        rows = [0, 1, 63, n - 1]
        o_ref, l_ref = O.shared_prefill_reference(qf[a], kh, vh, ka, va, cap, 1.0 / math.sqrt(D))
        H.check_attention(o_gpu[a, rows], l_gpu[a, rows], o_ref[rows], l_ref[rows], f"shared full a={a}")
