"""GPU parity of attn_decode_f16_merge: the fp16-tail decode whose split merge
also takes in a prior partial per row (the shared compressed prefix of the
pool fan-out), against the oracle's merge of the two attentions and against
the separate decode + lse_merge path. Both split merges (rendezvous and tree),
the row-parallel launch (one split, several row groups per CTA, the prior
merged in its epilogue), ragged and empty tails, and empty prior rows (lse
-inf) are covered."""
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


@pytest.mark.parametrize("D,A,P,TL,tails,n_split,n_q", [
    (512, 15, 4096, 512, None, 0, 1),                 # the fan-out workload's shapes
    (128, 5, 300, 208, [208, 0, 17, 200, 1], 0, 1),   # ragged and empty tails
    (256, 4, 0, 96, [96, 50, 96, 3], 3, 1),           # an empty prefix: every prior row is empty
    (128, 3, 160, 1024, [1024, 700, 5], 300, 1),      # more splits than fit at once: the tree merge
    (128, 3, 200, 96, [96, 40, 0], 1, 8),             # row-parallel CTAs (8 row groups), an empty tail
    (512, 2, 0, 64, [64, 17], 1, 4),                  # row-parallel, D=512, every prior row empty
])
def test_f16_merge_matches_oracle_and_separate_merge(D, A, P, TL, tails, n_split, n_q):
    _need_gpu()
    Hkv, Hq, seed = 2, 16, 60 + D + A
    scale = 1.0 / math.sqrt(D)
    outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), seed)
    signs = inputs.tbq_signs(D)
    tails = tails or [TL] * A
    qa = inputs.normal_tensor((A, n_q, Hq, D), seed, "m/q", outl)
    kt = inputs.normal_tensor((A, Hkv, TL, D), seed, "m/kt", outl)
    vt = inputs.normal_tensor((A, Hkv, TL, D), seed, "m/vt", outl)
    # Prior: the agents' attention over a packed prefix (agents' tokens as query tokens).
    o_pre = torch.empty((1, A * n_q, Hq, D), dtype=torch.float32, device=DEV)
    l_pre = torch.empty((1, A * n_q, Hq), dtype=torch.float32, device=DEV)
    if P > 0:
        kp = inputs.normal_tensor((1, P, Hkv, D), seed, "m/kp", outl)
        vp = inputs.normal_tensor((1, P, Hkv, D), seed, "m/vp", outl)
        cache = ckv.PackedCache(D, Hkv, 1, (P + 15) // 16 * 16, signs, device=DEV)
        ckv.kv_pack(cache, 0, torch.from_numpy(kp).to(DEV), torch.from_numpy(vp).to(DEV))
        ws = torch.zeros(ckv.attn_decode_workspace(cache, P, A * n_q, Hq), dtype=torch.uint8, device=DEV)
        ckv.attn_decode(cache, torch.full((1,), P, dtype=torch.int32, device=DEV), P,
                        torch.from_numpy(qa.reshape(1, A * n_q, Hq, D)).to(DEV), scale, o_pre, l_pre, ws)
        assert ckv.read_device_flag(ws) == 0
    else:
        o_pre.zero_()
        l_pre.fill_(float("-inf"))
    kd, vd = torch.from_numpy(kt).to(DEV), torch.from_numpy(vt).to(DEV)
    sl = torch.tensor(tails, dtype=torch.int32, device=DEV)
    qd = torch.from_numpy(qa).to(DEV)
    out = torch.full((A, n_q, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((A, n_q, Hq), float("nan"), dtype=torch.float32, device=DEV)
    ws_m = torch.zeros(ckv.attn_decode_f16_merge_workspace(D, Hkv, A, TL, n_q, Hq, n_split), dtype=torch.uint8,
                       device=DEV)
    ckv.attn_decode_f16_merge(kd, vd, sl, TL, qd, scale, o_pre.view(A, n_q, Hq, D), l_pre.view(A, n_q, Hq), out,
                              lse, ws_m, n_split=n_split)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws_m) == 0
    o_gpu, l_gpu = out.cpu().numpy(), lse.cpu().numpy()

    # The separate path: fp16 decode, then lse_merge of the two partials.
    o_t = torch.empty((A, n_q, Hq, D), dtype=torch.float32, device=DEV)
    l_t = torch.empty((A, n_q, Hq), dtype=torch.float32, device=DEV)
    ws_t = torch.zeros(ckv.attn_decode_f16_workspace(D, Hkv, A, TL, n_q, Hq, n_split), dtype=torch.uint8,
                       device=DEV)
    ckv.attn_decode_f16(kd, vd, sl, TL, qd, scale, o_t, l_t, ws_t, n_split=n_split)
    o_s = torch.empty((A * n_q * Hq, D), dtype=torch.float32, device=DEV)
    l_s = torch.empty(A * n_q * Hq, dtype=torch.float32, device=DEV)
    ckv.lse_merge([o_pre.view(-1, D), o_t.view(-1, D)], [l_pre.view(-1), l_t.view(-1)], o_s, l_s)
    torch.cuda.synchronize()
    H.check_attention(o_gpu, l_gpu, o_s.cpu().numpy().reshape(A, n_q, Hq, D).astype(np.float64),
                      l_s.cpu().numpy().reshape(A, n_q, Hq).astype(np.float64), "f16_merge vs decode + lse_merge")

    # Oracle: per agent, merge(prefix attention over the dequantised pool, tail attention).
    if P > 0:
        qs, d16, codes, n16, _ = H.oracle_quantize(np.swapaxes(kp[0], 0, 1), np.swapaxes(vp[0], 0, 1), signs)
        kh, vh = O.q8_0_dequantize(qs, d16), O.tbq3_dequantize(codes, n16, signs)
    o_ref = np.zeros((A, n_q, Hq, D))
    l_ref = np.zeros((A, n_q, Hq))
    for a in range(A):
        q = qa[a].astype(np.float64)
        ot, lt = O.decode_reference(q, kt[a].astype(np.float64), vt[a].astype(np.float64), tails[a], scale)
        if P > 0:
            op, lp = O.decode_reference(q, kh, vh, P, scale)
            om, lm = O.lse_merge([op.reshape(-1, D), ot.reshape(-1, D)], [lp.reshape(-1), lt.reshape(-1)])
            o_ref[a], l_ref[a] = om.reshape(n_q, Hq, D), lm.reshape(n_q, Hq)
        else:
            o_ref[a], l_ref[a] = ot, lt
    H.check_attention(o_gpu, l_gpu, o_ref, l_ref, "f16_merge vs oracle")


def test_fanout_back_to_back_matches_each_step_alone():
    """The fan-out step as the benchmark runs it: the prefix decode and the tail
    decode with the merge, with the fan-out plan's split counts, launched back
    to back for several steps with different queries and no synchronisation.
    The tail pass reads its tails and queries while the prefix pass runs and
    waits for it only to merge, so each step must still merge its own prefix
    partial (the prior buffers are reused by every step): every step's output
    equals, bit for bit, the same two calls run alone."""
    _need_gpu()
    D, Hkv, Hq, A, P, TL, N = 512, 2, 16, 15, 4096, 512, 6
    ps, ts = ckv.fanout_plan(A, Hkv, Hq)
    seed = 71
    outl = inputs.outlier_channels(D, 5, seed)
    kp = torch.from_numpy(inputs.normal_tensor((1, P, Hkv, D), seed, "b2b/kp", outl)).to(DEV)
    vp = torch.from_numpy(inputs.normal_tensor((1, P, Hkv, D), seed, "b2b/vp", outl)).to(DEV)
    cache = ckv.PackedCache(D, Hkv, 1, P, inputs.tbq_signs(D), device=DEV)
    ckv.kv_pack(cache, 0, kp, vp)
    kt = torch.from_numpy(inputs.normal_tensor((A, Hkv, TL, D), seed, "b2b/kt", outl)).to(DEV)
    vt = torch.from_numpy(inputs.normal_tensor((A, Hkv, TL, D), seed, "b2b/vt", outl)).to(DEV)
    qs = [torch.from_numpy(inputs.normal_tensor((A, Hq, D), seed + i, "b2b/q", outl)).to(DEV) for i in range(N)]
    seq_p = torch.full((1,), P, dtype=torch.int32, device=DEV)
    seq_t = torch.full((A,), TL, dtype=torch.int32, device=DEV)
    o_p = torch.empty((1, A, Hq, D), dtype=torch.float32, device=DEV)
    l_p = torch.empty((1, A, Hq), dtype=torch.float32, device=DEV)
    ws_p = torch.zeros(ckv.attn_decode_workspace(cache, P, A, Hq, ps), dtype=torch.uint8, device=DEV)
    ws_m = torch.zeros(ckv.attn_decode_f16_merge_workspace(D, Hkv, A, TL, 1, Hq, ts), dtype=torch.uint8, device=DEV)
    scale = 1.0 / math.sqrt(D)

    def step(q, out, lse):
        ckv.attn_decode(cache, seq_p, P, q[None], scale, o_p, l_p, ws_p, n_split=ps)
        ckv.attn_decode_f16_merge(kt, vt, seq_t, TL, q[:, None], scale, o_p.view(A, 1, Hq, D), l_p.view(A, 1, Hq),
                                  out, lse, ws_m, n_split=ts)

    outs = [torch.empty((A, 1, Hq, D), dtype=torch.float32, device=DEV) for _ in range(N)]
    lses = [torch.empty((A, 1, Hq), dtype=torch.float32, device=DEV) for _ in range(N)]
    for i in range(N):
        step(qs[i], outs[i], lses[i])
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws_p) == 0 and ckv.read_device_flag(ws_m) == 0
    out1 = torch.empty((A, 1, Hq, D), dtype=torch.float32, device=DEV)
    lse1 = torch.empty((A, 1, Hq), dtype=torch.float32, device=DEV)
    for i in range(N):
        step(qs[i], out1, lse1)
        torch.cuda.synchronize()
        assert torch.equal(outs[i], out1) and torch.equal(lses[i], lse1), f"step {i}"


def test_f16_merge_rejects_missing_or_aliased_prior():
    _need_gpu()
    D, Hkv, Hq, A, TL = 128, 1, 4, 2, 32
    k = torch.zeros((A, Hkv, TL, D), dtype=torch.float16, device=DEV)
    q = torch.zeros((A, 1, Hq, D), dtype=torch.float16, device=DEV)
    out = torch.zeros((A, 1, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.zeros((A, 1, Hq), dtype=torch.float32, device=DEV)
    sl = torch.full((A,), TL, dtype=torch.int32, device=DEV)
    ws = torch.zeros(ckv.attn_decode_f16_merge_workspace(D, Hkv, A, TL, 1, Hq), dtype=torch.uint8, device=DEV)
    with pytest.raises(ckv.CkvError):
        ckv.attn_decode_f16_merge(k, k, sl, TL, q, 0.1, None, lse, out, lse, ws)
    with pytest.raises(ckv.CkvError):
        ckv.attn_decode_f16_merge(k, k, sl, TL, q, 0.1, out, lse, out, lse, ws)
