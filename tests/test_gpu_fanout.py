"""GPU parity of attn_decode_fanout, the shared-pool fan-out decode step: each
agent's query over the shared compressed prefix and its own fp16 tail, in two
launches whose partials merge inside the tail decode. Checked against the
oracle's merge of the two attentions (ragged and empty tails, a prefix shorter
than its bound, an empty prefix, several head dims and agent counts), against
the composed form (the same step when other kernels may share the device),
back to back without synchronisation, and through the device flag."""
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


class _Fanout:
    """Seeded prefix (packed on the GPU), tails and queries of one fan-out step."""

    def __init__(self, D, Hkv, A, P_max, P, TL, tails, seed):
        self.D, self.Hkv, self.Hq, self.A, self.P_max, self.P, self.TL = D, Hkv, 8 * Hkv, A, P_max, P, TL
        self.tails = tails or [TL] * A
        outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), seed)
        self.signs = inputs.tbq_signs(D)
        cap_p = max(16, (P_max + 15) // 16 * 16)
        self.kp = inputs.normal_tensor((1, cap_p, Hkv, D), seed, "fan/kp", outl)
        self.vp = inputs.normal_tensor((1, cap_p, Hkv, D), seed, "fan/vp", outl)
        self.cache = ckv.PackedCache(D, Hkv, 1, cap_p, self.signs, device=DEV)
        ckv.kv_pack(self.cache, 0, torch.from_numpy(self.kp).to(DEV), torch.from_numpy(self.vp).to(DEV))
        self.kt = inputs.normal_tensor((A, Hkv, TL, D), seed, "fan/kt", outl)
        self.vt = inputs.normal_tensor((A, Hkv, TL, D), seed, "fan/vt", outl)
        self.q = inputs.normal_tensor((A, self.Hq, D), seed, "fan/q", outl)
        self.kt_d, self.vt_d = torch.from_numpy(self.kt).to(DEV), torch.from_numpy(self.vt).to(DEV)
        self.q_d = torch.from_numpy(self.q).to(DEV)
        self.p_len = torch.tensor([P], dtype=torch.int32, device=DEV)
        self.t_len = torch.tensor(self.tails, dtype=torch.int32, device=DEV)
        self.scale = 1.0 / math.sqrt(D)

    def workspace(self):
        n = ckv.attn_decode_fanout_workspace(self.cache, self.P_max, self.A, self.TL, self.Hq)
        assert n > 0
        return torch.zeros(n, dtype=torch.uint8, device=DEV)

    def run(self, ws, q=None, out=None, lse=None, sync=True):
        out = torch.full((self.A, self.Hq, self.D), float("nan"), device=DEV) if out is None else out
        lse = torch.full((self.A, self.Hq), float("nan"), device=DEV) if lse is None else lse
        ckv.attn_decode_fanout(self.cache, self.p_len, self.P_max, self.kt_d, self.vt_d, self.t_len, self.TL,
                               self.q_d if q is None else q, self.scale, out, lse, ws)
        if sync:
            torch.cuda.synchronize()
        return out, lse

    def oracle(self):
        A, Hq, D = self.A, self.Hq, self.D
        o_ref, l_ref = np.zeros((A, Hq, D)), np.zeros((A, Hq))
        if self.P > 0:
            qs, d16, codes, n16, _ = H.oracle_quantize(np.swapaxes(self.kp[0], 0, 1), np.swapaxes(self.vp[0], 0, 1),
                                                       self.signs)
            kh, vh = O.q8_0_dequantize(qs, d16), O.tbq3_dequantize(codes, n16, self.signs)
        for a in range(A):
            q = self.q[a][None].astype(np.float64)
            ot, lt = O.decode_reference(q, self.kt[a].astype(np.float64), self.vt[a].astype(np.float64),
                                        self.tails[a], self.scale)
            if self.P > 0:
                op, lp = O.decode_reference(q, kh, vh, self.P, self.scale)
                o_ref[a], l_ref[a] = O.lse_merge([op[0], ot[0]], [lp[0], lt[0]])
            else:
                o_ref[a], l_ref[a] = ot[0], lt[0]
        return o_ref, l_ref


@pytest.mark.parametrize("D,Hkv,A,P_max,P,TL,tails", [
    (512, 2, 15, 4096, 4096, 512, None),                     # the fan-out workload's shapes
    (128, 1, 5, 320, 300, 208, [208, 0, 17, 200, 1]),        # ragged and empty tails, prefix below its bound
    (256, 2, 4, 0, 0, 96, [96, 50, 96, 3]),                  # no prefix
    (64, 1, 40, 1000, 1000, 64, None),                       # many agents: two prefix splits
    (512, 1, 3, 48, 33, 32, [32, 1, 0]),                     # prefix and tails shorter than one record
    (64, 1, 80, 512, 512, 32, None),                         # too many tails to run beside: the composed form
])
def test_fanout_matches_oracle(D, Hkv, A, P_max, P, TL, tails):
    _need_gpu()
    f = _Fanout(D, Hkv, A, P_max, P, TL, tails, seed=80 + D + A)
    ws = f.workspace()
    out, lse = f.run(ws)
    assert ckv.read_device_flag(ws) == 0
    o_ref, l_ref = f.oracle()
    H.check_attention(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "fan-out vs oracle")


def test_fanout_composed_form_matches():
    """With other kernels declared on the device the step runs as the prefix
    decode into the workspace plus the tail decode with that prior; same
    attention as the fused form and the oracle."""
    _need_gpu()
    f = _Fanout(512, 2, 15, 4096, 4096, 512, None, seed=91)
    ws = f.workspace()
    fused, fused_lse = f.run(ws)
    ckv.set_concurrent_kernels(1)
    try:
        ws2 = f.workspace()
        assert ws2.numel() == ws.numel()  # one size for both forms
        comp, comp_lse = f.run(ws2)
    finally:
        ckv.set_concurrent_kernels(0)
    assert ckv.read_device_flag(ws) == 0 and ckv.read_device_flag(ws2) == 0
    H.check_attention(comp.cpu().numpy(), comp_lse.cpu().numpy(), fused.cpu().numpy().astype(np.float64),
                      fused_lse.cpu().numpy().astype(np.float64), "composed vs fused")
    o_ref, l_ref = f.oracle()
    H.check_attention(comp.cpu().numpy(), comp_lse.cpu().numpy(), o_ref, l_ref, "composed vs oracle")


def test_fanout_back_to_back_matches_each_step_alone():
    """Steps launched back to back with different queries and no
    synchronisation: the tail decode streams while the prefix decode runs and
    merges the prefix's partials only after it has finished, so every step
    equals, bit for bit, the same call run alone."""
    _need_gpu()
    f = _Fanout(512, 2, 15, 4096, 4096, 512, None, seed=93)
    ws = f.workspace()
    N = 6
    outl = inputs.outlier_channels(512, 5, 93)
    qs = [torch.from_numpy(inputs.normal_tensor((15, 16, 512), 93 + i, "fan/b2b", outl)).to(DEV) for i in range(N)]
    outs = [torch.empty((15, 16, 512), device=DEV) for _ in range(N)]
    lses = [torch.empty((15, 16), device=DEV) for _ in range(N)]
    for i in range(N):
        f.run(ws, qs[i], outs[i], lses[i], sync=False)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    for i in range(N):
        o1, l1 = f.run(ws, qs[i])
        assert torch.equal(outs[i], o1) and torch.equal(lses[i], l1), f"step {i}"


def test_fanout_flag_reports_out_of_range_lengths():
    """A prefix length above its bound, or a tail length above the tails'
    bound, raises the device flag (2) in the step's one flag word; that part
    counts as empty."""
    _need_gpu()
    f = _Fanout(128, 1, 3, 64, 64, 32, [32, 20, 5], seed=95)
    ws = f.workspace()
    f.p_len.fill_(100)  # > max_prefix_len 64
    out, lse = f.run(ws)
    assert ckv.read_device_flag(ws) == 2
    assert ckv.read_device_flag(ws) == 0
    f.P = 0
    o_ref, l_ref = f.oracle()
    H.check_attention(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "prefix out of range")
    f.p_len.fill_(64)
    f.P = 64
    f.t_len[1] = 40  # > max_tail_len 32
    out, lse = f.run(ws)
    assert ckv.read_device_flag(ws) == 2
    f.tails = [32, 0, 5]
    o_ref, l_ref = f.oracle()
    H.check_attention(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "tail out of range")


def test_fanout_refuses_other_head_ratios():
    _need_gpu()
    cache = ckv.PackedCache(128, 2, 1, 64, inputs.tbq_signs(128), device=DEV)
    assert ckv.attn_decode_fanout_workspace(cache, 64, 4, 32, 4) == 0
    k = torch.zeros((4, 2, 32, 128), dtype=torch.float16, device=DEV)
    q = torch.zeros((4, 4, 128), dtype=torch.float16, device=DEV)
    out = torch.zeros((4, 4, 128), device=DEV)
    lse = torch.zeros((4, 4), device=DEV)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    sl = torch.full((4,), 32, dtype=torch.int32, device=DEV)
    with pytest.raises(ckv.CkvError) as err:
        ckv.attn_decode_fanout(cache, sl[:1], 64, k, k, sl, 32, q, 0.1, out, lse, ws)
    assert err.value.status == -2
