"""With other kernels declared concurrent (ckv_set_concurrent_kernels), the
split decodes merge by the tree, in which no CTA waits for another. The
results match the oracle and the default (rendezvous) merge within the
attention tolerance, the device flag stays clear, and switching back restores
the default."""
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


def test_concurrent_mode_uses_a_merge_that_never_waits():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    D, Hkv, Hq, T, seed = 512, 2, 16, 8192, 71
    outl = inputs.outlier_channels(D, 5, seed)
    signs = inputs.tbq_signs(D)
    k = inputs.normal_tensor((1, T, Hkv, D), seed, "cc/k", outl)
    v = inputs.normal_tensor((1, T, Hkv, D), seed, "cc/v", outl)
    q = inputs.normal_tensor((1, 1, Hq, D), seed, "cc/q", outl)
    cache = ckv.PackedCache(D, Hkv, 1, T, signs, device=DEV)
    ckv.kv_pack(cache, 0, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    sl = torch.full((1,), T, dtype=torch.int32, device=DEV)
    qd = torch.from_numpy(q).to(DEV)
    ws = torch.zeros(ckv.attn_decode_workspace(cache, T, 1, Hq), dtype=torch.uint8, device=DEV)
    res = {}
    try:
        for mode in (True, False):
            ckv.set_concurrent_kernels(mode)
            for rep in range(3):  # repeated calls reuse the workspace's counters
                out = torch.full((1, 1, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
                lse = torch.full((1, 1, Hq), float("nan"), dtype=torch.float32, device=DEV)
                ckv.attn_decode(cache, sl, T, qd, 1 / math.sqrt(D), out, lse, ws)
            torch.cuda.synchronize()
            assert ckv.read_device_flag(ws) == 0
            assert torch.all(ws[64:256] == 0)  # the merge counters are back at zero
            res[mode] = (out.cpu().numpy()[0], lse.cpu().numpy()[0])
    finally:
        ckv.set_concurrent_kernels(False)
    kt, vt = np.swapaxes(k, 1, 2)[0], np.swapaxes(v, 1, 2)[0]
    qs, d16, codes, n16, _ = H.oracle_quantize(kt, vt, signs)
    o_ref, l_ref = O.decode_reference(q[0], O.q8_0_dequantize(qs, d16), O.tbq3_dequantize(codes, n16, signs), T,
                                      1 / math.sqrt(D))
    for mode, (o, l) in res.items():
        H.check_attention(o, l, o_ref, l_ref, f"concurrent={mode}")
    H.check_attention(res[True][0], res[True][1], res[False][0].astype(np.float64), res[False][1].astype(np.float64),
                      "tree vs rendezvous")
