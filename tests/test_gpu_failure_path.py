"""The failure path of the kernels' asynchronous waits, exercised without a
GPU fault: both wait forms (an mbarrier phase, a global counter) run on
events that never come, give up after their time limit, report through the
device flag, and the context keeps running work."""
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


def test_bounded_waits_report_and_the_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    ckv.selftest_bounded_waits(ws)
    torch.cuda.synchronize()
    flags = ws[:8].view(torch.int32).cpu().tolist()
    assert flags == [1, 1]                    # both waits ran out and said so
    # The same context then runs a decode normally.
    D, Hkv, Hq, T = 128, 1, 4, 100
    k, v, _ = PT._inputs(D, Hkv, Hq, 1, T, 1, seed=1400)
    outl = inputs.outlier_channels(D, 1, 1400)
    q = inputs.normal_tensor((1, 1, Hq, D), 1400, "fp/q", outl)
    cache = PT._cache(D, Hkv, 1, 112, 3, False)
    ckv.kv_pack(cache, 0, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    out = torch.empty((1, 1, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((1, 1, Hq), dtype=torch.float32, device=DEV)
    dws = torch.zeros(ckv.attn_decode_workspace(cache, T, 1, Hq), dtype=torch.uint8, device=DEV)
    ckv.attn_decode(cache, torch.tensor([T], dtype=torch.int32, device=DEV), T, torch.from_numpy(q).to(DEV),
                    1.0 / math.sqrt(D), out, lse, dws)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(dws) == 0
    kh, vh = PT.dequantised(k, v, 0, 3, False)
    o_ref, l_ref = O.decode_reference(q[0], kh, vh, T, 1.0 / math.sqrt(D))
    H.check_attention(out.cpu().numpy()[0], lse.cpu().numpy()[0], o_ref, l_ref, "decode after the wait check")
