"""GPU parity of the many-row decode (64 or more query rows per kv head, as
when many agents read one shared prefix): n_split -1 runs each 128-row tile on
the tcgen05 kernel split over the key range and merges the splits exactly; a
positive split count runs the mma.sync decode; 0 picks one of the two by the
library's cost model. All are checked against the float64 oracle, on caches
filled with 0xFF bytes before packing (never-written positions past seq_len),
with ragged and empty sequences, every V tier and both rotations."""
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


def _run(cache, q, seq_lens, maxs, n_split=0):
    B, n_q, Hq, D = q.shape
    out = torch.full((B, n_q, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((B, n_q, Hq), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ckv.attn_decode_workspace(cache, maxs, n_q, Hq, n_split), dtype=torch.uint8, device=DEV)
    sl = torch.tensor(seq_lens, dtype=torch.int32, device=DEV)
    ckv.attn_decode(cache, sl, maxs, torch.from_numpy(np.ascontiguousarray(q)).to(DEV), 1.0 / math.sqrt(D), out,
                    lse, ws, n_split=n_split)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy(), ckv.read_device_flag(ws)


@pytest.mark.parametrize("D,Hkv,Hq,n_q,bits,rot", [(512, 2, 16, 15, 3, False), (128, 1, 8, 8, 2, False),
                                                   (256, 2, 16, 10, 4, True), (64, 1, 16, 4, 3, False),
                                                   (512, 1, 8, 16, 2, True)])
def test_many_row_decode_matches_oracle(D, Hkv, Hq, n_q, bits, rot):
    _need_gpu()
    B, T, cap = 3, 1003, 1024
    seq_lens = [1003, 0, 517]
    k, v, _ = PT._inputs(D, Hkv, Hq, B, T, 1, seed=1300 + D + n_q)
    outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), 1300 + D)
    q = inputs.normal_tensor((B, n_q, Hq, D), 1300 + D, "rows/q", outl)
    cache = PT._cache(D, Hkv, B, cap, bits, rot, fill=0xFF)
    ckv.kv_pack(cache, 0, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    o_ref, l_ref = np.zeros((B, n_q, Hq, D)), np.zeros((B, n_q, Hq))
    for b in range(B):
        kh, vh = PT.dequantised(k, v, b, bits, rot)
        o_ref[b], l_ref[b] = O.decode_reference(q[b], kh, vh, seq_lens[b], 1.0 / math.sqrt(D))
    for n_split in (-1, 7, 0):   # -1: the tcgen05 tile path; 7: the mma.sync decode; 0: automatic
        o, l, flag = _run(cache, q, seq_lens, cap, n_split)
        assert flag == 0
        H.check_attention(o, l, o_ref, l_ref, f"rows D={D} n_q={n_q} b={bits} rot={rot} split={n_split}")


def test_many_row_decode_fanout_shape_full_rows():
    """The shared-prefix fan-out shape (15 agents x 16 heads over 4096 tokens),
    every row checked."""
    _need_gpu()
    D, Hkv, Hq, n_q, P = 512, 2, 16, 15, 4096
    k, v, _ = PT._inputs(D, Hkv, Hq, 1, P, 1, seed=1350)
    outl = inputs.outlier_channels(D, max(1, round(0.01 * D)), 1350)
    q = inputs.normal_tensor((1, n_q, Hq, D), 1350, "rows/qf", outl)
    cache = PT._cache(D, Hkv, 1, P, 3, False)
    ckv.kv_pack(cache, 0, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    kh, vh = PT.dequantised(k, v, 0, 3, False)
    o_ref, l_ref = O.decode_reference(q[0], kh, vh, P, 1.0 / math.sqrt(D))
    for n_split in (-1, 0):
        o, l, flag = _run(cache, q, [P], P, n_split)
        assert flag == 0
        H.check_attention(o[0], l[0], o_ref, l_ref, f"fan-out shape split={n_split}")


def test_many_row_decode_seq_len_out_of_range_sets_flag():
    """A seq_len above max_seq_len is reported through the device flag and the
    sequence is treated as empty; nothing is read out of range."""
    _need_gpu()
    D, Hkv, Hq, n_q, cap = 128, 1, 8, 8, 256
    k, v, _ = PT._inputs(D, Hkv, Hq, 2, 200, 1, seed=1360)
    q = inputs.normal_tensor((2, n_q, Hq, D), 1360, "rows/qo", inputs.outlier_channels(D, 1, 1360))
    cache = PT._cache(D, Hkv, 2, cap, 3, False)
    ckv.kv_pack(cache, 0, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    o, l, flag = _run(cache, q, [200, 250], 200, -1)
    assert flag == 2
    assert np.all(o[1] == 0.0) and np.all(np.isneginf(l[1]))
    kh, vh = PT.dequantised(k, v, 0, 3, False)
    o_ref, l_ref = O.decode_reference(q[0], kh, vh, 200, 1.0 / math.sqrt(D))
    H.check_attention(o[0], l[0], o_ref, l_ref, "in-range sequence beside an out-of-range one")


def test_tile_path_refuses_head_ratio_not_dividing_128():
    _need_gpu()
    D, Hkv, Hq, n_q = 128, 1, 12, 8    # 12 query heads per kv head
    cache = PT._cache(D, Hkv, 1, 64, 3, False)
    assert ckv.attn_decode_workspace(cache, 64, n_q, Hq, -1) == 0
    q = torch.zeros((1, n_q, Hq, D), dtype=torch.float16, device=DEV)
    out = torch.empty((1, n_q, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((1, n_q, Hq), dtype=torch.float32, device=DEV)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    sl = torch.tensor([64], dtype=torch.int32, device=DEV)
    with pytest.raises(ckv.CkvError):
        ckv.attn_decode(cache, sl, 64, q, 0.1, out, lse, ws, n_split=-1)
