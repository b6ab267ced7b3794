"""Guard regions around every buffer a kernel writes: each output, lse, cache
and workspace sits inside a larger allocation whose 4 KB head and tail hold a
sentinel; after the call the sentinels must be intact (no write outside the
buffer), on ragged shapes (token counts that are not a multiple of the tile,
fewer tokens than splits, a single token)."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import compressed_kv_attention_gb300 as ckv  # noqa: E402
from compressed_kv_attention_gb300 import inputs  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD_BYTES = 4096
F_SENT = -12345.0
B_SENT = 0xA5


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class Guarded:
    """A view of `shape` inside an allocation with GUARD_BYTES of sentinel on each side."""

    def __init__(self, shape, dtype, fill=None):
        self.n = int(np.prod(shape))
        esz = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD_BYTES // esz
        self.sent = F_SENT if dtype.is_floating_point else B_SENT
        self.buf = torch.full((self.n + 2 * self.g,), self.sent, dtype=dtype, device=DEV)
        self.view = self.buf[self.g:self.g + self.n].view(shape)
        if fill is not None:
            self.view.fill_(fill)

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.buf[:self.g] == self.sent).all()) and bool((self.buf[self.g + self.n:] == self.sent).all())


def _cache(D, Hkv, B, cap, bits=3, rot=False):
    signs2 = inputs.tbq_signs(D, seed=43) if rot else None
    data = Guarded((ckv.cache_bytes(D, Hkv, B, cap, bits, 128 if rot else 0),), torch.uint8, fill=0)
    return data, ckv.PackedCache(D, Hkv, B, cap, inputs.tbq_signs(D), data=data.view, v_bits=bits, signs2=signs2)


def _kv(D, Hkv, B, T, seed):
    outl = inputs.outlier_channels(D, 1, seed)
    k = inputs.normal_tensor((B, T, Hkv, D), seed, "cn/k", outl)
    v = inputs.normal_tensor((B, T, Hkv, D), seed, "cn/v", outl)
    return torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV), outl


@pytest.mark.parametrize("D,T,cap", [(128, 37, 48), (512, 1, 16), (256, 203, 208)])
def test_pack_and_decode_stay_inside_their_buffers(D, T, cap):
    _need_gpu()
    Hkv, Hq, B = 2, 16, 2
    k, v, outl = _kv(D, Hkv, B, T, seed=1500 + D)
    data, cache = _cache(D, Hkv, B, cap)
    ckv.kv_pack(cache, 0, k, v)
    assert data.intact()
    for n_q, n_split in ((1, 0), (1, 300), (4, 5), (8, 0), (8, -1)):
        q = torch.from_numpy(inputs.normal_tensor((B, n_q, Hq, D), 1500 + D, "cn/q", outl)).to(DEV)
        out = Guarded((B, n_q, Hq, D), torch.float32)
        lse = Guarded((B, n_q, Hq), torch.float32)
        ws = Guarded((ckv.attn_decode_workspace(cache, T, n_q, Hq, n_split),), torch.uint8, fill=0)
        sl = torch.tensor([T, max(T - 3, 0)], dtype=torch.int32, device=DEV)
        ckv.attn_decode(cache, sl, T, q, 1.0 / math.sqrt(D), out.view, lse.view, ws.view, n_split=n_split)
        assert out.intact() and lse.intact() and ws.intact() and data.intact(), (n_q, n_split)
        assert ckv.read_device_flag(ws.view) == 0


def test_prefill_stays_inside_its_buffers():
    _need_gpu()
    D, Hkv, Hq, B, nc, nn = 256, 1, 8, 2, 70, 45
    k, v, outl = _kv(D, Hkv, B, nc + nn, seed=1550)
    data, cache = _cache(D, Hkv, B, 128, bits=4, rot=True)
    ckv.kv_pack(cache, 0, k[:, :nc].contiguous(), v[:, :nc].contiguous())
    q = inputs.normal_tensor((B, nn, Hq, D), 1550, "cn/qp", outl, dtype="bfloat16", torch_out=True).to(DEV)
    out = Guarded((B, nn, Hq, D), torch.float32)
    lse = Guarded((B, nn, Hq), torch.float32)
    ws = Guarded((ckv.attn_prefill_workspace(cache, nn, Hq),), torch.uint8, fill=0)
    ckv.attn_prefill(cache, nc, q, k[:, nc:].contiguous(), v[:, nc:].contiguous(), 1.0 / math.sqrt(D), out.view,
                     lse.view, ws.view)
    assert out.intact() and lse.intact() and ws.intact() and data.intact()
    assert ckv.read_device_flag(ws.view) == 0


def test_f16_decode_and_merge_stay_inside_their_buffers():
    _need_gpu()
    D, Hkv, Hq, B, cap = 128, 2, 8, 3, 48
    outl = inputs.outlier_channels(D, 1, 1560)
    k16 = torch.from_numpy(inputs.normal_tensor((B, Hkv, cap, D), 1560, "cn/k16", outl)).to(DEV)
    v16 = torch.from_numpy(inputs.normal_tensor((B, Hkv, cap, D), 1560, "cn/v16", outl)).to(DEV)
    q = torch.from_numpy(inputs.normal_tensor((B, 1, Hq, D), 1560, "cn/q16", outl)).to(DEV)
    out = Guarded((B, 1, Hq, D), torch.float32)
    lse = Guarded((B, 1, Hq), torch.float32)
    ws = Guarded((ckv.attn_decode_f16_workspace(D, Hkv, B, cap, 1, Hq),), torch.uint8, fill=0)
    sl = torch.tensor([cap, 17, 0], dtype=torch.int32, device=DEV)
    ckv.attn_decode_f16(k16, v16, sl, cap, q, 1.0 / math.sqrt(D), out.view, lse.view, ws.view)
    assert out.intact() and lse.intact() and ws.intact()
    assert ckv.read_device_flag(ws.view) == 0
    rows = B * Hq
    mo = Guarded((rows, D), torch.float32)
    ml = Guarded((rows,), torch.float32)
    o2 = out.view.reshape(rows, D).clone() * 0.5
    l2 = lse.view.reshape(rows).clone() - 1.0
    ckv.lse_merge([out.view.reshape(rows, D), o2], [lse.view.reshape(rows), l2], mo.view, ml.view)
    assert mo.intact() and ml.intact()
