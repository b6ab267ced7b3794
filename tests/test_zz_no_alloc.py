"""The allocation-free decode entry point (ckv_attn_decode_noalloc).

Some callers cannot allocate device memory — a host framework that owns it all,
a loop that must not call cudaMalloc, a process that has already given the
device away — so the library offers one decode entry point whose scratch is a
fixed array inside the library instead of a caller workspace. Through the C
ABI this checks that:

* calls in a row give the results of the regular entry point (on a zeroed
  workspace) and of the oracle, within the attention tolerance, although each
  finds the array as the previous call left it: a small call before a call
  with many more row groups (whose merge counters then lie where the first
  call wrote partials), a tile-path call before a many-group call;
* a seq_len out of range raises the array's device flag, which
  ckv_read_noalloc_flag reads and clears, and the row counts as empty;
* a call whose scratch would not fit is refused without launching anything.

Collected last on purpose: it runs after every other test, and also passes in
a fresh process on its own.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import compressed_kv_attention_gb300 as ckv  # noqa: E402
from compressed_kv_attention_gb300 import inputs  # noqa: E402
from oracle import ckv_oracle as O  # noqa: E402
from tests import helpers as H  # noqa: E402

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class _Case:
    """Seeded K/V/Q (numpy, fp16), the GPU-packed cache and the oracle's result."""

    def __init__(self, D, Hkv, Hq, n_q, B, cap, seq_lens, seed):
        outl = inputs.outlier_channels(D, max(1, D // 100), seed)
        self.k = inputs.normal_tensor((B, cap, Hkv, D), seed, "noalloc/k", outl)
        self.v = inputs.normal_tensor((B, cap, Hkv, D), seed, "noalloc/v", outl)
        self.q = inputs.normal_tensor((B, n_q, Hq, D), seed, "noalloc/q", outl)
        self.signs = inputs.tbq_signs(D)
        self.cache = ckv.PackedCache(D, Hkv, B, cap, self.signs, device="cuda")
        ckv.kv_pack(self.cache, 0, torch.from_numpy(self.k).cuda(), torch.from_numpy(self.v).cuda())
        self.seq_lens = [int(s) for s in seq_lens]
        self.sl = torch.tensor(self.seq_lens, dtype=torch.int32, device="cuda")
        self.max_len = max(self.seq_lens)
        self.qd = torch.from_numpy(self.q).cuda()
        self.scale = 1.0 / math.sqrt(D)

    def oracle(self, valid=None):
        """Oracle decode; sequences with valid[b] False count as empty."""
        B, n_q, Hq, D = self.q.shape
        kt = np.ascontiguousarray(np.swapaxes(self.k, 1, 2))
        vt = np.ascontiguousarray(np.swapaxes(self.v, 1, 2))
        qs, d16, codes, n16, _ = H.oracle_quantize(kt, vt, self.signs)
        o = np.zeros((B, n_q, Hq, D))
        lse = np.full((B, n_q, Hq), -np.inf)
        for b, T in enumerate(self.seq_lens):
            if valid is not None and not valid[b]:
                continue
            kh = O.q8_0_dequantize(qs[b, :, :T], d16[b, :, :T])
            vh = O.tbq3_dequantize(codes[b, :, :T], n16[b, :, :T], self.signs)
            o[b], lse[b] = O.decode_reference(self.q[b].astype(np.float64), kh, vh, T, self.scale)
        return o, lse

    def _outputs(self, fill):
        B, n_q, Hq, D = self.q.shape
        return (torch.full((B, n_q, Hq, D), fill, dtype=torch.float32, device="cuda"),
                torch.full((B, n_q, Hq), fill, dtype=torch.float32, device="cuda"))

    def regular(self, n_split=0):
        B, n_q, Hq, D = self.q.shape
        out, lse = self._outputs(0.0)
        ws = torch.zeros(ckv.attn_decode_workspace(self.cache, self.max_len, n_q, Hq, n_split),
                         dtype=torch.uint8, device="cuda")
        ckv.attn_decode(self.cache, self.sl, self.max_len, self.qd, self.scale, out, lse, ws, n_split=n_split)
        torch.cuda.synchronize()
        assert ckv.read_device_flag(ws) == 0
        return out.cpu().numpy(), lse.cpu().numpy()

    def noalloc(self, n_split=0, max_len=None):
        out, lse = self._outputs(float("nan"))
        ckv.attn_decode_noalloc(self.cache, self.sl, self.max_len if max_len is None else max_len, self.qd,
                                self.scale, out, lse, n_split=n_split)
        torch.cuda.synchronize()
        return out.cpu().numpy(), lse.cpu().numpy()


def _check_call(case, what, n_split=0):
    o, l = case.noalloc(n_split)
    assert ckv.read_noalloc_flag() == 0, f"{what}: device flag raised"
    ro, rl = case.regular(n_split)
    H.check_attention(o, l, ro, rl, f"{what} vs attn_decode")
    oo, ol = case.oracle()
    H.check_attention(o, l, oo, ol, f"{what} vs oracle")


def test_noalloc_matches_regular_entry_point_twice():
    _need_gpu()
    ckv.read_noalloc_flag()  # start from a clear flag
    # First call: Gemma-4 global-layer shapes, 4096 cached tokens.
    _check_call(_Case(512, 2, 16, 1, 1, 4096, [4096], seed=31), "call 1")
    # Second call, different shapes, ragged and empty sequences: the array
    # still holds the first call's partials.
    _check_call(_Case(128, 1, 4, 2, 3, 208, [208, 0, 131], seed=32), "call 2")


def test_noalloc_after_calls_of_other_shapes():
    _need_gpu()
    ckv.read_noalloc_flag()
    # 2 row groups: counters in bytes [64, 80), partials from byte 256.
    _check_call(_Case(512, 2, 16, 1, 1, 2048, [2048], seed=33), "2 groups")
    # 64 row groups: counters up to byte 576 (2 splits, rendezvous merge) or
    # 832 (4 splits, tree merge), where the previous calls' partials lie.
    many = _Case(128, 1, 4, 1, 64, 256, list(np.random.default_rng(34).integers(1, 257, 64)), seed=34)
    _check_call(many, "64 groups after 2")
    _check_call(many, "64 groups, 4 splits", n_split=4)
    # The tile path (n_split -1) writes its partials from byte 256 and keeps no
    # counters; the many-group calls after it must not read them as counters.
    _check_call(_Case(128, 1, 8, 16, 1, 1024, [1024], seed=35), "tile path", n_split=-1)
    _check_call(many, "64 groups after the tile path")
    _check_call(many, "64 groups, 4 splits, after the tile path", n_split=4)


def test_noalloc_flag_reports_out_of_range_seq_len():
    _need_gpu()
    ckv.read_noalloc_flag()
    # max_seq_len 128 < capacity 256: a seq_len of 200 is out of range. The
    # kernel raises the flag (2) and counts that sequence as empty.
    case = _Case(128, 1, 4, 1, 2, 256, [100, 200], seed=36)
    o, l = case.noalloc(max_len=128)
    assert ckv.read_noalloc_flag() == 2
    assert ckv.read_noalloc_flag() == 0  # read clears it
    oo, ol = case.oracle(valid=[True, False])
    H.check_attention(o, l, oo, ol, "out-of-range sequence")
    # The next call on the same array is clean and correct.
    _check_call(_Case(128, 1, 4, 1, 2, 256, [100, 256], seed=37), "after the flag")


def test_noalloc_refuses_scratch_beyond_its_array():
    _need_gpu()
    cache = ckv.PackedCache(512, 2, 64, 16, inputs.tbq_signs(512), device="cuda")
    need = ckv.attn_decode_workspace(cache, 16, 1, 16, n_split=8)
    assert need > (4 << 20)
    q = torch.zeros((64, 1, 16, 512), dtype=torch.float16, device="cuda")
    out = torch.zeros((64, 1, 16, 512), dtype=torch.float32, device="cuda")
    lse = torch.zeros((64, 1, 16), dtype=torch.float32, device="cuda")
    sl = torch.full((64,), 16, dtype=torch.int32, device="cuda")
    with pytest.raises(ckv.CkvError) as err:
        ckv.attn_decode_noalloc(cache, sl, 16, q, 0.04, out, lse, n_split=8)
    assert err.value.status == -3 and "scratch" in str(err.value)
    torch.cuda.synchronize()
    assert torch.all(out == 0)   # nothing ran
