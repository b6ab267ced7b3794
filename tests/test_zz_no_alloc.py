"""The allocation-free decode entry point (ckv_attn_decode_noalloc).

Some callers cannot allocate device memory — a host framework that owns it all,
a loop that must not call cudaMalloc, a process that has already given the
device away — so the library offers one decode entry point whose scratch is a
fixed array inside the library instead of a caller workspace. This checks,
through the C ABI, that two calls in a row (the second reusing the array the
first one left behind, with different shapes) give the same results as the
regular entry point within the attention tolerance, and that a call whose
scratch would not fit is refused without launching anything.

Collected last on purpose: it runs after every other test, and also passes in
a fresh process on its own.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import compressed_kv_attention_gb300 as ckv  # noqa: E402
from compressed_kv_attention_gb300 import inputs  # noqa: E402
from tests import helpers as H  # noqa: E402

pytestmark = pytest.mark.gpu


def _case(D, Hkv, Hq, n_q, B, cap, seq_lens, seed):
    dev = "cuda"
    outl = inputs.outlier_channels(D, max(1, D // 100), seed)
    k = inputs.normal_tensor((B, cap, Hkv, D), seed, "noalloc/k", outl, device=dev)
    v = inputs.normal_tensor((B, cap, Hkv, D), seed, "noalloc/v", outl, device=dev)
    q = inputs.normal_tensor((B, n_q, Hq, D), seed, "noalloc/q", outl, device=dev)
    cache = ckv.PackedCache(D, Hkv, B, cap, inputs.tbq_signs(D), device=dev)
    ckv.kv_pack(cache, 0, k, v)
    sl = torch.tensor(seq_lens, dtype=torch.int32, device=dev)
    return cache, q, sl, max(seq_lens)


def _both(cache, q, sl, max_len):
    B, n_q, Hq, D = q.shape
    scale = 1.0 / math.sqrt(D)
    out_a = torch.empty((B, n_q, Hq, D), dtype=torch.float32, device="cuda")
    lse_a = torch.empty((B, n_q, Hq), dtype=torch.float32, device="cuda")
    ws = torch.zeros(ckv.attn_decode_workspace(cache, max_len, n_q, Hq), dtype=torch.uint8, device="cuda")
    ckv.attn_decode(cache, sl, max_len, q, scale, out_a, lse_a, ws)
    out_b = torch.full_like(out_a, float("nan"))
    lse_b = torch.full_like(lse_a, float("nan"))
    ckv.attn_decode_noalloc(cache, sl, max_len, q, scale, out_b, lse_b)
    torch.cuda.synchronize()
    return (out_a.cpu().numpy().astype(np.float64), lse_a.cpu().numpy().astype(np.float64),
            out_b.cpu().numpy(), lse_b.cpu().numpy())


def test_noalloc_matches_regular_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # First call: Gemma-4 global-layer shapes, 4096 cached tokens.
    ref_o, ref_l, o, l = _both(*_case(512, 2, 16, 1, 1, 4096, [4096], seed=31))
    H.check_attention(o, l, ref_o, ref_l, "noalloc call 1")
    # Second call, different shapes, ragged and empty sequences: the array still
    # holds the first call's partials.
    ref_o, ref_l, o, l = _both(*_case(128, 1, 4, 2, 3, 208, [208, 0, 131], seed=32))
    H.check_attention(o, l, ref_o, ref_l, "noalloc call 2")


def test_noalloc_refuses_scratch_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
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
