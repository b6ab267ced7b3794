"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
entry point include/ckv.h declares, and its argument checks return the
documented status before anything reaches the GPU."""
import ctypes
import os
import re

import pytest

from compressed_kv_attention_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from compressed_kv_attention_gb300 import build
        build.build()
    return B.load()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "ckv.h")).read()
    return sorted(set(re.findall(r"CKV_API\s+[\w\s\*]+?\b(ckv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_symbols()
    for required in ("ckv_kv_pack", "ckv_attn_decode", "ckv_attn_prefill", "ckv_lse_merge"):
        assert required in names
    assert len(names) >= 12


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name
        assert name in B.SIGNATURES, f"binding lacks {name}"


def test_version_and_cache_bytes(lib):
    assert lib.ckv_version() == 104
    assert lib.ckv_cache_bytes(512, 2, 1, 32768) == 2 * (32768 // 16) * (23 * 512 + 32)
    assert lib.ckv_cache_bytes(512, 2, 1, 32768) == 2 * 32768 * 738
    assert lib.ckv_cache_bytes(128, 1, 1, 256) == 256 * 186
    for bad in [(96, 1, 1, 16), (128, 0, 1, 16), (128, 1, 0, 16), (128, 1, 1, 20), (128, 1, 1, 0)]:
        assert lib.ckv_cache_bytes(*bad) == 0
    # other V bit widths: 17 D + 2 b D + 32 bytes per 16 positions
    assert lib.ckv_cache_bytes_v(512, 2, 1, 32768, 3, 0) == lib.ckv_cache_bytes(512, 2, 1, 32768)
    assert lib.ckv_cache_bytes_v(512, 2, 1, 32768, 2, 0) == 2 * 32768 * 674
    assert lib.ckv_cache_bytes_v(512, 2, 1, 32768, 4, 0) == 2 * 32768 * 802
    assert lib.ckv_cache_bytes_v(64, 1, 1, 16, 2, 0) == 17 * 64 + 4 * 64 + 32
    for bits in (0, 1, 5, 8):
        assert lib.ckv_cache_bytes_v(128, 1, 1, 256, bits, 0) == 0
    # block-diagonal rotation: one norm per 128 dims (744 B/token at D = 512, 3 bits)
    assert lib.ckv_cache_bytes_v(512, 2, 1, 32768, 3, 128) == 2 * 32768 * 744
    assert lib.ckv_cache_bytes_v(128, 1, 1, 16, 3, 128) == lib.ckv_cache_bytes(128, 1, 1, 16)
    assert lib.ckv_cache_bytes_v(64, 1, 1, 16, 3, 128) == 0
    assert lib.ckv_cache_bytes_v(256, 1, 1, 16, 3, 64) == 0


def _fake_cache(D=128, Hkv=1, batch=1, cap=256, data=0x10000, signs=0x20000, v_bits=0, signs2=0):
    return B.CkvCacheStruct(D, Hkv, batch, v_bits, cap, data, signs, signs2)


def test_pack_argument_checks(lib):
    fake = 0x7f0000000000  # 16-byte aligned, never dereferenced: checks fail first
    c = _fake_cache()
    assert lib.ckv_kv_pack(None, 0, 1, fake, fake, 128, 0, None) == -1
    assert lib.ckv_kv_pack(ctypes.byref(_fake_cache(D=96)), 0, 1, fake, fake, 128, 0, None) == -2
    assert lib.ckv_kv_pack(ctypes.byref(_fake_cache(cap=250)), 0, 1, fake, fake, 128, 0, None) == -1
    for bits in (1, 5, -1):
        assert lib.ckv_kv_pack(ctypes.byref(_fake_cache(v_bits=bits)), 0, 1, fake, fake, 128, 0, None) == -1
    assert b"v_bits" in lib.ckv_last_error()
    # the block-diagonal rotation needs a 128-dim group
    assert lib.ckv_kv_pack(ctypes.byref(_fake_cache(D=64, signs2=0x30000)), 0, 1, fake, fake, 128, 0, None) == -2
    assert lib.ckv_kv_pack(ctypes.byref(_fake_cache(data=0x10008)), 0, 1, fake, fake, 128, 0, None) == -1
    assert lib.ckv_kv_pack(ctypes.byref(c), 250, 10, fake, fake, 128, 0, None) == -1   # past capacity
    assert lib.ckv_kv_pack(ctypes.byref(c), -1, 1, fake, fake, 128, 0, None) == -1
    assert lib.ckv_kv_pack(ctypes.byref(c), 0, 4, None, fake, 128, 0, None) == -1
    assert lib.ckv_kv_pack(ctypes.byref(c), 0, 4, fake + 2, fake, 128, 0, None) == -1  # misaligned
    assert lib.ckv_kv_pack(ctypes.byref(c), 0, 4, fake, fake, 100, 0, None) == -1      # stride < row
    assert lib.ckv_kv_pack(ctypes.byref(c), 0, 0, None, None, 0, 0, None) == 0         # empty: no-op
    assert b"outside" in lib.ckv_last_error() or len(lib.ckv_last_error()) > 0


def test_decode_argument_checks(lib):
    fake = 0x7f0000000000
    c = _fake_cache(D=512, Hkv=2, cap=4096)
    need = lib.ckv_attn_decode_workspace(ctypes.byref(c), 4096, 1, 16, 8)
    # header (flag, 2 groups x (3 leaves + root) counters) in 256 bytes; per group
    # 8 partial slots + 3 leaf slots (leaves of ceil(sqrt(8)) = 3 splits) of 8 x 512 + 16 floats
    assert need == 256 + 2 * (8 + 3) * (8 * 512 + 16) * 4
    assert lib.ckv_attn_decode_workspace(ctypes.byref(c), 4096, 1, 15, 8) == 0  # 15 % 2 != 0
    args = lambda **kw: dict(dict(seq=fake, maxs=4096, q=fake, nq=1, hq=16, scale=0.04, ns=8, out=fake,
                                  lse=fake, ws=fake, wsb=need), **kw)
    def call(cache=c, **kw):
        a = args(**kw)
        return lib.ckv_attn_decode(ctypes.byref(cache), a["seq"], a["maxs"], a["q"], a["nq"], a["hq"],
                                   a["scale"], a["ns"], a["out"], a["lse"], a["ws"], a["wsb"], None)
    assert call(hq=15) == -2                      # 15 query heads over 2 kv heads
    assert call(nq=0) == -1
    assert call(seq=None) == -1
    assert call(q=fake + 4) == -1
    assert call(ws=None) == -3
    assert call(wsb=need - 1) == -3
    assert call(ws=fake + 16) == -3               # workspace must be 256-byte aligned
    assert call(scale=float("nan")) == -1
    assert call(ns=-1) == -3                      # -1: the tile path, whose workspace is larger
    assert call(ns=-2) == -1
    assert call(ns=1025) == -1                    # at most 1024 splits
    assert call(cache=_fake_cache(D=100)) == -2


def test_dca_and_verify_argument_checks(lib):
    fake = 0x7f0000000000
    c = _fake_cache(D=512, Hkv=2, cap=4096)
    need = lib.ckv_attn_decode_dca_workspace(ctypes.byref(c), 4096, 16, 8)
    # the decode's workspace for 2 + m regime rows plus their partials, for any piece count m in [1, 14]
    for m in (1, 14):
        dec = lib.ckv_attn_decode_workspace(ctypes.byref(c), 4096, 2 + m, 16, 8)
        assert need > dec > 0
    call = lambda chunk=64, hq=16, ws=fake, wsb=need: lib.ckv_attn_decode_dca(
        ctypes.byref(c), fake, 4096, chunk, fake, hq, 0.04, 8, fake, fake, ws, wsb, None)
    assert call(chunk=0) == -1
    assert call(hq=15) == -2
    assert call(wsb=need - 1) == -3
    assert call(ws=None) == -3
    assert lib.ckv_attn_decode_verify(ctypes.byref(c), fake, 4096, fake, 4, 15, 0.04, 8, fake, fake, fake,
                                      need, None) == -2


def test_decode_f16_and_merge_argument_checks(lib):
    fake = 0x7f0000000000
    need = lib.ckv_attn_decode_f16_workspace(512, 2, 15, 512, 1, 16, 4)
    # 30 groups: counters 64 + 30 x 3 x 4 bytes -> 512; 4 partial + 2 leaf slots each
    assert need == 512 + 15 * 2 * (4 + 2) * (8 * 512 + 16) * 4
    assert lib.ckv_attn_decode_f16(fake, fake, 512, 2, 15, 500, fake, 512, fake, 1, 16, 0.04, 4, fake, fake,
                                   fake, need, None) == -1  # capacity not a multiple of 16
    assert lib.ckv_attn_decode_f16(fake + 8, fake, 512, 2, 15, 512, fake, 512, fake, 1, 16, 0.04, 4, fake,
                                   fake, fake, need, None) == -1
    ptrs = (ctypes.c_void_p * 2)(fake, fake)
    assert lib.ckv_lse_merge(0, ptrs, ptrs, 10, 512, fake, fake, None) == -1
    assert lib.ckv_lse_merge(17, ptrs, ptrs, 10, 512, fake, fake, None) == -1
    nul = (ctypes.c_void_p * 2)(fake, None)
    assert lib.ckv_lse_merge(2, ptrs, nul, 10, 512, fake, fake, None) == -1
    assert lib.ckv_lse_merge(2, ptrs, ptrs, 10, 0, fake, fake, None) == -1


def test_fanout_step_argument_checks(lib):
    fake = 0x7f0000000000
    pre = _fake_cache(D=512, Hkv=2, batch=1, cap=4096)
    need = lib.ckv_attn_decode_fanout_workspace(ctypes.byref(pre), 4096, 15, 512, 16)
    assert need > 15 * 16 * 512 * 4  # holds at least the prefix partial of the composed form
    assert need % 256 == 0
    assert lib.ckv_attn_decode_fanout_workspace(ctypes.byref(pre), 4096, 15, 512, 8) == 0   # 4 heads per kv head
    assert lib.ckv_attn_decode_fanout_workspace(ctypes.byref(pre), 4096, 0, 512, 16) == 0
    two = _fake_cache(D=512, Hkv=2, batch=2, cap=4096)
    assert lib.ckv_attn_decode_fanout_workspace(ctypes.byref(two), 4096, 15, 512, 16) == 0  # prefix of 2 sequences

    def call(cache, n_q_heads=16, max_prefix=4096, cap=512, max_tail=512, k=fake, ws_bytes=need):
        return lib.ckv_attn_decode_fanout(ctypes.byref(cache), fake, max_prefix, k, fake, cap, fake, max_tail, 15,
                                          fake, n_q_heads, 0.04, fake, fake, fake, ws_bytes, None)
    assert call(pre, n_q_heads=8) == -2
    assert call(two) == -1
    assert call(pre, max_prefix=5000) == -1       # beyond the prefix capacity
    assert call(pre, max_tail=600) == -1          # beyond the tail capacity
    assert call(pre, cap=500, max_tail=400) == -1  # tail capacity not a multiple of 16
    assert call(pre, k=fake + 8) == -1
    assert call(pre, ws_bytes=need - 256) == -3


def test_fanout_plan_argument_checks(lib):
    ps, ts = ctypes.c_int32(7), ctypes.c_int32(7)
    assert lib.ckv_fanout_plan(15, 2, 16, None, ctypes.byref(ts)) == -1
    assert lib.ckv_fanout_plan(0, 2, 16, ctypes.byref(ps), ctypes.byref(ts)) == -1
    assert lib.ckv_fanout_plan(15, 0, 16, ctypes.byref(ps), ctypes.byref(ts)) == -1
    assert lib.ckv_fanout_plan(15, 3, 16, ctypes.byref(ps), ctypes.byref(ts)) == -2  # 16 heads over 3 kv heads


def test_read_device_flag_checks(lib):
    flag = ctypes.c_int32(7)
    assert lib.ckv_read_device_flag(None, ctypes.byref(flag), None) == -1
    assert lib.ckv_read_noalloc_flag(None, None) == -1
    assert lib.ckv_calibrate_stream(None, 16, 11808, 1, 1, 0, None, 0, None) == -1


def test_prefill_argument_checks(lib):
    fake = 0x7f0000000000
    c = _fake_cache(D=512, Hkv=2, cap=4096)
    ws = 256
    call = lambda cache=c, n_cached=0, q=fake, n_new=16, hq=16, k=fake, v=fake, out=fake, lse=fake, w=fake, wb=ws: \
        lib.ckv_attn_prefill(ctypes.byref(cache) if cache is not None else None, n_cached, q, n_new, hq, k, v,
                             0.04, out, lse, w, wb, None)
    assert call(cache=None) == -1
    assert call(cache=_fake_cache(D=32)) == -2       # prefill head dims: 64, 128, 256, 512
    assert call(n_cached=4090) == -1                 # past capacity
    assert call(hq=12) == -2                         # 6 heads per kv head does not divide 128
    for bits in (2, 3, 4):   # every tier passes the checks (then the workspace)
        assert call(cache=_fake_cache(D=512, Hkv=2, cap=4096, v_bits=bits)) == -3
        assert call(cache=_fake_cache(D=512, Hkv=2, cap=4096, v_bits=bits, signs2=0x30000)) == -3
    assert call(cache=_fake_cache(D=512, Hkv=2, cap=4096, v_bits=5)) == -1
    assert call(cache=_fake_cache(D=64, Hkv=2, cap=4096, signs2=0x30000)) == -2   # rotation needs D >= 128
    assert call(q=fake + 8) == -1
    assert call(out=None) == -1
    assert call(w=None) == -3
    assert call(wb=128) == -3
    assert call(n_new=0) == 0                        # nothing to do


def test_decode_append_argument_checks(lib):
    fake = 0x7f0000000000
    c = _fake_cache(D=512, Hkv=2, cap=4096)
    need = lib.ckv_attn_decode_workspace(ctypes.byref(c), 4096, 1, 16, 8)

    def call(nq=1, hq=16, k=fake, v=fake, n_new=1, ts=1024, bs=0, wsb=need):
        return lib.ckv_attn_decode_append(ctypes.byref(c), fake, 4096, k, v, n_new, ts, bs, fake, nq, hq, 0.04, 8,
                                          fake, fake, fake, wsb, None)
    assert call(nq=2) == -2          # 16 query rows per kv head: more than one row group
    assert call(n_new=0) == -1
    assert call(n_new=17) == -1
    assert call(k=None) == -1
    assert call(v=fake + 8) == -1    # not 16-byte aligned
    assert call(ts=1000) == -1       # token stride below one row of all kv heads
    assert call(ts=1028) == -1       # not a multiple of 8 elements
    assert call(bs=-8) == -1
    assert call(wsb=need - 1) == -3


def test_multitenant_prefill_argument_checks(lib):
    fake = 0x7f0000000000
    pre = _fake_cache(D=512, Hkv=2, cap=4096)
    two = _fake_cache(D=512, Hkv=2, batch=2, cap=4096)
    ws = lib.ckv_attn_prefill_shared_workspace(ctypes.byref(pre), 15, 1024, 64, 16)
    assert ws > 0
    assert lib.ckv_attn_prefill_shared_workspace(ctypes.byref(pre), 0, 1024, 64, 16) == 0

    def shared(cache=pre, n_prefix=4096, n_agents=15, n_new=64, hq=16, w=fake, wb=ws):
        return lib.ckv_attn_prefill_shared(ctypes.byref(cache), n_prefix, fake, fake, 1024, fake, n_agents, fake,
                                           fake, fake, n_new, hq, 0.04, fake, fake, w, wb, None)
    assert shared(cache=two) == -1          # the shared prefix is one sequence
    assert shared(n_prefix=4097) == -1      # past the prefix cache
    assert shared(n_agents=0) == -1
    assert shared(n_new=0) == 0             # nothing to do
    assert shared(wb=ws - 1) == -3
    assert shared(w=fake + 8) == -3         # workspace alignment
    # prefix-only prefill: at least one prefix token, inside the cache
    pf = lambda n_prefix, n_tok=16: lib.ckv_attn_prefill_prefix(ctypes.byref(pre), n_prefix, fake, n_tok, 16, 0.04,
                                                                 fake, fake, fake, 1 << 20, None)
    assert pf(0) == -1 and pf(4097) == -1 and pf(100, 0) == 0
    # tail append: strides and geometry
    ap = lambda ts, hd=512: lib.ckv_f16_append(fake, fake, hd, 2, 3, 1024, fake, fake, fake, 8, ts, ts * 8, None)
    assert ap(1000) == -1 and ap(1024, hd=96) == -2


def test_many_row_decode_path_selection(lib):
    """n_split 0 takes the 128-row tile path only where the cost model prefers
    it (long prefixes with many rows per kv head); -1 forces it; a head ratio
    that does not divide 128 cannot take it. The choice shows in the workspace
    size (the tile path keeps one 128 x (D + 1) float slot per tile and split)."""
    c_short = _fake_cache(D=512, Hkv=2, cap=4096)
    c_long = _fake_cache(D=512, Hkv=2, cap=65536)
    ws = lambda c, P, n_q, hq, ns: lib.ckv_attn_decode_workspace(ctypes.byref(c), P, n_q, hq, ns)  # noqa: E731
    tiles_short, auto_short = ws(c_short, 4096, 15, 16, -1), ws(c_short, 4096, 15, 16, 0)
    assert tiles_short > 256 + 2 * 128 * 513 * 4 and auto_short < tiles_short     # 4096 tokens: mma.sync
    tiles_long, auto_long = ws(c_long, 65536, 15, 16, -1), ws(c_long, 65536, 15, 16, 0)
    assert auto_long == tiles_long                                                # 65536 tokens: tiles
    assert ws(c_long, 65536, 8, 16, 0) < ws(c_long, 65536, 8, 16, -1)            # 64 rows: mma.sync
    assert ws(_fake_cache(D=128, Hkv=1, cap=64), 64, 8, 12, -1) == 0             # 12 heads per kv head
    fake = 0x7f0000000000
    c = _fake_cache(D=128, Hkv=1, cap=64)
    assert lib.ckv_attn_decode(ctypes.byref(c), fake, 64, fake, 8, 12, 0.1, -1, fake, fake, fake, 1 << 20,
                               None) == -2
    assert lib.ckv_attn_decode(ctypes.byref(c), fake, 64, fake, 8, 16, 0.1, -2, fake, fake, fake, 1 << 20,
                               None) == -1


def test_selftest_argument_checks(lib):
    assert lib.ckv_selftest_bounded_waits(None, 256, None) == -3
    assert lib.ckv_selftest_bounded_waits(0x7f0000000000, 128, None) == -3    # fewer than 256 bytes
    assert lib.ckv_selftest_bounded_waits(0x7f0000000010, 256, None) == -3    # not 256-byte aligned


def test_prefill_workspace_sizes(lib):
    """Flag (256 bytes) + one int32 per 128-row tile (rounded to 256 bytes) and,
    once there are more tiles than SMs, two partial slots of 128 x (D + 1)
    floats per SM for the tiles the stream-K schedule cuts."""
    c = _fake_cache(D=64, Hkv=2, cap=4096)
    small = lib.ckv_attn_prefill_workspace(ctypes.byref(c), 48, 16)          # 2 kv heads x 3 tiles of 16 tokens
    assert small == 256 + 256
    big = lib.ckv_attn_prefill_workspace(ctypes.byref(c), 2560, 16)         # 2 x 160 tiles
    slots = big - 256 - (4 * 320 + 255) // 256 * 256
    per_sm = 2 * 128 * 65 * 4
    assert slots > 0 and slots % per_sm == 0                               # whole SMs' worth of slot pairs
    assert lib.ckv_attn_prefill_workspace(None, 16, 16) == 256
