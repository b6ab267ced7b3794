"""ctypes binding of libckv.so (include/ckv.h): argument marshalling only.

Every function here has the name of the C entry point it calls, without the
``ckv_`` prefix, takes torch tensors for device memory, passes their pointers
and the current (or given) CUDA stream, and raises ``CkvError`` on a non-OK
status. No computation happens in Python: every step of the path runs in the
library's kernels. If the library is missing, loading it raises immediately.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libckv.so")

CKV_OK = 0
STATUS_NAMES = {0: "OK", -1: "INVALID_ARG", -2: "UNSUPPORTED", -3: "WORKSPACE", -4: "CUDA",
                -5: "DEVICE_FLAG"}


class CkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class CkvCacheStruct(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("v_bits", ctypes.c_int32),
                ("capacity", ctypes.c_int64), ("data", ctypes.c_void_p),
                ("v_signs", ctypes.c_void_p), ("v_signs2", ctypes.c_void_p)]


_lib = None

_c_int, _c_i64, _c_size, _c_f, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p
_cache_p = ctypes.POINTER(CkvCacheStruct)

SIGNATURES = {
    "ckv_version": (_c_int, []),
    "ckv_last_error": (ctypes.c_char_p, []),
    "ckv_cache_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_i64]),
    "ckv_cache_bytes_v": (_c_size, [_c_int, _c_int, _c_int, _c_i64, _c_int, _c_int]),
    "ckv_kv_pack": (_c_int, [_cache_p, _c_i64, _c_i64, _vp, _vp, _c_i64, _c_i64, _vp]),
    "ckv_attn_decode_workspace": (_c_size, [_cache_p, _c_i64, _c_int, _c_int, _c_int]),
    "ckv_attn_decode": (_c_int, [_cache_p, _vp, _c_i64, _vp, _c_int, _c_int, _c_f, _c_int, _vp, _vp,
                                 _vp, _c_size, _vp]),
    "ckv_attn_decode_dca_workspace": (_c_size, [_cache_p, _c_i64, _c_int, _c_int]),
    "ckv_attn_decode_dca": (_c_int, [_cache_p, _vp, _c_i64, _c_int, _vp, _c_int, _c_f, _c_int, _vp, _vp, _vp,
                                     _c_size, _vp]),
    "ckv_attn_decode_verify": (_c_int, [_cache_p, _vp, _c_i64, _vp, _c_int, _c_int, _c_f, _c_int, _vp, _vp,
                                        _vp, _c_size, _vp]),
    "ckv_attn_decode_append": (_c_int, [_cache_p, _vp, _c_i64, _vp, _vp, _c_int, _c_i64, _c_i64, _vp, _c_int,
                                        _c_int, _c_f, _c_int, _vp, _vp, _vp, _c_size, _vp]),
    "ckv_attn_decode_append_host": (_c_int, [_cache_p, _vp, _c_i64, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_f,
                                             _c_int, _vp, _vp, _vp, _c_size, _vp]),
    "ckv_attn_decode_noalloc": (_c_int, [_cache_p, _vp, _c_i64, _vp, _c_int, _c_int, _c_f, _c_int, _vp,
                                         _vp, _vp]),
    "ckv_attn_decode_f16_workspace": (_c_size, [_c_int, _c_int, _c_int, _c_i64, _c_int, _c_int, _c_int]),
    "ckv_attn_decode_f16_merge_workspace": (_c_size, [_c_int, _c_int, _c_int, _c_i64, _c_int, _c_int, _c_int]),
    "ckv_attn_decode_f16_merge": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_i64, _vp, _c_i64, _vp, _c_int,
                                           _c_int, _c_f, _c_int, _vp, _vp, _vp, _vp, _vp, _c_size, _vp]),
    "ckv_attn_decode_fanout_workspace": (_c_size, [_cache_p, _c_i64, _c_int, _c_i64, _c_int]),
    "ckv_attn_decode_fanout": (_c_int, [_cache_p, _vp, _c_i64, _vp, _vp, _c_i64, _vp, _c_i64, _c_int, _vp, _c_int,
                                        _c_f, _vp, _vp, _vp, _c_size, _vp]),
    "ckv_fanout_plan": (_c_int, [_c_int, _c_int, _c_int, ctypes.POINTER(ctypes.c_int32),
                                 ctypes.POINTER(ctypes.c_int32)]),
    "ckv_attn_decode_f16": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_i64, _vp, _c_i64, _vp, _c_int,
                                     _c_int, _c_f, _c_int, _vp, _vp, _vp, _c_size, _vp]),
    "ckv_lse_merge": (_c_int, [_c_int, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _c_i64, _c_int, _vp, _vp,
                               _vp]),
    "ckv_attn_prefill_workspace": (_c_size, [_cache_p, _c_int, _c_int]),
    "ckv_selftest_bounded_waits": (_c_int, [_vp, _c_size, _vp]),
    "ckv_attn_prefill": (_c_int, [_cache_p, _c_i64, _vp, _c_int, _c_int, _vp, _vp, _c_f, _vp, _vp, _vp,
                                  _c_size, _vp]),
    "ckv_attn_prefill_prefix": (_c_int, [_cache_p, _c_i64, _vp, _c_int, _c_int, _c_f, _vp, _vp, _vp, _c_size, _vp]),
    "ckv_f16_append": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_i64, _vp, _vp, _vp, _c_int, _c_i64, _c_i64,
                                _vp]),
    "ckv_attn_prefill_f16": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_i64, _vp, _c_i64, _vp, _c_int, _c_int,
                                      _c_f, _c_int, _vp, _vp, _vp, _c_size, _vp]),
    "ckv_attn_prefill_shared_workspace": (_c_size, [_cache_p, _c_int, _c_i64, _c_int, _c_int]),
    "ckv_attn_prefill_shared": (_c_int, [_cache_p, _c_i64, _vp, _vp, _c_i64, _vp, _c_int, _vp, _vp, _vp, _c_int,
                                         _c_int, _c_f, _vp, _vp, _vp, _c_size, _vp]),
    "ckv_read_device_flag": (_c_int, [_vp, ctypes.POINTER(_c_int), _vp]),
    "ckv_set_concurrent_kernels": (None, [_c_int]),
    "ckv_read_noalloc_flag": (_c_int, [ctypes.POINTER(_c_int), _vp]),
    "ckv_calibrate_stream": (_c_int, [_vp, _c_i64, _c_int, _c_int, _c_int, _c_int, _vp, _c_size, _vp]),
}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libckv.so (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with compressed_kv_attention_gb300/build.py "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != CKV_OK:
        raise CkvError(status, load().ckv_last_error().decode())


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


class PackedCache:
    """A packed q8_0-K / TBQ-V cache in device memory plus its geometry
    (``v_bits`` bits per V code: 3 is TBQ3, 2 and 4 the neighbouring tiers;
    ``signs2`` given: the block-diagonal rotation over 128-dim groups with
    ``signs`` before and ``signs2`` after the transform)."""

    def __init__(self, head_dim: int, n_kv_heads: int, batch: int, capacity: int, signs,
                 device="cuda", data=None, v_bits: int = 3, signs2=None):
        import torch
        self.head_dim, self.n_kv_heads, self.batch, self.capacity = head_dim, n_kv_heads, batch, capacity
        self.v_bits = v_bits
        self.rot_group = 128 if signs2 is not None else 0
        nbytes = cache_bytes(head_dim, n_kv_heads, batch, capacity, v_bits, self.rot_group)
        if nbytes == 0:
            raise CkvError(-1, "invalid cache geometry")
        self.data = data if data is not None else torch.zeros(nbytes, dtype=torch.uint8, device=device)
        self.signs = torch.as_tensor(signs, dtype=torch.int8).to(device)
        self.signs2 = None if signs2 is None else torch.as_tensor(signs2, dtype=torch.int8).to(device)
        self.struct = CkvCacheStruct(head_dim, n_kv_heads, batch, v_bits, capacity, _ptr(self.data),
                                     _ptr(self.signs), _ptr(self.signs2))

    def ref(self):
        return ctypes.byref(self.struct)


def version() -> int:
    return load().ckv_version()


def cache_bytes(head_dim: int, n_kv_heads: int, batch: int, capacity: int, v_bits: int = 3,
                rot_group: int = 0) -> int:
    return int(load().ckv_cache_bytes_v(head_dim, n_kv_heads, batch, capacity, v_bits, rot_group))


def kv_pack(cache: PackedCache, tok_offset: int, k, v, stream=None):
    """Pack fp16 K, V shaped [batch, n_tok, n_kv_heads, D] at positions [tok_offset, +n_tok)."""
    n_tok = k.shape[1]
    _check(load().ckv_kv_pack(cache.ref(), tok_offset, n_tok, _ptr(k), _ptr(v), k.stride(1), k.stride(0),
                              _stream(stream)))


def attn_decode_workspace(cache: PackedCache, max_seq_len: int, n_q: int, n_q_heads: int,
                          n_split: int = 0) -> int:
    return int(load().ckv_attn_decode_workspace(cache.ref(), max_seq_len, n_q, n_q_heads, n_split))


def attn_decode(cache: PackedCache, seq_len, max_seq_len: int, q, scale: float, out, lse, workspace,
                n_split: int = 0, stream=None):
    """q: fp16 [batch, n_q, n_q_heads, D]; out float32 like q; lse float32 [batch, n_q, n_q_heads].
    n_split: 0 automatic, > 0 that many key splits on the mma.sync decode, -1 the 128-row tcgen05
    tile path for many query rows per kv head (size the workspace with the same n_split)."""
    _, n_q, n_q_heads, _ = q.shape
    _check(load().ckv_attn_decode(cache.ref(), _ptr(seq_len), max_seq_len, _ptr(q), n_q, n_q_heads, scale,
                                  n_split, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                  _stream(stream)))


def attn_decode_dca_workspace(cache: PackedCache, max_seq_len: int, n_q_heads: int, n_split: int = 0) -> int:
    return int(load().ckv_attn_decode_dca_workspace(cache.ref(), max_seq_len, n_q_heads, n_split))


def attn_decode_dca(cache: PackedCache, seq_len, max_seq_len: int, chunk: int, q, scale: float, out, lse,
                    workspace, n_split: int = 0, stream=None):
    """Dual chunk attention: q fp16 [batch, 3, n_q_heads, D] holds the intra, successive and inter
    regime queries of the token at position seq_len - 1; out float32 [batch, n_q_heads, D], lse
    float32 [batch, n_q_heads]."""
    _, n_r, n_q_heads, _ = q.shape
    if n_r != 3:
        raise ValueError("q must hold the three regime queries on its second axis")
    _check(load().ckv_attn_decode_dca(cache.ref(), _ptr(seq_len), max_seq_len, chunk, _ptr(q), n_q_heads, scale,
                                      n_split, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                      _stream(stream)))


def attn_decode_verify(cache: PackedCache, seq_len, max_seq_len: int, q, scale: float, out, lse, workspace,
                       n_split: int = 0, stream=None):
    """Verify batch: q fp16 [batch, n_q, n_q_heads, D] are the last n_q positions of each
    sequence; query token i sees [0, seq_len - n_q + i]. Outputs as attn_decode."""
    _, n_q, n_q_heads, _ = q.shape
    _check(load().ckv_attn_decode_verify(cache.ref(), _ptr(seq_len), max_seq_len, _ptr(q), n_q, n_q_heads, scale,
                                         n_split, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                         _stream(stream)))


def attn_decode_append(cache: PackedCache, seq_len, max_seq_len: int, k_new, v_new, q, scale: float, out, lse,
                       workspace, n_split: int = 0, stream=None):
    """One decode step: pack k_new / v_new (fp16 [batch, n_new, n_kv_heads, D]) at positions
    [seq_len - n_new, seq_len) of every sequence, then attn_decode over [0, seq_len)."""
    _, n_q, n_q_heads, _ = q.shape
    n_new = k_new.shape[1]
    _check(load().ckv_attn_decode_append(cache.ref(), _ptr(seq_len), max_seq_len, _ptr(k_new), _ptr(v_new), n_new,
                                         k_new.stride(1), k_new.stride(0), _ptr(q), n_q, n_q_heads, scale, n_split,
                                         _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                         _stream(stream)))


def attn_decode_append_host(cache: PackedCache, seq_len, max_seq_len: int, k_new_host, v_new_host, q_host,
                            scale: float, out_host, lse_host, workspace, n_split: int = 0, stream=None):
    """One decode step on pinned host tensors (contiguous): q [B, n_q, Hq, D], k_new / v_new
    [B, n_new, Hkv, D] fp16 read, out [B, n_q, Hq, D] / lse [B, n_q, Hq] fp32 written by the kernel
    across the CPU-GPU interconnect; asynchronous on `stream`."""
    _, n_q, n_q_heads, _ = q_host.shape
    _check(load().ckv_attn_decode_append_host(cache.ref(), _ptr(seq_len), max_seq_len, _ptr(k_new_host),
                                              _ptr(v_new_host), k_new_host.shape[1], _ptr(q_host), n_q, n_q_heads,
                                              scale, n_split, _ptr(out_host), _ptr(lse_host), _ptr(workspace),
                                              workspace.numel(), _stream(stream)))


def attn_decode_noalloc(cache: PackedCache, seq_len, max_seq_len: int, q, scale: float, out, lse,
                        n_split: int = 0, stream=None):
    """attn_decode without a workspace: scratch lives in a fixed array inside the
    library (for callers that cannot allocate device memory; calls must not
    overlap on the GPU)."""
    _, n_q, n_q_heads, _ = q.shape
    _check(load().ckv_attn_decode_noalloc(cache.ref(), _ptr(seq_len), max_seq_len, _ptr(q), n_q, n_q_heads,
                                          scale, n_split, _ptr(out), _ptr(lse), _stream(stream)))


def attn_decode_f16_workspace(head_dim: int, n_kv_heads: int, batch: int, max_seq_len: int, n_q: int,
                              n_q_heads: int, n_split: int = 0) -> int:
    return int(load().ckv_attn_decode_f16_workspace(head_dim, n_kv_heads, batch, max_seq_len, n_q,
                                                    n_q_heads, n_split))


def attn_decode_f16_merge_workspace(head_dim: int, n_kv_heads: int, batch: int, max_seq_len: int, n_q: int,
                                    n_q_heads: int, n_split: int = 0) -> int:
    return int(load().ckv_attn_decode_f16_merge_workspace(head_dim, n_kv_heads, batch, max_seq_len, n_q,
                                                          n_q_heads, n_split))


def attn_decode_f16_merge(k, v, seq_len, max_seq_len: int, q, scale: float, prior_o, prior_lse, out, lse,
                          workspace, n_split: int = 0, stream=None):
    """attn_decode_f16 merged exactly with a prior partial (rows and lse laid out as out / lse)."""
    batch, n_kv_heads, capacity, D = k.shape
    _, n_q, n_q_heads, _ = q.shape
    _check(load().ckv_attn_decode_f16_merge(_ptr(k), _ptr(v), D, n_kv_heads, batch, capacity, _ptr(seq_len),
                                            max_seq_len, _ptr(q), n_q, n_q_heads, scale, n_split, _ptr(prior_o),
                                            _ptr(prior_lse), _ptr(out), _ptr(lse), _ptr(workspace),
                                            workspace.numel(), _stream(stream)))


def attn_decode_fanout_workspace(prefix: PackedCache, max_prefix_len: int, n_agents: int, max_tail_len: int,
                                 n_q_heads: int) -> int:
    return int(load().ckv_attn_decode_fanout_workspace(prefix.ref(), max_prefix_len, n_agents,
                                                       max_tail_len, n_q_heads))


def attn_decode_fanout(prefix: PackedCache, prefix_len, max_prefix_len: int, k_tail, v_tail, tail_len,
                       max_tail_len: int, q, scale: float, out, lse, workspace, stream=None):
    """One fan-out decode step: q fp16 [n_agents, n_q_heads, D] over the shared prefix and each agent's
    fp16 tail (k_tail, v_tail [n_agents, n_kv_heads, capacity, D]); out [n_agents, n_q_heads, D]."""
    n_agents, n_kv_heads, capacity, D = k_tail.shape
    _check(load().ckv_attn_decode_fanout(prefix.ref(), _ptr(prefix_len), max_prefix_len,
                                         _ptr(k_tail), _ptr(v_tail), capacity, _ptr(tail_len), max_tail_len,
                                         n_agents, _ptr(q), q.shape[1], scale, _ptr(out), _ptr(lse),
                                         _ptr(workspace), workspace.numel(), _stream(stream)))


def fanout_plan(n_agents: int, n_kv_heads: int, n_q_heads: int):
    """(prefix_splits, tail_splits) for the fan-out step on the current device (0, 0: automatic)."""
    ps, ts = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load().ckv_fanout_plan(n_agents, n_kv_heads, n_q_heads, ctypes.byref(ps), ctypes.byref(ts)))
    return ps.value, ts.value


def attn_decode_f16(k, v, seq_len, max_seq_len: int, q, scale: float, out, lse, workspace,
                    n_split: int = 0, stream=None):
    """k, v: fp16 [batch, n_kv_heads, capacity, D]; q fp16 [batch, n_q, n_q_heads, D]."""
    batch, n_kv_heads, capacity, D = k.shape
    _, n_q, n_q_heads, _ = q.shape
    _check(load().ckv_attn_decode_f16(_ptr(k), _ptr(v), D, n_kv_heads, batch, capacity, _ptr(seq_len),
                                      max_seq_len, _ptr(q), n_q, n_q_heads, scale, n_split, _ptr(out),
                                      _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)))


def lse_merge(o_parts, lse_parts, out, lse, stream=None):
    """Merge partials: each o part float32 [n_rows, d], each lse part float32 [n_rows]."""
    n = len(o_parts)
    optrs = (_vp * n)(*[_ptr(o) for o in o_parts])
    lptrs = (_vp * n)(*[_ptr(x) for x in lse_parts])
    n_rows = lse_parts[0].numel()
    d = o_parts[0].numel() // max(n_rows, 1)
    _check(load().ckv_lse_merge(n, optrs, lptrs, n_rows, d, _ptr(out), _ptr(lse), _stream(stream)))


def attn_prefill_workspace(cache: PackedCache, n_new: int, n_q_heads: int) -> int:
    return int(load().ckv_attn_prefill_workspace(cache.ref(), n_new, n_q_heads))


def attn_prefill(cache: PackedCache, n_cached: int, q, k_new, v_new, scale: float, out, lse, workspace,
                 stream=None):
    """q: bf16 [batch, n_new, n_q_heads, D]; k_new, v_new fp16 [batch, n_new, n_kv_heads, D]."""
    _, n_new, n_q_heads, _ = q.shape
    _check(load().ckv_attn_prefill(cache.ref(), n_cached, _ptr(q), n_new, n_q_heads, _ptr(k_new),
                                   _ptr(v_new), scale, _ptr(out), _ptr(lse), _ptr(workspace),
                                   workspace.numel(), _stream(stream)))


def read_device_flag(workspace, stream=None) -> int:
    flag = ctypes.c_int32(0)
    status = load().ckv_read_device_flag(_ptr(workspace), ctypes.byref(flag), _stream(stream))
    if status not in (CKV_OK, -5):
        _check(status)
    return int(flag.value)


def read_noalloc_flag(stream=None) -> int:
    """Read and clear the device flag of attn_decode_noalloc's built-in array."""
    flag = ctypes.c_int32(0)
    status = load().ckv_read_noalloc_flag(ctypes.byref(flag), _stream(stream))
    if status not in (CKV_OK, -5):
        _check(status)
    return int(flag.value)


def attn_prefill_prefix(cache: PackedCache, n_prefix: int, q, scale: float, out, lse, workspace, stream=None):
    """q: bf16 [batch, n_q_tokens, n_q_heads, D]; every query sees the packed prefix [0, n_prefix)."""
    _, n_tok, n_q_heads, _ = q.shape
    _check(load().ckv_attn_prefill_prefix(cache.ref(), n_prefix, _ptr(q), n_tok, n_q_heads, scale, _ptr(out),
                                          _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)))


def f16_append(k, v, capacity: int, seq_len, k_new, v_new, stream=None):
    """k, v: fp16 [batch, n_kv_heads, capacity, D]; k_new/v_new: fp16 [batch, n_new, n_kv_heads, D]."""
    batch, n_kv_heads, _, head_dim = k.shape
    _check(load().ckv_f16_append(_ptr(k), _ptr(v), head_dim, n_kv_heads, batch, capacity, _ptr(seq_len),
                                 _ptr(k_new), _ptr(v_new), k_new.shape[1], k_new.stride(1), k_new.stride(0),
                                 _stream(stream)))


def attn_prefill_f16(k, v, seq_len, max_seq_len: int, q, scale: float, out, lse, workspace, n_split: int = 0,
                     stream=None):
    """Causal prefill over fp16 caches [batch, n_kv_heads, capacity, D]; q: bf16 [batch, n_new, n_q_heads, D]."""
    batch, n_kv_heads, capacity, head_dim = k.shape
    _, n_new, n_q_heads, _ = q.shape
    _check(load().ckv_attn_prefill_f16(_ptr(k), _ptr(v), head_dim, n_kv_heads, batch, capacity, _ptr(seq_len),
                                       max_seq_len, _ptr(q), n_new, n_q_heads, scale, n_split, _ptr(out), _ptr(lse),
                                       _ptr(workspace), workspace.numel(), _stream(stream)))


def attn_prefill_shared_workspace(prefix: PackedCache, n_agents: int, tail_capacity: int, n_new: int,
                                  n_q_heads: int) -> int:
    return int(load().ckv_attn_prefill_shared_workspace(prefix.ref(), n_agents, tail_capacity, n_new, n_q_heads))


def attn_prefill_shared(prefix: PackedCache, n_prefix: int, k_tail, v_tail, tail_len, q, k_new, v_new,
                        scale: float, out, lse, workspace, stream=None):
    """Multi-tenant prefill: q bf16 [n_agents, n_new, n_q_heads, D]; tails fp16 [n_agents, Hkv, cap, D]."""
    n_agents, n_new, n_q_heads, _ = q.shape
    _check(load().ckv_attn_prefill_shared(prefix.ref(), n_prefix, _ptr(k_tail), _ptr(v_tail), k_tail.shape[2],
                                          _ptr(tail_len), n_agents, _ptr(q), _ptr(k_new), _ptr(v_new), n_new,
                                          n_q_heads, scale, _ptr(out), _ptr(lse), _ptr(workspace),
                                          workspace.numel(), _stream(stream)))


def selftest_bounded_waits(workspace, stream=None):
    """Run the kernels' two bounded-wait forms on events that never come; afterwards the int32
    words at workspace bytes 0 and 4 read 1 (workspace: >= 256 zero-filled device bytes)."""
    _check(load().ckv_selftest_bounded_waits(_ptr(workspace), workspace.numel(), _stream(stream)))


def calibrate_stream(src, n_tiles: int, record_bytes: int, n_streams: int, n_split: int, rendezvous: bool,
                     workspace, stream=None):
    """Stream the records at `src` (a device tensor) through the decode's staging without computing."""
    _check(load().ckv_calibrate_stream(_ptr(src), n_tiles, record_bytes, n_streams, n_split, int(rendezvous),
                                       _ptr(workspace), workspace.numel(), _stream(stream)))


def set_concurrent_kernels(on: bool) -> None:
    """Declare that other kernels may run on the device concurrently (split merges then never wait)."""
    load().ckv_set_concurrent_kernels(int(bool(on)))
