"""Compressed-KV attention for NVIDIA GB300: q8_0 keys, 3-bit TurboQuant-MSE values,
attention computed in-kernel over the packed cache.

The CUDA library (libckv.so, C ABI in include/ckv.h) does all the work; the
binding marshals torch tensors into it. Importing this package does not load
the library; the first call does, and fails loudly if it was not built.
"""
from ._binding import (CkvError, PackedCache, attn_decode, attn_decode_append, attn_decode_f16,  # noqa: F401
                       attn_decode_f16_merge, attn_decode_f16_merge_workspace, attn_decode_append_host,
                       attn_decode_dca, attn_decode_dca_workspace, attn_decode_fanout, attn_decode_fanout_workspace,
                       attn_decode_noalloc, attn_decode_verify,
                       attn_decode_f16_workspace, attn_decode_workspace, attn_prefill, attn_prefill_f16,
                       attn_prefill_prefix, attn_prefill_shared, attn_prefill_shared_workspace,
                       attn_prefill_workspace, cache_bytes, calibrate_stream, f16_append, fanout_plan, kv_pack, load,
                       lse_merge, read_device_flag, read_noalloc_flag, set_concurrent_kernels, selftest_bounded_waits,
                       version)
