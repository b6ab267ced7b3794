"""Float64 CPU oracle (test infrastructure only; see ckv_oracle.py)."""
from .ckv_oracle import (LLOYD_MAX_3BIT, QK8_0, attention, decode_reference, fwht,  # noqa: F401
                         fwht_orthonormal, kv_head_of, lse_merge, nearest_centroid,
                         prefill_reference, q8_0_dequantize, q8_0_quantize, tbq3_dequantize,
                         tbq3_quantize, to_fp16)
from . import layout  # noqa: F401
