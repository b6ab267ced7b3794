// attn_decode.cu — the compressed decode at 3 bits per V code (TBQ3), and the
// dispatch over the V bit widths. The kernel is in attn_decode_kernel.cuh; the
// 2- and 4-bit tiers are instantiated in their own translation units.
#include "attn_decode_kernel.cuh"

namespace ckv {

cudaError_t launch_attn_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.rot) {
    switch (a.v_bits) {
      case 2: return launch_attn_decode_rot2(a, stream);
      case 3: return launch_attn_decode_rot3(a, stream);
      case 4: return launch_attn_decode_rot4(a, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.v_bits) {
    case 2: return launch_attn_decode_tbq2(a, stream);
    case 3: return launch_decode_bits<3>(a, stream);
    case 4: return launch_attn_decode_tbq4(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ckv
