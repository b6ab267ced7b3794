// attn_decode_tbq2.cu — the compressed decode at 2 bits per V code (the
// TurboQuant tier of 4 Lloyd-Max levels); kernel in attn_decode_kernel.cuh.
#include "attn_decode_kernel.cuh"

namespace ckv {

cudaError_t launch_attn_decode_tbq2(const DecodeArgs& a, cudaStream_t stream) {
  return launch_decode_bits<2>(a, stream);
}

}  // namespace ckv
