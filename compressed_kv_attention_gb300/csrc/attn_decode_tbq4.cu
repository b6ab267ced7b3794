// attn_decode_tbq4.cu — the compressed decode at 4 bits per V code (the
// TurboQuant tier of 16 Lloyd-Max levels); kernel in attn_decode_kernel.cuh.
#include "attn_decode_kernel.cuh"

namespace ckv {

cudaError_t launch_attn_decode_tbq4(const DecodeArgs& a, cudaStream_t stream) {
  return launch_decode_bits<4>(a, stream);
}

}  // namespace ckv
