// attn_decode_rot4.cu — the compressed decode at 4 bits per V code with the
// block-diagonal rotation (128-dim groups, two sign diagonals, one norm per
// group); kernel in attn_decode_kernel.cuh.
#include "attn_decode_kernel.cuh"

namespace ckv {

cudaError_t launch_attn_decode_rot4(const DecodeArgs& a, cudaStream_t stream) {
  return launch_decode_bits<4, 1>(a, stream);
}

}  // namespace ckv
