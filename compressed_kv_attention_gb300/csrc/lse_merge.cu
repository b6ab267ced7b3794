// lse_merge.cu — exact merge of normalised (output, lse) partials computed over
// disjoint key sets, e.g. a shared compressed prefix and a private fp16 tail.
// DCA page ("Feature — Gemma-4 A4B Dual Chunk Attention (DCA), training-free 1M
// context"), section "Implementation progress + Section-D simplification":
// M = max_r lse_r, w_r = exp(lse_r - M), O = sum_r w_r O_r / sum_r w_r;
// section "Section C2b": an empty partial has lse = -inf and weighs 0.
#include "ckv_kernels.cuh"

namespace ckv {

// One CTA per row; threads stride over the d columns (float4 where possible).
__global__ void __launch_bounds__(128) lse_merge_kernel(LseMergeArgs a) {
  const int64_t row = blockIdx.x;
  const int64_t grp = row / a.rows_per_group, j = row % a.rows_per_group;
  const int64_t orow = grp * a.o_group_stride + j * a.d, lrow = grp * a.l_group_stride + j;
  float M = -INFINITY;
  for (int r = 0; r < a.n_parts; ++r) M = fmaxf(M, a.l[r][lrow]);
  float w[16];
  float W = 0.0f;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    w[r] = 0.0f;
    if (r < a.n_parts && M != -INFINITY) {
      const float lr = a.l[r][lrow];
      w[r] = (lr == -INFINITY) ? 0.0f : expf(lr - M);
      W += w[r];
    }
  }
  const float inv = (W > 0.0f) ? 1.0f / W : 0.0f;
  for (int c = threadIdx.x; c < a.d; c += blockDim.x) {
    float s = 0.0f;
#pragma unroll
    for (int r = 0; r < 16; ++r)
      if (r < a.n_parts && w[r] != 0.0f) s = fmaf(w[r], a.o[r][orow + c], s);
    a.out[row * a.d + c] = s * inv;
  }
  __syncthreads();  // every read of the lse parts is done before lse may be overwritten
  if (threadIdx.x == 0) a.lse[row] = (W > 0.0f) ? M + logf(W) : -INFINITY;
}

cudaError_t launch_lse_merge(const LseMergeArgs& a, cudaStream_t stream) {
  if (a.n_rows == 0) return cudaSuccess;
  lse_merge_kernel<<<static_cast<unsigned>(a.n_rows), 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ckv
