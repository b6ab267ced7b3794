// prefill_common.cuh — arguments shared by the prefill kernels.
#pragma once

#include <cuda_bf16.h>

#include "ckv_device.cuh"

namespace ckv {

struct PrefillArgs {
  const uint8_t* cache;
  int64_t capacity;
  int n_kv_heads, batch;
  int64_t n_cached;
  int n_new, n_q_heads;
  const __nv_bfloat16* q;  // [batch][n_new][n_q_heads][D]
  float scale_log2;
  float* out;              // [batch][n_new][n_q_heads][D]
  float* lse;              // [batch][n_new][n_q_heads]
  int32_t* flag;
};

}  // namespace ckv
