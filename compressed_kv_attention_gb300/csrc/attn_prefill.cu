// attn_prefill.cu — chunked causal prefill over the packed cache (tcgen05).
#include <cuda_runtime.h>

#include "../../include/ckv.h"
#include "ckv_kernels.cuh"

extern "C" {

size_t ckv_attn_prefill_workspace(const ckv_cache* cache, int32_t n_new, int32_t n_q_heads) {
  (void)cache; (void)n_new; (void)n_q_heads;
  return 256;
}

ckv_status ckv_attn_prefill(const ckv_cache* cache, int64_t n_cached, const void* q_bf16, int32_t n_new,
                            int32_t n_q_heads, const void* k_new_f16, const void* v_new_f16, float scale,
                            float* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  (void)cache; (void)n_cached; (void)q_bf16; (void)n_new; (void)n_q_heads; (void)k_new_f16;
  (void)v_new_f16; (void)scale; (void)out; (void)lse; (void)workspace; (void)ws_bytes; (void)stream;
  return CKV_ERR_UNSUPPORTED;
}

}  // extern "C"
