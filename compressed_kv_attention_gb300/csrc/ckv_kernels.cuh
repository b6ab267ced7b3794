// ckv_kernels.cuh — argument blocks and launchers of the library's kernels.
// Internal to the CUDA library: the public boundary is include/ckv.h.
#pragma once

#include <cuda_runtime.h>

#include "ckv_device.cuh"

namespace ckv {

struct PackArgs {
  uint8_t* cache;
  int64_t capacity;
  int head_dim, n_kv_heads, batch;
  int64_t tok_offset, n_tok;
  const __half* k;
  const __half* v;
  int64_t token_stride, batch_stride;  // in elements
  const int8_t* signs;
};
cudaError_t launch_kv_pack(const PackArgs& a, cudaStream_t stream);

// Split-K decode. Rows of one (sequence, kv head) are the G * n_q query vectors
// that read it, ordered (query token, head in group); they are processed in
// groups of 8 ("row groups"). Each CTA writes one partial to the workspace:
//   part[group][split][8][D]  float32, sum_j p_j V_j in true space, relative to
//                             the CTA's running max (unnormalised)
//   ml  [group][split][8][2]  float32, (running max in log2 units, row sum)
// group = (b * n_kv_heads + kv_head) * n_row_groups + row_group. With a
// cooperative launch the CTAs of a group then merge the splits themselves;
// otherwise launch_decode_merge does it.
struct DecodeArgs {
  const uint8_t* cache;      // packed records (compressed decode) or nullptr
  const __half* k16;         // dense fp16 keys (fp16 decode) or nullptr
  const __half* v16;
  const int8_t* signs;       // sign diagonal (compressed decode) or nullptr
  int64_t capacity;
  int head_dim, n_kv_heads, batch;
  const int32_t* seq_len;
  int64_t max_seq_len;
  const __half* q;
  int n_q, n_q_heads;
  float scale_log2;          // logit scale * log2(e)
  int n_split, n_row_groups;
  float* part;
  float* ml;
  int32_t* flag;
  uint32_t* counters;        // [groups], zero at launch (cooperative merge)
  int merge_in_kernel;       // 1: cooperative launch, CTAs merge their group
  float* out;
  float* lse;
  // Append (compressed decode, one row group): before its tiles are read, the
  // CTA that owns positions [seq_len - n_new, seq_len) of a sequence and kv
  // head quantises those rows of k_new / v_new into the cache.
  int n_new;                 // 0: plain decode
  uint8_t* cache_w;          // the same cache, writable
  const __half* k_new;       // [batch][n_new][n_kv_heads][D] with the strides below
  const __half* v_new;
  int64_t new_token_stride, new_batch_stride;  // in elements
};

struct MergeArgs {
  const float* part;
  const float* ml;
  int head_dim, n_kv_heads, batch, n_q, n_q_heads, n_split, n_row_groups;
  float* out;
  float* lse;
};

// Largest split count the in-kernel merge handles (its shared scratch).
constexpr int kMaxInKernelSplits = 512;

// Launch the decode kernel; `cooperative` requests the in-kernel merge (all
// CTAs co-resident). Returns cudaErrorCooperativeLaunchTooLarge when the grid
// cannot be co-resident, without launching.
cudaError_t launch_attn_decode(DecodeArgs a, bool cooperative, cudaStream_t stream);
cudaError_t launch_attn_decode_f16(DecodeArgs a, bool cooperative, cudaStream_t stream);
cudaError_t launch_decode_merge(const MergeArgs& a, cudaStream_t stream);
// Zero the first `bytes` (a multiple of 4) of a workspace.
cudaError_t launch_ws_reset(void* header, size_t bytes, cudaStream_t stream);

struct LseMergeArgs {
  const float* o[16];
  const float* l[16];
  int n_parts;
  int64_t n_rows;
  int d;
  float* out;
  float* lse;
};
cudaError_t launch_lse_merge(const LseMergeArgs& a, cudaStream_t stream);

// Shared-memory bytes the compressed decode kernel needs for a head dim.
size_t decode_smem_bytes(int head_dim);

// Record a failure message for ckv_last_error() on this thread; returns `status`.
int set_last_error(int status, const char* fmt, ...);

}  // namespace ckv
