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
  int v_bits;                          // bits per V code: 2, 3 or 4
  int rot;                             // 0: full D-point transform; 1: 128-dim groups, two sign diagonals
  int64_t tok_offset, n_tok;
  const __half* k;
  const __half* v;
  int64_t token_stride, batch_stride;  // in elements
  const int8_t* signs;
  const int8_t* signs2;                // second diagonal (rot = 1)
};
cudaError_t launch_kv_pack(const PackArgs& a, cudaStream_t stream);

// Split-K decode. Rows of one (sequence, kv head) are the G * n_q query vectors
// that read it, ordered (query token, head in group); they are processed in
// groups of 8 ("row groups"). Each CTA writes its partial to a workspace slot
// and the CTAs that finish last merge them (decode_common.cuh, split merge
// tree). Workspace regions (floats, slot = 8 D + 16 floats):
//   part[group][split][slot]   one partial per CTA
//   sub [group][leaf][slot]    one merged partial per leaf of splits
//   counters[group][stride]    u32: rendezvous arrivals and departures, or
//                              the tree's leaf and root counters
// group = (b * n_kv_heads + kv_head) * n_row_groups + row_group.
struct DecodeArgs {
  const uint8_t* cache;      // packed records (compressed decode) or nullptr
  const __half* k16;         // dense fp16 keys (fp16 decode) or nullptr
  const __half* v16;
  const int8_t* signs;       // sign diagonal (compressed decode) or nullptr
  const int8_t* signs2;      // second diagonal of the block-diagonal rotation (rot = 1)
  int rot;                   // 0: full D-point transform; 1: 128-dim groups, two diagonals
  int64_t capacity;
  int head_dim, n_kv_heads, batch;
  int v_bits;                // bits per V code of the compressed cache: 2, 3 or 4
  const int32_t* seq_len;
  int64_t max_seq_len;
  const __half* q;
  int q_bf16;                // fp16 decode only: q holds bf16 values (converted exactly on load)
  int n_q, n_q_heads;
  int causal_q;              // 1: query token qi sees [0, seq_len - n_q + qi + 1) (verify batch)
  int dca_chunk;             // > 0: dual chunk attention regimes as query rows (decode_common.cuh)
  int dca_parts;             // DCA: the inter regime's range is split into this many rows (n_q = 2 + parts)
  float scale_log2;          // logit scale * log2(e)
  int n_split, n_row_groups;
  float* part;
  float* sub;                // merge-tree leaf slots, sub_stride per group
  int sub_stride;            // merge_nl, plus one slot for the prior partial when there is one
  int merge_ls, merge_nl;    // leaf size and leaf count of the merge tree
  // Optional prior partial per output row (fp16 decode only), computed over
  // other keys: normalised rows and lse laid out as out and lse. The split
  // merge combines it with the splits exactly; it enters as one more slot
  // (sub + (group * sub_stride + merge_nl) * slot), written by split 0.
  const float* prior_o;
  const float* prior_lse;
  // DCA with 8 query heads per kv head: the regime pieces are row groups with
  // the same 8 heads, so with dca_fold the split rendezvous spans all row
  // groups of a (sequence, kv head) and merges every (piece, split) slot:
  // the result is the DCA output itself, written to fold_out / fold_lse
  // ([batch][n_q_heads][D], [batch][n_q_heads]) instead of per-piece rows.
  // The launcher keeps it only for a rendezvous launch and reports the
  // choice in *host_folded (host memory).
  int dca_fold;
  float* fold_out;
  float* fold_lse;
  int* host_folded;
  // Fan-out, prefix side (compressed decode): the CTAs write their split slots
  // and leave; another decode merges them.
  int slots_only;
  // Fan-out, tail side (fp16 decode, one query token, 8 query heads per kv
  // head): the split merge of row group (b, kvh) also takes in ext_n slots of
  // a slots_only decode of one sequence whose row group b of kv head kvh holds
  // the same 8 rows: ext_part + ((kvh * ext_nrg + b) * ext_n + s) * slot.
  const float* ext_part;
  int ext_n, ext_nrg;
  // Compressed decode: q, k_new and v_new are written by no kernel (page-locked
  // host buffers), so they are loaded before the wait for the previous grid.
  int early_inputs;
  int rendezvous;            // 1: every CTA resident at once, merge by rendezvous
  int32_t* flag;
  uint32_t* counters;        // ctr_stride words per group, zero between calls
  int ctr_stride;
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

// Largest split count: the merge tree merges at most 32 slots at a time.
constexpr int kMaxSplits = 1024;

// Floats of one slot: [8][D] accumulators, then 8 maxima and 8 row sums.
__host__ __device__ constexpr int64_t merge_slot_floats(int D) { return 8 * (int64_t)D + 16; }

// The tree shape for n_split partials: leaves of ls splits (the last may be
// shorter), nl leaves, ls = ceil(sqrt(n_split)).
struct MergeTree {
  int ls, nl;
};
__host__ __device__ inline MergeTree merge_tree(int n_split) {
  int ls = 1;
  while (ls * ls < n_split) ++ls;
  return MergeTree{ls, (n_split + ls - 1) / ls};
}


cudaError_t launch_attn_decode(const DecodeArgs& a, cudaStream_t stream);       // dispatches on v_bits
cudaError_t launch_attn_decode_tbq2(const DecodeArgs& a, cudaStream_t stream);  // v_bits 2
cudaError_t launch_attn_decode_tbq4(const DecodeArgs& a, cudaStream_t stream);  // v_bits 4
cudaError_t launch_attn_decode_rot2(const DecodeArgs& a, cudaStream_t stream);  // rot 1, v_bits 2
cudaError_t launch_attn_decode_rot3(const DecodeArgs& a, cudaStream_t stream);  // rot 1, v_bits 3
cudaError_t launch_attn_decode_rot4(const DecodeArgs& a, cudaStream_t stream);  // rot 1, v_bits 4
cudaError_t launch_attn_decode_f16(const DecodeArgs& a, cudaStream_t stream);

// New rows into dense fp16 K/V caches [batch][n_kv_heads][capacity][D].
struct F16AppendArgs {
  __half* k;
  __half* v;
  int head_dim, n_kv_heads, batch;
  int64_t capacity;
  const int32_t* seq_len;       // per sequence, counting the new rows
  const __half* k_new;          // [batch][n_new][n_kv_heads][D] with the strides below
  const __half* v_new;
  int n_new;
  int64_t token_stride, batch_stride;  // in elements
};
cudaError_t launch_f16_append(const F16AppendArgs& a, cudaStream_t stream);

struct LseMergeArgs {
  const float* o[16];
  const float* l[16];
  int n_parts;
  int64_t n_rows;
  int d;
  // Row i of part r is o[r] + (i / rows_per_group) * o_group_stride +
  // (i % rows_per_group) * d (lse likewise with l_group_stride and 1); the
  // output row i is out + i * d. One group of n_rows rows: contiguous parts.
  int64_t rows_per_group, o_group_stride, l_group_stride;
  float* out;
  float* lse;
};
cudaError_t launch_lse_merge(const LseMergeArgs& a, cudaStream_t stream);

// Decode with many query rows per kv head (a shared prefix read by many
// agents): the tcgen05 prefill kernel runs every 128-row tile split over the
// key range (each CTA a share of the 64-key steps, writing one partial slot),
// then a merge kernel combines each row's slots. Used by attn_decode when
// rows_decode_applies() (n_split 0: where a fitted cost model prefers it; -1:
// forced); the workspace holds the flag (bytes 0..255) and the slots.
bool rows_decode_applies(int batch, int n_kv_heads, int n_q_heads, int n_q, int n_split, int64_t max_seq_len);
size_t rows_decode_ws_bytes(int head_dim, int n_kv_heads, int batch, int n_q_heads, int n_q, int64_t max_seq_len);
// The mma.sync decode's automatic split count for this call (>= 1; 1 on invalid input).
int decode_auto_split(const void* cache, int64_t max_seq_len, int n_q, int n_q_heads);
// Bytes at the start of the workspace that ckv_attn_decode uses for the device
// flag (bytes 0..3) and its split-merge counters (from byte 64) for this call:
// 256 on the tile path, which keeps no counters.
size_t decode_header_bytes(const void* cache, int64_t max_seq_len, int n_q, int n_q_heads, int n_split);
cudaError_t launch_rows_decode(const void* cache, int64_t key_end, const int32_t* seq_len, const void* q_f16,
                               int n_q, int n_q_heads, float scale, float* out, float* lse, void* ws,
                               cudaStream_t stream);

// Record a failure message for ckv_last_error() on this thread; returns `status`.
int set_last_error(int status, const char* fmt, ...);

}  // namespace ckv
