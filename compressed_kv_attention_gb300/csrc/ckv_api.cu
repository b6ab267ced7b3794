// ckv_api.cu — the extern "C" entry points declared in include/ckv.h: argument
// checks, workspace sizing and kernel launches on the caller's stream.
#include <cuda_runtime.h>

#include <atomic>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/ckv.h"
#include "ckv_kernels.cuh"

namespace {

thread_local char g_err[512] = "";

ckv_status fail(ckv_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

ckv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(CKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_dim(int d) { return d == 64 || d == 128 || d == 256 || d == 512; }

// Workspace header: the device flag at byte 0, one split-merge counter per row
// group from byte 64, rounded up to 256 bytes; both are cleared by every call.
// Decode workspace: the device flag (bytes 0..3), the merge-tree counters from
// byte 64, then the partial slots and the leaf slots (decode_common.cuh).
// Counter words per group: two for the rendezvous merge, nl + 1 for the tree.
int ctr_stride(int n_split) {
  const int t = ckv::merge_tree(n_split).nl + 1;
  return t > 2 ? t : 2;
}
size_t ws_header_bytes(int64_t groups, int n_split) {
  return (64 + 4 * static_cast<size_t>(groups) * ctr_stride(n_split) + 255) / 256 * 256;
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

int cache_v_bits(const ckv_cache* c) { return c->v_bits == 0 ? 3 : c->v_bits; }

ckv_status check_cache(const ckv_cache* c) {
  if (!c) return fail(CKV_ERR_INVALID_ARG, "cache is null");
  if (!supported_dim(c->head_dim))
    return fail(CKV_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256,512}", c->head_dim);
  if (c->n_kv_heads <= 0 || c->batch <= 0)
    return fail(CKV_ERR_INVALID_ARG, "n_kv_heads and batch must be positive");
  if (c->v_bits != 0 && (c->v_bits < 2 || c->v_bits > 4))
    return fail(CKV_ERR_INVALID_ARG, "v_bits must be 2, 3 or 4 (or 0 for 3), got %d", c->v_bits);
  if (c->v_signs2 && c->head_dim < ckv::kRotGroup)
    return fail(CKV_ERR_UNSUPPORTED, "the block-diagonal rotation needs head_dim >= 128 (got %d)", c->head_dim);
  if (c->capacity <= 0 || c->capacity % 16)
    return fail(CKV_ERR_INVALID_ARG, "capacity must be a positive multiple of 16");
  if (!c->data || !aligned(c->data, 16)) return fail(CKV_ERR_INVALID_ARG, "cache data null or not 16-byte aligned");
  if (!c->v_signs) return fail(CKV_ERR_INVALID_ARG, "v_signs is null");
  return CKV_OK;
}

// Split count: one CTA per SM in a single wave (measured best: a CTA streams
// its splits' tiles through the whole kernel); no more splits than tiles.
int auto_split(int64_t units, int64_t max_seq_len, int tiles_per_cta_iter) {
  const int64_t tiles = (max_seq_len + 15) / 16;
  if (tiles == 0) return 1;
  // A sequence that one CTA covers in two iterations runs as one split: its
  // rows then go straight to the output, with no merge (a 256-token decode at
  // head dim 128: 6.96 us in one split against 8.74 in two).
  if (tiles <= 2 * tiles_per_cta_iter) return 1;
  const int sms = num_sms();
  int64_t s = sms / units;
  const int64_t by_tiles = (tiles + tiles_per_cta_iter - 1) / tiles_per_cta_iter;
  if (s > by_tiles) s = by_tiles;
  if (s < 1) s = 1;
  if (s > ckv::kMaxSplits) s = ckv::kMaxSplits;
  return static_cast<int>(s);
}

// prior: one more slot per group for a prior partial (after the leaf slots).
size_t decode_ws_bytes(int D, int64_t groups, int n_split, int prior = 0) {
  const ckv::MergeTree tr = ckv::merge_tree(n_split);
  return ws_header_bytes(groups, n_split) +
         static_cast<size_t>(groups) * (n_split + tr.nl + prior) * ckv::merge_slot_floats(D) * sizeof(float);
}

struct DecodePlan {
  int n_row_groups, n_split;
  int64_t groups;
  size_t ws;
};

ckv_status plan_decode(int D, int n_kv_heads, int batch, int64_t max_seq_len, int n_q, int n_q_heads,
                       int n_split, DecodePlan* p, int prior = 0) {
  if (n_q <= 0 || n_q_heads <= 0) return fail(CKV_ERR_INVALID_ARG, "n_q and n_q_heads must be positive");
  if (n_q_heads % n_kv_heads)
    return fail(CKV_ERR_UNSUPPORTED, "n_q_heads %d not a multiple of n_kv_heads %d", n_q_heads, n_kv_heads);
  if (max_seq_len < 0) return fail(CKV_ERR_INVALID_ARG, "max_seq_len negative");
  if (n_split < 0 || n_split > ckv::kMaxSplits) return fail(CKV_ERR_INVALID_ARG, "n_split out of range");
  const int64_t rows = static_cast<int64_t>(n_q_heads / n_kv_heads) * n_q;
  const int64_t nrg = (rows + 7) / 8;
  if (nrg > 65535) return fail(CKV_ERR_UNSUPPORTED, "too many query rows per kv head");
  p->n_row_groups = static_cast<int>(nrg);
  p->groups = static_cast<int64_t>(batch) * n_kv_heads * nrg;
  const int per_iter = (D == 512) ? 4 : 8;
  p->n_split = n_split ? n_split : auto_split(p->groups, max_seq_len, per_iter);
  p->ws = decode_ws_bytes(D, p->groups, p->n_split, prior);
  return CKV_OK;
}

ckv_status check_ws(void* ws, size_t have, size_t need) {
  if (!ws || !aligned(ws, 256)) return fail(CKV_ERR_WORKSPACE, "workspace null or not 256-byte aligned");
  if (have < need) return fail(CKV_ERR_WORKSPACE, "workspace %zu bytes, need %zu", have, need);
  return CKV_OK;
}

}  // namespace

namespace ckv {
static std::atomic<int> g_concurrent{0};
bool concurrent_kernels() { return g_concurrent.load(std::memory_order_relaxed) != 0; }

int set_last_error(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return status;
}
}  // namespace ckv

extern "C" {

int32_t ckv_version(void) { return 104; }

void ckv_set_concurrent_kernels(int32_t on) { ckv::g_concurrent.store(on ? 1 : 0, std::memory_order_relaxed); }

const char* ckv_last_error(void) { return g_err; }

size_t ckv_cache_bytes_v(int32_t head_dim, int32_t n_kv_heads, int32_t batch, int64_t capacity,
                         int32_t v_bits, int32_t rot_group) {
  if (!supported_dim(head_dim) || n_kv_heads <= 0 || batch <= 0 || capacity <= 0 || capacity % 16 ||
      v_bits < 2 || v_bits > 4 || (rot_group != 0 && rot_group != ckv::kRotGroup) ||
      (rot_group && head_dim < ckv::kRotGroup))
    return 0;
  const int ng = rot_group ? head_dim / rot_group : 1;
  return static_cast<size_t>(batch) * n_kv_heads * (capacity / 16) * ckv::record_bytes(head_dim, v_bits, ng);
}

size_t ckv_cache_bytes(int32_t head_dim, int32_t n_kv_heads, int32_t batch, int64_t capacity) {
  return ckv_cache_bytes_v(head_dim, n_kv_heads, batch, capacity, 3, 0);
}

ckv_status ckv_kv_pack(const ckv_cache* cache, int64_t tok_offset, int64_t n_tok, const void* k_f16,
                       const void* v_f16, int64_t token_stride, int64_t batch_stride, void* stream) {
  ckv_status s = check_cache(cache);
  if (s != CKV_OK) return s;
  if (n_tok < 0 || tok_offset < 0 || tok_offset + n_tok > cache->capacity)
    return fail(CKV_ERR_INVALID_ARG, "token range [%lld, %lld) outside [0, %lld)", (long long)tok_offset,
                (long long)(tok_offset + n_tok), (long long)cache->capacity);
  if (n_tok == 0) return CKV_OK;
  if (!k_f16 || !v_f16 || !aligned(k_f16, 16) || !aligned(v_f16, 16))
    return fail(CKV_ERR_INVALID_ARG, "k/v null or not 16-byte aligned");
  const int64_t row = static_cast<int64_t>(cache->n_kv_heads) * cache->head_dim;
  if (token_stride < row || token_stride % 8 || batch_stride < 0 || batch_stride % 8 ||
      (cache->batch > 1 && batch_stride < token_stride * n_tok))
    return fail(CKV_ERR_INVALID_ARG, "bad strides (token %lld, batch %lld)", (long long)token_stride,
                (long long)batch_stride);
  const int64_t tiles = (tok_offset + n_tok - 1) / 16 - tok_offset / 16 + 1;
  if (tiles > 0x7fffffffLL) return fail(CKV_ERR_UNSUPPORTED, "too many tiles in one pack");
  ckv::PackArgs a{};
  a.cache = static_cast<uint8_t*>(cache->data);
  a.capacity = cache->capacity;
  a.head_dim = cache->head_dim;
  a.n_kv_heads = cache->n_kv_heads;
  a.batch = cache->batch;
  a.v_bits = cache_v_bits(cache);
  a.rot = cache->v_signs2 ? 1 : 0;
  a.signs2 = cache->v_signs2;
  a.tok_offset = tok_offset;
  a.n_tok = n_tok;
  a.k = static_cast<const __half*>(k_f16);
  a.v = static_cast<const __half*>(v_f16);
  a.token_stride = token_stride;
  a.batch_stride = batch_stride;
  a.signs = cache->v_signs;
  cudaError_t e = ckv::launch_kv_pack(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_pack launch");
  return CKV_OK;
}

// Workspace of the mma.sync decode family (decode, verify, DCA, append).
static size_t mma_decode_ws(const ckv_cache* cache, int64_t max_seq_len, int32_t n_q, int32_t n_q_heads,
                            int32_t n_split) {
  if (check_cache(cache) != CKV_OK) return 0;
  DecodePlan p;
  if (plan_decode(cache->head_dim, cache->n_kv_heads, cache->batch, max_seq_len, n_q, n_q_heads, n_split,
                  &p) != CKV_OK)
    return 0;
  return p.ws;
}

}  // extern "C"

namespace ckv {
int decode_auto_split(const void* cache_v, int64_t max_seq_len, int n_q, int n_q_heads) {
  const ckv_cache* cache = static_cast<const ckv_cache*>(cache_v);
  DecodePlan p;
  if (check_cache(cache) != CKV_OK ||
      plan_decode(cache->head_dim, cache->n_kv_heads, cache->batch, max_seq_len, n_q, n_q_heads, 0, &p) != CKV_OK)
    return 1;
  return p.n_split;
}

size_t decode_header_bytes(const void* cache_v, int64_t max_seq_len, int n_q, int n_q_heads, int n_split) {
  const ckv_cache* cache = static_cast<const ckv_cache*>(cache_v);
  if (check_cache(cache) != CKV_OK) return 256;
  if (rows_decode_applies(cache->batch, cache->n_kv_heads, n_q_heads, n_q, n_split, max_seq_len)) return 256;
  DecodePlan p;
  if (plan_decode(cache->head_dim, cache->n_kv_heads, cache->batch, max_seq_len, n_q, n_q_heads, n_split, &p) !=
      CKV_OK)
    return 256;
  return ws_header_bytes(p.groups, p.n_split);
}
}  // namespace ckv

extern "C" {

// Key range the many-row decode splits: seq_len never exceeds this.
static int64_t rows_key_end(const ckv_cache* cache, int64_t max_seq_len) {
  return max_seq_len < cache->capacity ? max_seq_len : cache->capacity;
}

size_t ckv_attn_decode_workspace(const ckv_cache* cache, int64_t max_seq_len, int32_t n_q,
                                 int32_t n_q_heads, int32_t n_split) {
  if (check_cache(cache) != CKV_OK) return 0;
  const bool rows = ckv::rows_decode_applies(cache->batch, cache->n_kv_heads, n_q_heads, n_q, n_split, max_seq_len);
  if (n_split == -1) {
    if (!rows || n_q_heads <= 0 || n_q_heads % cache->n_kv_heads) return 0;
    return ckv::rows_decode_ws_bytes(cache->head_dim, cache->n_kv_heads, cache->batch, n_q_heads, n_q,
                                     rows_key_end(cache, max_seq_len));
  }
  const size_t ws = mma_decode_ws(cache, max_seq_len, n_q, n_q_heads, n_split);
  if (ws == 0 || !rows) return ws;
  const size_t rw = ckv::rows_decode_ws_bytes(cache->head_dim, cache->n_kv_heads, cache->batch, n_q_heads, n_q,
                                              rows_key_end(cache, max_seq_len));
  return rw > ws ? rw : ws;
}

// New rows appended by the decode kernel itself (ckv_attn_decode_append).
struct AppendRows {
  const void* k;
  const void* v;
  int n_new;
  int64_t token_stride, batch_stride;
};

// Launch options beyond the common arguments. The fan-out's link between its
// two decodes (see ckv_attn_decode_fanout): the prefix decode writes slots
// only; the tail decode merges ext_n of them per row group and raises its
// errors in the prefix decode's flag word. early_inputs: Q and the new rows
// are page-locked host buffers, read before the wait for the previous grid.
struct DecodeExtras {
  int slots_only;
  const float* ext_part;
  int ext_n, ext_nrg;
  int32_t* flag;
  int early_inputs;
};

static ckv_status run_decode(bool compressed, const ckv_cache* cache, const void* k16, const void* v16,
                             int D, int Hkv, int B, int64_t capacity, const int32_t* seq_len,
                             int64_t max_seq_len, const void* q, int n_q, int n_q_heads, float scale,
                             int n_split, float* out, float* lse, void* ws, size_t ws_bytes,
                             void* stream, const AppendRows* app = nullptr, int causal_q = 0,
                             int dca_chunk = 0, int q_bf16 = 0, int dca_parts = 0,
                             const float* prior_o = nullptr, const float* prior_lse = nullptr,
                             float* fold_out = nullptr, float* fold_lse = nullptr, int* host_folded = nullptr,
                             const DecodeExtras* link = nullptr) {
  DecodePlan p;
  ckv_status s = plan_decode(D, Hkv, B, max_seq_len, n_q, n_q_heads, n_split, &p, prior_o ? 1 : 0);
  if (s != CKV_OK) return s;
  if (app) {
    if (p.n_row_groups != 1)
      return fail(CKV_ERR_UNSUPPORTED, "append needs at most 8 query rows per kv head (n_q * group = %d)",
                  (n_q_heads / Hkv) * n_q);
    if (app->n_new < 1 || app->n_new > 16) return fail(CKV_ERR_INVALID_ARG, "n_new must be in [1, 16]");
    if (app->n_new > max_seq_len) return fail(CKV_ERR_INVALID_ARG, "n_new exceeds max_seq_len");
    if (!app->k || !app->v || !aligned(app->k, 16) || !aligned(app->v, 16))
      return fail(CKV_ERR_INVALID_ARG, "k_new/v_new null or not 16-byte aligned");
    const int64_t row = static_cast<int64_t>(Hkv) * D;
    if (app->token_stride < row || app->token_stride % 8 || app->batch_stride < 0 || app->batch_stride % 8 ||
        (B > 1 && app->batch_stride < app->token_stride * app->n_new))
      return fail(CKV_ERR_INVALID_ARG, "bad strides (token %lld, batch %lld)", (long long)app->token_stride,
                  (long long)app->batch_stride);
  }
  if (!seq_len || !q || !out || !lse) return fail(CKV_ERR_INVALID_ARG, "null seq_len/q/out/lse");
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(seq_len, 4))
    return fail(CKV_ERR_INVALID_ARG, "q/out must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(CKV_ERR_INVALID_ARG, "scale not finite");
  s = check_ws(ws, ws_bytes, p.ws);
  if (s != CKV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t header = ws_header_bytes(p.groups, p.n_split);
  const ckv::MergeTree tr = ckv::merge_tree(p.n_split);
  uint8_t* base = static_cast<uint8_t*>(ws);
  ckv::DecodeArgs a{};
  a.cache = compressed ? static_cast<const uint8_t*>(cache->data) : nullptr;
  a.k16 = static_cast<const __half*>(k16);
  a.v16 = static_cast<const __half*>(v16);
  a.signs = compressed ? cache->v_signs : nullptr;
  a.capacity = capacity;
  a.head_dim = D;
  a.n_kv_heads = Hkv;
  a.batch = B;
  a.v_bits = compressed ? cache_v_bits(cache) : 0;
  a.rot = (compressed && cache->v_signs2) ? 1 : 0;
  a.signs2 = compressed ? cache->v_signs2 : nullptr;
  a.seq_len = seq_len;
  a.max_seq_len = max_seq_len;
  a.q = static_cast<const __half*>(q);
  a.q_bf16 = q_bf16;
  a.n_q = n_q;
  a.n_q_heads = n_q_heads;
  a.causal_q = causal_q;
  a.dca_chunk = dca_chunk;
  a.dca_parts = dca_parts;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.n_split = p.n_split;
  a.n_row_groups = p.n_row_groups;
  a.part = reinterpret_cast<float*>(base + header);
  a.sub = a.part + static_cast<size_t>(p.groups) * p.n_split * ckv::merge_slot_floats(D);
  a.merge_ls = tr.ls;
  a.merge_nl = tr.nl;
  a.sub_stride = tr.nl + (prior_o ? 1 : 0);
  a.prior_o = prior_o;
  a.prior_lse = prior_lse;
  a.dca_fold = fold_out ? 1 : 0;
  a.fold_out = fold_out;
  a.fold_lse = fold_lse;
  a.host_folded = host_folded;
  a.ctr_stride = ctr_stride(p.n_split);
  a.flag = reinterpret_cast<int32_t*>(base);
  if (link) {
    a.slots_only = link->slots_only;
    a.ext_part = link->ext_part;
    a.ext_n = link->ext_n;
    a.ext_nrg = link->ext_nrg;
    if (link->flag) a.flag = link->flag;
    a.early_inputs = link->early_inputs;
  }
  a.counters = reinterpret_cast<uint32_t*>(base + 64);
  a.out = out;
  a.lse = lse;
  if (app) {
    a.n_new = app->n_new;
    a.cache_w = static_cast<uint8_t*>(cache->data);
    a.k_new = static_cast<const __half*>(app->k);
    a.v_new = static_cast<const __half*>(app->v);
    a.new_token_stride = app->token_stride;
    a.new_batch_stride = app->batch_stride;
  }
  const cudaError_t e = compressed ? ckv::launch_attn_decode(a, st) : ckv::launch_attn_decode_f16(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return CKV_OK;
}

ckv_status ckv_attn_decode(const ckv_cache* cache, const int32_t* seq_len, int64_t max_seq_len,
                           const void* q_f16, int32_t n_q, int32_t n_q_heads, float scale, int32_t n_split,
                           float* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  ckv_status s = check_cache(cache);
  if (s != CKV_OK) return s;
  if (n_split == -1 &&
      !ckv::rows_decode_applies(cache->batch, cache->n_kv_heads, n_q_heads, n_q, n_split, max_seq_len))
    return fail(CKV_ERR_UNSUPPORTED, "n_split -1 (tile path) needs n_q_heads / n_kv_heads dividing 128 and "
                                     "max_seq_len > 0");
  if (ckv::rows_decode_applies(cache->batch, cache->n_kv_heads, n_q_heads, n_q, n_split, max_seq_len)) {
    // Many query rows per kv head: the tcgen05 tile path (same checks as below).
    DecodePlan p;
    s = plan_decode(cache->head_dim, cache->n_kv_heads, cache->batch, max_seq_len, n_q, n_q_heads, 0, &p);
    if (s != CKV_OK) return s;
    if (!seq_len || !q_f16 || !out || !lse) return fail(CKV_ERR_INVALID_ARG, "null seq_len/q/out/lse");
    if (!aligned(q_f16, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(seq_len, 4))
      return fail(CKV_ERR_INVALID_ARG, "q/out must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail(CKV_ERR_INVALID_ARG, "scale not finite");
    s = check_ws(workspace, ws_bytes, ckv_attn_decode_workspace(cache, max_seq_len, n_q, n_q_heads, n_split));
    if (s != CKV_OK) return s;
    const cudaError_t e = ckv::launch_rows_decode(cache, rows_key_end(cache, max_seq_len), seq_len, q_f16, n_q,
                                                  n_q_heads, scale, out, lse, workspace,
                                                  static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return CKV_OK;
  }
  return run_decode(true, cache, nullptr, nullptr, cache->head_dim, cache->n_kv_heads, cache->batch,
                    cache->capacity, seq_len, max_seq_len, q_f16, n_q, n_q_heads, scale, n_split, out, lse,
                    workspace, ws_bytes, stream);
}

// DCA: the inter regime's range, up to max_seq_len - 2 chunk keys, is cut into
// pieces of about one chunk (1 to 14: the merge takes 16 parts), so that its
// rows' CTAs carry about as many keys as the intra and successive regimes'.
static int dca_parts_for(int64_t max_seq_len, int chunk) {
  const int64_t inter = max_seq_len > 2LL * chunk ? max_seq_len - 2LL * chunk : 0;
  int64_t m = (inter + chunk / 2) / chunk;
  if (m < 1) m = 1;
  if (m > 14) m = 14;
  return static_cast<int>(m);
}

// DCA workspace: the decode's (2 + parts query rows per query head, one row
// group each), then the rows' partial outputs [batch][2 + parts][n_q_heads][D]
// and lse values.
static size_t dca_ws_parts(const ckv_cache* cache, int n_rows_per_head, int n_q_heads, size_t* o_off,
                           size_t* l_off) {
  const size_t rows = static_cast<size_t>(cache->batch) * n_rows_per_head * n_q_heads;
  *o_off = 0;
  *l_off = (rows * cache->head_dim * sizeof(float) + 255) / 256 * 256;
  return *l_off + (rows * sizeof(float) + 255) / 256 * 256;
}

static size_t dca_ws_for(const ckv_cache* cache, int64_t max_seq_len, int n_q_heads, int n_split, int parts,
                         size_t* dec_out) {
  const size_t dec = mma_decode_ws(cache, max_seq_len, 2 + parts, n_q_heads, n_split);
  if (dec_out) *dec_out = dec;
  if (dec == 0) return 0;
  size_t o_off, l_off;
  return (dec + 255) / 256 * 256 + dca_ws_parts(cache, 2 + parts, n_q_heads, &o_off, &l_off);
}

size_t ckv_attn_decode_dca_workspace(const ckv_cache* cache, int64_t max_seq_len, int32_t n_q_heads,
                                     int32_t n_split) {
  // Enough for any chunk: the largest need over the piece counts a call can choose.
  size_t need = 0;
  for (int parts = 1; parts <= 14; ++parts) {
    const size_t w = dca_ws_for(cache, max_seq_len, n_q_heads, n_split, parts, nullptr);
    if (w == 0) return 0;
    need = w > need ? w : need;
  }
  return need;
}

ckv_status ckv_attn_decode_dca(const ckv_cache* cache, const int32_t* seq_len, int64_t max_seq_len,
                               int32_t chunk, const void* q_f16, int32_t n_q_heads, float scale, int32_t n_split,
                               float* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  ckv_status s = check_cache(cache);
  if (s != CKV_OK) return s;
  if (chunk < 1) return fail(CKV_ERR_INVALID_ARG, "chunk must be positive (got %d)", chunk);
  if (!out || !lse) return fail(CKV_ERR_INVALID_ARG, "null out/lse");
  const int parts = dca_parts_for(max_seq_len, chunk);
  const int n_rows = 2 + parts;
  size_t dec = 0;
  const size_t need = dca_ws_for(cache, max_seq_len, n_q_heads, n_split, parts, &dec);
  if (dec == 0) {
    // Invalid geometry: the decode's own checks give the status and message.
    return run_decode(true, cache, nullptr, nullptr, cache->head_dim, cache->n_kv_heads, cache->batch,
                      cache->capacity, seq_len, max_seq_len, q_f16, n_rows, n_q_heads, scale, n_split, out, lse,
                      workspace, ws_bytes, stream, nullptr, 0, chunk, 0, parts);
  }
  s = check_ws(workspace, ws_bytes, need);
  if (s != CKV_OK) return s;
  size_t o_off, l_off;
  dca_ws_parts(cache, n_rows, n_q_heads, &o_off, &l_off);
  uint8_t* pbase = static_cast<uint8_t*>(workspace) + (dec + 255) / 256 * 256;
  float* po = reinterpret_cast<float*>(pbase + o_off);
  float* pl = reinterpret_cast<float*>(pbase + l_off);
  // The regimes (the inter one in pieces) as the query tokens of one decode.
  // With 8 query heads per kv head every row group is one piece of the same
  // 8 heads, and a rendezvous launch merges the pieces inside the decode
  // (folded: the output lands in out / lse directly); otherwise the pieces'
  // rows go to the workspace and lse_merge combines them.
  const bool fold = n_q_heads == 8 * cache->n_kv_heads;
  int folded = 0;
  s = run_decode(true, cache, nullptr, nullptr, cache->head_dim, cache->n_kv_heads, cache->batch,
                 cache->capacity, seq_len, max_seq_len, q_f16, n_rows, n_q_heads, scale, n_split, po, pl, workspace,
                 dec, stream, nullptr, 0, chunk, 0, parts, nullptr, nullptr, fold ? out : nullptr,
                 fold ? lse : nullptr, &folded);
  if (s != CKV_OK) return s;
  if (folded) return CKV_OK;
  const int D = cache->head_dim;
  ckv::LseMergeArgs m{};
  for (int r = 0; r < n_rows; ++r) {
    m.o[r] = po + static_cast<size_t>(r) * n_q_heads * D;
    m.l[r] = pl + static_cast<size_t>(r) * n_q_heads;
  }
  m.n_parts = n_rows;
  m.n_rows = static_cast<int64_t>(cache->batch) * n_q_heads;
  m.d = D;
  m.rows_per_group = n_q_heads;
  m.o_group_stride = static_cast<int64_t>(n_rows) * n_q_heads * D;
  m.l_group_stride = static_cast<int64_t>(n_rows) * n_q_heads;
  m.out = out;
  m.lse = lse;
  const cudaError_t e = ckv::launch_lse_merge(m, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lse_merge launch");
  return CKV_OK;
}

ckv_status ckv_attn_decode_verify(const ckv_cache* cache, const int32_t* seq_len, int64_t max_seq_len,
                                  const void* q_f16, int32_t n_q, int32_t n_q_heads, float scale, int32_t n_split,
                                  float* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  ckv_status s = check_cache(cache);
  if (s != CKV_OK) return s;
  return run_decode(true, cache, nullptr, nullptr, cache->head_dim, cache->n_kv_heads, cache->batch,
                    cache->capacity, seq_len, max_seq_len, q_f16, n_q, n_q_heads, scale, n_split, out, lse,
                    workspace, ws_bytes, stream, nullptr, 1);
}

ckv_status ckv_attn_decode_append(const ckv_cache* cache, const int32_t* seq_len, int64_t max_seq_len,
                                  const void* k_new_f16, const void* v_new_f16, int32_t n_new,
                                  int64_t token_stride, int64_t batch_stride, const void* q_f16, int32_t n_q,
                                  int32_t n_q_heads, float scale, int32_t n_split, float* out, float* lse,
                                  void* workspace, size_t ws_bytes, void* stream) {
  ckv_status s = check_cache(cache);
  if (s != CKV_OK) return s;
  const AppendRows app{k_new_f16, v_new_f16, n_new, token_stride, batch_stride};
  return run_decode(true, cache, nullptr, nullptr, cache->head_dim, cache->n_kv_heads, cache->batch,
                    cache->capacity, seq_len, max_seq_len, q_f16, n_q, n_q_heads, scale, n_split, out, lse,
                    workspace, ws_bytes, stream, &app);
}

// The device address of a page-locked host buffer (mapped into the device's
// address space), or nullptr for memory the device cannot reach this way.
static void* mapped_host(const void* p) {
  if (!p) return nullptr;
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // clear the error of an unregistered pointer
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

ckv_status ckv_attn_decode_append_host(const ckv_cache* cache, const int32_t* seq_len, int64_t max_seq_len,
                                       const void* k_new_host, const void* v_new_host, int32_t n_new,
                                       const void* q_host, int32_t n_q, int32_t n_q_heads, float scale,
                                       int32_t n_split, float* out_host, float* lse_host, void* workspace,
                                       size_t ws_bytes, void* stream) {
  ckv_status s = check_cache(cache);
  if (s != CKV_OK) return s;
  void* k = mapped_host(k_new_host);
  void* v = mapped_host(v_new_host);
  void* q = mapped_host(q_host);
  void* o = mapped_host(out_host);
  void* l = mapped_host(lse_host);
  if (!k || !v || !q || !o || !l)
    return fail(CKV_ERR_INVALID_ARG, "host buffers must be page-locked and mapped (cudaHostAlloc / pinned)");
  const int64_t tok = static_cast<int64_t>(cache->n_kv_heads) * cache->head_dim;
  const AppendRows app{k, v, n_new, tok, tok * n_new};
  const DecodeExtras ex{0, nullptr, 0, 0, nullptr, 1};
  return run_decode(true, cache, nullptr, nullptr, cache->head_dim, cache->n_kv_heads, cache->batch,
                    cache->capacity, seq_len, max_seq_len, q, n_q, n_q_heads, scale, n_split, static_cast<float*>(o),
                    static_cast<float*>(l), workspace, ws_bytes, stream, &app, 0, 0, 0, 0, nullptr, nullptr, nullptr,
                    nullptr, nullptr, &ex);
}

size_t ckv_attn_decode_f16_workspace(int32_t head_dim, int32_t n_kv_heads, int32_t batch,
                                     int64_t max_seq_len, int32_t n_q, int32_t n_q_heads, int32_t n_split) {
  if (!supported_dim(head_dim) || n_kv_heads <= 0 || batch <= 0) return 0;
  DecodePlan p;
  if (plan_decode(head_dim, n_kv_heads, batch, max_seq_len, n_q, n_q_heads, n_split, &p) != CKV_OK) return 0;
  return p.ws;
}

ckv_status ckv_attn_decode_f16(const void* k_f16, const void* v_f16, int32_t head_dim, int32_t n_kv_heads,
                               int32_t batch, int64_t capacity, const int32_t* seq_len, int64_t max_seq_len,
                               const void* q_f16, int32_t n_q, int32_t n_q_heads, float scale,
                               int32_t n_split, float* out, float* lse, void* workspace, size_t ws_bytes,
                               void* stream) {
  if (!supported_dim(head_dim))
    return fail(CKV_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256,512}", head_dim);
  if (n_kv_heads <= 0 || batch <= 0) return fail(CKV_ERR_INVALID_ARG, "n_kv_heads and batch must be positive");
  if (capacity <= 0 || capacity % 16) return fail(CKV_ERR_INVALID_ARG, "capacity must be a positive multiple of 16");
  if (!k_f16 || !v_f16 || !aligned(k_f16, 16) || !aligned(v_f16, 16))
    return fail(CKV_ERR_INVALID_ARG, "k/v null or not 16-byte aligned");
  return run_decode(false, nullptr, k_f16, v_f16, head_dim, n_kv_heads, batch, capacity, seq_len, max_seq_len,
                    q_f16, n_q, n_q_heads, scale, n_split, out, lse, workspace, ws_bytes, stream);
}

size_t ckv_attn_decode_f16_merge_workspace(int32_t head_dim, int32_t n_kv_heads, int32_t batch,
                                           int64_t max_seq_len, int32_t n_q, int32_t n_q_heads, int32_t n_split) {
  if (!supported_dim(head_dim) || n_kv_heads <= 0 || batch <= 0) return 0;
  DecodePlan p;
  if (plan_decode(head_dim, n_kv_heads, batch, max_seq_len, n_q, n_q_heads, n_split, &p, 1) != CKV_OK) return 0;
  return p.ws;
}

ckv_status ckv_attn_decode_f16_merge(const void* k_f16, const void* v_f16, int32_t head_dim, int32_t n_kv_heads,
                                     int32_t batch, int64_t capacity, const int32_t* seq_len, int64_t max_seq_len,
                                     const void* q_f16, int32_t n_q, int32_t n_q_heads, float scale, int32_t n_split,
                                     const float* prior_o, const float* prior_lse, float* out, float* lse,
                                     void* workspace, size_t ws_bytes, void* stream) {
  if (!supported_dim(head_dim))
    return fail(CKV_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256,512}", head_dim);
  if (n_kv_heads <= 0 || batch <= 0) return fail(CKV_ERR_INVALID_ARG, "n_kv_heads and batch must be positive");
  if (capacity <= 0 || capacity % 16) return fail(CKV_ERR_INVALID_ARG, "capacity must be a positive multiple of 16");
  if (!k_f16 || !v_f16 || !aligned(k_f16, 16) || !aligned(v_f16, 16))
    return fail(CKV_ERR_INVALID_ARG, "k/v null or not 16-byte aligned");
  if (!prior_o || !prior_lse || !aligned(prior_o, 16) || !aligned(prior_lse, 4))
    return fail(CKV_ERR_INVALID_ARG, "prior_o (16-byte aligned) and prior_lse are required");
  if (prior_o == out || prior_lse == lse) return fail(CKV_ERR_INVALID_ARG, "prior and output must not alias");
  return run_decode(false, nullptr, k_f16, v_f16, head_dim, n_kv_heads, batch, capacity, seq_len, max_seq_len,
                    q_f16, n_q, n_q_heads, scale, n_split, out, lse, workspace, ws_bytes, stream, nullptr, 0, 0, 0,
                    0, prior_o, prior_lse);
}

// Split counts that let the fan-out's tail decode run beside its prefix decode
// on `sms` SMs (0, 0: each decode's automatic count).
static void fanout_splits(int64_t n_agents, int64_t n_kv_heads, int64_t group_q, int sms, int* ps_out, int* ts_out) {
  // Tail pass: batch n_agents, one query token; prefix pass: batch 1, n_agents query tokens.
  const int64_t tail_groups = n_agents * n_kv_heads * ((group_q + 7) / 8);
  const int64_t prefix_groups = n_kv_heads * ((group_q * n_agents + 7) / 8);
  *ps_out = 0;
  *ts_out = 0;
  if (2 * tail_groups >= sms) return;
  const int64_t ps = (sms - tail_groups) / prefix_groups;
  if (ps < 1) return;
  *ps_out = static_cast<int>(ps < ckv::kMaxSplits ? ps : ckv::kMaxSplits);
  *ts_out = 1;
}

ckv_status ckv_fanout_plan(int32_t n_agents, int32_t n_kv_heads, int32_t n_q_heads, int32_t* prefix_splits,
                           int32_t* tail_splits) {
  if (!prefix_splits || !tail_splits) return fail(CKV_ERR_INVALID_ARG, "null output");
  if (n_agents <= 0 || n_kv_heads <= 0 || n_q_heads <= 0) return fail(CKV_ERR_INVALID_ARG, "counts must be positive");
  if (n_q_heads % n_kv_heads)
    return fail(CKV_ERR_UNSUPPORTED, "n_q_heads %d not a multiple of n_kv_heads %d", n_q_heads, n_kv_heads);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return fail(CKV_ERR_CUDA, "cannot query the device");
  int ps, ts;
  fanout_splits(n_agents, n_kv_heads, n_q_heads / n_kv_heads, sms, &ps, &ts);
  *prefix_splits = ps;
  *tail_splits = ts;
  return CKV_OK;
}

// Fan-out workspace: [prefix decode][tail decode][prefix partial O, lse (composed form)].
struct FanoutWs {
  size_t pre, tail, o_pre, l_pre, total;
  int ps, ts;       // split counts (0: automatic)
  bool fused;       // the tail decode merges the prefix decode's slots
};
static bool fanout_ws(const ckv_cache* prefix, int64_t max_prefix_len, int32_t n_agents, int64_t max_tail_len,
                      int32_t n_q_heads, FanoutWs* w) {
  if (!prefix || check_cache(prefix) != CKV_OK || prefix->batch != 1 || n_agents <= 0 || n_q_heads <= 0 ||
      max_prefix_len < 0 || max_tail_len < 0 || n_q_heads != 8 * prefix->n_kv_heads)
    return false;
  const int D = prefix->head_dim, Hkv = prefix->n_kv_heads;
  int ps = 0, ts = 0;
  fanout_splits(n_agents, Hkv, 8, num_sms(), &ps, &ts);
  // The fused form needs the prefix on the mma.sync decode (the tile path's
  // cost model may prefer 128-row tiles for a long prefix) and the tail grid
  // resident at once (its merge is the rendezvous).
  const int64_t tail_grid = static_cast<int64_t>(n_agents) * Hkv * (ts ? ts : 1);
  w->fused = !ckv::concurrent_kernels() && ts > 0 && tail_grid <= num_sms() &&
             !ckv::rows_decode_applies(1, Hkv, n_q_heads, n_agents, 0, max_prefix_len);
  w->ps = w->fused ? ps : 0;
  w->ts = w->fused ? ts : 0;
  // Regions sized for both forms, so that the size does not depend on which
  // one a call takes.
  const size_t pre_f = ts > 0 ? mma_decode_ws(prefix, max_prefix_len, n_agents, n_q_heads, ps) : 0;
  const size_t pre_c = ckv_attn_decode_workspace(prefix, max_prefix_len, n_agents, n_q_heads, 0);
  const size_t tail_f = ts > 0 ? ckv_attn_decode_f16_workspace(D, Hkv, n_agents, max_tail_len, 1, n_q_heads, ts) : 0;
  const size_t tail_c = ckv_attn_decode_f16_merge_workspace(D, Hkv, n_agents, max_tail_len, 1, n_q_heads, 0);
  if (pre_c == 0 || tail_c == 0 || (ts > 0 && (pre_f == 0 || tail_f == 0))) return false;
  const size_t pre = pre_f > pre_c ? pre_f : pre_c;
  const size_t tail = tail_f > tail_c ? tail_f : tail_c;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = static_cast<size_t>(n_agents) * n_q_heads;
  w->pre = 0;
  w->tail = up(pre);
  w->o_pre = w->tail + up(tail);
  w->l_pre = w->o_pre + up(rows * D * sizeof(float));
  w->total = w->l_pre + up(rows * sizeof(float));
  return true;
}

size_t ckv_attn_decode_fanout_workspace(const ckv_cache* prefix, int64_t max_prefix_len, int32_t n_agents,
                                        int64_t max_tail_len, int32_t n_q_heads) {
  FanoutWs w;
  return fanout_ws(prefix, max_prefix_len, n_agents, max_tail_len, n_q_heads, &w) ? w.total : 0;
}

ckv_status ckv_attn_decode_fanout(const ckv_cache* prefix, const int32_t* prefix_len, int64_t max_prefix_len,
                                  const void* k_tail, const void* v_tail, int64_t tail_capacity,
                                  const int32_t* tail_len, int64_t max_tail_len, int32_t n_agents, const void* q_f16,
                                  int32_t n_q_heads, float scale, float* out, float* lse, void* workspace,
                                  size_t ws_bytes, void* stream) {
  ckv_status s = check_cache(prefix);
  if (s != CKV_OK) return s;
  if (prefix->batch != 1) return fail(CKV_ERR_INVALID_ARG, "the shared prefix cache holds one sequence (batch 1)");
  if (n_agents <= 0 || n_q_heads <= 0) return fail(CKV_ERR_INVALID_ARG, "n_agents and n_q_heads must be positive");
  if (n_q_heads != 8 * prefix->n_kv_heads)
    return fail(CKV_ERR_UNSUPPORTED, "the fan-out step needs 8 query heads per kv head (%d over %d)", n_q_heads,
                prefix->n_kv_heads);
  if (max_prefix_len < 0 || max_prefix_len > prefix->capacity) return fail(CKV_ERR_INVALID_ARG, "max_prefix_len outside the cache");
  if (max_tail_len < 0 || max_tail_len > tail_capacity) return fail(CKV_ERR_INVALID_ARG, "max_tail_len outside the tails");
  if (tail_capacity <= 0 || tail_capacity % 16) return fail(CKV_ERR_INVALID_ARG, "tail capacity must be a positive multiple of 16");
  if (!k_tail || !v_tail || !aligned(k_tail, 16) || !aligned(v_tail, 16))
    return fail(CKV_ERR_INVALID_ARG, "tail k/v null or not 16-byte aligned");
  if (!prefix_len || !aligned(prefix_len, 4)) return fail(CKV_ERR_INVALID_ARG, "prefix_len null or misaligned");
  FanoutWs w;
  if (!fanout_ws(prefix, max_prefix_len, n_agents, max_tail_len, n_q_heads, &w))
    return fail(CKV_ERR_INVALID_ARG, "invalid fan-out geometry");
  s = check_ws(workspace, ws_bytes, w.total);
  if (s != CKV_OK) return s;
  const int D = prefix->head_dim, Hkv = prefix->n_kv_heads;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  if (!w.fused) {
    // Composed form: the prefix partial goes through the workspace and the
    // tail decode merges it as its prior.
    float* o_pre = reinterpret_cast<float*>(base + w.o_pre);
    float* l_pre = reinterpret_cast<float*>(base + w.l_pre);
    s = ckv_attn_decode(prefix, prefix_len, max_prefix_len, q_f16, n_agents, n_q_heads, scale, 0, o_pre, l_pre,
                        base + w.pre, w.tail - w.pre, stream);
    if (s != CKV_OK) return s;
    DecodeExtras fl{0, nullptr, 0, 0, reinterpret_cast<int32_t*>(base + w.pre), 0};  // one flag word for the step
    return run_decode(false, nullptr, k_tail, v_tail, D, Hkv, n_agents, tail_capacity, tail_len, max_tail_len, q_f16,
                      1, n_q_heads, scale, 0, out, lse, base + w.tail, w.o_pre - w.tail, stream, nullptr, 0, 0, 0, 0,
                      o_pre, l_pre, nullptr, nullptr, nullptr, &fl);
  }
  // Fused form: the prefix decode writes its split slots and leaves; the tail
  // decode, beside it on the SMs it leaves free, merges its own split with the
  // prefix's slots of the same rows.
  DecodePlan pp;
  s = plan_decode(D, Hkv, 1, max_prefix_len, n_agents, n_q_heads, w.ps, &pp);
  if (s != CKV_OK) return s;
  DecodeExtras pl{1, nullptr, 0, 0, nullptr, 0};
  s = run_decode(true, prefix, nullptr, nullptr, D, Hkv, 1, prefix->capacity, prefix_len, max_prefix_len, q_f16,
                 n_agents, n_q_heads, scale, w.ps, out, lse, base + w.pre, w.tail - w.pre, stream, nullptr, 0, 0, 0,
                 0, nullptr, nullptr, nullptr, nullptr, nullptr, &pl);
  if (s != CKV_OK) return s;
  DecodeExtras tl{0, reinterpret_cast<const float*>(base + w.pre + ws_header_bytes(pp.groups, pp.n_split)),
                  pp.n_split, pp.n_row_groups, reinterpret_cast<int32_t*>(base + w.pre), 0};
  return run_decode(false, nullptr, k_tail, v_tail, D, Hkv, n_agents, tail_capacity, tail_len, max_tail_len, q_f16,
                    1, n_q_heads, scale, w.ts, out, lse, base + w.tail, w.o_pre - w.tail, stream, nullptr, 0, 0, 0, 0,
                    nullptr, nullptr, nullptr, nullptr, nullptr, &tl);
}

ckv_status ckv_f16_append(void* k_f16, void* v_f16, int32_t head_dim, int32_t n_kv_heads, int32_t batch,
                          int64_t capacity, const int32_t* seq_len, const void* k_new_f16, const void* v_new_f16,
                          int32_t n_new, int64_t token_stride, int64_t batch_stride, void* stream) {
  if (!supported_dim(head_dim)) return fail(CKV_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256,512}", head_dim);
  if (n_kv_heads <= 0 || batch <= 0 || capacity <= 0 || n_new < 0)
    return fail(CKV_ERR_INVALID_ARG, "bad geometry");
  if (n_new == 0) return CKV_OK;
  if (!k_f16 || !v_f16 || !seq_len || !k_new_f16 || !v_new_f16 || !aligned(k_f16, 16) || !aligned(v_f16, 16) ||
      !aligned(k_new_f16, 16) || !aligned(v_new_f16, 16) || !aligned(seq_len, 4))
    return fail(CKV_ERR_INVALID_ARG, "null or misaligned pointer");
  const int64_t row = static_cast<int64_t>(n_kv_heads) * head_dim;
  if (token_stride < row || token_stride % 8 || batch_stride < 0 || batch_stride % 8 ||
      (batch > 1 && batch_stride < token_stride * n_new))
    return fail(CKV_ERR_INVALID_ARG, "bad strides (token %lld, batch %lld)", (long long)token_stride,
                (long long)batch_stride);
  if (n_new > 65535 || batch > 65535) return fail(CKV_ERR_UNSUPPORTED, "n_new and batch must be at most 65535");
  ckv::F16AppendArgs a{};
  a.k = static_cast<__half*>(k_f16);
  a.v = static_cast<__half*>(v_f16);
  a.head_dim = head_dim;
  a.n_kv_heads = n_kv_heads;
  a.batch = batch;
  a.capacity = capacity;
  a.seq_len = seq_len;
  a.k_new = static_cast<const __half*>(k_new_f16);
  a.v_new = static_cast<const __half*>(v_new_f16);
  a.n_new = n_new;
  a.token_stride = token_stride;
  a.batch_stride = batch_stride;
  const cudaError_t e = ckv::launch_f16_append(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "f16_append launch");
  return CKV_OK;
}

ckv_status ckv_attn_prefill_f16(const void* k_f16, const void* v_f16, int32_t head_dim, int32_t n_kv_heads,
                                int32_t batch, int64_t capacity, const int32_t* seq_len, int64_t max_seq_len,
                                const void* q_bf16, int32_t n_new, int32_t n_q_heads, float scale, int32_t n_split,
                                float* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  if (!supported_dim(head_dim))
    return fail(CKV_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256,512}", head_dim);
  if (n_kv_heads <= 0 || batch <= 0) return fail(CKV_ERR_INVALID_ARG, "n_kv_heads and batch must be positive");
  if (capacity <= 0 || capacity % 16) return fail(CKV_ERR_INVALID_ARG, "capacity must be a positive multiple of 16");
  if (!k_f16 || !v_f16 || !aligned(k_f16, 16) || !aligned(v_f16, 16))
    return fail(CKV_ERR_INVALID_ARG, "k/v null or not 16-byte aligned");
  return run_decode(false, nullptr, k_f16, v_f16, head_dim, n_kv_heads, batch, capacity, seq_len, max_seq_len,
                    q_bf16, n_new, n_q_heads, scale, n_split, out, lse, workspace, ws_bytes, stream, nullptr, 1, 0,
                    1);
}

// Shared-prefix prefill workspace: [prefix prefill][tail pass][prefix O, lse].
struct SharedWs {
  size_t pre, tail, o_pre, l_pre, total;
};
static bool shared_ws(const ckv_cache* prefix, int32_t n_agents, int64_t tail_capacity, int32_t n_new,
                      int32_t n_q_heads, SharedWs* w) {
  if (!prefix || n_agents <= 0 || n_new <= 0 || tail_capacity <= 0) return false;
  const size_t pre = ckv_attn_prefill_workspace(prefix, n_agents * n_new, n_q_heads);
  const size_t tail = ckv_attn_decode_f16_merge_workspace(prefix->head_dim, prefix->n_kv_heads, n_agents,
                                                          tail_capacity, n_new, n_q_heads, 0);
  if (tail == 0) return false;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = static_cast<size_t>(n_agents) * n_new * n_q_heads;
  w->pre = 0;
  w->tail = up(pre);
  w->o_pre = w->tail + up(tail);
  w->l_pre = w->o_pre + up(rows * prefix->head_dim * sizeof(float));
  w->total = w->l_pre + up(rows * sizeof(float));
  return true;
}

size_t ckv_attn_prefill_shared_workspace(const ckv_cache* prefix, int32_t n_agents, int64_t tail_capacity,
                                         int32_t n_new, int32_t n_q_heads) {
  SharedWs w;
  return shared_ws(prefix, n_agents, tail_capacity, n_new, n_q_heads, &w) ? w.total : 0;
}

ckv_status ckv_attn_prefill_shared(const ckv_cache* prefix, int64_t n_prefix, void* k_tail, void* v_tail,
                                   int64_t tail_capacity, const int32_t* tail_len, int32_t n_agents,
                                   const void* q_bf16, const void* k_new_f16, const void* v_new_f16, int32_t n_new,
                                   int32_t n_q_heads, float scale, float* out, float* lse, void* workspace,
                                   size_t ws_bytes, void* stream) {
  if (!prefix) return fail(CKV_ERR_INVALID_ARG, "prefix cache is null");
  if (prefix->batch != 1) return fail(CKV_ERR_INVALID_ARG, "the shared prefix cache holds one sequence (batch 1)");
  if (n_prefix < 0 || n_prefix > prefix->capacity) return fail(CKV_ERR_INVALID_ARG, "n_prefix outside the cache");
  if (n_agents <= 0 || n_new < 0) return fail(CKV_ERR_INVALID_ARG, "n_agents must be positive, n_new >= 0");
  if (n_new == 0) return CKV_OK;
  if (!out || !lse || !aligned(out, 16) || !aligned(lse, 4)) return fail(CKV_ERR_INVALID_ARG, "null or misaligned out/lse");
  SharedWs w;
  if (!shared_ws(prefix, n_agents, tail_capacity, n_new, n_q_heads, &w))
    return fail(CKV_ERR_INVALID_ARG, "invalid shared-prefix prefill geometry");
  ckv_status s = check_ws(workspace, ws_bytes, w.total);
  if (s != CKV_OK) return s;
  const int D = prefix->head_dim, Hkv = prefix->n_kv_heads;
  if (tail_capacity % 16) return fail(CKV_ERR_INVALID_ARG, "tail capacity must be a multiple of 16");
  if (!k_tail || !v_tail || !aligned(k_tail, 16) || !aligned(v_tail, 16))
    return fail(CKV_ERR_INVALID_ARG, "tail k/v null or not 16-byte aligned");
  uint8_t* base = static_cast<uint8_t*>(workspace);
  // 1. The new rows join each agent's fp16 tail at [tail_len - n_new, tail_len).
  const int64_t row = static_cast<int64_t>(Hkv) * D;
  s = ckv_f16_append(k_tail, v_tail, D, Hkv, n_agents, tail_capacity, tail_len, k_new_f16, v_new_f16, n_new, row,
                     row * n_new, stream);
  if (s != CKV_OK) return s;
  // 2. All agents' queries over the shared compressed prefix, one sequence of n_agents * n_new tokens
  //    (its rows are laid out as the output's).
  float* o_pre = reinterpret_cast<float*>(base + w.o_pre);
  float* l_pre = reinterpret_cast<float*>(base + w.l_pre);
  if (n_prefix > 0) {
    s = ckv_attn_prefill_prefix(prefix, n_prefix, q_bf16, n_agents * n_new, n_q_heads, scale, o_pre, l_pre,
                                base + w.pre, w.tail - w.pre, stream);
    if (s != CKV_OK) return s;
  }
  // 3. Every agent's queries over its own tail, causal (token i sees [0, tail_len - n_new + i]), merged
  //    exactly with the prefix partial inside the same launch.
  return run_decode(false, nullptr, k_tail, v_tail, D, Hkv, n_agents, tail_capacity, tail_len, tail_capacity, q_bf16,
                    n_new, n_q_heads, scale, 0, out, lse, base + w.tail, w.o_pre - w.tail, stream, nullptr, 1, 0, 1, 0,
                    n_prefix > 0 ? o_pre : nullptr, n_prefix > 0 ? l_pre : nullptr);
}

ckv_status ckv_lse_merge(int32_t n_parts, const float* const* o_parts, const float* const* lse_parts,
                         int64_t n_rows, int32_t d, float* out, float* lse, void* stream) {
  if (n_parts < 1 || n_parts > 16) return fail(CKV_ERR_INVALID_ARG, "n_parts must be in [1, 16]");
  if (!o_parts || !lse_parts || !out || !lse) return fail(CKV_ERR_INVALID_ARG, "null pointer argument");
  if (n_rows < 0 || n_rows > 0x7fffffffLL || d <= 0) return fail(CKV_ERR_INVALID_ARG, "bad n_rows or d");
  ckv::LseMergeArgs a{};
  for (int r = 0; r < n_parts; ++r) {
    if (!o_parts[r] || !lse_parts[r]) return fail(CKV_ERR_INVALID_ARG, "part %d is null", r);
    a.o[r] = o_parts[r];
    a.l[r] = lse_parts[r];
  }
  a.n_parts = n_parts;
  a.n_rows = n_rows;
  a.d = d;
  a.rows_per_group = n_rows > 0 ? n_rows : 1;
  a.out = out;
  a.lse = lse;
  cudaError_t e = ckv::launch_lse_merge(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "lse_merge launch");
  return CKV_OK;
}

ckv_status ckv_read_device_flag(const void* workspace, int32_t* flag, void* stream) {
  if (!workspace || !flag) return fail(CKV_ERR_INVALID_ARG, "null argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream sync");
  e = cudaMemcpy(flag, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "flag read");
  if (*flag != 0) {
    e = cudaMemset(const_cast<void*>(workspace), 0, sizeof(int32_t));
    if (e != cudaSuccess) return cuda_fail(e, "flag clear");
    return fail(CKV_ERR_DEVICE_FLAG, "device flag %d", *flag);
  }
  return CKV_OK;
}

}  // extern "C"
