/*
 * ckv.h — C ABI of the compressed-KV attention library for NVIDIA GB300 (sm_103a).
 *
 * The library runs attention directly over an asymmetrically compressed KV
 * cache: keys are q8_0 (blocks of 32 int8 codes with one fp16 scale) and values
 * are 3-bit TurboQuant-MSE ("TBQ3": a +/-1 sign diagonal, an orthonormal fast
 * Walsh-Hadamard transform, one fp16 norm per vector, 3-bit Lloyd-Max codes).
 * The scheme is the one on the PolyKV page ("F5 M6 — PolyKV (shared compressed
 * KV pool)", section "What PolyKV is (reference)"); attention reads the packed
 * bytes in-kernel rather than decompressing the cache first (same page,
 * sections "S2 perf-path Level B" and "S2 perf-path — turbo-MMA verify kernel +
 * scalar-K/turbo-V fused decode": K is read in true space, V in the rotated
 * basis, and one inverse transform runs on the output).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller. The library
 *    never allocates or frees memory. Scratch space ("workspace") is sized by
 *    the matching *_workspace() query and passed in by the caller, zero-filled
 *    once before its first use (e.g. cudaMemsetAsync); calls leave its header
 *    as they found it, so it is reused without clearing.
 *  - Work is enqueued asynchronously on the caller's CUDA stream (`stream` is a
 *    cudaStream_t; NULL means the legacy default stream). Arguments are checked
 *    on the host before anything is launched; a failed check returns a status
 *    and launches nothing. No call aborts or exits the process.
 *  - ckv_last_error() returns a message for the last failure on this thread.
 *  - Kernels that wait on asynchronous copies bound every wait; a wait that
 *    runs out (or a device-side range check that fails) sets a flag in the first
 *    4 bytes of the workspace instead of hanging. The flag keeps the first
 *    error of any call since it was last read: ckv_read_device_flag() reads it
 *    after the stream has drained and clears it.
 *  - Head dims supported: 64, 128, 256, 512. The number of query heads must be
 *    a multiple of the number of KV heads; query head h reads KV head
 *    floor(h / G), G = n_q_heads / n_kv_heads (grouped-query attention, as the
 *    Upstream Sync page's entry 0080 describes for Gemma-4: 16 heads, 2 KV heads).
 *  - Outputs are float32: the normalised attention output and the natural-log
 *    log-sum-exp of every query row, the "FA output packed with per-row LSE"
 *    contract of the DCA page ("Feature — Gemma-4 A4B Dual Chunk Attention (DCA),
 *    training-free 1M context", section "Implementation progress + Section-D
 *    simplification"). A row that sees no key returns output 0 and lse -inf
 *    (same page, section "Section C2b": empty regimes drop out of the merge).
 */
#ifndef CKV_H
#define CKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CKV_API __attribute__((visibility("default")))
#else
#define CKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CKV_OK = 0,
  CKV_ERR_INVALID_ARG = -1,  /* null pointer, misalignment, bad size or range   */
  CKV_ERR_UNSUPPORTED = -2,  /* valid but not supported (head_dim, head ratio)  */
  CKV_ERR_WORKSPACE = -3,    /* workspace pointer null or smaller than needed   */
  CKV_ERR_CUDA = -4,         /* a CUDA call or launch failed (see last_error)   */
  CKV_ERR_DEVICE_FLAG = -5   /* a kernel reported a bounded-wait or range fault */
} ckv_status;

/*
 * The packed cache. One allocation of ckv_cache_bytes() bytes, 16-byte aligned.
 *
 * V codes have b = v_bits bits (3: TBQ3, the default; 2 and 4: the neighbouring
 * TurboQuant tiers, PolyKV page section "S2 — TurboQuant tier family": the same
 * rotation and Lloyd-Max scheme at another bit width). A record is
 * R = 17*D + 2*b*D + 32 bytes (23*D + 32 at b = 3).
 *
 * Each (sequence b, kv head h) owns capacity/16 consecutive "tile records";
 * record t holds token positions [16 t, 16 t + 16) and starts at byte
 * ((b * n_kv_heads + h) * (capacity / 16) + t) * R. Inside a record
 * (p = position in the tile, i = dim, D = head_dim):
 *
 *   [0, 16D)       K q8_0 codes, each stored as the byte q + 128. (p, i) is at
 *                  ((i/32)*32 + L)*16 + (p/8)*8 + (i%8), L = 4*(p%8) + (i%32)/8.
 *   [16D, 17D)     K q8_0 scales (fp16), row-major [16][D/32].
 *   [17D, 17D+2bD) V codes, b bits each. With G = D/8, L = 4*(i/G) + (p%8)/2
 *                  and pair index k = 4*((i%G)/2) + (i%G)%2 + 2*(p/8), the code of
 *                  (p, i) is bits [2bk + b*(p%2), +b) (LSB first) of lane L's
 *                  bD/16-byte stream; stream byte s of lane L is at
 *                  17D + ((s/gr)*32 + L)*gr + s%gr, gr = the largest of 16, 8, 4
 *                  that divides bD/16. Codes index the ascending Lloyd-Max table
 *                  of N(0,1) with 2^b levels; b = 3:
 *                  (-2.1520, -1.3439, -0.7560, -0.2451, 0.2451, 0.7560, 1.3439, 2.1520),
 *                  b = 2: (-1.5104, -0.4528, 0.4528, 1.5104), b = 4: +/-(0.1284,
 *                  0.3880, 0.6568, 0.9423, 1.2562, 1.6180, 2.0690, 2.7326).
 *   [17D+2bD, R)   V norms (fp16), one per position.
 *
 * The layout puts every lane's share of a tile contiguous so that a tile moves
 * into shared memory with one bulk copy and each lane's mma fragments come out
 * of conflict-free 16-byte shared loads. Positions that were never packed hold
 * whatever the allocation held; attention never reads past seq_len.
 *
 * v_signs: the +/-1 sign diagonal (int8, D entries, device), one vector shared
 * by every head and token.
 *
 * v_signs2: NULL for the transform above (one sign diagonal, the full D-point
 * FWHT, one norm per vector). Non-NULL selects the block-diagonal rotation of
 * the fork the PolyKV page builds on (sections "S2 perf-path Level A/B" and
 * "S2 perf-path D=512 fused turbo-vec": the WHT runs on each 128-dim group,
 * with a sign diagonal before it and one after it, and each group keeps its
 * own norm): for every group g of 128 dims, u_g = s2_g * H_128 (s1_g * x_g) /
 * ||x_g|| with s1 = v_signs, s2 = v_signs2 (device, head_dim entries each), and
 * the record holds D/128 norms per position, group-major: norm (p, j) at
 * 17D + 2bD + 2*(16*j + p); R = 17D + 2bD + 32*D/128. Needs head_dim >= 128.
 */
typedef struct {
  int32_t head_dim;      /* D */
  int32_t n_kv_heads;    /* Hkv */
  int32_t batch;         /* B sequences */
  int32_t v_bits;        /* bits per V code: 2, 3 or 4; 0 means 3 */
  int64_t capacity;      /* token positions per sequence, multiple of 16 */
  void* data;            /* device, ckv_cache_bytes(...) bytes, 16-byte aligned */
  const int8_t* v_signs; /* device, head_dim entries of +1 / -1 */
  const int8_t* v_signs2; /* NULL, or device, head_dim entries: the block-diagonal rotation */
} ckv_cache;

/* Bytes of the packed cache at 3 bits per V code: batch * n_kv_heads * capacity/16 * (23*D + 32).
 * 0 if invalid. */
CKV_API size_t ckv_cache_bytes(int32_t head_dim, int32_t n_kv_heads, int32_t batch, int64_t capacity);
/* The same at v_bits (2, 3 or 4) bits per V code and rotation: rot_group 0 for
 * the full transform (... * (17*D + 2*v_bits*D + 32)) or 128 for the
 * block-diagonal rotation (... * (17*D + 2*v_bits*D + 32*D/128)). 0 if invalid. */
CKV_API size_t ckv_cache_bytes_v(int32_t head_dim, int32_t n_kv_heads, int32_t batch, int64_t capacity,
                                 int32_t v_bits, int32_t rot_group);

/*
 * kv_pack — quantise n_tok new K and V rows of every sequence into the cache at
 * token positions [tok_offset, tok_offset + n_tok).
 *
 * K rows become q8_0 (PolyKV page, "What PolyKV is (reference)": K -> int8 q8_0):
 * per block of 32, d16 = fp16(amax/127), q = x/d16 rounded half away from zero
 * (fp32 division, correctly rounded), clamped to [-127, 127]; d16 == 0 stores 0.
 * V rows become TBQ3 (same section: FWHT rotation, then Lloyd-Max; "Phase-0 fork
 * recon": warp-shuffle group transform and bit-packed codes on write): y = s*x,
 * u = H_D y / ||x|| (H_D the Sylvester Hadamard matrix; this equals the
 * orthonormal transform times sqrt(D)/||x||), each u_i snapped to the nearest
 * centroid (ties at midpoints to the smaller magnitude, u = 0 to +0.2451),
 * n16 = fp16(||x||). A zero vector stores codes 4 and norm 0. With v_bits 2 or
 * 4 the same steps use that tier's table (u = 0 and the zero vector take code
 * 2^(b-1), the smallest positive centroid).
 *
 * k_f16, v_f16: fp16, element (b, j, h, i) of token j of sequence b at
 *   b*batch_stride + j*token_stride + h*D + i (in elements). token_stride >= Hkv*D.
 * Errors: INVALID_ARG for null/misaligned pointers (inputs 16-byte aligned,
 * strides multiples of 8 elements), a range outside [0, capacity), or negative n_tok.
 */
CKV_API ckv_status ckv_kv_pack(const ckv_cache* cache, int64_t tok_offset, int64_t n_tok,
                       const void* k_f16, const void* v_f16,
                       int64_t token_stride, int64_t batch_stride, void* stream);

/*
 * selftest_bounded_waits — the failure path of the library's asynchronous
 * waits. Every wait in its kernels (an mbarrier phase, a global counter
 * written by other CTAs) gives up after 2 s of wall time, raises the device
 * flag (1 = a bounded wait ran out) and lets the kernel finish, so a lost
 * event becomes an error status instead of a hung context. This call runs
 * both forms on events that never come: after it, the int32 at workspace
 * byte 0 (the mbarrier form) and at byte 4 (the counter form) read 1.
 * workspace: device, at least 256 bytes, 256-byte aligned, zero-filled (the
 * counter at byte 64 must stay 0). Takes about 4 s of GPU time.
 */
CKV_API ckv_status ckv_selftest_bounded_waits(void* workspace, size_t ws_bytes, void* stream);

/*
 * calibrate_stream — a measuring aid with no counterpart in the pages: the
 * decode's data movement alone. Streams n_streams runs of n_tiles records of
 * record_bytes each (device memory at src, 16-byte aligned, record_bytes a
 * multiple of 16, 4 x 4 records <= 200 KB), split over n_split CTAs per run,
 * through the decode's staging (bulk copies of 4 records into a 4-stage
 * shared-memory ring, programmatic launch) and computes nothing; with
 * rendezvous != 0 the CTAs of a run then meet on a counter as the decode's
 * split merge does (refused with CKV_ERR_UNSUPPORTED unless the grid fits on
 * the device at once). Its time per launch, back to back, is the floor of any
 * kernel with that launch shape on those bytes. workspace: 64 + 8 n_streams
 * zero-filled device bytes, 256-byte aligned (flag at 0, counters from 64,
 * left at zero). Asynchronous on `stream`.
 */
CKV_API ckv_status ckv_calibrate_stream(const void* src, int64_t n_tiles, int32_t record_bytes, int32_t n_streams,
                                        int32_t n_split, int32_t rendezvous, void* workspace, size_t ws_bytes,
                                        void* stream);

/*
 * attn_decode — attention of n_q query tokens per sequence over the packed
 * cache, every query seeing cached positions [0, seq_len[b]).
 *
 * Split-K flash-decode: each CTA streams a contiguous range of tile records
 * through shared memory, computes S = Q K_hat^T on tensor cores from the int8
 * codes (scales applied per 32-block), runs the online softmax, and accumulates
 * P V_hat in the rotated basis straight from the b-bit codes. Each CTA writes
 * its partial to the workspace; the CTAs that finish last merge the partials
 * of their row group with the exact log-sum-exp combine (a two-level tree,
 * no CTA waiting for another) and apply the inverse transform and sign flip
 * once per output row (valid because the rotation is linear and shared within
 * a head: PolyKV page, "S2 perf-path Level B" — the transform runs only on the
 * small FA output). One kernel launch; it may begin while the previous kernel
 * on the stream finishes, and waits for it before touching global memory.
 *
 * seq_len: device int32 [batch], each in [0, min(capacity, max_seq_len)]; a
 *   value outside that range raises the device flag and counts as 0.
 *   max_seq_len (host) sizes the split grid: the splits divide
 *   [0, min(capacity, max_seq_len)), and tiles past seq_len are skipped.
 * q_f16: device fp16 [batch][n_q][n_q_heads][D].
 * scale: logit scale (e.g. 1/sqrt(D)).
 * n_split: KV splits per (sequence, kv head, row group), at most 1024; 0 picks
 *   one that fills the GPU. out: float32 [batch][n_q][n_q_heads][D]; lse:
 *   float32 [batch][n_q][n_q_heads].
 * workspace: ckv_attn_decode_workspace() bytes, 256-byte aligned, zero-filled
 *   before first use; its merge counters are back at zero after every call.
 *
 * Many query rows per kv head (n_q * n_q_heads / n_kv_heads >= 64, as when
 * many agents read one shared prefix: PolyKV page, section "S2 perf-path
 * Level B" — large-n_q attention over turbo KV belongs on the tensor cores):
 * the row groups above dequantise every tile once per 8 rows, so with n_split
 * 0 the call instead runs the tcgen05 prefill kernel on 128-row tiles (query
 * heads / kv heads must divide 128), each CTA taking a share of the 64-key
 * steps and writing one partial, then a merge kernel (two launches) — where a
 * cost model fitted on GB300 at head_dim 512 says it is faster (long prefixes:
 * 1.3x at 32768 tokens and 1.6x at 65536 with 120 rows per kv head). n_split
 * -1 forces that path (CKV_ERR_UNSUPPORTED if the head ratio does not divide
 * 128 or max_seq_len is 0); its workspace is one 128 x (D + 1) float slot per
 * tile and split.
 */
CKV_API size_t ckv_attn_decode_workspace(const ckv_cache* cache, int64_t max_seq_len, int32_t n_q,
                                 int32_t n_q_heads, int32_t n_split);
CKV_API ckv_status ckv_attn_decode(const ckv_cache* cache, const int32_t* seq_len, int64_t max_seq_len,
                           const void* q_f16, int32_t n_q, int32_t n_q_heads, float scale,
                           int32_t n_split, float* out, float* lse, void* workspace,
                           size_t ws_bytes, void* stream);

/*
 * attn_decode_verify — attention of a verify batch: the n_q query tokens of a
 * sequence are its last n_q positions, so query token i sees cached positions
 * [0, seq_len[b] - n_q + i] (causal among the batch; a token whose range is
 * empty gets O = 0 and lse = -inf). This is the multi-query decode that checks
 * n_q drafted tokens at once (PolyKV page, section "WorkStream-1": the
 * "turbo-MMA verify (n_q>1)" path for MTP verify batches). The drafts' K/V rows
 * must already be in the cache (ckv_kv_pack). Arguments, workspace and errors
 * as attn_decode; the same kernel runs with per-row key limits.
 */
CKV_API ckv_status ckv_attn_decode_verify(const ckv_cache* cache, const int32_t* seq_len, int64_t max_seq_len,
                                          const void* q_f16, int32_t n_q, int32_t n_q_heads, float scale,
                                          int32_t n_split, float* out, float* lse, void* workspace,
                                          size_t ws_bytes, void* stream);

/*
 * attn_decode_dca — dual chunk attention of one query token per sequence (the
 * token at position i = seq_len[b] - 1) over the packed cache. DCA page
 * ("Feature — Gemma-4 A4B Dual Chunk Attention (DCA), training-free 1M
 * context"), section "Section C design": with chunk c and k = i / c, three
 * regimes partition the keys [0, seq_len[b]):
 *   intra       [k c, seq_len)        query q_f16[b][0]
 *   successive  [(k - 1) c, k c)      query q_f16[b][1]
 *   inter       [0, (k - 1) c)        query q_f16[b][2]
 * (each query roped for its regime by the caller; the keys are cached as
 * roped once), and their softmaxes are merged exactly by log-sum-exp.
 * q_f16: fp16 [batch][3][n_q_heads][D]; out: float32 [batch][n_q_heads][D];
 * lse: float32 [batch][n_q_heads]. chunk >= 1. Two launches: the decode
 * kernel with the regimes as its query rows (each row group reads only its
 * regime's tiles; the inter range is cut into m equal pieces of about one
 * chunk, m = clamp(round((max_seq_len - 2 chunk) / chunk), 1, 14), rows that
 * all use the inter query, so that no regime's CTAs carry more keys than the
 * others) and the exact merge of the 2 + m rows. workspace:
 * ckv_attn_decode_dca_workspace() bytes (enough for any chunk), zero-filled
 * before first use.
 */
CKV_API size_t ckv_attn_decode_dca_workspace(const ckv_cache* cache, int64_t max_seq_len, int32_t n_q_heads,
                                             int32_t n_split);
CKV_API ckv_status ckv_attn_decode_dca(const ckv_cache* cache, const int32_t* seq_len, int64_t max_seq_len,
                                       int32_t chunk, const void* q_f16, int32_t n_q_heads, float scale,
                                       int32_t n_split, float* out, float* lse, void* workspace,
                                       size_t ws_bytes, void* stream);

/*
 * attn_decode_append — one decode step: quantise n_new new K/V rows of every
 * sequence into the cache at positions [seq_len[b] - n_new, seq_len[b]) (the
 * same bytes ckv_kv_pack writes), then attend as attn_decode over
 * [0, seq_len[b]). The rows are packed inside the decode kernel by the CTA whose
 * KV range holds them, before it reads those tiles, so the step is a single
 * kernel. seq_len is the length after the append.
 *
 * k_new_f16, v_new_f16: fp16, element (b, j, h, i) of new row j at
 *   b*batch_stride + j*token_stride + h*D + i (elements), 16-byte aligned,
 *   strides multiples of 8. n_new in [1, 16], <= max_seq_len.
 * Other arguments and the workspace as attn_decode.
 * Errors: as attn_decode and ckv_kv_pack; UNSUPPORTED when a kv head has more
 * than 8 query rows (n_q * n_q_heads / n_kv_heads > 8): use ckv_kv_pack then
 * ckv_attn_decode. A seq_len[b] below n_new raises the device flag (nothing is
 * written for that sequence).
 */
CKV_API ckv_status ckv_attn_decode_append(const ckv_cache* cache, const int32_t* seq_len,
                                          int64_t max_seq_len, const void* k_new_f16, const void* v_new_f16,
                                          int32_t n_new, int64_t token_stride, int64_t batch_stride,
                                          const void* q_f16, int32_t n_q, int32_t n_q_heads, float scale,
                                          int32_t n_split, float* out, float* lse, void* workspace,
                                          size_t ws_bytes, void* stream);

/*
 * attn_decode_append_host — one decode step (attn_decode_append) on HOST
 * buffers, with no staging copies: the kernel reads q
 * [batch][n_q][n_q_heads][D] and k_new, v_new [batch][n_new][n_kv_heads][D]
 * (fp16, packed, 16-byte aligned) from page-locked host memory and writes out
 * [batch][n_q][n_q_heads][D] and lse [batch][n_q][n_q_heads] (fp32) back to
 * it, across the CPU-GPU interconnect (on GB300, NVLink-C2C with the Grace
 * host's memory). Host buffers must be page-locked and mapped into the device
 * address space (cudaHostAlloc or cudaHostRegister; with unified addressing
 * their device address is the host address): anything else is refused with
 * CKV_ERR_INVALID_ARG before any launch. The results are in host memory once
 * `stream` has completed. seq_len stays a device array. The kernel reads q,
 * k_new and v_new before it waits for the previous kernel on the stream (no
 * kernel writes them), so their trips across the interconnect overlap that
 * kernel's last work; the host must have written them before this call, as
 * for any launch. Other arguments and errors as attn_decode_append. No
 * counterpart in the pages: it is the host side of a serving loop.
 */
CKV_API ckv_status ckv_attn_decode_append_host(const ckv_cache* cache, const int32_t* seq_len, int64_t max_seq_len,
                                               const void* k_new_host, const void* v_new_host, int32_t n_new,
                                               const void* q_host, int32_t n_q, int32_t n_q_heads, float scale,
                                               int32_t n_split, float* out_host, float* lse_host, void* workspace,
                                               size_t ws_bytes, void* stream);

/*
 * attn_decode_noalloc — attn_decode for callers that cannot allocate device
 * memory. The pages have no counterpart to this entry point; it exists for
 * callers with no way to hand in a workspace: a host framework that owns all
 * device memory and gives a plug-in none of it, a latency-critical loop that
 * must not call cudaMalloc (it can block and synchronise the device), or a
 * process whose memory planner has already handed out the whole device.
 *
 * Same arguments and results as attn_decode, without the workspace. The
 * scratch is a 4 MiB array compiled into the library (held on every device that
 * loads it until the process exits); a call whose scratch would exceed it (see
 * ckv_attn_decode_workspace) returns CKV_ERR_WORKSPACE. Nothing is allocated.
 * Every call shares that one array, which keeps the last call's contents: each
 * call first clears, on its stream, the counter words its own shape uses
 * (cudaMemsetAsync of at most a few KB), so a call of any shape may follow a
 * call of any other, or a call whose bounded wait timed out. Calls that overlap
 * on the GPU race on the array and give wrong results (order them on one
 * stream or with events). The device flag (first 4 bytes of the array) is not
 * cleared by a call; read and clear it with ckv_read_noalloc_flag. The first
 * call on a device looks up the array's address on that device; make that
 * first call before any stream capture on the device.
 */
CKV_API ckv_status ckv_attn_decode_noalloc(const ckv_cache* cache, const int32_t* seq_len,
                                           int64_t max_seq_len, const void* q_f16, int32_t n_q,
                                           int32_t n_q_heads, float scale, int32_t n_split, float* out,
                                           float* lse, void* stream);

/*
 * read_noalloc_flag — ckv_read_device_flag for the built-in array of
 * attn_decode_noalloc, whose address callers never see. Drains `stream`, stores
 * the flag word in *flag (host memory), and when it is nonzero (1 = a bounded
 * wait ran out, 2 = a seq_len outside [0, min(capacity, max_seq_len)], counted
 * as 0) clears it and returns CKV_ERR_DEVICE_FLAG. No counterpart in the pages.
 */
CKV_API ckv_status ckv_read_noalloc_flag(int32_t* flag, void* stream);

/*
 * attn_decode_f16 — the same decode over a dense fp16 KV cache (the private,
 * uncompressed tails of the shared-pool fan-out: PolyKV page, section "S1 —
 * SharedKVPool": one shared prefix plus a private suffix per agent).
 * k_f16, v_f16: device fp16 [batch][n_kv_heads][capacity][D], 16-byte aligned.
 * Other arguments as attn_decode.
 */
CKV_API size_t ckv_attn_decode_f16_workspace(int32_t head_dim, int32_t n_kv_heads, int32_t batch,
                                     int64_t max_seq_len, int32_t n_q, int32_t n_q_heads,
                                     int32_t n_split);
CKV_API ckv_status ckv_attn_decode_f16(const void* k_f16, const void* v_f16, int32_t head_dim,
                               int32_t n_kv_heads, int32_t batch, int64_t capacity,
                               const int32_t* seq_len, int64_t max_seq_len, const void* q_f16,
                               int32_t n_q, int32_t n_q_heads, float scale, int32_t n_split,
                               float* out, float* lse, void* workspace, size_t ws_bytes,
                               void* stream);

/*
 * attn_decode_f16_merge — attn_decode_f16 whose split merge also takes in one
 * prior partial per output row, computed over other keys: the result is the
 * attention over the union of the two key sets (the exact log-sum-exp combine
 * of lse_merge, done inside the decode's own merge, so no separate merge
 * launch). For the shared-pool fan-out, the prior is each agent's attention
 * over the shared compressed prefix and the fp16 keys are its private tail
 * (PolyKV page, section "S1 — SharedKVPool": shared prefix plus private
 * suffix; DCA page, "Implementation progress + Section-D simplification":
 * partials packed with their per-row lse and combined by the LSE merge).
 * prior_o: device fp32 rows laid out as out ([batch][n_q][n_q_heads][D],
 * 16-byte aligned), prior_lse as lse; an empty prior row has lse -inf. Neither
 * may alias out or lse. Workspace: ckv_attn_decode_f16_merge_workspace (one
 * more merge slot per row group than attn_decode_f16). Other arguments and
 * errors as attn_decode_f16.
 * Ordering: the kernel streams K, V and Q (and reads seq_len) before it waits
 * for the previous kernel on the stream, and waits only before it merges, so
 * that a prefix decode launched just before it (which writes prior_o and
 * prior_lse) overlaps its tail pass. So K, V, Q and seq_len must not be
 * written by the kernel just before it on the stream; kernels that write them
 * (ckv_f16_append, kv_pack, the caller's own) are fully ordered before it as
 * usual, because only this library's decode kernels let a following kernel
 * start early, and only after their own wait.
 */
CKV_API size_t ckv_attn_decode_f16_merge_workspace(int32_t head_dim, int32_t n_kv_heads, int32_t batch,
                                                   int64_t max_seq_len, int32_t n_q, int32_t n_q_heads,
                                                   int32_t n_split);
CKV_API ckv_status ckv_attn_decode_f16_merge(const void* k_f16, const void* v_f16, int32_t head_dim,
                                             int32_t n_kv_heads, int32_t batch, int64_t capacity,
                                             const int32_t* seq_len, int64_t max_seq_len, const void* q_f16,
                                             int32_t n_q, int32_t n_q_heads, float scale, int32_t n_split,
                                             const float* prior_o, const float* prior_lse, float* out, float* lse,
                                             void* workspace, size_t ws_bytes, void* stream);

/*
 * fanout_plan — split counts for the shared-pool fan-out step (PolyKV page,
 * section "S1 — SharedKVPool"): the prefix decode (ckv_attn_decode over the
 * shared cache, batch 1, the n_agents agents' single query tokens as n_q =
 * n_agents) followed on the same stream by ckv_attn_decode_f16_merge over the
 * agents' private fp16 tails (batch n_agents, n_q 1). The tail grid streams
 * its tails on the SMs that the prefix grid leaves free and waits for it only
 * to merge, so the two run side by side: the plan gives the tail pass one
 * split per (agent, kv head) row group and the prefix pass as many splits per
 * row group as fit on the remaining SMs of the current device. When the tail
 * grid alone would take half of the SMs or more, both counts are 0 (each
 * call's own automatic choice). This is a host computation: it launches
 * nothing. Errors: CKV_ERR_INVALID_ARG for non-positive counts or null
 * outputs, CKV_ERR_UNSUPPORTED if n_q_heads is not a multiple of n_kv_heads,
 * CKV_ERR_CUDA if the device cannot be queried.
 */
CKV_API ckv_status ckv_fanout_plan(int32_t n_agents, int32_t n_kv_heads, int32_t n_q_heads,
                                   int32_t* prefix_splits, int32_t* tail_splits);

/*
 * attn_decode_fanout — one decode step of the shared-pool fan-out (PolyKV
 * page, section "S1 — SharedKVPool": one compressed prefix counted once, a
 * private fp16 suffix per agent; DCA page, "Implementation progress +
 * Section-D simplification": partials over disjoint key sets combined by the
 * LSE merge). Agent a's query token (n_q_heads heads) attends the prefix
 * positions [0, prefix_len[0]) of `prefix` (a packed cache of one sequence)
 * and its own tail positions [0, tail_len[a]). Two launches: the prefix
 * decode (the agents as n_agents query tokens of one sequence) writes its
 * split partials and no output; the fp16 tail decode, with the split counts
 * of ckv_fanout_plan so that it runs beside the prefix decode on the SMs it
 * leaves free, merges its own partial with the prefix decode's partials of
 * the same 8 rows in its split merge. When that form does not apply (the
 * tile path's cost model picks 128-row tiles for a long prefix, the tail grid
 * does not fit on the device at once, or ckv_set_concurrent_kernels is on)
 * the step runs as ckv_attn_decode into the workspace followed by
 * ckv_attn_decode_f16_merge; the result is the same attention.
 * n_q_heads must be 8 * prefix->n_kv_heads (one row group of 8 query heads
 * per agent and kv head), else CKV_ERR_UNSUPPORTED: compose ckv_attn_decode
 * and ckv_attn_decode_f16_merge instead.
 * prefix_len: device int32 [1], <= max_prefix_len <= prefix capacity.
 * k_tail, v_tail: device fp16 [n_agents][n_kv_heads][tail_capacity][D]
 * (tail_capacity a multiple of 16); tail_len: device int32 [n_agents], each
 * <= max_tail_len <= tail_capacity. q_f16: device fp16 [n_agents][n_q_heads][D].
 * out: float32 [n_agents][n_q_heads][D]; lse: float32 [n_agents][n_q_heads].
 * workspace: ckv_attn_decode_fanout_workspace bytes (0: invalid geometry),
 * 256-byte aligned, zero-filled before first use and left reusable by each
 * call; ckv_read_device_flag on it reports both launches' device errors.
 * Ordering as ckv_attn_decode_f16_merge: K, V, Q and tail_len must not be
 * written by the kernel just before this call on the stream.
 */
CKV_API size_t ckv_attn_decode_fanout_workspace(const ckv_cache* prefix, int64_t max_prefix_len,
                                                int32_t n_agents, int64_t max_tail_len, int32_t n_q_heads);
CKV_API ckv_status ckv_attn_decode_fanout(const ckv_cache* prefix, const int32_t* prefix_len,
                                          int64_t max_prefix_len, const void* k_tail, const void* v_tail,
                                          int64_t tail_capacity, const int32_t* tail_len, int64_t max_tail_len,
                                          int32_t n_agents, const void* q_f16, int32_t n_q_heads, float scale,
                                          float* out, float* lse, void* workspace, size_t ws_bytes,
                                          void* stream);

/*
 * lse_merge — exact merge of n_parts normalised partials computed over
 * disjoint key sets (DCA page, "Implementation progress + Section-D
 * simplification": M = max lse_r, w_r = exp(lse_r - M), O = sum w_r O_r / sum w_r,
 * lse = M + ln sum w_r). Partials with lse = -inf weigh 0; all empty -> O = 0,
 * lse = -inf.
 * o_parts, lse_parts: HOST arrays of n_parts DEVICE pointers, each o part
 * float32 [n_rows][d], each lse part float32 [n_rows]. 1 <= n_parts <= 16.
 * out: float32 [n_rows][d]; lse: float32 [n_rows] (may alias a part).
 */
CKV_API ckv_status ckv_lse_merge(int32_t n_parts, const float* const* o_parts,
                         const float* const* lse_parts, int64_t n_rows, int32_t d,
                         float* out, float* lse, void* stream);

/*
 * attn_prefill — chunked prefill: pack n_new new K/V rows of every sequence at
 * positions [n_cached, n_cached + n_new) (as kv_pack), then causal attention of
 * the n_new queries over the packed cache: query i sees positions
 * [0, n_cached + i] (the cache stores what the packer is handed and attention
 * reads it back). S = Q K_hat^T and P V_hat run on tcgen05 tensor cores.
 * q_bf16: device bf16 [batch][n_new][n_q_heads][D]. k_new_f16, v_new_f16: device
 * fp16 [batch][n_new][n_kv_heads][D]. out: float32 [batch][n_new][n_q_heads][D];
 * lse: float32 [batch][n_new][n_q_heads]. head_dim 64, 128, 256 or 512 and
 * the query-to-kv head ratio dividing 128, else CKV_ERR_UNSUPPORTED. Every V
 * tier (v_bits 2, 3, 4) and both rotations (v_signs2 NULL, or the
 * block-diagonal one at head_dim >= 128) are read; positions past
 * n_cached + n_new may hold any bytes.
 */
CKV_API size_t ckv_attn_prefill_workspace(const ckv_cache* cache, int32_t n_new, int32_t n_q_heads);
CKV_API ckv_status ckv_attn_prefill(const ckv_cache* cache, int64_t n_cached, const void* q_bf16,
                            int32_t n_new, int32_t n_q_heads, const void* k_new_f16,
                            const void* v_new_f16, float scale, float* out, float* lse,
                            void* workspace, size_t ws_bytes, void* stream);

/*
 * attn_prefill_prefix — every one of n_q_tokens query tokens attends to the
 * whole packed prefix [0, n_prefix) of each sequence (no causal limit, nothing
 * packed): the shared-pool part of a multi-tenant prefill, where the queries of
 * several agents that share one compressed prefix run as one sequence (PolyKV
 * page, section "S1 — SharedKVPool": shared prefix cells are attended by every
 * agent). Same kernels, arguments, layouts, limits and workspace
 * (ckv_attn_prefill_workspace(cache, n_q_tokens, n_q_heads)) as
 * ckv_attn_prefill; n_prefix in [1, capacity].
 */
CKV_API ckv_status ckv_attn_prefill_prefix(const ckv_cache* cache, int64_t n_prefix, const void* q_bf16,
                                   int32_t n_q_tokens, int32_t n_q_heads, float scale, float* out,
                                   float* lse, void* workspace, size_t ws_bytes, void* stream);

/*
 * f16_append — copy n_new rows per sequence into dense fp16 K/V caches laid out
 * [batch][n_kv_heads][capacity][D] (the layout of ckv_attn_decode_f16) at
 * positions [seq_len[b] - n_new, seq_len[b]); seq_len (device, int32 [batch])
 * counts the new rows. Rows whose position falls outside [0, capacity) are
 * skipped. k_new/v_new: fp16 with the strides of ckv_kv_pack.
 */
CKV_API ckv_status ckv_f16_append(void* k_f16, void* v_f16, int32_t head_dim, int32_t n_kv_heads,
                          int32_t batch, int64_t capacity, const int32_t* seq_len,
                          const void* k_new_f16, const void* v_new_f16, int32_t n_new,
                          int64_t token_stride, int64_t batch_stride, void* stream);

/*
 * attn_prefill_f16 — causal prefill over dense fp16 caches (a private,
 * uncompressed per-agent tail: PolyKV page, section "S1 — SharedKVPool", the
 * private suffix): query token i of n_new sees positions [0, seq_len[b] - n_new
 * + i] (the new rows are the sequence's last n_new positions, already in the
 * cache). q_bf16: bf16 [batch][n_new][n_q_heads][D], converted exactly to fp16
 * for the tensor cores (|q| < 65504). Runs the fp16 decode kernel with n_new
 * query tokens; workspace as ckv_attn_decode_f16_workspace(..., n_q = n_new, ...).
 */
CKV_API ckv_status ckv_attn_prefill_f16(const void* k_f16, const void* v_f16, int32_t head_dim,
                                int32_t n_kv_heads, int32_t batch, int64_t capacity,
                                const int32_t* seq_len, int64_t max_seq_len, const void* q_bf16,
                                int32_t n_new, int32_t n_q_heads, float scale, int32_t n_split,
                                float* out, float* lse, void* workspace, size_t ws_bytes, void* stream);

/*
 * attn_prefill_shared — multi-tenant prefill over a shared compressed prefix
 * plus private fp16 tails (PolyKV page, section "S1 — SharedKVPool": one
 * shared prefix counted once, a private suffix per agent). n_agents agents each
 * prefill n_new tokens; query token i of agent a sees the whole prefix
 * [0, n_prefix) of `prefix` (a packed cache holding one sequence, batch 1) and
 * its own tail positions [0, tail_len[a] - n_new + i]. Steps, all on the device:
 * the new K/V rows are copied into the tails (ckv_f16_append), the prefix part
 * runs as one sequence of n_agents * n_new query tokens
 * (ckv_attn_prefill_prefix), and the tail part runs causally with the prefix
 * partial of every row merged exactly into its epilogue (the kernel of
 * ckv_attn_decode_f16_merge, bf16 queries); n_prefix = 0 leaves only the tail
 * part. Three launches.
 * k_tail, v_tail: fp16 [n_agents][Hkv][tail_capacity][D] (written: new rows).
 * tail_len: device int32 [n_agents], each tail's length counting the new rows.
 * q_bf16: [n_agents][n_new][n_q_heads][D]; k_new_f16, v_new_f16: fp16
 * [n_agents][n_new][Hkv][D]; out: float32 [n_agents][n_new][n_q_heads][D];
 * lse: float32 [n_agents][n_new][n_q_heads]. Head dim, head ratio and the V
 * format follow ckv_attn_prefill.
 */
CKV_API size_t ckv_attn_prefill_shared_workspace(const ckv_cache* prefix, int32_t n_agents,
                                         int64_t tail_capacity, int32_t n_new, int32_t n_q_heads);
CKV_API ckv_status ckv_attn_prefill_shared(const ckv_cache* prefix, int64_t n_prefix, void* k_tail,
                                   void* v_tail, int64_t tail_capacity, const int32_t* tail_len,
                                   int32_t n_agents, const void* q_bf16, const void* k_new_f16,
                                   const void* v_new_f16, int32_t n_new, int32_t n_q_heads,
                                   float scale, float* out, float* lse, void* workspace,
                                   size_t ws_bytes, void* stream);

/*
 * set_concurrent_kernels — declare (on != 0) that other kernels may run on the
 * device at the same time as this library's, e.g. on another stream or in
 * another process under MPS; process-wide, default off. A split decode whose
 * grid fits on the device merges its splits by a rendezvous in which every
 * CTA waits for the others; with other kernels holding SMs, part of the grid
 * may not be resident and the wait would run out (2 s, device flag 1, rows
 * left unmerged). With this set, the split decodes use the tree merge, in
 * which no CTA waits for another (slower: about 30 against 21 us for the
 * Gemma-4 step). Takes effect for launches after the call.
 */
CKV_API void ckv_set_concurrent_kernels(int32_t on);

/* Synchronously read the device flag (first 4 bytes of a workspace) after draining
 * `stream`. *flag receives it; when it is nonzero the flag is cleared and
 * CKV_ERR_DEVICE_FLAG returned. */
CKV_API ckv_status ckv_read_device_flag(const void* workspace, int32_t* flag, void* stream);

/* Message for the last failure on the calling thread ("" if none). */
CKV_API const char* ckv_last_error(void);

/* Library ABI version (major * 100 + minor). */
CKV_API int32_t ckv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CKV_H */
