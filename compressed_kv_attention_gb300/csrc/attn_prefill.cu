// attn_prefill.cu — chunked causal prefill over the packed cache on tcgen05.
//
// PolyKV page ("F5 M6 — PolyKV (shared compressed KV pool)"), section "S2
// perf-path Level B": large-n_q prefill over turbo KV is a tensor-core job
// (the vector kernel is 2-3x slower than f16 MMA there). Here the n_new new
// K/V rows are packed first (q8_0 / TBQ3, as kv_pack), then every query tile
// attends over the packed cache through fifth-generation tensor cores.
//
// One CTA owns 128 query rows (128 / G query tokens x G heads of one kv head)
// and walks the cache in 64-token steps:
//   S  = Q K_hat^T        M = 128, N = 64, K = D, in TMEM columns [0, 64).
//        K_hat = q * d16 has up to 18 significant bits, so it enters the tensor
//        core as an exact fp16 pair hi + lo (two passes of MMAs into the same
//        accumulator); Q is bf16, which converts to fp16 exactly.
//   online softmax, one row per thread (warps 0-3), the running max moving
//        only when it grows by more than 2^4 (O in TMEM is rescaled then);
//        P' = p * norm as fp16 into shared memory.
//   O += P' C             C = the Lloyd-Max centroids of the V codes (the
//        rotated basis); dims [0, 448) accumulate in TMEM columns [64, 512); at
//        D = 512 the last 64 dims go through columns [0, 64) each step and are
//        summed in registers.
// Operands live in shared memory in the 128-byte-swizzle K-major layout. The
// output leaves the kernel normalised but still in the rotated basis; a
// per-row kernel then applies the inverse Walsh-Hadamard transform and the
// sign flip in place (the transform runs once per output row, never on the
// cache).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <type_traits>

#include "../../include/ckv.h"
#include "ckv_kernels.cuh"

namespace ckv {

namespace {

struct PrefillArgs {
  const uint8_t* cache;
  int64_t capacity;
  int n_kv_heads, batch;
  int64_t n_cached;
  int n_new, n_q_heads;
  // 0: causal chunked prefill (query i sees [0, n_cached + i]); 1: every query
  // sees exactly [0, n_cached) (queries of other sequences over a shared prefix).
  int prefix_only;
  const __nv_bfloat16* q;  // [batch][n_new][n_q_heads][D]
  float scale_log2;
  float* out;              // [batch][n_new][n_q_heads][D]
  float* lse;              // [batch][n_new][n_q_heads]
  int32_t* flag;
  // Stream-K schedule (stream_k = 1): CTA c takes the 64-key steps
  // [c W / grid, (c + 1) W / grid) of all tiles laid end to end (tile
  // t = (b * n_kv_heads + kv_head) * n_q_tiles + q_tile); a tile is cut at
  // most once. The part before a cut at CTA c goes to slot 2c, the part after
  // it to slot 2c + 1 (slot: [128 rows][D] normalised rotated-basis rows, then
  // [128] lse), and tile_split[t] = c; whole tiles write their rows to `out`
  // and tile_split[t] = -1. Otherwise (stream_k = 0) CTA t runs tile t.
  int stream_k;
  float* part;
  int32_t* tile_split;
  // Decode over many query rows (n_split > 0, with prefix_only = 1): the
  // queries of sequence b see [0, seq_len[b]) (device array, each entry in
  // [0, n_cached]); CTA c runs tile c / n_split over its share c % n_split of
  // the ceil(n_cached / 64) steps and writes its rows to slot c; the
  // de-rotation kernel merges a row's n_split slots.
  const int32_t* seq_len;
  int n_split;
  int q_f16;  // queries are fp16 (else bf16)
};

// B: bits per V code (2, 3 or 4). ROT: the block-diagonal rotation (one V
// norm per 128-dim group and position; the norms then scale the centroids in
// C^T instead of entering P').
template <int D, int B, bool ROT>
struct PCfg {
  static constexpr int M = 128;                  // query rows per CTA
  static constexpr int NKV = 64;                 // cached tokens per step
  static constexpr int NB = D / 32;              // q8_0 blocks per vector
  static constexpr int OT = D < 448 ? D : 448;   // output dims accumulated in TMEM
  static constexpr int OR = D - OT;              // output dims summed in registers (0 or 64)
  static constexpr int NG = ROT ? D / kRotGroup : 1;
  static constexpr int REC = record_bytes(D, B, NG);
  // Value table: 3 bits, 64 entries, one per 6-bit field (a pair of codes);
  // 2 bits, 16 entries per 4-bit field; 4 bits, 16 entries, one per code
  // (two loads per field).
  static constexpr int LUT_N = B == 3 ? 64 : 16;
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = M * D * 2;                 // K_hat hi, then lo, then C^T
  static constexpr int P_OFF = KV_OFF + NKV * D * 2;
  static constexpr int NORM_OFF = P_OFF + M * NKV * 2;
  static constexpr int LUT_OFF = NORM_OFF + NKV * 4;        // LUT_N table words x 32 lanes
  static constexpr int SCALE_OFF = LUT_OFF + LUT_N * 32 * 4; // two steps' q8_0 scales
  // Up to head dim 128, P' enters the P.V product as the fp16 pair hi (P_OFF)
  // + lo (P_LO_OFF): fp16 rounding of P' alone costs up to 2.7e-3 of |o|_inf
  // at head dim 64 over long rows (2.1e-3 at 128; 1.4e-3 at 256, 8e-4 at 512).
  static constexpr bool PSPLIT = D <= 128;
  static constexpr int P_LO_OFF = (SCALE_OFF + 2 * NKV * NB * 2 + 1023) / 1024 * 1024;
  static constexpr int BYTES = PSPLIT ? P_LO_OFF + M * NKV * 2 : SCALE_OFF + 2 * NKV * NB * 2;
  // At least half the SM's shared memory, so that one CTA (and its 512 TMEM
  // columns) owns each SM.
  static constexpr int SMEM = (BYTES + 1024 > 120 * 1024 ? BYTES + 1024 : 120 * 1024);
  static constexpr int THREADS = 256;
};

// TMEM column of output dim chunk c, and the chunks' (first dim, width, column):
// dims [0, 256) -> column 64, dims [256, OT) -> column 320, dims [OT, D) -> column 0.
struct OChunk {
  int dim0, n, col;
};

}  // namespace

// SPLIT: the split many-row decode (one segment per CTA, keys per sequence
// from seq_len); otherwise the causal or prefix-only prefill, whose key end is
// a launch constant (kept out of shared memory: the step loop reads it).
template <int D, int B, bool ROT, bool SPLIT>
__global__ void __launch_bounds__(256, 1) attn_prefill_kernel(PrefillArgs a) {
  using C = PCfg<D, B, ROT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sQ = smem + C::Q_OFF;
  uint8_t* sKV = smem + C::KV_OFF;
  uint8_t* sP = smem + C::P_OFF;
  float* sNorm = reinterpret_cast<float*>(smem + C::NORM_OFF);
  uint32_t* sLut = reinterpret_cast<uint32_t*>(smem + C::LUT_OFF);
  __half* sScale = reinterpret_cast<__half*>(smem + C::SCALE_OFF);

  const int group_q = a.n_q_heads / a.n_kv_heads;
  const int QT = C::M / group_q;  // query tokens per tile
  const int n_qt = (a.n_new + QT - 1) / QT;
  const int64_t n_rec = a.capacity / kTile;
  // 64-key steps of query tile qt: its rows see keys [0, n_cached + last row]
  // (prefix_only: [0, n_cached)).
  auto steps_of = [&](int qt) {
    const int64_t kv_end = a.prefix_only ? a.n_cached : a.n_cached + min((qt + 1) * QT, a.n_new);
    return static_cast<int>((kv_end + C::NKV - 1) / C::NKV);
  };

  // The tile being run, set per segment (CTA-uniform, kept in shared memory
  // so that the step loop does not hold it in registers). s_kv_end: the end
  // of the keys every query sees (prefix_only) and of the packed rows; the
  // positions after it in the last step may hold any bytes, so their V norms
  // enter as zero (a NaN there would reach O through P' = 0).
  __shared__ int s_q0, s_kvh, s_b, s_s0;
  __shared__ long long s_kv_end;  // SPLIT only
  // The key end of the other modes, read from the launch arguments at each use.
  auto kv_end_const = [&]() -> int64_t { return a.prefix_only ? a.n_cached : a.n_cached + a.n_new; };
  __shared__ const uint8_t* s_stream;
  __shared__ float* s_slot;  // nullptr: rows to `out`

  // Split decode: the sequence length of this CTA's tile, loaded now so that
  // its latency overlaps the setup below.
  int split_len = 0;
  if constexpr (SPLIT) {
    if (tid == 0) {
      const int64_t bh = (blockIdx.x / a.n_split) / n_qt;
      split_len = a.seq_len[bh / a.n_kv_heads];
    }
  }
  if (warp == 0) tmem_alloc(&s_tmem, 512);
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  // Value table, one copy per lane, in units of the tier's centroid scale
  // (the de-rotation multiplies it back). 3 bits: entry f (6 bits) =
  // fp16x2(c[f & 7], c[f >> 3]); 2 bits: entry f (4 bits) = fp16x2(c[f & 3],
  // c[f >> 2]); 4 bits: entry k = fp16x2(c[k], c[k]).
  for (int e = tid; e < C::LUT_N * 32; e += C::THREADS) {
    const int f = e >> 5;
    constexpr float inv = 1.0f / centroid_scale(B);
    if constexpr (B == 3)
      sLut[e] = pack_half2(tbq_centroid<3>(f & 7) * inv, tbq_centroid<3>(f >> 3) * inv);
    else if constexpr (B == 2)
      sLut[e] = pack_half2(tbq_centroid<2>(f & 3) * inv, tbq_centroid<2>(f >> 2) * inv);
    else
      sLut[e] = pack_half2(tbq_centroid<4>(f) * inv, tbq_centroid<4>(f) * inv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t q_base = smem_u32(sQ), kv_base = smem_u32(sKV), p_base = smem_u32(sP);

  // ---- Q tile: bf16 -> fp16 (exact in range), 128-byte swizzled K-major ----
  // fp16 queries arrive by asynchronous copies that the caller waits for
  // (q_wait) after issuing the first step's code loads, so the two overlap.
  // Many CTAs load the same tile at once (the splits of a many-row decode):
  // each starts its walk over the tile's 16-byte pieces at its own offset, so
  // that they do not all request the same L2 lines together.
  constexpr int QPIECES = C::M * (D / 8);
  const int q_rot = static_cast<int>((blockIdx.x * 37u) % (QPIECES / C::THREADS)) * C::THREADS;
  auto load_q = [&]() {
  if (a.q_f16) {
    // fp16 queries go to shared memory as they are: 16-byte asynchronous
    // copies, all in flight at once (a split decode runs few steps per CTA,
    // so this load is not amortised).
    for (int pc = tid; pc < QPIECES; pc += C::THREADS) {
      const int piece = pc + q_rot < QPIECES ? pc + q_rot : pc + q_rot - QPIECES;
      const int r = piece / (D / 8), k0 = (piece % (D / 8)) * 8;
      const int qi = s_q0 + r / group_q, h = s_kvh * group_q + r % group_q;
      const uint32_t dst = smem_u32(sQ + sw128_offset(r, k0, C::M));
      if (qi < a.n_new) {
        const void* src = a.q + (((int64_t)s_b * a.n_new + qi) * a.n_q_heads + h) * D + k0;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
      } else {
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    return;
  }
  for (int piece = tid; piece < C::M * (D / 8); piece += C::THREADS) {
    const int r = piece / (D / 8), k0 = (piece % (D / 8)) * 8;
    const int qi = s_q0 + r / group_q, h = s_kvh * group_q + r % group_q;
    uint4 outv = make_uint4(0, 0, 0, 0);
    if (qi < a.n_new) {
      const uint4 v =
          *reinterpret_cast<const uint4*>(a.q + (((int64_t)s_b * a.n_new + qi) * a.n_q_heads + h) * D + k0);
      if (a.q_f16) {
        outv = v;
      } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
          o[i] = pack_half2(__low2float(x), __high2float(x));
        }
        outv = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    *reinterpret_cast<uint4*>(sQ + sw128_offset(r, k0, C::M)) = outv;
  }
  };

  // Rows: warps 0-3, thread = row (query token s_q0 + row / G, head row % G).
  const bool softmax_warp = warp < 4;
  const int row = tid & 127;
  const uint32_t row_tmem = tmem + ((uint32_t)(warp & 3) * 32u << 16);

  uint32_t phase = 0;
  auto wait_mma = [&]() {
    if (!*(volatile int*)&s_abort) {
      if (!mbar_wait(&s_bar, phase & 1)) {
        *(volatile int*)&s_abort = 1;
        raise_flag(a.flag, kFlagWaitTimeout);
      }
    }
    ++phase;
    tc_fence_after();
  };
  auto sync_for_mma = [&]() {  // generic-proxy shared writes and TMEM stores -> tensor core
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };
  auto issue_s = [&]() {  // S (+)= Q K^T over D, from the K tile in sKV
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint64_t ad = umma_desc_sw128(q_base + (ks >> 2) * (C::M * 128) + (ks & 3) * 32);
      const uint64_t bd = umma_desc_sw128(kv_base + (ks >> 2) * (C::NKV * 128) + (ks & 3) * 32);
      umma_f16(tmem, ad, bd, umma_idesc_f16_f32(C::M, C::NKV), true);
    }
  };
  const OChunk chunks[3] = {{0, C::OT < 256 ? C::OT : 256, 64},
                            {256, C::OT > 256 ? C::OT - 256 : 0, 320},
                            {C::OT, C::OR, 0}};

  // Codes of a step are fetched into registers one step ahead, so their
  // global-memory latency overlaps the rest of the previous step.
  //  K: the step's 4 records hold 4D 16-byte code chunks; round r of warp w
  //     loads chunks [256r + 32w, +32), one (record, 32-dim block) with its
  //     32 lanes L, 512 contiguous bytes. Lane l takes L = 4 (l & 7) + (l >> 3):
  //     the chunk holds 8 dims of tokens l & 7 and (l & 7) + 8, and a quarter
  //     warp (fixed l >> 3) then stores 8 rows of one swizzle column, which
  //     land on distinct bank groups. The scales go to shared memory.
  //  V: threads 128..255; warp w takes lane streams [8w, 8w + 8) of the
  //     step's 4 records (lane = 8 * record + stream), which spreads one
  //     store instruction over 16 banks.
  constexpr int G = D / 8, LB = v_lane_bytes(D, B), GR = v_granule(D, B), NW = LB / 4;
  constexpr int KR = 4 * D / C::THREADS;    // code chunks per thread per step
  constexpr int NSW = C::NKV * C::NB / 4;   // 8-byte scale words per step
  constexpr int VPRE = G;                   // value fields whose table loads overlap the second S pass
  static_assert(NSW <= C::THREADS, "one scale word per thread");
  const int kq = lane >> 3, kpp = lane & 7;
  const int vu = tid - 128, vr4 = (vu & 31) >> 3, vL = 8 * (vu >> 5) + (vu & 7);
  uint4 kw[KR];
  uint2 ksc = make_uint2(0, 0);
  float nrm = 0.0f;
  auto fetch = [&](int step) {
    const uint8_t* stream = s_stream;
    const int64_t rec0 = (int64_t)step * (C::NKV / kTile);
#pragma unroll
    for (int r = 0; r < KR; ++r) {
      const int g = r * C::THREADS + warp * 32;
      const int64_t rec = rec0 + g / D;
      const int blk = (g % D) / 32;
      kw[r] = rec < n_rec ? *reinterpret_cast<const uint4*>(stream + rec * C::REC + (blk * 32 + 4 * kpp + kq) * 16)
                          : make_uint4(0, 0, 0, 0);
    }
    if (tid < NSW) {
      const int h0 = tid * 4;  // first of the word's 4 scales, [record][token][block] order
      const int64_t rec = rec0 + h0 / (kTile * C::NB);
      ksc = rec < n_rec ? *reinterpret_cast<const uint2*>(stream + rec * C::REC + k_scale_offset(D) +
                                                          2 * (h0 % (kTile * C::NB)))
                        : make_uint2(0, 0);
    }
    if (!ROT && tid < C::NKV) {
      const int64_t rec = rec0 + tid / kTile;
      nrm = (rec < n_rec && rec0 * kTile + tid < (SPLIT ? s_kv_end : kv_end_const()))
                ? __half2float(*reinterpret_cast<const __half*>(stream + rec * C::REC + v_norm_offset(D, B) +
                                                                2 * (tid % kTile)))
                : 0.0f;
    }
  };
  // V codes of a step (value warps), loaded once the previous step's build
  // has consumed them. ROT: also the thread's group norms of positions
  // (p0, p0 + 1) and (p0 + 8, p0 + 9), p0 = 2 (vL & 3), as fp16 pairs (its
  // dims [G (vL >> 2), + G) lie in one 128-dim group).
  auto fetch_v = [&](uint32_t (&vw)[NW], uint32_t (&vn)[2], int step) {
    const uint8_t* stream = s_stream;
    const int64_t rec0 = (int64_t)step * (C::NKV / kTile);
    if constexpr (ROT) {
      const int64_t rec = rec0 + vr4;
      const int p0 = 2 * (vL & 3), grp = G * (vL >> 2) / kRotGroup;
      const uint8_t* nb = stream + rec * C::REC + v_norm_offset(D, B) + 2 * (kTile * grp + p0);
      const int64_t r = (SPLIT ? s_kv_end : kv_end_const()) - rec * kTile - p0;  // positions p0 + i, i < r, hold rows
      vn[0] = (rec < n_rec && r > 0) ? *reinterpret_cast<const uint32_t*>(nb) & (r >= 2 ? 0xffffffffu : 0xffffu)
                                     : 0u;
      vn[1] = (rec < n_rec && r > 8) ? *reinterpret_cast<const uint32_t*>(nb + 16) & (r >= 10 ? 0xffffffffu : 0xffffu)
                                     : 0u;
    }
    {
      const int64_t rec = rec0 + vr4;
      const uint8_t* vb = stream + rec * C::REC + v_code_offset(D);
      if constexpr (GR == 16) {
#pragma unroll
        for (int k = 0; k < NW / 4; ++k) {
          const uint4 v = (rec < n_rec) ? *reinterpret_cast<const uint4*>(vb + (k * 32 + vL) * 16)
                                        : make_uint4(0, 0, 0, 0);
          vw[4 * k] = v.x;
          vw[4 * k + 1] = v.y;
          vw[4 * k + 2] = v.z;
          vw[4 * k + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int s4 = 0; s4 < NW; ++s4) {
          const int sbyte = s4 * 4;
          vw[s4] = (rec < n_rec)
                       ? *reinterpret_cast<const uint32_t*>(vb + ((sbyte / GR) * 32 + vL) * GR + (sbyte % GR))
                       : 0u;
        }
      }
    }
  };
  // Scales of a fetched step into buffer `buf` (read after the next barrier).
  auto put_scales = [&](int buf) {
    if (tid < NSW) *reinterpret_cast<uint2*>(sScale + buf * C::NKV * C::NB + tid * 4) = ksc;
  };

  // C^T (centroids, rotated basis): rows = dims, K = tokens. A field of 2B
  // bits pairs the codes of two adjacent positions of one dim (the even
  // position in the low bits), which is one fp16x2 word of C^T: one table
  // load per field at 2 and 3 bits, two at 4 bits (v_field), one store
  // (v_store). ROT: the word is scaled by the positions' group norms.
  const uint32_t v_lut = smem_u32(sLut) + (uint32_t)(lane << 2);
  const int v_g = vL >> 2, v_tok0 = vr4 * 16 + 2 * (vL & 3);
  auto v_field = [&](const uint32_t (&vc)[NW], int pi) -> uint32_t {
    if constexpr (B == 3) {
      const int bit = 6 * pi;
      const int wi = bit >> 5, sh = bit & 31;
      uint32_t f = vc[wi] >> sh;
      if (sh > 26 && wi + 1 < NW) f |= vc[wi + 1] << (32 - sh);
      return lds32(v_lut + ((f & 63u) << 7));
    } else if constexpr (B == 2) {
      const uint32_t f = (vc[pi >> 3] >> (4 * (pi & 7))) & 15u;
      return lds32(v_lut + (f << 7));
    } else {
      const uint32_t f = (vc[pi >> 2] >> (8 * (pi & 3))) & 255u;
      const uint32_t lo = lds32(v_lut + ((f & 15u) << 7)), hi = lds32(v_lut + ((f >> 4) << 7));
      return __byte_perm(lo, hi, 0x7610);  // (c[even], c[odd])
    }
  };
  auto v_store = [&](int pi, uint32_t val, const uint32_t (&vn)[2]) {
    const int mt = pi >> 2, rh = pi & 1, h2 = (pi >> 1) & 1;
    const int dim = G * v_g + 2 * mt + rh;
    const int tok = v_tok0 + 8 * h2;  // even position; the odd one follows it in K
    if constexpr (ROT) val = hmul2_u32(val, vn[h2]);
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(smem_u32(sKV) + sw128_offset(dim, tok, D)), "r"(val));
  };

  // The two roles run the same barriers and MMA waits; each role's state
  // (the softmax rows' running max, sum and register tail; the value warps'
  // code words) exists only on its own path.
  // Steps [s_s0, s1) of the current tile; the rows go to `out` (s_slot
  // nullptr) or to a partial slot of the stream-K schedule.
  auto role_loop = [&](auto role, int s1) {
    constexpr bool SM = decltype(role)::value;  // softmax warps (rows) or value warps
    float m_used = -INFINITY, l_sum = 0.0f;
    float otail[SM && C::OR > 0 ? C::OR : 1];
#pragma unroll
    for (int i = 0; i < (SM && C::OR > 0 ? C::OR : 1); ++i) otail[i] = 0.0f;
    uint32_t vw[SM ? 1 : NW];
    uint32_t vn[2] = {0u, 0u};
    if constexpr (!SM) {
      if (s_s0 < s1) fetch_v(vw, vn, s_s0);
    }
    for (int step = s_s0; step < s1; ++step) {
      const int64_t j0 = (int64_t)step * C::NKV;
      // ---- K_hat = q * d16 split into fp16 hi (to shared memory) + lo (kept) ----
      // q is an exact fp16 integer; hi = q*d rounded once (HMUL2 of exact fp16
      // operands) and lo = fma(q, d, -hi), the exact residual (HFMA2).
      uint32_t lo_keep[KR][8];
      const __half* scb = sScale + (step & 1) * C::NKV * C::NB;
#pragma unroll
      for (int r = 0; r < KR; ++r) {
        const int g = r * C::THREADS + warp * 32;
        const int blk = (g % D) / 32;
        const int row0 = (g / D) * kTile + kpp;  // tokens row0 and row0 + 8 of the step
        const uint32_t w[4] = {kw[r].x, kw[r].y, kw[r].z, kw[r].w};
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          const __half d = scb[(row0 + 8 * hs) * C::NB + blk];
          const __half2 dd = __halves2half2(d, d);
          uint32_t qh[4], hi[4];
          i8x4_to_half2x2(w[2 * hs], qh[0], qh[1]);
          i8x4_to_half2x2(w[2 * hs + 1], qh[2], qh[3]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __half2 qv = *reinterpret_cast<const __half2*>(&qh[e]);
            const __half2 h = __hmul2(qv, dd);
            const __half2 l = __hfma2(qv, dd, __hneg2(h));
            hi[e] = *reinterpret_cast<const uint32_t*>(&h);
            lo_keep[r][4 * hs + e] = *reinterpret_cast<const uint32_t*>(&l);
          }
          *reinterpret_cast<uint4*>(sKV + sw128_offset(row0 + 8 * hs, blk * 32 + 8 * kq, C::NKV)) =
              make_uint4(hi[0], hi[1], hi[2], hi[3]);
        }
      }
      if (!ROT && tid < C::NKV) sNorm[tid] = nrm;
      sync_for_mma();
      if (SM && tid == 0) {
        // First pass of S overwrites the accumulator (columns [0, 64)).
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t ad = umma_desc_sw128(q_base + (ks >> 2) * (C::M * 128) + (ks & 3) * 32);
          const uint64_t bd = umma_desc_sw128(kv_base + (ks >> 2) * (C::NKV * 128) + (ks & 3) * 32);
          umma_f16(tmem, ad, bd, umma_idesc_f16_f32(C::M, C::NKV), ks > 0);
        }
        umma_commit(&s_bar);
      }
      // The next step's loads are issued while the tensor core runs this pass;
      // warp 0, whose MMA issue blocks until the pass drains, loads during the
      // second pass instead (its softmax has slack against the value build).
      if (warp != 0 && step + 1 < s1) fetch(step + 1);
      wait_mma();
      // ---- lo pass ----
#pragma unroll
      for (int r = 0; r < KR; ++r) {
        const int g = r * C::THREADS + warp * 32;
        const int blk = (g % D) / 32;
        const int row0 = (g / D) * kTile + kpp;
#pragma unroll
        for (int hs = 0; hs < 2; ++hs)
          *reinterpret_cast<uint4*>(sKV + sw128_offset(row0 + 8 * hs, blk * 32 + 8 * kq, C::NKV)) =
              make_uint4(lo_keep[r][4 * hs], lo_keep[r][4 * hs + 1], lo_keep[r][4 * hs + 2], lo_keep[r][4 * hs + 3]);
      }
      sync_for_mma();
      if (SM && tid == 0) {
        issue_s();
        umma_commit(&s_bar);
      }
      if (warp == 0 && step + 1 < s1) fetch(step + 1);
      // While the second pass runs, the value warps load the table entries of
      // their first VPRE fields (the stores wait for the K tile to free).
      uint32_t vpre[SM ? 1 : VPRE];
      if constexpr (!SM) {
#pragma unroll
        for (int u = 0; u < VPRE; ++u) vpre[u] = v_field(vw, u);
      }
      wait_mma();
      if (step + 1 < s1) put_scales((step + 1) & 1);  // read after this step's last barrier

      if constexpr (SM) {
        // ---- online softmax of this step's 64 columns, one row per thread ----
        uint32_t sv[2][32];
        tmem_ld32(row_tmem + 0, sv[0]);
        tmem_ld32(row_tmem + 32, sv[1]);
        tmem_ld_wait();
        // Columns [0, nvis) are visible to the row: all of them except near the diagonal.
        const int row_qi = s_q0 + row / group_q;
        const int64_t rel = row_qi >= a.n_new     ? 0
                            : a.prefix_only ? (SPLIT ? s_kv_end : a.n_cached) - j0
                                            : a.n_cached + row_qi - j0 + 1;
        const int nvis = rel <= 0 ? 0 : (rel >= C::NKV ? C::NKV : static_cast<int>(rel));
        const bool all_vis = __all_sync(0xffffffffu, nvis == C::NKV);
        float x[C::NKV];
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < C::NKV; ++j) {
          const float v = __uint_as_float(sv[j >> 5][j & 31]) * a.scale_log2;
          x[j] = (all_vis || j < nvis) ? v : -INFINITY;
          mt = fmaxf(mt, x[j]);
        }
        const float m_new = fmaxf(m_used, mt);
        const bool need = (m_new > m_used + 4.0f);  // also true when m_used is -inf and a key is visible
        if (__any_sync(0xffffffffu, need)) {
          const float f = need ? ((m_used == -INFINITY) ? 0.0f : fast_exp2(m_used - m_new)) : 1.0f;
          if (step > s_s0) {
            // Rescale O in TMEM (initialised by the first P.V) and the register tail.
#pragma unroll 1
            for (int c0 = 64; c0 < 64 + C::OT; c0 += 32) {
              uint32_t ov[32];
              tmem_ld32(row_tmem + c0, ov);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
              tmem_st32(row_tmem + c0, ov);
            }
            tmem_st_wait();
          }
#pragma unroll
          for (int i = 0; i < C::OR; ++i) otail[i] *= f;
          l_sum *= f;
          if (need) m_used = m_new;
        }
        // With no visible key so far m_used is -inf and every x is -inf: all p are 0.
        const float mref = (m_used == -INFINITY) ? 0.0f : m_used;
        float ps = 0.0f;
        uint32_t pw[C::NKV / 2];
        [[maybe_unused]] uint32_t pwl[C::PSPLIT ? C::NKV / 2 : 1];
        const float4* n4 = reinterpret_cast<const float4*>(sNorm);
        auto pack_p = [&](int i, float y0, float y1) {  // P' pair i: fp16 hi, and lo when split
          pw[i] = pack_half2(y0, y1);
          if constexpr (C::PSPLIT) {
            const __half2 h = *reinterpret_cast<const __half2*>(&pw[i]);
            pwl[i] = pack_half2(y0 - __low2float(h), y1 - __high2float(h));
          }
        };
#pragma unroll
        for (int j = 0; j < C::NKV; j += 4) {
          const float4 nn = ROT ? make_float4(1.0f, 1.0f, 1.0f, 1.0f) : n4[j / 4];
          const float p0 = fast_exp2(x[j] - mref), p1 = fast_exp2(x[j + 1] - mref);
          const float p2 = fast_exp2(x[j + 2] - mref), p3 = fast_exp2(x[j + 3] - mref);
          ps += (p0 + p1) + (p2 + p3);
          pack_p(j / 2, p0 * nn.x, p1 * nn.y);
          pack_p(j / 2 + 1, p2 * nn.z, p3 * nn.w);
        }
        l_sum += ps;
#pragma unroll
        for (int c = 0; c < C::NKV / 8; ++c) {
          *reinterpret_cast<uint4*>(sP + sw128_offset(row, 8 * c, C::M)) =
              make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
          if constexpr (C::PSPLIT)
            *reinterpret_cast<uint4*>(smem + C::P_LO_OFF + sw128_offset(row, 8 * c, C::M)) =
                make_uint4(pwl[4 * c], pwl[4 * c + 1], pwl[4 * c + 2], pwl[4 * c + 3]);
        }
      } else {
        // ---- C^T for the step: the prefetched fields, then the rest ----
#pragma unroll
        for (int u = 0; u < VPRE; ++u) v_store(u, vpre[u], vn);
        // Table loads are issued in batches ahead of their stores, so one
        // shared-memory latency is exposed per batch rather than per field.
        constexpr int VB = G < 16 ? G : 16;  // divides the G fields left
#pragma unroll
        for (int pb = VPRE; pb < 2 * G; pb += VB) {
          uint32_t val[VB];
#pragma unroll
          for (int u = 0; u < VB; ++u) val[u] = v_field(vw, pb + u);
#pragma unroll
          for (int u = 0; u < VB; ++u) v_store(pb + u, val[u], vn);
        }
        if (step + 1 < s1) fetch_v(vw, vn, step + 1);
      }
      sync_for_mma();
      if (SM && tid == 0) {
        // ---- O += P' C over the step's 64 tokens ----
        for (int ks = 0; ks < C::NKV / 16; ++ks) {
          const uint64_t ad = umma_desc_sw128(p_base + ks * 32);
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            if (chunks[c].n == 0) continue;
            const uint64_t bd = umma_desc_sw128(kv_base + chunks[c].dim0 * 128 + ks * 32);
            const bool acc = (c == 2) ? (ks > 0) : (step > s_s0 || ks > 0);
            umma_f16(tmem + chunks[c].col, ad, bd, umma_idesc_f16_f32(C::M, chunks[c].n), acc);
            if constexpr (C::PSPLIT)  // the lo half of P' into the same accumulator
              umma_f16(tmem + chunks[c].col, umma_desc_sw128(smem_u32(smem + C::P_LO_OFF) + ks * 32), bd,
                       umma_idesc_f16_f32(C::M, chunks[c].n), true);
          }
        }
        umma_commit(&s_bar);
      }
      wait_mma();
      if constexpr (SM && C::OR > 0) {
        uint32_t tv[2][32];
        tmem_ld32(row_tmem + 0, tv[0]);
        tmem_ld32(row_tmem + 32, tv[1]);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < C::OR; ++i) otail[i] += __uint_as_float(tv[i >> 5][i & 31]);
      }
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }

    // ---- normalise and write the rotated-basis rows; lse ----
    // A thread holds one row, so row-wise global stores would scatter each
    // warp instruction over 32 rows. The rows pass through shared memory
    // instead (the Q tile, free after the last step until the next segment
    // loads its own), CW columns at a time, 16-byte units XOR-swizzled by the
    // row, and each warp then writes whole contiguous row pieces.
    if constexpr (SM) {
      constexpr int CW = D / 2 < 128 ? D / 2 : 128;  // columns per pass: 128 rows x CW floats fit in the Q tile
      constexpr int U = CW / 4;                     // 16-byte units per row piece
      constexpr int RPI = 32 / U;                   // rows one warp instruction covers
      const float inv = l_sum > 0.0f ? 1.0f / l_sum : 0.0f;
      float* const slot = s_slot;
      float* const sT = reinterpret_cast<float*>(sQ);
      static_assert(C::M * CW * 4 <= C::M * D * 2 && CW % 32 == 0, "transpose buffer");
      // Output row of tile row rr (nullptr: a row past the last query token).
      auto out_row = [&](int rr) -> float* {
        if (slot) return slot + (int64_t)rr * D;
        const int qi = s_q0 + rr / group_q;
        if (qi >= a.n_new) return nullptr;
        return a.out + (((int64_t)s_b * a.n_new + qi) * a.n_q_heads + s_kvh * group_q + rr % group_q) * D;
      };
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += CW) {
#pragma unroll
        for (int j = 0; j < CW; j += 32) {
          uint32_t ov[32];
          const int c = c0 + j;
          if (c < C::OT) {
            if (s_s0 < s1) {
              tmem_ld32(row_tmem + 64 + c, ov);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = 0u;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(otail[(c - C::OT + i) % (C::OR > 0 ? C::OR : 1)]);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int u = j / 4 + q;
            *reinterpret_cast<float4*>(sT + row * CW + 4 * (u ^ (row % U))) =
                make_float4(__uint_as_float(ov[4 * q]) * inv, __uint_as_float(ov[4 * q + 1]) * inv,
                            __uint_as_float(ov[4 * q + 2]) * inv, __uint_as_float(ov[4 * q + 3]) * inv);
          }
        }
        named_bar(1, 128);
        {
          const int sub = lane / U, ul = lane % U;
          for (int r0 = warp * 32; r0 < warp * 32 + 32; r0 += RPI) {
            const int rr = r0 + sub;
            float* orow = out_row(rr);
            const float4 v = *reinterpret_cast<const float4*>(sT + rr * CW + 4 * (ul ^ (rr % U)));
            if (orow) *reinterpret_cast<float4*>(orow + c0 + 4 * ul) = v;
          }
        }
        named_bar(1, 128);
      }
      float* orow = out_row(row);
      if (orow) {
        float* olse = slot ? slot + (int64_t)C::M * D + row
                           : a.lse + (((int64_t)s_b * a.n_new + s_q0 + row / group_q) * a.n_q_heads +
                                      s_kvh * group_q + row % group_q);
        *olse = l_sum > 0.0f ? (m_used + log2f(l_sum)) * 0.6931471805599453f : -INFINITY;
      }
    }
  };

  // ---- the CTA's step range, walked tile by tile ----
  // The walk state is uniform over the CTA and kept in shared memory (thread
  // 0 advances it), so the step loop does not carry it in registers.
  __shared__ long long s_walk[4];  // steps left, (sequence, kv head), query tile, first step
  if (tid == 0) {
    int64_t S_bh = 0;  // steps of all query tiles of one (sequence, kv head)
    for (int q = 0; q < n_qt; ++q) S_bh += steps_of(q);
    const int64_t n_bh = (int64_t)a.batch * a.n_kv_heads;
    if (a.stream_k) {
      const int64_t W = n_bh * S_bh;
      const int64_t w0 = (int64_t)blockIdx.x * W / gridDim.x;
      const int64_t w1 = (int64_t)(blockIdx.x + 1) * W / gridDim.x;
      const int64_t bh0 = S_bh > 0 ? w0 / S_bh : n_bh;
      int64_t rem = w0 - bh0 * S_bh;
      int q = 0;
      while (q < n_qt && rem >= steps_of(q)) rem -= steps_of(q++);
      s_walk[0] = w1 - w0;
      s_walk[1] = bh0;
      s_walk[2] = q;
      s_walk[3] = rem;
    } else {
      s_walk[0] = steps_of(static_cast<int>(blockIdx.x % n_qt));
      s_walk[1] = blockIdx.x / n_qt;
      s_walk[2] = blockIdx.x % n_qt;
      s_walk[3] = 0;
    }
  }
  __syncthreads();
  const int64_t n_bh = (int64_t)a.batch * a.n_kv_heads;
  if constexpr (SPLIT) {
    // One segment: tile blockIdx / n_split, share blockIdx % n_split of the steps.
    __shared__ int s_s1;
    if (tid == 0) {
      const int64_t t = blockIdx.x / a.n_split;
      const int sp = static_cast<int>(blockIdx.x % a.n_split);
      const int64_t bh = t / n_qt;
      const int qt = static_cast<int>(t % n_qt);
      const int b = static_cast<int>(bh / a.n_kv_heads);
      const int64_t S = (a.n_cached + C::NKV - 1) / C::NKV;
      int64_t len = split_len;
      if (len < 0 || len > a.n_cached) {
        raise_flag(a.flag, kFlagSeqLenRange);
        len = 0;
      }
      const int64_t sb = (len + C::NKV - 1) / C::NKV;  // steps this sequence has
      const int64_t s0 = sp * S / a.n_split;
      int64_t s1 = (sp + 1) * S / a.n_split;
      if (s1 > sb) s1 = sb;
      if (s1 < s0) s1 = s0;
      s_b = b;
      s_kvh = static_cast<int>(bh % a.n_kv_heads);
      s_q0 = qt * QT;
      s_s0 = static_cast<int>(s0);
      s_s1 = static_cast<int>(s1);
      s_kv_end = len;
      s_stream = a.cache + bh * n_rec * C::REC;
      s_slot = a.part + (int64_t)blockIdx.x * (C::M * (D + 1));
    }
    __syncthreads();
    const int s0 = s_s0, s1 = s_s1;
    load_q();
    if (s0 < s1) fetch(s0);
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (s0 < s1) put_scales(s0 & 1);
    __syncthreads();
    if (softmax_warp)
      role_loop(std::true_type{}, s1);
    else
      role_loop(std::false_type{}, s1);
  }
  if constexpr (!SPLIT) while (true) {
    const int64_t left = s_walk[0], bh = s_walk[1];
    const int qt = static_cast<int>(s_walk[2]), s0 = static_cast<int>(s_walk[3]);
    if (left <= 0 || bh >= n_bh) break;
    const int n_steps = steps_of(qt);
    const int s1 = (s0 + left < n_steps) ? static_cast<int>(s0 + left) : n_steps;
    const int64_t t = bh * n_qt + qt;
    float* slot = nullptr;  // this segment's rows: `out`, or a partial slot
    if (s0 > 0 || s1 < n_steps) {
      // Cut tile: the head part before the cut at CTA blockIdx + 1, the tail
      // part after the cut at this CTA.
      const int cut = (s0 == 0) ? blockIdx.x + 1 : blockIdx.x;
      if (!a.stream_k || (s0 > 0 && s1 < n_steps)) {
        if (tid == 0) raise_flag(a.flag, kFlagInternal);
        break;
      }
      slot = a.part + (int64_t)(2 * cut + (s0 == 0 ? 0 : 1)) * (C::M * (D + 1));
      if (tid == 0) a.tile_split[t] = cut;
    } else if (a.tile_split && tid == 0) {
      a.tile_split[t] = -1;
    }
    if (tid == 0) {
      s_b = static_cast<int>(bh / a.n_kv_heads);
      s_kvh = static_cast<int>(bh % a.n_kv_heads);
      s_q0 = qt * QT;
      s_s0 = s0;
      s_stream = a.cache + bh * n_rec * C::REC;
      s_slot = slot;
    }
    __syncthreads();
    load_q();
    if (s0 < s1) fetch(s0);
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (s0 < s1) put_scales(s0 & 1);
    __syncthreads();  // also: every thread has read the walk state
    if (tid == 0) {
      s_walk[0] = left - (s1 - s0);
      s_walk[3] = 0;
      if (qt + 1 == n_qt) {
        s_walk[2] = 0;
        s_walk[1] = bh + 1;
      } else {
        s_walk[2] = qt + 1;
      }
    }
    if (softmax_warp)
      role_loop(std::true_type{}, s1);
    else
      role_loop(std::false_type{}, s1);
    tc_fence_before();
    __syncthreads();  // TMEM read and Q tile free before the next segment
    tc_fence_after();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// Inverse transform of one row held by a warp (v[e] = dim 32 e + lane) into p:
// p = s * H_D(v) * scale_B / D, or per 128-dim group s1 * H_128(s2 * v) *
// scale_B / 128.
template <int D, int B, bool ROT>
__device__ __forceinline__ void derotate_row(float (&v)[D / 32], int lane, const int8_t* signs,
                                             const int8_t* signs2, float* p) {
  constexpr int E = D / 32;
  if constexpr (ROT) {
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (signs2[32 * e + lane] < 0) v[e] = -v[e];
  }
#pragma unroll
  for (int hl = 1; hl < 32; hl <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, v[e], hl);
      v[e] = (lane & hl) ? (o - v[e]) : (v[e] + o);
    }
  }
  // Butterflies across registers: dims 32 e + lane, e < E; the rotation's
  // groups are 4 registers wide.
  constexpr int EW = ROT ? kRotGroup / 32 : E;
#pragma unroll
  for (int hh = 1; hh < EW; hh <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if ((e & hh) == 0) {
        const float x0 = v[e], x1 = v[e + hh];
        v[e] = x0 + x1;
        v[e + hh] = x0 - x1;
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int d = 32 * e + lane;
    p[d] = (signs[d] < 0 ? -v[e] : v[e]) * (centroid_scale(B) / (ROT ? kRotGroup : D));
  }
}

// Inverse transform of the prefill output rows in place:
// row = s * H_D(row) * scale_B / D (scale_B: the tier's centroid scale); with
// the block-diagonal rotation, per 128-dim group, row = s1 * H_128(s2 * row) *
// scale_B / 128.
// Rows of a tile cut by the stream-K schedule are first merged from the two
// partial slots (exact log-sum-exp combine), and their lse written.
template <int D, int B, bool ROT>
__global__ void __launch_bounds__(256) derotate_rows_kernel(PrefillArgs a, const int8_t* signs, const int8_t* signs2,
                                                            int QT) {
  constexpr int E = D / 32;
  const int64_t n_rows = (int64_t)a.batch * a.n_new * a.n_q_heads;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= n_rows) return;
  float* p = a.out + r * D;
  float v[E];
  int cut = -1, rin = 0;
  if (a.stream_k) {
    const int group_q = a.n_q_heads / a.n_kv_heads;
    const int h = static_cast<int>(r % a.n_q_heads);
    const int64_t bq = r / a.n_q_heads;
    const int qi = static_cast<int>(bq % a.n_new);
    const int64_t b = bq / a.n_new;
    const int n_qt = (a.n_new + QT - 1) / QT;
    const int64_t t = (b * a.n_kv_heads + h / group_q) * n_qt + qi / QT;
    cut = a.tile_split[t];
    rin = (qi % QT) * group_q + h % group_q;
  }
  if (cut < 0) {
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = p[32 * e + lane];
  } else {
    constexpr int64_t SLOT = 128 * (int64_t)(D + 1);
    const float* s0 = a.part + (2 * (int64_t)cut) * SLOT;
    const float* s1 = s0 + SLOT;
    const float l0 = s0[128 * D + rin], l1 = s1[128 * D + rin];
    const float M = fmaxf(l0, l1);
    const float w0 = (l0 == -INFINITY) ? 0.0f : __expf(l0 - M);
    const float w1 = (l1 == -INFINITY) ? 0.0f : __expf(l1 - M);
    const float L = w0 + w1;
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e)
      v[e] = (w0 * s0[(int64_t)rin * D + 32 * e + lane] + w1 * s1[(int64_t)rin * D + 32 * e + lane]) * inv;
    if (lane == 0) a.lse[r] = L > 0.0f ? M + logf(L) : -INFINITY;
  }
  derotate_row<D, B, ROT>(v, lane, signs, signs2, p);
}

// Split many-row decode: one CTA per output row merges the row's n_split
// slots exactly (log-sum-exp; slots of an empty key range carry lse = -inf,
// zero rows, and weigh 0), then one warp applies the inverse transform. The
// weights go to shared memory first, so the slot loads of the accumulation
// depend on nothing and several are in flight per thread.
constexpr int kMaxRowSplits = 1024;
template <int D, int B, bool ROT>
__global__ void __launch_bounds__(512) merge_split_rows_kernel(PrefillArgs a, const int8_t* signs,
                                                               const int8_t* signs2, int QT) {
  // One CTA per output row. The row's n_split partial slots sit in L2; every
  // thread takes one 16-byte unit of the row over a strided subset of the
  // slots with all its loads in flight, so the merge costs about one L2 round
  // trip; the subsets are then summed in shared memory.
  constexpr int64_t SLOT = 128 * (int64_t)(D + 1);
  constexpr int NT = 512, UNITS = D / 4, SG = NT / UNITS, PER = 20;  // loads in flight per thread and batch
  __shared__ float s_w[kMaxRowSplits];
  __shared__ __align__(16) float4 s_acc[SG][UNITS];
  __shared__ __align__(16) float s_o[D];
  __shared__ float s_red[NT / 32];
  const int64_t r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_split = a.n_split;
  const int group_q = a.n_q_heads / a.n_kv_heads;
  const int h = static_cast<int>(r % a.n_q_heads);
  const int64_t bq = r / a.n_q_heads;
  const int qi = static_cast<int>(bq % a.n_new);
  const int64_t b = bq / a.n_new;
  const int n_qt = (a.n_new + QT - 1) / QT;
  const int64_t t = (b * a.n_kv_heads + h / group_q) * n_qt + qi / QT;
  const int rin = (qi % QT) * group_q + h % group_q;
  const float* base = a.part + t * n_split * SLOT;
  // The row's partial units, issued before the weights are known.
  const int u = tid % UNITS, g = tid / UNITS;
  float4 x[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int sp = g + j * SG;
    x[j] = sp < n_split ? __ldcg(reinterpret_cast<const float4*>(base + sp * SLOT + (int64_t)rin * D + 4 * u))
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  float M = -INFINITY;
  for (int sp = tid; sp < n_split; sp += NT) {
    const float l = __ldcg(base + sp * SLOT + 128 * D + rin);
    s_w[sp] = l;
    M = fmaxf(M, l);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) s_red[warp] = M;
  __syncthreads();
  M = s_red[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) M = fmaxf(M, s_red[w]);
  __syncthreads();
  for (int sp = tid; sp < n_split; sp += NT) {
    const float l = s_w[sp];
    s_w[sp] = (l == -INFINITY) ? 0.0f : __expf(l - M);
  }
  __syncthreads();
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int sp0 = 0; sp0 < n_split; sp0 += PER * SG) {
    if (sp0 > 0) {  // further batches (more than PER * SG splits)
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int sp = sp0 + g + j * SG;
        x[j] = sp < n_split ? __ldcg(reinterpret_cast<const float4*>(base + sp * SLOT + (int64_t)rin * D + 4 * u))
                            : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int sp = sp0 + g + j * SG;
      if (sp < n_split) {
        const float w = s_w[sp];
        acc.x += w * x[j].x;
        acc.y += w * x[j].y;
        acc.z += w * x[j].z;
        acc.w += w * x[j].w;
      }
    }
  }
  s_acc[g][u] = acc;
  __syncthreads();
  float L = 0.0f;
  for (int sp = 0; sp < n_split; ++sp) L += s_w[sp];
  if (tid < UNITS) {
    float4 y = s_acc[0][tid];
#pragma unroll
    for (int gg = 1; gg < SG; ++gg) {
      const float4 z = s_acc[gg][tid];
      y.x += z.x;
      y.y += z.y;
      y.z += z.z;
      y.w += z.w;
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    *reinterpret_cast<float4*>(s_o + 4 * tid) = make_float4(y.x * inv, y.y * inv, y.z * inv, y.w * inv);
  }
  __syncthreads();
  if (warp == 0) {
    float v[D / 32];
#pragma unroll
    for (int e = 0; e < D / 32; ++e) v[e] = s_o[32 * e + lane];
    derotate_row<D, B, ROT>(v, lane, signs, signs2, a.out + r * D);
    if (lane == 0) a.lse[r] = L > 0.0f ? M + logf(L) : -INFINITY;
  }
}

// SMs of the current device (cached per device).
static int device_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// Work layout of one prefill call: query tiles of qt tokens (128 rows), 64-key
// steps per tile, and whether the stream-K schedule runs (more tiles than SMs,
// and every CTA's step range at least as long as any tile, so a tile is cut at
// most once).
struct PrefillPlan {
  int qt, n_qt;
  int64_t n_tiles;
  int grid;
  int stream_k;
};
static PrefillPlan plan_prefill(int batch, int n_kv_heads, int n_q_heads, int64_t n_cached, int n_new,
                                int prefix_only) {
  PrefillPlan p{};
  p.qt = 128 / (n_q_heads / n_kv_heads);
  p.n_qt = (n_new + p.qt - 1) / p.qt;
  p.n_tiles = (int64_t)batch * n_kv_heads * p.n_qt;
  p.grid = device_sms();
  int64_t s_bh = 0, max_steps = 0;
  for (int t = 0; t < p.n_qt; ++t) {
    const int64_t kv_end = prefix_only ? n_cached : n_cached + std::min((t + 1) * p.qt, n_new);
    const int64_t st = (kv_end + 63) / 64;
    s_bh += st;
    max_steps = std::max(max_steps, st);
  }
  const int64_t W = (int64_t)batch * n_kv_heads * s_bh;
  p.stream_k = (p.n_tiles > p.grid && W / p.grid >= max_steps) ? 1 : 0;
  return p;
}

// Workspace bytes: the device flag, tile_split, and (when the schedule may be
// stream-K) two partial slots per CTA.
static size_t prefill_ws_bytes(int D, int batch, int n_kv_heads, int n_q_heads, int n_new) {
  const int qt = 128 / (n_q_heads / n_kv_heads);
  const int64_t n_tiles = (int64_t)batch * n_kv_heads * ((n_new + qt - 1) / qt);
  size_t bytes = 256 + (4 * static_cast<size_t>(n_tiles) + 255) / 256 * 256;
  const int sms = device_sms();
  if (n_tiles > sms) bytes += 2 * static_cast<size_t>(sms) * 128 * (D + 1) * sizeof(float);
  return bytes;
}

template <int D, int B, bool ROT>
static cudaError_t launch_prefill_d(const PrefillArgs& a, const int8_t* signs, const int8_t* signs2,
                                    cudaStream_t stream) {
  using Cf = PCfg<D, B, ROT>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_prefill_kernel<D, B, ROT, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_prefill_kernel<D, B, ROT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cf::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const PrefillPlan pl = plan_prefill(a.batch, a.n_kv_heads, a.n_q_heads, a.n_cached, a.n_new, a.prefix_only);
  PrefillArgs k = a;
  k.stream_k = a.n_split > 0 ? 0 : pl.stream_k;
  const unsigned grid = static_cast<unsigned>(a.n_split > 0 ? pl.n_tiles * a.n_split
                                                            : (pl.stream_k ? pl.grid : pl.n_tiles));
  if (a.n_split > 0)
    attn_prefill_kernel<D, B, ROT, true><<<grid, Cf::THREADS, Cf::SMEM, stream>>>(k);
  else
    attn_prefill_kernel<D, B, ROT, false><<<grid, Cf::THREADS, Cf::SMEM, stream>>>(k);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t rows = (int64_t)a.batch * a.n_new * a.n_q_heads;
  if (a.n_split > 0)
    merge_split_rows_kernel<D, B, ROT><<<static_cast<unsigned>(rows), 512, 0, stream>>>(k, signs, signs2, pl.qt);
  else
    derotate_rows_kernel<D, B, ROT><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(k, signs, signs2,
                                                                                              pl.qt);
  return cudaGetLastError();
}

// Instantiation for the cache's V code width and rotation (checked before).
template <int D>
static cudaError_t launch_prefill_v(const PrefillArgs& a, const ckv_cache* cache, cudaStream_t stream) {
  const int bits = cache->v_bits == 0 ? 3 : cache->v_bits;
  if (cache->v_signs2) {
    if constexpr (D >= kRotGroup) {
      if (bits == 2) return launch_prefill_d<D, 2, true>(a, cache->v_signs, cache->v_signs2, stream);
      if (bits == 4) return launch_prefill_d<D, 4, true>(a, cache->v_signs, cache->v_signs2, stream);
      return launch_prefill_d<D, 3, true>(a, cache->v_signs, cache->v_signs2, stream);
    }
    return cudaErrorInvalidValue;
  }
  if (bits == 2) return launch_prefill_d<D, 2, false>(a, cache->v_signs, nullptr, stream);
  if (bits == 4) return launch_prefill_d<D, 4, false>(a, cache->v_signs, nullptr, stream);
  return launch_prefill_d<D, 3, false>(a, cache->v_signs, nullptr, stream);
}

// ---- decode with many query rows per kv head ----
// With many rows per kv head (for example 15 agents x 8 heads over one shared
// prefix) the mma.sync decode, 8 rows per CTA, dequantises every tile once per
// 8 rows; a 128-row tile dequantises it once but pays about 28 us of fixed
// cost (Q load, a 256 KB partial slot per CTA, the merge; the slots cross
// between the two dies' L2 halves). Measured at head_dim 512 (B * Hkv = 2,
// 120 rows), tiles against mma.sync: 34 against 24 us at 4096 tokens, 57
// against 70 at 16384, 81 against 129 at 32768, 133 against 248 at 65536.
// Fitted costs in us, X = batch * n_kv_heads * max_seq_len / 1024: mma.sync
// 10 + 0.125 X per row group of 8, tiles 28 + 0.82 X per 128-row tile. n_split
// 0 takes the tiles only where they save at least 30 us (near a tie the
// mma.sync decode, measured more widely, is kept); -1 forces the tiles.
bool rows_decode_applies(int batch, int n_kv_heads, int n_q_heads, int n_q, int n_split, int64_t max_seq_len) {
  if ((n_split != 0 && n_split != -1) || max_seq_len <= 0 || n_kv_heads <= 0 || batch <= 0 || n_q <= 0 ||
      n_q_heads % n_kv_heads)
    return false;
  const int g = n_q_heads / n_kv_heads;
  if (128 % g) return false;
  if (n_split == -1) return true;
  const double rows = static_cast<double>(g) * n_q;
  const double groups = std::ceil(rows / 8.0), tiles = std::ceil(n_q / (128.0 / g));
  const double x = static_cast<double>(batch) * n_kv_heads * static_cast<double>(max_seq_len) / 1024.0;
  return rows >= 64 && (0.125 * groups - 0.82 * tiles) * x > 30.0;
}

struct RowsPlan {
  int qt, n_split;
  int64_t n_tiles;
  size_t ws;
};
static RowsPlan plan_rows(int D, int n_kv_heads, int batch, int n_q_heads, int n_q, int64_t key_end) {
  RowsPlan p{};
  p.qt = 128 / (n_q_heads / n_kv_heads);
  p.n_tiles = static_cast<int64_t>(batch) * n_kv_heads * ((n_q + p.qt - 1) / p.qt);
  const int64_t steps = (key_end + 63) / 64;
  int64_t s = device_sms() / (p.n_tiles > 0 ? p.n_tiles : 1);  // one wave
  if (s > steps) s = steps;
  if (s > kMaxRowSplits) s = kMaxRowSplits;
  if (s < 1) s = 1;
  p.n_split = static_cast<int>(s);
  p.ws = 256 + static_cast<size_t>(p.n_tiles) * p.n_split * 128 * (D + 1) * sizeof(float);
  return p;
}

size_t rows_decode_ws_bytes(int head_dim, int n_kv_heads, int batch, int n_q_heads, int n_q, int64_t max_seq_len) {
  return plan_rows(head_dim, n_kv_heads, batch, n_q_heads, n_q, max_seq_len).ws;
}

cudaError_t launch_rows_decode(const void* cache_v, int64_t key_end, const int32_t* seq_len, const void* q_f16,
                               int n_q, int n_q_heads, float scale, float* out, float* lse, void* ws,
                               cudaStream_t stream) {
  const ckv_cache* cache = static_cast<const ckv_cache*>(cache_v);
  const RowsPlan pl = plan_rows(cache->head_dim, cache->n_kv_heads, cache->batch, n_q_heads, n_q, key_end);
  PrefillArgs a{};
  a.cache = static_cast<const uint8_t*>(cache->data);
  a.capacity = cache->capacity;
  a.n_kv_heads = cache->n_kv_heads;
  a.batch = cache->batch;
  a.n_cached = key_end;
  a.n_new = n_q;
  a.n_q_heads = n_q_heads;
  a.prefix_only = 1;
  a.q = static_cast<const __nv_bfloat16*>(q_f16);
  a.q_f16 = 1;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  a.lse = lse;
  a.flag = static_cast<int32_t*>(ws);
  a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 256);
  a.seq_len = seq_len;
  a.n_split = pl.n_split;
  switch (cache->head_dim) {
    case 64: return launch_prefill_v<64>(a, cache, stream);
    case 128: return launch_prefill_v<128>(a, cache, stream);
    case 256: return launch_prefill_v<256>(a, cache, stream);
    case 512: return launch_prefill_v<512>(a, cache, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ckv

extern "C" {

CKV_API size_t ckv_attn_prefill_workspace(const ckv_cache* cache, int32_t n_new, int32_t n_q_heads) {
  if (!cache || n_new < 0 || cache->n_kv_heads <= 0 || n_q_heads <= 0 || n_q_heads % cache->n_kv_heads ||
      128 % (n_q_heads / cache->n_kv_heads))
    return 256;
  return ckv::prefill_ws_bytes(cache->head_dim, cache->batch, cache->n_kv_heads, n_q_heads, n_new);
}

}  // extern "C"

namespace {

ckv_status prefill_fail(ckv_status st, const char* msg) {
  return static_cast<ckv_status>(ckv::set_last_error(st, "%s", msg));
}

// Checks shared by both prefill entry points (n_new > 0 queries over a cache
// whose keys end at n_cached, or n_cached + n_new for the causal prefill).
ckv_status prefill_checks(const ckv_cache* cache, int64_t kv_end, const void* q_bf16, int32_t n_new,
                          int32_t n_q_heads, float* out, float* lse) {
  if (!cache) return prefill_fail(CKV_ERR_INVALID_ARG, "cache is null");
  if (n_new < 0 || kv_end < 0 || kv_end > cache->capacity || cache->capacity % 16)
    return prefill_fail(CKV_ERR_INVALID_ARG, "token range outside the cache");
  if (cache->head_dim != 64 && cache->head_dim != 128 && cache->head_dim != 256 && cache->head_dim != 512)
    return static_cast<ckv_status>(
        ckv::set_last_error(CKV_ERR_UNSUPPORTED, "prefill supports head_dim 64, 128, 256, 512 (got %d)",
                            static_cast<int>(cache->head_dim)));
  if (n_q_heads <= 0 || cache->n_kv_heads <= 0 || cache->batch <= 0 || n_q_heads % cache->n_kv_heads ||
      128 % (n_q_heads / cache->n_kv_heads))
    return prefill_fail(CKV_ERR_UNSUPPORTED, "prefill needs n_q_heads / n_kv_heads dividing 128");
  if (cache->v_bits != 0 && cache->v_bits != 2 && cache->v_bits != 3 && cache->v_bits != 4)
    return static_cast<ckv_status>(ckv::set_last_error(CKV_ERR_INVALID_ARG, "v_bits must be 2, 3 or 4 (got %d)",
                                                       static_cast<int>(cache->v_bits)));
  if (cache->v_signs2 && cache->head_dim < ckv::kRotGroup)
    return prefill_fail(CKV_ERR_UNSUPPORTED, "the block-diagonal rotation needs head_dim >= 128");
  if (!cache->data || !cache->v_signs || (reinterpret_cast<uintptr_t>(cache->data) & 15))
    return prefill_fail(CKV_ERR_INVALID_ARG, "cache data / signs");
  if (n_new == 0) return CKV_OK;
  if (!q_bf16 || !out || !lse || (reinterpret_cast<uintptr_t>(q_bf16) & 15) ||
      (reinterpret_cast<uintptr_t>(out) & 15))
    return prefill_fail(CKV_ERR_INVALID_ARG, "null or misaligned tensor");
  return CKV_OK;
}

ckv_status run_prefill(const ckv_cache* cache, int64_t n_cached, const void* q_bf16, int32_t n_new,
                       int32_t n_q_heads, float scale, float* out, float* lse, void* workspace, size_t ws_bytes,
                       void* stream, int prefix_only) {
  const size_t need = ckv::prefill_ws_bytes(cache->head_dim, cache->batch, cache->n_kv_heads, n_q_heads, n_new);
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return static_cast<ckv_status>(ckv::set_last_error(
        CKV_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned", need));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  ckv::PrefillArgs a{};
  a.cache = static_cast<const uint8_t*>(cache->data);
  a.capacity = cache->capacity;
  a.n_kv_heads = cache->n_kv_heads;
  a.batch = cache->batch;
  a.n_cached = n_cached;
  a.n_new = n_new;
  a.n_q_heads = n_q_heads;
  a.prefix_only = prefix_only;
  a.q = static_cast<const __nv_bfloat16*>(q_bf16);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  a.lse = lse;
  a.flag = static_cast<int32_t*>(workspace);
  {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int qt = 128 / (n_q_heads / cache->n_kv_heads);
    const int64_t n_tiles = (int64_t)cache->batch * cache->n_kv_heads * ((n_new + qt - 1) / qt);
    a.tile_split = reinterpret_cast<int32_t*>(ws + 256);
    a.part = reinterpret_cast<float*>(ws + 256 + (4 * n_tiles + 255) / 256 * 256);
  }
  switch (cache->head_dim) {
    case 64: e = ckv::launch_prefill_v<64>(a, cache, st); break;
    case 128: e = ckv::launch_prefill_v<128>(a, cache, st); break;
    case 256: e = ckv::launch_prefill_v<256>(a, cache, st); break;
    case 512: e = ckv::launch_prefill_v<512>(a, cache, st); break;
    default:
      return static_cast<ckv_status>(
          ckv::set_last_error(CKV_ERR_UNSUPPORTED, "head_dim %d", static_cast<int>(cache->head_dim)));
  }
  if (e != cudaSuccess)
    return static_cast<ckv_status>(ckv::set_last_error(CKV_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e)));
  return CKV_OK;
}

}  // namespace

extern "C" {

CKV_API ckv_status ckv_attn_prefill(const ckv_cache* cache, int64_t n_cached, const void* q_bf16, int32_t n_new,
                                    int32_t n_q_heads, const void* k_new_f16, const void* v_new_f16, float scale,
                                    float* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  if (n_cached < 0) return prefill_fail(CKV_ERR_INVALID_ARG, "token range outside the cache");
  ckv_status s = prefill_checks(cache, n_cached + (n_new > 0 ? n_new : 0), q_bf16, n_new, n_q_heads, out, lse);
  if (s != CKV_OK || n_new == 0) return s;
  if (!k_new_f16 || !v_new_f16 || (reinterpret_cast<uintptr_t>(k_new_f16) & 15) ||
      (reinterpret_cast<uintptr_t>(v_new_f16) & 15))
    return prefill_fail(CKV_ERR_INVALID_ARG, "null or misaligned tensor");
  const size_t need = ckv::prefill_ws_bytes(cache->head_dim, cache->batch, cache->n_kv_heads, n_q_heads, n_new);
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return static_cast<ckv_status>(ckv::set_last_error(
        CKV_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned", need));
  // Pack the new rows (same quantisers as kv_pack) at [n_cached, n_cached + n_new).
  const int64_t row = static_cast<int64_t>(cache->n_kv_heads) * cache->head_dim;
  s = ckv_kv_pack(cache, n_cached, n_new, k_new_f16, v_new_f16, row, row * n_new, stream);
  if (s != CKV_OK) return s;
  return run_prefill(cache, n_cached, q_bf16, n_new, n_q_heads, scale, out, lse, workspace, ws_bytes, stream, 0);
}

CKV_API ckv_status ckv_attn_prefill_prefix(const ckv_cache* cache, int64_t n_prefix, const void* q_bf16,
                                           int32_t n_q_tokens, int32_t n_q_heads, float scale, float* out,
                                           float* lse, void* workspace, size_t ws_bytes, void* stream) {
  if (n_prefix < 1) return prefill_fail(CKV_ERR_INVALID_ARG, "n_prefix must be at least 1");
  ckv_status s = prefill_checks(cache, n_prefix, q_bf16, n_q_tokens, n_q_heads, out, lse);
  if (s != CKV_OK || n_q_tokens == 0) return s;
  return run_prefill(cache, n_prefix, q_bf16, n_q_tokens, n_q_heads, scale, out, lse, workspace, ws_bytes, stream,
                     1);
}

}  // extern "C"
