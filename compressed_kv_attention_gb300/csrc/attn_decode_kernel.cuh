// attn_decode_kernel.cuh — split-K flash-decode over the packed q8_0-K /
// TBQ-V cache (B = 2, 3 or 4 bits per V code), and the split merge that
// applies the inverse transform once per output row. Each bit width is
// instantiated in its own translation unit (attn_decode.cu: 3 bits,
// attn_decode_tbq2.cu / attn_decode_tbq4.cu: the other tiers).
//
// The pages' decode reads the compressed cache in-register inside the
// attention kernel rather than materialising it (PolyKV page, "F5 M6 — PolyKV
// (shared compressed KV pool)", section "S2 perf-path Level B": K and V read
// in-register, the transform applied only to the small output; section "S2
// perf-path — turbo-MMA verify kernel + scalar-K/turbo-V fused decode": K in
// true space, V in the rotated basis, output inverse only). The design here:
//
//  * One CTA = one (sequence, kv head, row group of 8 query vectors, KV split).
//    A producer warp streams the split's tile records (16 tokens each, one
//    contiguous bulk copy per stage of NP records) into a 4-stage shared-memory
//    ring guarded by mbarriers; 8 consumer warps take one record each.
//  * S^T = K_hat Q^T on tensor cores (mma.sync m16n8k16): the codes (bytes
//    q + 128) turn into fp16 subnormals (q + 128) 2^-24 with two byte permutes
//    per four codes (the 128 offset is removed through the accumulator), each
//    32-dim block is multiplied into its own accumulator and scaled by its fp16
//    scale (so K_hat = q * d16 is exact, never rounded to fp16).
//  * P'^T = exp2(S - m) * norm / (fp16) and O^T += C^T P'^T where C holds the
//    Lloyd-Max centroids selected by the B-bit codes. At 3 bits two codes (same
//    dim, two adjacent positions) index a 64-entry fp16x2 table replicated per
//    lane in shared memory, so every lookup is conflict-free; at 2 bits the
//    pair table has 16 entries; at 4 bits each code indexes a 16-entry table
//    and a byte permute joins the pair.
//  * The CTA merges its tile groups and writes one partial (m, l, O_rot) per
//    row; the merge kernel combines the splits exactly (log-sum-exp), divides,
//    runs one inverse Walsh-Hadamard transform and the sign flip per row.
#pragma once

#include "ckv_kernels.cuh"
#include "decode_common.cuh"
#include "pack_common.cuh"

namespace ckv {

namespace {

// ROT = 1: the block-diagonal rotation (128-dim groups, two sign diagonals,
// one norm per group). The group norms then scale V's fp16 pairs on the
// A side (a lane's dims all lie in one group), P' carries no norm and is split
// into hi + lo up to head dim 256.
template <int D, int B, int ROT = 0>
struct CDec : DecodeShape<D> {
  using Sh = DecodeShape<D>;
  static constexpr int NGRP = ROT ? D / kRotGroup : 1;  // V norms per position
  static constexpr int REC = record_bytes(D, B, NGRP);
  static constexpr int STAGE = Sh::NP * REC;
  static constexpr int NSTAGE = 4;
  // Stages issued at once at the start; each later first-round stage waits
  // until the stage EARLY before it has landed, so that the first data of
  // every CTA does not queue behind the other CTAs' later stages.
  static constexpr int EARLY = 2;
  static constexpr int THREADS = (Sh::NCW + 1) * 32;
  static constexpr int VW = B * Sh::MT_W / 4;   // V-code words per lane per warp
  static constexpr int GR = v_granule(D, B);    // stream granule bytes
  static constexpr int NG = VW * 4 / GR;        // granules per lane per warp
  static constexpr int LUT = (B == 3) ? 64 : 16;  // table entries (each replicated per lane)
  static constexpr bool PSPLIT = ROT ? D <= 256 : D <= 128;  // P' as an fp16 hi + lo pair
  static constexpr int RED_BYTES = Sh::NP * Sh::RED_FLOATS * 4;
  static constexpr int RING = (NSTAGE * STAGE > RED_BYTES) ? NSTAGE * STAGE : RED_BYTES;
  static constexpr int OFF_XCHG = (RING + 127) / 128 * 128;
  static constexpr int OFF_ML = OFF_XCHG + Sh::XCHG_BYTES;
  static constexpr int OFF_QB = OFF_ML + Sh::NP * 16 * 4;          // [NCW][NB_W][4][2] query-block biases
  static constexpr int OFF_BAR = OFF_QB + Sh::NCW * Sh::NB_W * 4 * 2 * 4;
  static constexpr int SMEM = OFF_BAR + 2 * NSTAGE * 8 + 16;
};

// Load `n` bytes (4, 8 or 16) from shared memory into consecutive words.
template <int N>
__device__ __forceinline__ void lds_words(uint32_t* w, uint32_t addr) {
  if constexpr (N == 16) {
    const uint4 v = lds128(addr);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (N == 8) {
    const uint2 v = lds64(addr);
    w[0] = v.x; w[1] = v.y;
  } else {
    w[0] = lds32(addr);
  }
}

// Bits [bit, bit + 6) of the little-endian word array, moved to bits [7, 13).
template <int VW>
__device__ __forceinline__ uint32_t field_x128(const uint32_t* w, int bit) {
  const int wi = bit >> 5, sh = bit & 31;
  uint32_t x;
  if (sh < 7) {
    x = w[wi] << (7 - sh);
  } else if (sh <= 26) {
    x = w[wi] >> (sh - 7);
  } else {
    x = __funnelshift_r(w[wi], (wi + 1 < VW) ? w[wi + 1] : 0u, sh - 7);
  }
  return x & 0x1F80u;
}

// Bits [bit, bit + 4) of the word array (a field that does not cross a word),
// moved to bits [7, 11).
__device__ __forceinline__ uint32_t nib_x128(const uint32_t* w, int bit) {
  const int wi = bit >> 5, sh = bit & 31;
  const uint32_t x = (sh < 7) ? (w[wi] << (7 - sh)) : (w[wi] >> (sh - 7));
  return x & 0x780u;
}

}  // namespace

// S^T = K_hat Q^T for one tile record at shared address `rb`: this warp's
// blocks, one accumulator per 32-dim block scaled by the block's fp16 scale.
// The codes enter the tensor core as fp16 subnormals (q + 128) * 2^-24, the
// accumulator starts at qbias = -2^-17 * (block sum of the query row), so each
// block product is 2^-24 q.Q exactly up to fp32 accumulation; the 2^24 goes
// into the softmax scale.
template <int D>
__device__ __forceinline__ void qk_tile(uint32_t rb, int wh, int lane, const uint32_t (&qf)[DecodeShape<D>::NB_W][4],
                                        uint32_t qb, float (&S)[4]) {
  using C = DecodeShape<D>;
  const int g = lane >> 2;
  uint32_t sc0[C::NB_W / 2], sc1[C::NB_W / 2];
  lds_words<C::NB_W * 2>(sc0, rb + k_scale_offset(D) + g * 2 * C::NB + wh * 2 * C::NB_W);
  lds_words<C::NB_W * 2>(sc1, rb + k_scale_offset(D) + (g + 8) * 2 * C::NB + wh * 2 * C::NB_W);
  S[0] = S[1] = S[2] = S[3] = 0.0f;
#pragma unroll
  for (int i = 0; i < C::NB_W; ++i) {
    const int blk = wh * C::NB_W + i;
    const uint4 kk = lds128(rb + (blk * 32 + lane) * 16);
    uint32_t a0s0, a2s0, a0s1, a2s1, a1s0, a3s0, a1s1, a3s1;
    i8x4_to_sub_half2x2(kk.x, a0s0, a2s0);
    i8x4_to_sub_half2x2(kk.y, a0s1, a2s1);
    i8x4_to_sub_half2x2(kk.z, a1s0, a3s0);
    i8x4_to_sub_half2x2(kk.w, a1s1, a3s1);
    const uint2 bq = lds64(qb + i * 32);
    float c[4] = {__uint_as_float(bq.x), __uint_as_float(bq.y), __uint_as_float(bq.x), __uint_as_float(bq.y)};
    mma16816(c, a0s0, a1s0, a2s0, a3s0, qf[i][0], qf[i][1]);
    mma16816(c, a0s1, a1s1, a2s1, a3s1, qf[i][2], qf[i][3]);
    const __half2 d0h = *reinterpret_cast<const __half2*>(&sc0[i >> 1]);
    const __half2 d1h = *reinterpret_cast<const __half2*>(&sc1[i >> 1]);
    const float d0 = (i & 1) ? __high2float(d0h) : __low2float(d0h);
    const float d1 = (i & 1) ? __high2float(d1h) : __low2float(d1h);
    S[0] = fmaf(d0, c[0], S[0]);
    S[1] = fmaf(d0, c[1], S[1]);
    S[2] = fmaf(d1, c[2], S[2]);
    S[3] = fmaf(d1, c[3], S[3]);
  }
}

// Bias of the subnormal code encoding for rows 2t, 2t+1 of each of the warp's
// blocks: -2^-17 times the sum of the block's query values. Each lane sums its
// B fragments, the four lanes of a row reduce, and lanes 0..3 (t = lane) store
// the pair for rows 2t, 2t+1 at qb[i][t] (shared, [NBW][4] float2).
template <int NBW>
__device__ __forceinline__ void q_block_bias(const uint32_t (&qf)[NBW][4], int lane, float* qb) {
  const int t = lane & 3;
#pragma unroll
  for (int i = 0; i < NBW; ++i) {
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&qf[i][j]));
      s += f.x + f.y;
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    const float r0 = __shfl_sync(0xffffffffu, s, 8 * t);
    const float r1 = __shfl_sync(0xffffffffu, s, 8 * t + 4);
    if (lane < 4) {
      qb[(i * 4 + t) * 2] = -r0 * 7.62939453125e-06f;  // 2^-17
      qb[(i * 4 + t) * 2 + 1] = -r1 * 7.62939453125e-06f;
    }
  }
  __syncwarp();
}

// O^T += C^T P'^T for one tile record, straight from the B-bit codes. `lut`
// is the shared centroid table; entry f of lane l sits at byte f * 128 + 4 l,
// so the address is one AND-OR of the shifted field with the lane offset.
// Pair field k (2B bits, codes of two adjacent positions, same dim) feeds
// A-fragment register k % 4 of m-tile k / 4.
// ROT: nA / nB are the lane's group norms of positions (2t, 2t + 1) and
// (2t + 8, 2t + 9) as fp16 pairs, multiplied into the A registers.
template <int D, int B, int ROT>
__device__ __forceinline__ void pv_tile(uint32_t rb, const uint8_t* lut, uint32_t lane4, int wh, int lane,
                                        uint32_t pb0, uint32_t pb1, const uint32_t (&pl)[2],
                                        float (&acc)[CDec<D, B, ROT>::MT_W][4], uint32_t nA, uint32_t nB) {
  using C = CDec<D, B, ROT>;
  uint32_t vw[C::VW];
#pragma unroll
  for (int c = 0; c < C::NG; ++c)
    lds_words<C::GR>(vw + c * (C::GR / 4), rb + v_code_offset(D) + ((wh * C::NG + c) * 32 + lane) * C::GR);
#pragma unroll
  for (int i = 0; i < C::MT_W; ++i) {
    uint32_t av[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = 4 * i + j;
      if constexpr (B == 3) {
        av[j] = *reinterpret_cast<const uint32_t*>(lut + (field_x128<C::VW>(vw, 6 * k) | lane4));
      } else if constexpr (B == 2) {
        av[j] = *reinterpret_cast<const uint32_t*>(lut + (nib_x128(vw, 4 * k) | lane4));
      } else {
        const uint32_t lo = *reinterpret_cast<const uint32_t*>(lut + (nib_x128(vw, 8 * k) | lane4));
        const uint32_t hi = *reinterpret_cast<const uint32_t*>(lut + (nib_x128(vw, 8 * k + 4) | lane4));
        av[j] = __byte_perm(lo, hi, 0x5410);
      }
    }
    if constexpr (ROT) {
      av[0] = hmul2_u32(av[0], nA);
      av[1] = hmul2_u32(av[1], nA);
      av[2] = hmul2_u32(av[2], nB);
      av[3] = hmul2_u32(av[3], nB);
    }
    mma16816(acc[i], av[0], av[1], av[2], av[3], pb0, pb1);
    if constexpr (C::PSPLIT) mma16816(acc[i], av[0], av[1], av[2], av[3], pl[0], pl[1]);
  }
}

// DCA: built with the regime key ranges' lower limits and tile narrowing
// (the other decodes compile without them).
template <int D, int B, bool DCA, int ROT>
__global__ void __launch_bounds__(CDec<D, B, ROT>::THREADS, 1) attn_decode_kernel(DecodeArgs a) {
  using C = CDec<D, B, ROT>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(16) uint32_t s_lut[C::LUT * 32];
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, rg = blockIdx.y, bh = blockIdx.z;
  const int b = bh / a.n_kv_heads, kvh = bh % a.n_kv_heads;
  const int group_q = a.n_q_heads / a.n_kv_heads;
  const int R = group_q * a.n_q;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::NSTAGE;
  float4* xbuf = reinterpret_cast<float4*>(smem + C::OFF_XCHG);
  float* mlbuf = reinterpret_cast<float*>(smem + C::OFF_ML);

  // The split boundaries come from the host-side bound min(capacity,
  // max_seq_len), so the producer can start streaming before the sequence's
  // length has arrived from memory; tiles past the length are masked (and not
  // fetched once the length is known).
  __shared__ int s_seq;
  const int64_t lim = a.capacity < a.max_seq_len ? a.capacity : a.max_seq_len;
  const int64_t n_tiles_max = (lim + kTile - 1) / kTile;
  const int64_t tile_begin = split * n_tiles_max / a.n_split;
  // Without an append or a DCA regime the first stages are issued before the
  // length is known; otherwise the tile range depends on it.
  const bool defer = a.n_new > 0 || DCA;
  int64_t tb = tile_begin;  // first tile actually run (DCA: at or after the regime's first key)
  const int64_t tile_end_max = (split + 1) * n_tiles_max / a.n_split;
  const int n_iters_max = static_cast<int>((tile_end_max - tile_begin + C::NP - 1) / C::NP);
  const uint8_t* gbase = a.cache + (int64_t)(b * a.n_kv_heads + kvh) * (a.capacity / kTile) * C::REC;

  // Setup that reads no global memory runs while the previous grid on the
  // stream may still be finishing: the producer lane sets up the barriers,
  // the consumers fill the centroid table, one copy per lane. B <= 3: entry f
  // (2B bits) = fp16x2(c[f % 2^B], c[f / 2^B]); B = 4: entry f = c[f] in
  // both halves. Values are c / centroid_scale(B).
  if (warp == C::NCW) {
    if (lane == 0) {
      for (int s = 0; s < C::NSTAGE; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], C::NCW);
      }
      s_abort = 0;
      fence_barrier_init();
    }
  } else {
    constexpr float inv = 1.0f / centroid_scale(B);
    for (int e = threadIdx.x; e < C::LUT * 32; e += C::NCW * 32) {
      const int f = e >> 5;
      const int klo = (B == 4) ? f : (f & ((1 << B) - 1));
      const int khi = (B == 4) ? f : (f >> B);
      const __half lo = __float2half_rn(tbq_centroid<B>(klo) * inv);
      const __half hi = __float2half_rn(tbq_centroid<B>(khi) * inv);
      s_lut[e] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
    }
  }
  // Inputs that no kernel writes (early_inputs: the page-locked host Q and
  // new rows of a host-buffer step) are loaded before the wait, so their
  // trips across the host link overlap the previous grid's last work.
  if (!a.early_inputs) {
    griddep_wait();
    // The next grid may begin only now: a grid that reads its inputs before
    // its own wait (the fp16 decode with a prior partial) then runs beside
    // this one alone, never beside the grids before it, which may still
    // write them.
    griddep_launch_dependents();
    if (threadIdx.x == 0) s_seq = a.seq_len[b];
  }

  // Query fragments first: issued before the producer starts its bulk copies,
  // these small loads do not queue behind them. The sequence length is read by
  // one thread per CTA (every CTA of the grid reads the same few words) and
  // shared; for an append the producer warp also fetches the newest row now.
  pack::PositionInput<D> new_row;
  if (warp == C::NCW && a.n_new > 0) {
    const int64_t j = a.n_new - 1;
    pack::load_position<D>(a.k_new + b * a.new_batch_stride + j * a.new_token_stride + (int64_t)kvh * D,
                           a.v_new + b * a.new_batch_stride + j * a.new_token_stride + (int64_t)kvh * D, a.signs,
                           lane, new_row);
  }
  uint32_t qf[C::NB_W][4];
  if (warp < C::NCW) {
    const int g = lane >> 2, t = lane & 3, wh = warp % C::WT;
    const int rr = rg * 8 + g;
    int qi = 0, h = 0;
    const bool ok = rr < R;
    if (ok) row_to_query(rr, group_q, kvh, qi, h);
    // DCA: rows qi >= 2 are pieces of the inter regime and share its query (q holds 3 tokens).
    const int q_tokens = DCA ? 3 : a.n_q;
    const int q_src = (DCA && qi > 2) ? 2 : qi;
    const __half* qrow = a.q + ((int64_t)(b * q_tokens + q_src) * a.n_q_heads + h) * D;
    load_q_frags<C::NB_W>(qf, qrow, ok, wh * C::NB_W, t);
  }
  if (a.early_inputs) {
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) s_seq = a.seq_len[b];
  }

  // For a plain decode the producer lane issues the first stages before the
  // CTA-wide barrier; the consumers meanwhile load Q.
  int issued = 0;  // producer lane
  auto issue = [&](int it, int64_t end) {
    const int s = it % C::NSTAGE;
    const int64_t first = tb + (int64_t)it * C::NP;
    const int64_t left = end - first;
    const uint32_t cnt = left < C::NP ? (uint32_t)left : (uint32_t)C::NP;
    mbar_arrive_expect_tx(&full[s], cnt * C::REC);
    bulk_g2s(smem + s * C::STAGE, gbase + first * C::REC, cnt * C::REC, &full[s]);
    ++issued;
  };
  int pre = 0;
  if (warp == C::NCW && !defer) {
    pre = n_iters_max < C::EARLY ? n_iters_max : C::EARLY;
    if (lane == 0)
      for (int it = 0; it < pre; ++it) issue(it, tile_end_max);
  }
  __syncthreads();

  if (warp == C::NCW) {
    // ------------------------------------------------------------ producer --
    const int seq_raw = s_seq;
    const int64_t sl = (seq_raw < 0 || seq_raw > lim) ? 0 : seq_raw;
    const int64_t nt = (sl + kTile - 1) / kTile;
    int64_t tile_end = nt < tile_end_max ? (nt > tile_begin ? nt : tile_begin) : tile_end_max;
    if constexpr (DCA) dca_tiles(a, rg, static_cast<int>(sl), split, tb, tile_end);
    const int n_iters = static_cast<int>((tile_end - tb + C::NP - 1) / C::NP);
    // Later first-round stages wait for an earlier one to land (EARLY), except
    // in the CTA that appends: it issues every stage before its new rows at
    // once and quantises while they stream.
    bool hold = true;
    if (defer) {
      int64_t n0 = 0, n1 = 0;
      if (a.n_new > 0) {
        n0 = sl - a.n_new;
        n1 = sl;
        if (n0 < tile_begin * kTile) n0 = tile_begin * kTile;
        if (n1 > tile_end * kTile) n1 = tile_end * kTile;
        if (sl < a.n_new) {
          if (lane == 0) raise_flag(a.flag, kFlagSeqLenRange);
          n1 = n0;
        }
      }
      if (n0 < n1) {
        hold = false;
        const int it_new = static_cast<int>((n0 / kTile - tile_begin) / C::NP);
        pre = it_new < n_iters ? it_new : n_iters;
        if (pre > C::NSTAGE) pre = C::NSTAGE;
      } else {
        pre = n_iters < C::EARLY ? n_iters : C::EARLY;
      }
      if (lane == 0)
        for (int it = 0; it < pre; ++it) issue(it, tile_end);
      // New positions inside this CTA's tiles, written into the cache before
      // the stages holding them are issued.
      for (int64_t pos = n0; pos < n1; ++pos) {
        const int64_t j = pos - (sl - a.n_new);
        const __half* krow = a.k_new + b * a.new_batch_stride + j * a.new_token_stride + (int64_t)kvh * D;
        const __half* vrow = a.v_new + b * a.new_batch_stride + j * a.new_token_stride + (int64_t)kvh * D;
        uint8_t* grec = a.cache_w + ((int64_t)(b * a.n_kv_heads + kvh) * (a.capacity / kTile) + pos / kTile) * C::REC;
        pack::PositionCodes<D, B> pc;
        if (pos == sl - 1) {
          pack::quantise_loaded<D, B, ROT>(new_row, static_cast<int>(pos % kTile), lane, pc, a.signs2);
        } else {
          pack::quantise_position<D, B, ROT>(krow, vrow, a.signs, static_cast<int>(pos % kTile), lane, pc,
                                             a.signs2);
        }
        pack::store_position_global<D, B, ROT>(grec, static_cast<int>(pos % kTile), lane, pc);
      }
      if (n0 < n1) {
        // The rows were written through the generic proxy; the bulk copies that
        // read them back run in the async proxy.
        __threadfence();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
      }
    }
    if (lane == 0) {
      for (int it = pre; it < n_iters; ++it) {
        const int s = it % C::NSTAGE;
        if (it >= C::NSTAGE && !*(volatile int*)&s_abort) {
          if (!mbar_wait(&empty[s], ((it / C::NSTAGE) - 1) & 1)) {
            *(volatile int*)&s_abort = 1;
            raise_flag(a.flag, kFlagWaitTimeout);
          }
        } else if (hold && it >= C::EARLY && !*(volatile int*)&s_abort) {
          if (!mbar_wait(&full[it - C::EARLY], 0)) {
            *(volatile int*)&s_abort = 1;
            raise_flag(a.flag, kFlagWaitTimeout);
          }
        }
        if (*(volatile int*)&s_abort) break;
        issue(it, tile_end);
      }
      // Do not leave while a copy may still be landing in this CTA's memory.
      const int k0 = issued > C::NSTAGE ? issued - C::NSTAGE : 0;
      for (int k = k0; k < issued; ++k) {
        if (!mbar_wait(&full[k % C::NSTAGE], (k / C::NSTAGE) & 1)) {
          raise_flag(a.flag, kFlagWaitTimeout);
          break;
        }
      }
    }
    return;
  }

  int seqlen = s_seq;
  if (seqlen < 0 || seqlen > lim) {
    if (threadIdx.x == 0) raise_flag(a.flag, kFlagSeqLenRange);
    seqlen = 0;
  }
  const int64_t n_tiles = (seqlen + kTile - 1) / kTile;
  int64_t tile_end = n_tiles < tile_end_max ? (n_tiles > tile_begin ? n_tiles : tile_begin) : tile_end_max;
  if constexpr (DCA) dca_tiles(a, rg, seqlen, split, tb, tile_end);
  const int n_iters = static_cast<int>((tile_end - tb + C::NP - 1) / C::NP);

  // -------------------------------------------------------------- consumers --
  const int tid = threadIdx.x;  // 0 .. 255
  const int group = warp / C::WT, wh = warp % C::WT;
  const int g = lane >> 2;
  // Key ranges of this lane's two rows (2t, 2t + 1) of the row group.
  int lo0, lim0, lo1, lim1;
  row_key_range(a, rg * 8 + 2 * (lane & 3), seqlen, lo0, lim0);
  row_key_range(a, rg * 8 + 2 * (lane & 3) + 1, seqlen, lo1, lim1);

  float* qb_warp = reinterpret_cast<float*>(smem + C::OFF_QB) + warp * C::NB_W * 8;
  q_block_bias<C::NB_W>(qf, lane, qb_warp);
  const uint32_t qb = smem_u32(qb_warp) + (lane & 3) * 8;
  const float scale_log2 = a.scale_log2 * 16777216.0f;  // S carries 2^-24
  float acc[C::MT_W][4];
#pragma unroll
  for (int i = 0; i < C::MT_W; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
  SoftmaxState st{-INFINITY, -INFINITY, 0.0f, 0.0f};

  const uint32_t ring = smem_u32(smem);
  const uint8_t* lut_bytes = reinterpret_cast<const uint8_t*>(s_lut);
  const uint32_t lane4 = (uint32_t)lane << 2;

  // Bounded wait for stage `it`; after a timeout every later wait is skipped
  // (results are then flagged invalid) so that the CTA still finishes.
  auto wait_stage = [&](int it) {
    if (!*(volatile int*)&s_abort) {
      if (!mbar_wait(&full[it % C::NSTAGE], (it / C::NSTAGE) & 1)) {
        *(volatile int*)&s_abort = 1;
        raise_flag(a.flag, kFlagWaitTimeout);
      }
    }
  };
  auto record = [&](int it) { return ring + (it % C::NSTAGE) * C::STAGE + group * C::REC; };

  // Software pipeline: while the softmax and P.V of tile `it` run, the
  // S = K_hat Q^T of tile `it + 1` is already in flight. With two warps per
  // tile, each warp's half of the next S goes to shared memory before the
  // current P.V and is summed with the partner's half after it.
  float S[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (n_iters > 0) {
    wait_stage(0);
    if (tb + group < tile_end) {
      qk_tile<D>(record(0), wh, lane, qf, qb, S);
      if constexpr (C::WT == 2) exchange_S<2>(S, xbuf, group, wh, 0, lane);
    }
  }
  for (int it = 0; it < n_iters; ++it) {
    const int64_t tile = tb + (int64_t)it * C::NP + group;
    const bool next = (it + 1 < n_iters) && (tile + C::NP < tile_end);
    float Sn[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (it + 1 < n_iters) wait_stage(it + 1);
    if (next) {
      qk_tile<D>(record(it + 1), wh, lane, qf, qb, Sn);
      if constexpr (C::WT == 2)
        xbuf[((group * 2 + ((it + 1) & 1)) * 2 + wh) * 32 + lane] = make_float4(Sn[0], Sn[1], Sn[2], Sn[3]);
    }
    if (tile < tile_end) {
      const uint32_t rb = record(it);
      const int64_t tpos = tile * kTile;
      float n0 = 1.0f, n1 = 1.0f;
      uint32_t nA = 0u, nB = 0u;
      if constexpr (ROT) {
        // This lane's dims lie in group (D / 8) g / 128; its positions 2t, 2t+1 and 2t+8, 2t+9.
        const uint32_t nb = rb + v_norm_offset(D, B) + 2 * (16 * ((D / 8) * (lane >> 2) / kRotGroup) + 2 * (lane & 3));
        nA = lds32(nb);
        nB = lds32(nb + 16);
        // Positions at or past seq_len may hold any bytes (a NaN norm would
        // reach O through P' = 0): their norms enter as zero. r >= 10 on every
        // tile but a sequence's last.
        const int r = seqlen - static_cast<int>(tpos) - 2 * (lane & 3);
        nA &= r >= 2 ? 0xffffffffu : r == 1 ? 0xffffu : 0u;
        nB &= r >= 10 ? 0xffffffffu : r == 9 ? 0xffffu : 0u;
      } else {
        n0 = __half2float(__ushort_as_half((unsigned short)lds16(rb + v_norm_offset(D, B) + 2 * g)));
        n1 = __half2float(__ushort_as_half((unsigned short)lds16(rb + v_norm_offset(D, B) + 2 * (g + 8))));
      }
      uint32_t pb0, pb1, pl[2] = {0u, 0u};
      softmax_tile<C::MT_W, C::PSPLIT, DCA>(S, tpos, g, lo0, lim0, lo1, lim1, scale_log2, n0, n1, st, acc, pb0,
                                            pb1, pl);
      pv_tile<D, B, ROT>(rb, lut_bytes, lane4, wh, lane, pb0, pb1, pl, acc, nA, nB);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[it % C::NSTAGE]);
    if constexpr (C::WT == 2) {
      if (next) {
        named_bar(2 + group, 64);
        const float4 o = xbuf[((group * 2 + ((it + 1) & 1)) * 2 + (1 - wh)) * 32 + lane];
        Sn[0] += o.x;
        Sn[1] += o.y;
        Sn[2] += o.z;
        Sn[3] += o.w;
      }
    }
    S[0] = Sn[0];
    S[1] = Sn[1];
    S[2] = Sn[2];
    S[3] = Sn[3];
  }

  // The epilogue reuses the ring. Stages the producer issued before the length
  // was known but that hold none of this CTA's tiles may still be landing:
  // wait for them first.
  if (!defer) {
    const int pre = n_iters_max < C::EARLY ? n_iters_max : C::EARLY;
    for (int it = n_iters; it < pre; ++it) wait_stage(it);
  }

  const int64_t gid = (int64_t)(b * a.n_kv_heads + kvh) * a.n_row_groups + rg;
  // One split and nothing to merge across row groups: the rows go out directly.
  const bool direct = a.n_split == 1 && !a.dca_fold && !a.slots_only;
  decode_epilogue<typename C::Sh, C::MT_W, ROT>(st, acc, reinterpret_cast<float*>(smem), mlbuf, group, wh, warp,
                                                lane, a.signs, a.part + (gid * a.n_split + split) * merge_slot_floats(D),
                                                centroid_scale(B), a.signs2, direct ? &a : nullptr, b, kvh, rg);
  if (direct || a.slots_only) return;  // slots_only: the fan-out's tail decode merges these slots
  decode_split_tail<D, C::RING, 256>(a, split, gid, b, kvh, rg, tid, smem);
}

template <int D, int B, bool DCA, int ROT>
static cudaError_t launch_decode_d(const DecodeArgs& a, cudaStream_t stream) {
  using C = CDec<D, B, ROT>;
  static bool configured = false;  // per process; the attribute is per function
  static ResidencyCache cap{};  // per device
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<D, B, DCA, ROT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_split_decode(attn_decode_kernel<D, B, DCA, ROT>, a, C::THREADS, C::SMEM, &cap, stream);
}

template <int D, int B, int ROT>
static cudaError_t launch_decode_dim(const DecodeArgs& a, cudaStream_t stream) {
  return a.dca_chunk > 0 ? launch_decode_d<D, B, true, ROT>(a, stream) : launch_decode_d<D, B, false, ROT>(a, stream);
}

// Every head dim of one bit width and rotation (the block-diagonal rotation
// needs at least one 128-dim group).
template <int B, int ROT = 0>
static cudaError_t launch_decode_bits(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.head_dim) {
    case 64:
      if constexpr (ROT) return cudaErrorInvalidValue;
      else return launch_decode_dim<64, B, 0>(a, stream);
    case 128: return launch_decode_dim<128, B, ROT>(a, stream);
    case 256: return launch_decode_dim<256, B, ROT>(a, stream);
    case 512: return launch_decode_dim<512, B, ROT>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ckv
