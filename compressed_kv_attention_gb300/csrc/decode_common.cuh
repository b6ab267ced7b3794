// decode_common.cuh — pieces shared by the split-K decode kernels.
//
// Warp-level formulation (one 16-token tile, up to 8 query rows of one kv head):
//   S^T[16 x 8]  = K_hat[16 x D] * Q^T[D x 8]            (mma m16n8k16, K as A)
//   online softmax over the 16 positions of every row      (rows = mma columns)
//   O^T[D x 8]  += V_hat^T[D x 16] * P'^T[16 x 8]          (V as A, P' as B)
// The softmax probabilities leave the S^T accumulator as fp16 pairs and become
// the B operand of the second product through one movmatrix transpose per
// 8x8 block. WT warps may share a tile: each multiplies 1/WT of the 32-dim
// blocks for S and owns 1/WT of the output dims for O, and the partial S are
// summed through shared memory.
#pragma once

#include "ckv_device.cuh"
#include "ckv_kernels.cuh"

namespace ckv {

template <int D, int NCW_ = 8, int WT_ = (D == 512) ? 2 : 1>
struct DecodeShape {
  static constexpr int DIM = D;
  static constexpr int NB = D / 32;                 // q8_0 blocks per vector
  static constexpr int MT = D / 16;                 // 16-dim m-tiles of O^T
  static constexpr int WT = WT_;                    // warps sharing one tile
  static constexpr int NCW = NCW_;                  // consumer warps per CTA
  static constexpr int NP = NCW / WT;               // tiles in flight per CTA
  static constexpr int NB_W = NB / WT;              // blocks per warp (S)
  static constexpr int MT_W = MT / WT;              // m-tiles per warp (O)
  static constexpr int GD = D / 8;                  // output dims owned per lane row
  // Per-group reduction buffer [8 rows][RP]: dim d of row r at
  // r*RP + d + 2*PS*(d / GD). Dims are written and read in pairs (float2). With
  // PS = (1 - GD/2) mod 16 and RP = 4 (mod 16) the fragment-order pair writes
  // of a half-warp fall on 16 different bank pairs.
  static constexpr int PS = ((1 - GD / 2) % 16 + 16) % 16;
  static constexpr int RP0 = D + 14 * PS + 2;
  static constexpr int RP = RP0 + ((4 - RP0 % 16) + 16) % 16;
  static constexpr int RED_FLOATS = 8 * RP;
  static constexpr int XCHG_BYTES = (WT >= 2) ? NP * 2 * WT * 32 * 16 : 0;  // [NP][2][WT][32] float4
};

// Per-row online-softmax state of one lane: rows 2t and 2t+1 of the row group.
struct SoftmaxState {
  float m0, m1, l0, l1;
};

__device__ __forceinline__ float warp_max_over_gid(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
  return x;
}

// One tile of the online softmax. S holds the logits of positions (g, g+8) x
// rows (2t, 2t+1) in the mma C layout; position p is visible to row 2t when
// lo0 <= p < lim0 and to row 2t+1 when lo1 <= p < lim1 (tpos: the tile's first
// position);
// n0/n1 multiply the probabilities of positions g / g+8 (the V norms; 1 for
// dense values). Rescales acc when the
// running max grows and returns the two B-operand registers of P'. With
// SPLIT, P' is the exact-to-2^-22 pair hi + lo of fp16 values (hi in pb,
// lo in pl) and the caller multiplies both: rounding P' to fp16 alone costs up
// to 2.7e-3 of |o|_inf at head dim 64 over long rows (2.1e-3 at 128, 1.4e-3 at
// 256, 8e-4 at 512), so the kernels split at head dims up to 128.
template <int MTW, bool SPLIT = false, bool LOWER = false>
__device__ __forceinline__ void softmax_tile(const float (&S)[4], int64_t tpos, int g, int lo0, int lim0, int lo1,
                                             int lim1, float scale_log2, float n0, float n1,
                                             SoftmaxState& st, float (&acc)[MTW][4],
                                             uint32_t& pb0, uint32_t& pb1, uint32_t* pl = nullptr) {
  const float ninf = -INFINITY;
  // Position g for rows 2t / 2t+1 (v0, v1), position g + 8 (v2, v3); the
  // lower limits are checked only in the kernels built for them (LOWER).
  const int64_t pos_g = tpos + g, pos_g8 = tpos + g + 8;
  bool v0 = pos_g < lim0, v1 = pos_g < lim1, v2 = pos_g8 < lim0, v3 = pos_g8 < lim1;
  if constexpr (LOWER) {
    v0 = v0 && pos_g >= lo0;
    v1 = v1 && pos_g >= lo1;
    v2 = v2 && pos_g8 >= lo0;
    v3 = v3 && pos_g8 >= lo1;
  }
  const float x0 = v0 ? S[0] * scale_log2 : ninf;
  const float x1 = v1 ? S[1] * scale_log2 : ninf;
  const float x2 = v2 ? S[2] * scale_log2 : ninf;
  const float x3 = v3 ? S[3] * scale_log2 : ninf;
  const float t0 = warp_max_over_gid(fmaxf(x0, x2));
  const float t1 = warp_max_over_gid(fmaxf(x1, x3));
  const float mn0 = fmaxf(st.m0, t0), mn1 = fmaxf(st.m1, t1);
  if (__any_sync(0xffffffffu, (mn0 > st.m0) || (mn1 > st.m1))) {
    const float a0 = (st.m0 == ninf) ? 0.0f : fast_exp2(st.m0 - mn0);
    const float a1 = (st.m1 == ninf) ? 0.0f : fast_exp2(st.m1 - mn1);
#pragma unroll
    for (int i = 0; i < MTW; ++i) {
      acc[i][0] *= a0;
      acc[i][1] *= a1;
      acc[i][2] *= a0;
      acc[i][3] *= a1;
    }
    st.l0 *= a0;
    st.l1 *= a1;
    st.m0 = mn0;
    st.m1 = mn1;
  }
  const float p0 = v0 ? fast_exp2(x0 - st.m0) : 0.0f;
  const float p1 = v1 ? fast_exp2(x1 - st.m1) : 0.0f;
  const float p2 = v2 ? fast_exp2(x2 - st.m0) : 0.0f;
  const float p3 = v3 ? fast_exp2(x3 - st.m1) : 0.0f;
  st.l0 += p0 + p2;
  st.l1 += p1 + p3;
  const float y0 = v0 ? p0 * n0 : 0.0f, y1 = v1 ? p1 * n0 : 0.0f;
  const float y2 = v2 ? p2 * n1 : 0.0f, y3 = v3 ? p3 * n1 : 0.0f;
  const uint32_t X0 = pack_half2(y0, y1);
  const uint32_t X1 = pack_half2(y2, y3);
  pb0 = movmatrix_trans(X0);
  pb1 = movmatrix_trans(X1);
  if constexpr (SPLIT) {
    const __half2 h0 = *reinterpret_cast<const __half2*>(&X0);
    const __half2 h1 = *reinterpret_cast<const __half2*>(&X1);
    pl[0] = movmatrix_trans(pack_half2(y0 - __low2float(h0), y1 - __high2float(h0)));
    pl[1] = movmatrix_trans(pack_half2(y2 - __low2float(h1), y3 - __high2float(h1)));
  }
}

// Partial S of a tile shared by WT warps: each warp stores its float4 into
// slot [group][parity][wh] (xchg_put), then after the group's named barrier
// every warp sums the WT slots in the same order (xchg_get), so all of them
// hold bit-identical S. Parity alternates per tile so that a warp that runs
// ahead never overwrites a slot a partner is still reading.
template <int WT>
__device__ __forceinline__ void xchg_put(const float (&S)[4], float4* xbuf, int group, int wh, int parity,
                                         int lane) {
  xbuf[((group * 2 + parity) * WT + wh) * 32 + lane] = make_float4(S[0], S[1], S[2], S[3]);
}

template <int WT>
__device__ __forceinline__ void xchg_get(float (&S)[4], const float4* xbuf, int group, int parity, int lane) {
  named_bar(2 + group, 32 * WT);
  const float4* p = xbuf + ((group * 2 + parity) * WT) * 32 + lane;
  float4 v = p[0];
#pragma unroll
  for (int w = 1; w < WT; ++w) {
    const float4 o = p[w * 32];
    v.x += o.x;
    v.y += o.y;
    v.z += o.z;
    v.w += o.w;
  }
  S[0] = v.x;
  S[1] = v.y;
  S[2] = v.z;
  S[3] = v.w;
}

template <int WT>
__device__ __forceinline__ void exchange_S(float (&S)[4], float4* xbuf, int group, int wh, int parity, int lane) {
  xchg_put<WT>(S, xbuf, group, wh, parity, lane);
  xchg_get<WT>(S, xbuf, group, parity, lane);
}

// Inverse rotation of one output row held by a warp (lane: dims 64 e + 2 lane
// + c, c < 2), then the sign flip and vscale / D, stored to `orow`:
// the unnormalised Walsh-Hadamard transform pairs the two values of a float2
// (dim bit 0), lanes (bits 1..5, shuffles) and registers (bits 6..); one
// 1/sqrt(D) comes from the orthonormal inverse, one from the norm scaling
// folded into P', and vscale (the centroid table's scale) undoes the
// table's scaling. Without `signs` (dense values) the row is stored as is.
// ROT = 1 (block-diagonal rotation): the second diagonal `signs2` comes first,
// the butterfly stays inside 128-dim groups (the register stages stop at dim
// bit 6), and the scale is vscale / 128 (the norms were applied to V itself).
template <int D, int ROT = 0>
__device__ __forceinline__ void derotate_store_row(float2 (&v)[D / 64], int lane, const int8_t* signs,
                                                   float* orow, float vscale = kCentroidScale,
                                                   const int8_t* signs2 = nullptr) {
  constexpr int E2 = D / 64;
  constexpr int EG = ROT ? kRotGroup / 64 : E2;   // register stages inside one transform group
  constexpr float GSCALE = ROT ? 1.0f / kRotGroup : 1.0f / D;
  if (signs) {
    if constexpr (ROT) {
#pragma unroll
      for (int e = 0; e < E2; ++e) {
        const char2 sg = *reinterpret_cast<const char2*>(signs2 + 64 * e + 2 * lane);
        if (sg.x < 0) v[e].x = -v[e].x;
        if (sg.y < 0) v[e].y = -v[e].y;
      }
    }
#pragma unroll
    for (int e = 0; e < E2; ++e) {
      const float a0 = v[e].x, a1 = v[e].y;
      v[e] = make_float2(a0 + a1, a0 - a1);
    }
#pragma unroll
    for (int hl = 1; hl < 32; hl <<= 1) {
#pragma unroll
      for (int e = 0; e < E2; ++e) {
        const float ox = __shfl_xor_sync(0xffffffffu, v[e].x, hl);
        const float oy = __shfl_xor_sync(0xffffffffu, v[e].y, hl);
        v[e].x = (lane & hl) ? (ox - v[e].x) : (v[e].x + ox);
        v[e].y = (lane & hl) ? (oy - v[e].y) : (v[e].y + oy);
      }
    }
#pragma unroll
    for (int hh = 1; hh < EG; hh <<= 1) {
#pragma unroll
      for (int e = 0; e < E2; ++e) {
        if ((e & hh) == 0) {
          const float2 x0 = v[e], x1 = v[e + hh];
          v[e] = make_float2(x0.x + x1.x, x0.y + x1.y);
          v[e + hh] = make_float2(x0.x - x1.x, x0.y - x1.y);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < E2; ++e) {
      const int d = 64 * e + 2 * lane;
      const char2 sg = *reinterpret_cast<const char2*>(signs + d);
      v[e].x = (sg.x < 0 ? -v[e].x : v[e].x) * (vscale * GSCALE);
      v[e].y = (sg.y < 0 ? -v[e].y : v[e].y) * (vscale * GSCALE);
    }
  }
  if (orow) {
    float2* o2 = reinterpret_cast<float2*>(orow) + lane;
#pragma unroll
    for (int e = 0; e < E2; ++e) o2[32 * e] = v[e];
  }
}

// CTA epilogue. Merges the NP tile groups' softmax states and accumulators
// into one partial per row, applies the inverse transform and sign flip (when
// `signs` is set: the values were accumulated in the rotated basis), and
// writes the partial to the CTA's workspace slot:
//   slot[r * D + d]   sum_j p_j V_j of row r relative to the CTA's running
//                     max, true space
//   slot[8 D + r]     running max of row r in log2 units
//   slot[8 D + 8 + r] row sum of row r
// De-rotating each partial here is exact: the transform is linear and the
// split merge only forms per-row weighted sums of partials.
// Runs on the Sh::NCW consumer warps (named barrier 1). `red` holds
// NP * RED_FLOATS floats (stage memory is reused), `mlbuf` NP * 16 floats.
// Each group stores its unscaled accumulators with its own (m, l); warp r < 8
// owns row r and rescales the groups while summing them (other warps are done
// after the second barrier).
__device__ __forceinline__ void row_outputs(const DecodeArgs& a, int b, int kvh, int rg, int r, float** o,
                                            float** l);

// With `direct` (a launch of one split and nothing to merge) the rows go
// straight to the outputs of row group (b, kvh, rg), normalised, with their
// lse, instead of to the slot.
template <typename Sh, int MTW, int ROT = 0>
__device__ __forceinline__ void decode_epilogue(SoftmaxState st, float (&acc)[MTW][4], float* red,
                                                float* mlbuf, int group, int wh, int warp, int lane,
                                                const int8_t* signs, float* slot,
                                                float vscale = kCentroidScale, const int8_t* signs2 = nullptr,
                                                const DecodeArgs* direct = nullptr, int b = 0, int kvh = 0,
                                                int rg = 0) {
  constexpr int D = Sh::DIM;
  const int g = lane >> 2, t = lane & 3;
  // Reduce the row sums over the 8 lanes that share rows (2t, 2t+1).
  st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 4);
  st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 8);
  st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 16);
  st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 4);
  st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 8);
  st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 16);
  named_bar(1, Sh::NCW * 32);  // every consumer is done with the stage memory
  if (wh == 0 && lane < 4) {
    mlbuf[group * 16 + (2 * t) * 2 + 0] = st.m0;
    mlbuf[group * 16 + (2 * t) * 2 + 1] = st.l0;
    mlbuf[group * 16 + (2 * t + 1) * 2 + 0] = st.m1;
    mlbuf[group * 16 + (2 * t + 1) * 2 + 1] = st.l1;
  }
  float* myred = red + group * Sh::RED_FLOATS;
#pragma unroll
  for (int i = 0; i < MTW; ++i) {
    const int pd = Sh::GD * g + 2 * (wh * MTW + i) + 2 * Sh::PS * g;  // dim pair d, d+1 with d / GD == g
    *reinterpret_cast<float2*>(myred + (2 * t) * Sh::RP + pd) = make_float2(acc[i][0], acc[i][2]);
    *reinterpret_cast<float2*>(myred + (2 * t + 1) * Sh::RP + pd) = make_float2(acc[i][1], acc[i][3]);
  }
  named_bar(1, Sh::NCW * 32);
  if (warp >= 8) return;
  // Warp r owns row r: lane holds dims d = 64 e + 2 lane + c (e < D/64, c < 2).
  const int r = warp;
  float mq[Sh::NP], mc = -INFINITY;
#pragma unroll
  for (int q = 0; q < Sh::NP; ++q) {
    mq[q] = mlbuf[q * 16 + r * 2];
    mc = fmaxf(mc, mq[q]);
  }
  float fq[Sh::NP], lc = 0.0f;
#pragma unroll
  for (int q = 0; q < Sh::NP; ++q) {
    fq[q] = (mq[q] == -INFINITY) ? 0.0f : exp2f(mq[q] - mc);
    lc = fmaf(fq[q], mlbuf[q * 16 + r * 2 + 1], lc);
  }
  constexpr int E2 = D / 64;
  float2 v[E2];
#pragma unroll
  for (int e = 0; e < E2; ++e) {
    const int d = 64 * e + 2 * lane;
    const int pd = d + 2 * Sh::PS * (d / Sh::GD);
    float2 x = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int q = 0; q < Sh::NP; ++q) {
      const float2 y = *reinterpret_cast<const float2*>(red + q * Sh::RED_FLOATS + r * Sh::RP + pd);
      x.x = fmaf(fq[q], y.x, x.x);
      x.y = fmaf(fq[q], y.y, x.y);
    }
    v[e] = x;
  }
  if (direct) {
    float* orow;
    float* lrow;
    row_outputs(*direct, b, kvh, rg, r, &orow, &lrow);
    if (!orow) return;
    const float inv = lc > 0.0f ? 1.0f / lc : 0.0f;
#pragma unroll
    for (int e = 0; e < E2; ++e) v[e] = make_float2(v[e].x * inv, v[e].y * inv);
    derotate_store_row<D, ROT>(v, lane, signs, orow, vscale, signs2);
    if (lane == 0) *lrow = lc > 0.0f ? (mc + log2f(lc)) * 0.6931471805599453f : -INFINITY;
    return;
  }
  derotate_store_row<D, ROT>(v, lane, signs, slot + r * D, vscale, signs2);
  if (lane == 0) {
    slot[8 * D + r] = mc;
    slot[8 * D + 8 + r] = lc;
  }
}


// Keys [lo, hi) visible to row `rr` (query token qi = rr / G) of a sequence
// of length seqlen:
//  * plain decode: [0, seqlen);
//  * causal_q (a verify batch: the n_q tokens are the last n_q positions):
//    [0, seqlen - n_q + qi + 1);
//  * dca_chunk = c (dual chunk attention of the query at position
//    i = seqlen - 1, chunk k = i / c): intra [k c, seqlen) (qi = 0),
//    successive [(k - 1) c, k c) (qi = 1), inter [0, (k - 1) c) — the three
//    partition [0, seqlen) (DCA page, "Section C design"). The inter range is
//    cut into dca_parts equal pieces, rows qi = 2 .. 1 + dca_parts (all with
//    the inter query), so that its CTAs carry no more keys than the others;
//    the exact merge of the pieces is the inter regime's attention.
__device__ __forceinline__ void row_key_range(const DecodeArgs& a, int rr, int seqlen, int& lo, int& hi) {
  const int qi = rr / (a.n_q_heads / a.n_kv_heads);
  lo = 0;
  hi = seqlen;
  if (a.causal_q) {
    hi = seqlen - a.n_q + qi + 1;
    if (hi < 0) hi = 0;
  } else if (a.dca_chunk > 0) {
    if (seqlen == 0) return;
    const int c = a.dca_chunk, k = (seqlen - 1) / c;
    if (qi == 0) {
      lo = k * c;
    } else if (qi == 1) {
      lo = k >= 1 ? (k - 1) * c : 0;
      hi = k >= 1 ? k * c : 0;
    } else {
      const int64_t L = k >= 2 ? (int64_t)(k - 1) * c : 0;
      const int m = a.dca_parts > 0 ? a.dca_parts : 1, p = qi - 2;
      lo = static_cast<int>(p * L / m);
      hi = static_cast<int>((p + 1) * L / m);
    }
  }
}

// Union of the key ranges of the row group's real rows (tiles outside it are
// neither fetched nor read): [glo, ghi), empty when glo >= ghi.
__device__ __forceinline__ void group_key_range(const DecodeArgs& a, int rg, int seqlen, int& glo, int& ghi) {
  const int R = (a.n_q_heads / a.n_kv_heads) * a.n_q;
  glo = seqlen;
  ghi = 0;
  for (int r = 0; r < 8 && rg * 8 + r < R; ++r) {
    int lo, hi;
    row_key_range(a, rg * 8 + r, seqlen, lo, hi);
    if (lo < hi) {
      glo = lo < glo ? lo : glo;
      ghi = hi > ghi ? hi : ghi;
    }
  }
}

// DCA: the n_split CTAs of a row group divide its regime's key range (not
// the whole cache), so every CTA of every regime streams: tiles [tb, te).
__device__ __forceinline__ void dca_tiles(const DecodeArgs& a, int rg, int seqlen, int split, int64_t& tb,
                                          int64_t& te) {
  int glo, ghi;
  group_key_range(a, rg, seqlen, glo, ghi);
  const int64_t lo_t = glo / kTile, hi_t = ghi > glo ? (ghi + kTile - 1) / kTile : lo_t;
  const int64_t n = hi_t - lo_t;
  tb = lo_t + (int64_t)split * n / a.n_split;
  te = lo_t + (int64_t)(split + 1) * n / a.n_split;
}

// Which query vector row `rr` (0 <= rr < G * n_q) of kv head `kvh` is: the
// query token and the query head.
__device__ __forceinline__ void row_to_query(int rr, int group_q, int kvh, int& qi, int& h) {
  qi = rr / group_q;
  h = kvh * group_q + (rr % group_q);
}

// Load the Q B-fragments of one lane: row `gid` of the row group, blocks
// [blk0, blk0 + NBW), dims blk*32 + 8t .. +8 (zeros for rows past the end).
template <int NBW>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[NBW][4], const __half* qrow, bool ok,
                                             int blk0, int t) {
#pragma unroll
  for (int i = 0; i < NBW; ++i) {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (ok) v = __ldg(reinterpret_cast<const uint4*>(qrow + (blk0 + i) * 32 + 8 * t));
    qf[i][0] = v.x;
    qf[i][1] = v.y;
    qf[i][2] = v.z;
    qf[i][3] = v.w;
  }
}


// Output pointers of the 8 rows of row group `rg` (nullptr for padding rows).
__device__ __forceinline__ void row_outputs(const DecodeArgs& a, int b, int kvh, int rg, int r,
                                            float** o, float** l) {
  const int group_q = a.n_q_heads / a.n_kv_heads;
  const int rr = rg * 8 + r;
  if (rr >= group_q * a.n_q) {
    *o = nullptr;
    *l = nullptr;
    return;
  }
  int qi, h;
  row_to_query(rr, group_q, kvh, qi, h);
  const int64_t orow = (int64_t)(b * a.n_q + qi) * a.n_q_heads + h;
  *o = a.out + orow * a.head_dim;
  *l = a.lse + orow;
}

// The prior partial of row group (b, kvh, rg) as one more merge slot: rows
// o (normalised) with m = lse log2(e) and l = 1 (an empty row: 0, -inf, 0).
// Written by split 0 of the group before it counts its own slot in, so the
// merge's release/acquire covers it. nthr threads.
template <int D>
__device__ __forceinline__ void write_prior_slot(const DecodeArgs& a, int64_t gid, int b, int kvh, int rg, int tid,
                                                 int nthr) {
  float* slot = a.sub + (gid * a.sub_stride + a.merge_nl) * merge_slot_floats(D);
  for (int i = tid; i < 8 * (D / 4); i += nthr) {
    const int r = i / (D / 4), c = i % (D / 4);
    float* orow;
    float* lrow;
    row_outputs(a, b, kvh, rg, r, &orow, &lrow);
    const float4 v = orow ? __ldg(reinterpret_cast<const float4*>(a.prior_o + (orow - a.out)) + c)
                          : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    reinterpret_cast<float4*>(slot)[i] = v;
  }
  if (tid < 8) {
    float* orow;
    float* lrow;
    row_outputs(a, b, kvh, rg, tid, &orow, &lrow);
    const float l = lrow ? __ldg(a.prior_lse + (lrow - a.lse)) : -INFINITY;
    slot[8 * D + tid] = (l == -INFINITY) ? -INFINITY : l * 1.4426950408889634f;
    slot[8 * D + 8 + tid] = (l == -INFINITY) ? 0.0f : 1.0f;
  }
}

// ------------------------------------------------------------ split merge --
//
// Merging is exact: with M = max_s m_s and w_s = 2^(m_s - M), the merge of
// slots s is (sum_s w_s O_s, M, L = sum_s w_s l_s); the output is O / L and
// lse = (M + log2 L) ln 2, and a row with no key gives O = 0, lse = -inf.
// Two ways to get there, both leaving the group's counters at zero:
//  * Rendezvous (every CTA of the grid resident at once, the host checks
//    occupancy): the CTAs of a group meet on a counter, then each merges a
//    slice of the group's 8 x D output, all slices at once. A second counter
//    counts departures; the last CTA to leave zeroes both.
//  * Tree (any grid): the splits form NL leaves of up to LS consecutive
//    splits. A CTA counts itself into its leaf; the CTA that completes a leaf
//    merges the leaf's slots into a leaf slot and counts the leaf into the
//    group's root; the CTA that completes the root merges the leaf slots and
//    writes the output rows. No CTA waits for another; each merger zeroes the
//    counter it completed.

// Merge `cnt` slots (slot s at src + s * merge_slot_floats(D)), cnt <= 32.
// The accumulators arrive through bulk copies, at most SCR / (32 D) slots at
// a time, into `scratch` (SCR bytes of shared memory no longer in use). On
// return unit u = tid + 256 k (u < 2 D: row u / (D/4), dims 4 (u % (D/4)) ..)
// of the weighted sum is in acc[k]; s_M / s_L hold the row maxima and sums.
// 256 threads, named barrier 1. False when a copy wait ran out (the device
// flag is raised; the sums are then incomplete).
// Most slots one merge_slots call combines: the tree's 32 leaves and a prior.
constexpr int kMergeSlots = 33;

template <int D, int SCR>
__device__ __forceinline__ bool merge_slots(const float* src, int cnt, uint8_t* scratch, uint64_t* mbar,
                                            uint32_t& mphase, int tid, float* s_w, float* s_M, float* s_L,
                                            int32_t* flag, float4 (&acc)[(2 * D + 255) / 256]) {
  constexpr int64_t SLOT = merge_slot_floats(D);
  constexpr int NK = (2 * D + 255) / 256;
  constexpr int KC = SCR / (32 * D);
  static_assert(KC >= 1, "merge scratch holds at least one slot");
  // Maxima and sums of every slot and row (s_w: kMergeSlots * 8 maxima, then
  // as many sums), then the weights.
  for (int i = tid; i < cnt * 8; i += 256) {
    const float* ml = src + (i >> 3) * SLOT + 8 * D;
    s_w[i] = __ldcg(ml + (i & 7));
    s_w[kMergeSlots * 8 + i] = __ldcg(ml + 8 + (i & 7));
  }
  named_bar(1, 256);
  if (tid < 8) {
    float M = -INFINITY;
    for (int q = 0; q < cnt; ++q) M = fmaxf(M, s_w[q * 8 + tid]);
    float L = 0.0f;
    for (int q = 0; q < cnt; ++q) {
      const float m = s_w[q * 8 + tid];
      const float w = (m == -INFINITY) ? 0.0f : exp2f(m - M);
      s_w[q * 8 + tid] = w;
      L = fmaf(w, s_w[kMergeSlots * 8 + q * 8 + tid], L);
    }
    s_M[tid] = M;
    s_L[tid] = L;
  }
#pragma unroll
  for (int k = 0; k < NK; ++k) acc[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  bool ok = true;
  for (int c0 = 0; c0 < cnt; c0 += KC) {
    const int kc = (cnt - c0 < KC) ? cnt - c0 : KC;
    fence_proxy_async_all();  // this thread's reads of the scratch precede the copies into it
    named_bar(1, 256);        // weights written; the previous chunk fully read
    if (tid == 0) {
      fence_proxy_async_all();
      mbar_arrive_expect_tx(mbar, (uint32_t)kc * 32u * D);
      for (int q = 0; q < kc; ++q) bulk_g2s(scratch + q * 32 * D, src + (c0 + q) * SLOT, 32u * D, mbar);
    }
    if (!mbar_wait(mbar, mphase & 1)) {
      ok = false;
      if (tid == 0) raise_flag(flag, kFlagWaitTimeout);
      mbar_wait(mbar, mphase & 1);  // a second bounded wait for copies still landing
    }
    ++mphase;
    const float4* chunk = reinterpret_cast<const float4*>(scratch);
#pragma unroll
    for (int k = 0; k < NK; ++k) {
      const int u = tid + 256 * k;
      if (u < 2 * D) {
        const int row = u / (D / 4);
        for (int q = 0; q < kc; ++q) {
          const float w = s_w[(c0 + q) * 8 + row];
          const float4 x = chunk[q * 2 * D + u];
          acc[k].x = fmaf(w, x.x, acc[k].x);
          acc[k].y = fmaf(w, x.y, acc[k].y);
          acc[k].z = fmaf(w, x.z, acc[k].z);
          acc[k].w = fmaf(w, x.w, acc[k].w);
        }
      }
    }
  }
  named_bar(1, 256);  // every thread is done with the scratch and the weights
  return ok;
}

// Tree merge, after the epilogue has written this CTA's slot: count into the
// leaf and, when this CTA completes the leaf (and then the root), merge. 256
// consumer threads, named barrier 1. `scratch` (SCR bytes) is the stage memory.
template <int D, int SCR>
__device__ __forceinline__ void tree_merge_tail(const DecodeArgs& a, int split, int64_t gid, int b, int kvh,
                                                int rg, int tid, uint8_t* scratch) {
  constexpr int64_t SLOT = merge_slot_floats(D);
  constexpr int NK = (2 * D + 255) / 256;
  __shared__ __align__(8) uint64_t s_mbar;
  __shared__ float s_w[2 * kMergeSlots * 8], s_M[8], s_L[8];
  __shared__ int s_last;
  __shared__ float* s_out[8];
  __shared__ float* s_lse[8];
  const MergeTree tr{a.merge_ls, a.merge_nl};
  const int leaf = split / tr.ls;
  const int leaf_cnt = (leaf + 1 < tr.nl) ? tr.ls : a.n_split - leaf * tr.ls;
  uint32_t* ctr = a.counters + gid * a.ctr_stride;
  const int warp = tid >> 5, lane = tid & 31;

  // 1. Count into the leaf (the slot stores are released first; mergers read
  //    them back through bulk copies).
  fence_proxy_async_all();
  __threadfence();
  named_bar(1, 256);
  if (tid == 0) {
    const uint32_t t = atomicAdd(ctr + leaf, 1u);
    s_last = (t + 1 == (uint32_t)leaf_cnt);
    if (s_last) {
      ctr[leaf] = 0u;
      __threadfence();  // acquire: the leaf's slots are complete
      mbar_init(&s_mbar, 1);
      fence_barrier_init();
    }
  }
  named_bar(1, 256);
  if (!s_last) return;
  uint32_t mphase = 0;
  float4 acc[NK];
  const float* leaf_src = a.part + (gid * a.n_split + (int64_t)leaf * tr.ls) * SLOT;
  merge_slots<D, SCR>(leaf_src, leaf_cnt, scratch, &s_mbar, mphase, tid, s_w, s_M, s_L, a.flag, acc);

  // 2. Write the leaf slot and count it into the root.
  float* lslot = a.sub + (gid * a.sub_stride + leaf) * SLOT;
#pragma unroll
  for (int k = 0; k < NK; ++k) {
    const int u = tid + 256 * k;
    if (u < 2 * D) reinterpret_cast<float4*>(lslot)[u] = acc[k];
  }
  if (tid < 8) {
    lslot[8 * D + tid] = s_M[tid];
    lslot[8 * D + 8 + tid] = s_L[tid];
  }
  fence_proxy_async_all();
  __threadfence();
  named_bar(1, 256);
  if (tid == 0) {
    const uint32_t t = atomicAdd(ctr + tr.nl, 1u);
    s_last = (t + 1 == (uint32_t)tr.nl);
    if (s_last) {
      ctr[tr.nl] = 0u;
      __threadfence();
    }
  }
  if (tid < 8) row_outputs(a, b, kvh, rg, tid, &s_out[tid], &s_lse[tid]);
  named_bar(1, 256);
  if (!s_last) return;

  // 3. Merge the leaves; normalise; rows through shared memory to the warp
  //    that stores each.
  merge_slots<D, SCR>(a.sub + gid * a.sub_stride * SLOT, a.sub_stride, scratch, &s_mbar, mphase, tid, s_w, s_M, s_L, a.flag,
                      acc);
  float* rows = reinterpret_cast<float*>(scratch);
#pragma unroll
  for (int k = 0; k < NK; ++k) {
    const int u = tid + 256 * k;
    if (u < 2 * D) {
      const float L = s_L[u / (D / 4)];
      const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
      reinterpret_cast<float4*>(rows)[u] =
          make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
    }
  }
  named_bar(1, 256);
  {
    const int r = warp;  // 8 warps, 8 rows
    float2 v[D / 64];
#pragma unroll
    for (int e = 0; e < D / 64; ++e) v[e] = reinterpret_cast<const float2*>(rows + r * D)[32 * e + lane];
    derotate_store_row<D>(v, lane, nullptr, s_out[r]);
    if (lane == 0 && s_lse[r]) {
      const float L = s_L[r];
      *s_lse[r] = (L > 0.0f) ? (s_M[r] + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
  }
}

// ---------------------------------------------------------- host launch --

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Rendezvous merge of one slice of the group's output: floats units [u0, u1)
// of the 8 x D rows (unit u: row u / (D/4), dims 4 (u % (D/4)) .. +4), from the
// n_split slots at `slots`. Threads tid < nthr (a multiple of 32, >= 256) take
// part and synchronise on named barrier `bar_id`; `sm` holds
// 8 (n_split + n_extra) + 16 nthr / 32 floats. The partials sit in L2, so the cost is
// dependent round trips: every thread issues its (m, l) loads and its first
// batch of partial loads before it waits on any; row maxima and sums are
// reduced by all threads at once (the (m, l) entries a thread holds all belong
// to row tid % 8); each output unit is summed by k consecutive lanes and
// reduced with shuffles.
template <int D>
__device__ __forceinline__ void merge_slice(const float* slots, int n_split, int u0, int u1, int tid, int nthr,
                                            float* sm, float* const* out_rows, float* const* lse_rows,
                                            bool write_lse, int bar_id, const float* extra = nullptr,
                                            int n_extra = 1) {
  constexpr int U = D / 4;                               // float4 units per row
  constexpr int64_t SLOT = merge_slot_floats(D);
  constexpr int MLR = 4;                                 // (m, l) pairs per thread in registers
  constexpr int PB = 8;                                  // partial loads per thread per batch
  // Slot s < n_split at slots + s SLOT; with `extra`, slots n_split ..
  // n_split + n_extra - 1 follow at extra, extra + SLOT, ...
  const int n_real = n_split;
  if (extra) n_split += n_extra;
  const int nw = nthr >> 5;
  float* w = sm;                   // [n_split][8] weights (every slot, the extra ones included)
  float* wmax = w + n_split * 8;   // [nw][8] per-warp row maxima
  float* wsum = wmax + nw * 8;     // [nw][8] per-warp row sums
  auto slot_at = [&](int sidx) {
    return sidx < n_real ? slots + (int64_t)sidx * SLOT : extra + (int64_t)(sidx - n_real) * SLOT;
  };
  const int n_ml = n_split * 8;
  const int nu = u1 - u0;
  const int lane = tid & 31, warp = tid >> 5;
  int k = 1;  // lanes per unit: a power of two, so a unit's lanes share a warp
  while (k < 32 && 2 * k * nu <= nthr) k *= 2;
  const int cs = nthr / k;
  const int ui = tid / k, sub = tid % k;
  auto ml_at = [&](int i) {  // (max, sum) of entry i = slot * 8 + row
    const float* p = slot_at(i >> 3) + 8 * D + (i & 7);
    return make_float2(__ldcg(p), __ldcg(p + 8));
  };

  // 1. Loads in flight together.
  float2 mlv[MLR];
#pragma unroll
  for (int j = 0; j < MLR; ++j) {
    const int i = tid + j * nthr;
    mlv[j] = (i < n_ml) ? ml_at(i) : make_float2(-INFINITY, 0.0f);
  }
  float4 x[PB];
#pragma unroll
  for (int j = 0; j < PB; ++j) {
    const int s = sub + j * k;
    x[j] = (ui < nu && s < n_split) ? __ldcg(reinterpret_cast<const float4*>(slot_at(s)) + u0 + ui)
                                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  // 2. Row maxima.
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < MLR; ++j) m = fmaxf(m, mlv[j].x);
  for (int i = tid + MLR * nthr; i < n_ml; i += nthr) m = fmaxf(m, ml_at(i).x);
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
  if (lane < 8) wmax[warp * 8 + lane] = m;
  named_bar(bar_id, nthr);
  float M = -INFINITY;
  for (int ww = 0; ww < nw; ++ww) M = fmaxf(M, wmax[ww * 8 + (tid & 7)]);
  // 3. Weights and row sums.
  float Ls = 0.0f;
#pragma unroll
  for (int j = 0; j < MLR; ++j) {
    const int i = tid + j * nthr;
    if (i < n_ml) {
      const float ws = (mlv[j].x == -INFINITY || M == -INFINITY) ? 0.0f : exp2f(mlv[j].x - M);
      w[i] = ws;
      Ls = fmaf(ws, mlv[j].y, Ls);
    }
  }
  for (int i = tid + MLR * nthr; i < n_ml; i += nthr) {
    const float2 v = ml_at(i);
    const float ws = (v.x == -INFINITY || M == -INFINITY) ? 0.0f : exp2f(v.x - M);
    w[i] = ws;
    Ls = fmaf(ws, v.y, Ls);
  }
  Ls += __shfl_xor_sync(0xffffffffu, Ls, 8);
  Ls += __shfl_xor_sync(0xffffffffu, Ls, 16);
  if (lane < 8) wsum[warp * 8 + lane] = Ls;
  named_bar(bar_id, nthr);
  if (write_lse && tid < 8 && lse_rows[tid]) {
    float L = 0.0f;
    for (int ww = 0; ww < nw; ++ww) L += wsum[ww * 8 + tid];
    *lse_rows[tid] = (L > 0.0f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
  // 4. Weighted sums, reduced over each unit's k lanes.
  for (int base = 0; base < nu; base += cs) {
    const int el = base + ui;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    int r = 0;
    if (el < nu) {
      const int u = u0 + el;
      r = u / U;
      int s0 = sub;
      if (base == 0) {
#pragma unroll
        for (int j = 0; j < PB; ++j) {
          const int s = sub + j * k;
          if (s < n_split) {
            const float ws = w[s * 8 + r];
            acc.x = fmaf(ws, x[j].x, acc.x);
            acc.y = fmaf(ws, x[j].y, acc.y);
            acc.z = fmaf(ws, x[j].z, acc.z);
            acc.w = fmaf(ws, x[j].w, acc.w);
          }
        }
        s0 = sub + PB * k;
      }
      for (; s0 < n_split; s0 += PB * k) {
#pragma unroll
        for (int j = 0; j < PB; ++j) {
          const int s = s0 + j * k;
          x[j] = (s < n_split) ? __ldcg(reinterpret_cast<const float4*>(slot_at(s)) + u)
                               : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int j = 0; j < PB; ++j) {
          const int s = s0 + j * k;
          if (s < n_split) {
            const float ws = w[s * 8 + r];
            acc.x = fmaf(ws, x[j].x, acc.x);
            acc.y = fmaf(ws, x[j].y, acc.y);
            acc.z = fmaf(ws, x[j].z, acc.z);
            acc.w = fmaf(ws, x[j].w, acc.w);
          }
        }
      }
    }
    for (int off = 1; off < k; off <<= 1) {
      acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
      acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
      acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
      acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
    }
    if (sub == 0 && el < nu && out_rows[r]) {
      float L = 0.0f;
      for (int ww = 0; ww < nw; ++ww) L += wsum[ww * 8 + r];
      const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
      float* o = out_rows[r] + 4 * ((u0 + el) % U);
      o[0] = acc.x * inv;
      o[1] = acc.y * inv;
      o[2] = acc.z * inv;
      o[3] = acc.w * inv;
    }
  }
}

// Rendezvous merge, after the epilogue has written this CTA's slot (NT
// consumer threads, NT >= 256, named barrier 1, `scratch` holds the merge's
// shared floats). The wait is bounded: on timeout the device flag is raised
// and the CTA leaves without merging (the counters are then left non-zero: a
// workspace whose flag was raised is zeroed before reuse).
template <int D, int NT>
__device__ __forceinline__ void rendezvous_merge_tail(const DecodeArgs& a, int split, int64_t gid, int b, int kvh,
                                                      int rg, int tid, float* scratch) {
  __shared__ int s_ok;
  __shared__ float* s_out[8];
  __shared__ float* s_lse[8];
  // Fold (DCA): the merge group is the (sequence, kv head), its members every
  // (row group, split) CTA, whose slots are contiguous.
  const int64_t mg = a.dca_fold ? gid / a.n_row_groups : gid;
  const int nm = a.dca_fold ? a.n_split * a.n_row_groups : a.n_split;
  const int cm = a.dca_fold ? rg * a.n_split + split : split;
  uint32_t* arrive = a.counters + mg * a.ctr_stride;
  uint32_t* depart = arrive + 1;
  const uint32_t n = (uint32_t)nm;
  __threadfence();  // this CTA's slot, released to the group
  named_bar(1, NT);
  uint32_t dep = 0;
  if (tid == 0) {
    atomicAdd(arrive, 1u);
    int ok = 1;
    if (ld_acquire_u32(arrive) < n) {
      const uint64_t t0 = global_timer_ns();
      for (uint32_t it = 1;; ++it) {
        if (ld_acquire_u32(arrive) >= n) break;
        if ((it & 255u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
          raise_flag(a.flag, kFlagWaitTimeout);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    // Departure count; its result is needed only at the end.
    if (ok) dep = atomicAdd(depart, 1u);
    s_ok = ok;
  }
  if (tid < 8) {
    if (a.dca_fold) {  // row tid of the group: head kvh * 8 + tid of the single output token
      const int64_t orow = (int64_t)b * a.n_q_heads + kvh * 8 + tid;
      s_out[tid] = a.fold_out + orow * a.head_dim;
      s_lse[tid] = a.fold_lse + orow;
    } else {
      row_outputs(a, b, kvh, rg, tid, &s_out[tid], &s_lse[tid]);
    }
  }
  named_bar(1, NT);
  if (!s_ok) return;
  const int u0 = (int)((int64_t)cm * 2 * D / nm);
  const int u1 = (int)((int64_t)(cm + 1) * 2 * D / nm);
  const float* extra = nullptr;
  int n_extra = 1;
  if (a.prior_o) {
    extra = a.sub + (gid * a.sub_stride + a.merge_nl) * merge_slot_floats(D);
  } else if (a.ext_part) {
    extra = a.ext_part + ((int64_t)kvh * a.ext_nrg + b) * a.ext_n * merge_slot_floats(D);
    n_extra = a.ext_n;
  }
  merge_slice<D>(a.part + mg * nm * merge_slot_floats(D), nm, u0, u1, tid, NT, scratch, s_out, s_lse, cm == 0, 1,
                 extra, n_extra);
  if (tid == 0 && dep + 1 == n) {  // the last CTA to leave: nobody reads the counters any more
    *arrive = 0u;
    *depart = 0u;
  }
}

// The split merge after the epilogue: rendezvous when the host found the grid
// co-resident (on all NT consumer threads), else the tree (on threads < 256;
// the others leave).
template <int D, int SCR, int NT>
__device__ __forceinline__ void decode_split_tail(const DecodeArgs& a, int split, int64_t gid, int b, int kvh,
                                                  int rg, int tid, uint8_t* scratch) {
  if (a.rendezvous) {
    rendezvous_merge_tail<D, NT>(a, split, gid, b, kvh, rg, tid, reinterpret_cast<float*>(scratch));
  } else if (tid < 256) {
    tree_merge_tail<D, SCR>(a, split, gid, b, kvh, rg, tid, scratch);
  }
}

// Whether the caller declared that other kernels may run concurrently with
// this library's on the device (ckv_set_concurrent_kernels; process-wide).
bool concurrent_kernels();

// Blocks of `kernel` that can be resident at once on the current device.
template <typename K>
static inline int coresident_blocks(K kernel, int threads, size_t smem) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess) return 0;
  return sms * per_sm;
}

// Per-device residency figures of one kernel (blocks resident at once).
constexpr int kMaxDevices = 64;
struct ResidencyCache {
  int blocks[kMaxDevices];
};

// Launch a split decode kernel. The splits merge by rendezvous when the whole
// grid fits on the device at once, else by the tree. With programmatic stream
// serialisation the grid may begin while the previous grid on the stream
// finishes; the kernel waits for it (griddep_wait) before touching global
// memory, and every one of this grid's CTAs has started before the next grid
// can begin, so the rendezvous never waits on a CTA that cannot run. When the
// caller has declared that other kernels may run at the same time on the
// device (ckv_set_concurrent_kernels), a grid that fits may still not be
// resident all at once, so the tree merge, which never waits for another
// CTA, is used instead.
template <typename K>
static inline cudaError_t launch_split_decode(K kernel, DecodeArgs a, int threads, size_t smem, ResidencyCache* cache,
                                              cudaStream_t stream) {
  const int64_t grid_total = (int64_t)a.n_split * a.n_row_groups * a.batch * a.n_kv_heads;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  if (cache->blocks[dev] == 0) cache->blocks[dev] = coresident_blocks(kernel, threads, smem);
  a.rendezvous = (!concurrent_kernels() && grid_total <= cache->blocks[dev]) ? 1 : 0;
  // Another decode's slots (ext_part) are merged only by the rendezvous; the
  // caller checks residency before it asks for them.
  if (a.ext_part && !a.rendezvous) return cudaErrorNotSupported;
  if (!a.rendezvous) a.dca_fold = 0;
  if (a.host_folded) *a.host_folded = a.dca_fold;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_split, a.n_row_groups, a.batch * a.n_kv_heads);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace ckv
