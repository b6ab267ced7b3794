// decode_common.cuh — pieces shared by the split-K decode kernels.
//
// Warp-level formulation (one 16-token tile, up to 8 query rows of one kv head):
//   S^T[16 x 8]  = K_hat[16 x D] * Q^T[D x 8]            (mma m16n8k16, K as A)
//   online softmax over the 16 positions of every row      (rows = mma columns)
//   O^T[D x 8]  += V_hat^T[D x 16] * P'^T[16 x 8]          (V as A, P' as B)
// The softmax probabilities leave the S^T accumulator as fp16 pairs and become
// the B operand of the second product through one movmatrix transpose per
// 8x8 block. With D = 512 two warps share a tile: each multiplies half of the
// 32-dim blocks for S and owns half of the output dims for O, and the two
// partial S are summed through shared memory.
#pragma once

#include "ckv_device.cuh"

namespace ckv {

template <int D>
struct DecodeShape {
  static constexpr int NB = D / 32;                 // q8_0 blocks per vector
  static constexpr int MT = D / 16;                 // 16-dim m-tiles of O^T
  static constexpr int WT = (D == 512) ? 2 : 1;     // warps sharing one tile
  static constexpr int NCW = 8;                     // consumer warps per CTA
  static constexpr int NP = NCW / WT;               // tiles in flight per CTA
  static constexpr int NB_W = NB / WT;              // blocks per warp (S)
  static constexpr int MT_W = MT / WT;              // m-tiles per warp (O)
  static constexpr int GD = D / 8;                  // output dims owned per lane row
  static constexpr int RED_FLOATS = 8 * (D + 8);    // per-group reduction buffer
  static constexpr int XCHG_BYTES = (WT == 2) ? NP * 2 * 2 * 32 * 16 : 0;
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
// rows (2t, 2t+1) in the mma C layout; n0/n1 multiply the probabilities of
// positions g / g+8 (the V norms; 1 for dense values). Rescales acc when the
// running max grows and returns the two B-operand registers of P'.
template <int MTW>
__device__ __forceinline__ void softmax_tile(const float (&S)[4], bool valid0, bool valid1,
                                             float scale_log2, float n0, float n1,
                                             SoftmaxState& st, float (&acc)[MTW][4],
                                             uint32_t& pb0, uint32_t& pb1) {
  const float ninf = -INFINITY;
  const float x0 = valid0 ? S[0] * scale_log2 : ninf;
  const float x1 = valid0 ? S[1] * scale_log2 : ninf;
  const float x2 = valid1 ? S[2] * scale_log2 : ninf;
  const float x3 = valid1 ? S[3] * scale_log2 : ninf;
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
  const float p0 = valid0 ? fast_exp2(x0 - st.m0) : 0.0f;
  const float p1 = valid0 ? fast_exp2(x1 - st.m1) : 0.0f;
  const float p2 = valid1 ? fast_exp2(x2 - st.m0) : 0.0f;
  const float p3 = valid1 ? fast_exp2(x3 - st.m1) : 0.0f;
  st.l0 += p0 + p2;
  st.l1 += p1 + p3;
  const uint32_t X0 = pack_half2(valid0 ? p0 * n0 : 0.0f, valid0 ? p1 * n0 : 0.0f);
  const uint32_t X1 = pack_half2(valid1 ? p2 * n1 : 0.0f, valid1 ? p3 * n1 : 0.0f);
  pb0 = movmatrix_trans(X0);
  pb1 = movmatrix_trans(X1);
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Sum the two warps' partial S of a shared tile (D = 512). Both warps end
// with the same values (IEEE addition is commutative).
__device__ __forceinline__ void exchange_S(float (&S)[4], float4* xbuf, int group, int wh,
                                           int parity, int lane) {
  float4* mine = xbuf + ((group * 2 + parity) * 2 + wh) * 32 + lane;
  const float4* other = xbuf + ((group * 2 + parity) * 2 + (1 - wh)) * 32 + lane;
  *mine = make_float4(S[0], S[1], S[2], S[3]);
  named_bar(2 + group, 64);
  const float4 o = *other;
  S[0] += o.x;
  S[1] += o.y;
  S[2] += o.z;
  S[3] += o.w;
}

// CTA epilogue: merge the NP tile groups' states and accumulators into one
// partial and write it to the workspace. Runs on the 256 consumer threads
// (named barrier 1). `red` must hold NP * RED_FLOATS floats (stage memory is
// reused), `mlbuf` NP * 16 floats.
template <int D, int MTW>
__device__ __forceinline__ void decode_epilogue(SoftmaxState st, float (&acc)[MTW][4], float* red,
                                                float* mlbuf, int group, int wh, int lane,
                                                int tid, float* part_out, float* ml_out) {
  using Sh = DecodeShape<D>;
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
  named_bar(1, Sh::NCW * 32);
  float mc0 = -INFINITY, mc1 = -INFINITY;
#pragma unroll
  for (int q = 0; q < Sh::NP; ++q) {
    mc0 = fmaxf(mc0, mlbuf[q * 16 + (2 * t) * 2]);
    mc1 = fmaxf(mc1, mlbuf[q * 16 + (2 * t + 1) * 2]);
  }
  const float f0 = (st.m0 == -INFINITY) ? 0.0f : exp2f(st.m0 - mc0);
  const float f1 = (st.m1 == -INFINITY) ? 0.0f : exp2f(st.m1 - mc1);
  float* myred = red + group * Sh::RED_FLOATS;
#pragma unroll
  for (int i = 0; i < MTW; ++i) {
    const int d0 = Sh::GD * g + 2 * (wh * MTW + i);
    *reinterpret_cast<float2*>(myred + d0 * 8 + 8 * g + 2 * t) =
        make_float2(acc[i][0] * f0, acc[i][1] * f1);
    *reinterpret_cast<float2*>(myred + (d0 + 1) * 8 + 8 * g + 2 * t) =
        make_float2(acc[i][2] * f0, acc[i][3] * f1);
  }
  named_bar(1, Sh::NCW * 32);
  for (int d = tid; d < D; d += Sh::NCW * 32) {
    float s[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) s[r] = 0.0f;
#pragma unroll
    for (int q = 0; q < Sh::NP; ++q) {
      const float* src = red + q * Sh::RED_FLOATS + d * 8 + 8 * (d / Sh::GD);
      const float4 x = *reinterpret_cast<const float4*>(src);
      const float4 y = *reinterpret_cast<const float4*>(src + 4);
      s[0] += x.x; s[1] += x.y; s[2] += x.z; s[3] += x.w;
      s[4] += y.x; s[5] += y.y; s[6] += y.z; s[7] += y.w;
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) part_out[r * D + d] = s[r];
  }
  if (tid < 8) {
    float mc = -INFINITY;
#pragma unroll
    for (int q = 0; q < Sh::NP; ++q) mc = fmaxf(mc, mlbuf[q * 16 + tid * 2]);
    float lc = 0.0f;
#pragma unroll
    for (int q = 0; q < Sh::NP; ++q) {
      const float mq = mlbuf[q * 16 + tid * 2];
      if (mq != -INFINITY) lc += exp2f(mq - mc) * mlbuf[q * 16 + tid * 2 + 1];
    }
    ml_out[tid * 2 + 0] = mc;
    ml_out[tid * 2 + 1] = lc;
  }
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

}  // namespace ckv
