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
#include "ckv_kernels.cuh"

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
  // Per-group reduction buffer [8 rows][RP]: dim d of row r at
  // r*RP + d + 2*PS*(d / GD). Dims are written and read in pairs (float2). With
  // PS = (1 - GD/2) mod 16 and RP = 4 (mod 16) the fragment-order pair writes
  // of a half-warp fall on 16 different bank pairs.
  static constexpr int PS = ((1 - GD / 2) % 16 + 16) % 16;
  static constexpr int RP0 = D + 14 * PS + 2;
  static constexpr int RP = RP0 + ((4 - RP0 % 16) + 16) % 16;
  static constexpr int RED_FLOATS = 8 * RP;
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

// CTA epilogue. Merges the NP tile groups' softmax states and accumulators
// into one partial per row, applies the inverse transform and sign flip (when
// `signs` is set: the values were accumulated in the rotated basis), and
// writes the partial to the workspace:
//   part_out[8][D]  sum_j p_j V_j relative to the CTA's running max, true space
//   ml_out[8][2]    (running max in log2 units, row sum)
// De-rotating each partial here is exact: the transform is linear and the
// split merge only forms per-row weighted sums of partials. Runs on the 256
// consumer threads (named barrier 1). `red` holds NP * RED_FLOATS floats (stage
// memory is reused), `mlbuf` NP * 16 floats. Each group stores its unscaled
// accumulators with its own (m, l); the warp that owns a row rescales the
// groups while summing them.
template <int D, int MTW>
__device__ __forceinline__ void decode_epilogue(SoftmaxState st, float (&acc)[MTW][4], float* red,
                                                float* mlbuf, int group, int wh, int warp, int lane,
                                                int tid, const int8_t* signs, float* part_out,
                                                float* ml_out) {
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
  float* myred = red + group * Sh::RED_FLOATS;
#pragma unroll
  for (int i = 0; i < MTW; ++i) {
    const int pd = Sh::GD * g + 2 * (wh * MTW + i) + 2 * Sh::PS * g;  // dim pair d, d+1 with d / GD == g
    *reinterpret_cast<float2*>(myred + (2 * t) * Sh::RP + pd) = make_float2(acc[i][0], acc[i][2]);
    *reinterpret_cast<float2*>(myred + (2 * t + 1) * Sh::RP + pd) = make_float2(acc[i][1], acc[i][3]);
  }
  named_bar(1, Sh::NCW * 32);
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
  if (signs) {
    // Unnormalised Walsh-Hadamard transform of the row: the stage on dim bit 0
    // pairs the two values of a float2, bits 1..5 pair lanes (shuffles), bits
    // 6.. pair registers; then the sign flip and 1/D (one 1/sqrt(D) from the
    // orthonormal inverse, one from the norm scaling folded into P').
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
    for (int hh = 1; hh < E2; hh <<= 1) {
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
      v[e].x = (sg.x < 0 ? -v[e].x : v[e].x) * (1.0f / D);
      v[e].y = (sg.y < 0 ? -v[e].y : v[e].y) * (1.0f / D);
    }
  }
  float2* prow = reinterpret_cast<float2*>(part_out + r * D) + lane;
#pragma unroll
  for (int e = 0; e < E2; ++e) prow[32 * e] = v[e];
  if (lane == 0) {
    ml_out[r * 2 + 0] = mc;
    ml_out[r * 2 + 1] = lc;
  }
  (void)tid;
}

// Floats of shared scratch that merge_rows needs.
__host__ __device__ constexpr int merge_scratch_floats(int n_split, int nthr) {
  return 8 * n_split + 16 * (nthr / 32);
}

// Exact merge of the n_split partials of one row group (8 rows x D):
// M = max_s m_s, w_s = 2^(m_s - M), O = sum_s w_s part_s / sum_s w_s l_s,
// lse = (M + log2 sum_s w_s l_s) ln 2; a row with no key gives O = 0, lse = -inf.
// part: [n_split][8][D], ml: [n_split][8][2] of the group. This CTA produces
// the float4 units [u0, u1) of the 8 x D output (unit u: row u / (D/4), dims
// 4 (u % (D/4)) .. +4). Threads tid < nthr (nthr a multiple of 32, >= 256)
// take part and synchronise on named barrier `bar_id`; `sm` provides
// merge_scratch_floats(n_split, nthr) floats. out_rows / lse_rows: where each
// row goes (nullptr for padding rows); lse is written when write_lse.
//
// The partials sit in L2, so the cost is dependent round trips and barriers:
// every thread issues its (m, l) loads and its first batch of partial loads
// before it waits on any of them; row maxima and sums are reduced by all
// threads at once (the (m, l) entries a thread holds all belong to row tid % 8);
// each output unit is summed by k consecutive lanes and reduced with shuffles.
template <int D>
__device__ __forceinline__ void merge_rows(const float* part, const float* ml, int n_split, int u0, int u1,
                                           int tid, int nthr, float* sm, float* const* out_rows,
                                           float* const* lse_rows, bool write_lse, int bar_id) {
  constexpr int U = D / 4;        // float4 units per row
  constexpr int MLR = 4;          // (m, l) pairs per thread held in registers
  constexpr int PB = 8;           // partial loads per thread per batch
  const int nw = nthr >> 5;
  float* w = sm;                  // [n_split][8] weights
  float* wmax = w + n_split * 8;  // [nw][8] per-warp row maxima
  float* wsum = wmax + nw * 8;    // [nw][8] per-warp row sums
  const float2* ml2 = reinterpret_cast<const float2*>(ml);
  const float4* part4 = reinterpret_cast<const float4*>(part);
  const int n_ml = n_split * 8;
  const int nu = u1 - u0;
  const int lane = tid & 31, warp = tid >> 5;
  int k = 1;  // lanes per unit: a power of two, so a unit's lanes share a warp
  while (k < 32 && 2 * k * nu <= nthr) k *= 2;
  const int cs = nthr / k;
  const int ui = tid / k, sub = tid % k;

  // 1. Loads in flight together.
  float2 mlv[MLR];
#pragma unroll
  for (int j = 0; j < MLR; ++j) {
    const int i = tid + j * nthr;
    mlv[j] = (i < n_ml) ? __ldcg(ml2 + i) : make_float2(-INFINITY, 0.0f);
  }
  float4 x[PB];
#pragma unroll
  for (int j = 0; j < PB; ++j) {
    const int s = sub + j * k;
    x[j] = (ui < nu && s < n_split) ? __ldcg(part4 + (size_t)s * 8 * U + u0 + ui)
                                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  // 2. Row maxima.
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < MLR; ++j) m = fmaxf(m, mlv[j].x);
  for (int i = tid + MLR * nthr; i < n_ml; i += nthr) m = fmaxf(m, __ldcg(ml2 + i).x);
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
    const float2 v = __ldcg(ml2 + i);
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
          x[j] = (s < n_split) ? __ldcg(part4 + (size_t)s * 8 * U + u) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
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

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Split-merge rendezvous of a cooperative launch: every CTA of the row group
// has written its partial; the last of them to arrive releases the others.
// The wait is bounded; on timeout the device flag is raised and false returned.
__device__ __forceinline__ bool group_rendezvous(uint32_t* counter, uint32_t n_split, int tid, int nthr,
                                                 int bar_id, int32_t* flag, int* s_ok) {
  __threadfence();
  named_bar(bar_id, nthr);
  if (tid == 0) {
    atomicAdd(counter, 1u);
    int ok = 1;
    if (ld_acquire_u32(counter) < n_split) {
      const uint64_t t0 = global_timer_ns();
      for (uint32_t it = 1;; ++it) {
        if (ld_acquire_u32(counter) >= n_split) break;
        if ((it & 255u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
          raise_flag(flag, kFlagWaitTimeout);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    *s_ok = ok;
  }
  named_bar(bar_id, nthr);
  return *(volatile int*)s_ok != 0;
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

// After the epilogue: when the launch is cooperative, meet the group's other
// CTAs and merge this CTA's slice of the group's output (256 consumer threads).
template <int D>
__device__ __forceinline__ void decode_merge_tail(const DecodeArgs& a, int split, int rg, int b, int kvh,
                                                  int tid, float* sm, int* s_ok, float** s_out,
                                                  float** s_lse) {
  if (!a.merge_in_kernel) return;
  const int64_t gid = (int64_t)(b * a.n_kv_heads + kvh) * a.n_row_groups + rg;
  if (!group_rendezvous(a.counters + gid, (uint32_t)a.n_split, tid, 256, 1, a.flag, s_ok)) return;
  if (tid < 8) row_outputs(a, b, kvh, rg, tid, &s_out[tid], &s_lse[tid]);
  named_bar(1, 256);
  const int u0 = (int)((int64_t)split * 2 * D / a.n_split);
  const int u1 = (int)((int64_t)(split + 1) * 2 * D / a.n_split);
  merge_rows<D>(a.part + (size_t)gid * a.n_split * 8 * D, a.ml + (size_t)gid * a.n_split * 16, a.n_split,
                u0, u1, tid, 256, sm, s_out, s_lse, split == 0, 1);
}


// ---------------------------------------------------------- host launch --

// Blocks of `kernel` that can be resident at once on the current device.
template <typename K>
static inline int coresident_blocks(K kernel, int threads, size_t smem) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess) return 0;
  return sms * per_sm;
}

template <typename K>
static inline cudaError_t launch_split_decode(K kernel, DecodeArgs a, bool cooperative, int threads, size_t smem,
                                int* cap_cache, cudaStream_t stream) {
  const int64_t grid_total = (int64_t)a.n_split * a.n_row_groups * a.batch * a.n_kv_heads;
  if (cooperative) {
    if (*cap_cache == 0) *cap_cache = coresident_blocks(kernel, threads, smem);
    if (grid_total > *cap_cache || a.n_split > kMaxInKernelSplits) return cudaErrorCooperativeLaunchTooLarge;
  }
  a.merge_in_kernel = cooperative ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_split, a.n_row_groups, a.batch * a.n_kv_heads);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = cooperative ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace ckv
