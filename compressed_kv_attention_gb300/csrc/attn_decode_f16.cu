// attn_decode_f16.cu — split-K decode over a dense fp16 KV cache, emitting
// (partial) outputs and log-sum-exps in the same form as the compressed
// decode. It serves the private, uncompressed per-agent tails of a shared pool
// (PolyKV page, "F5 M6 — PolyKV (shared compressed KV pool)", section "S1 —
// SharedKVPool": one shared prefix plus a private suffix per agent; the
// per-agent cost is just the suffix).
//
// Same warp formulation as the compressed decode (see decode_common.cuh); the
// operands come straight from global memory as fp16 fragments (16-byte loads
// per lane), so no staging ring and no producer warp.
#include "ckv_kernels.cuh"
#include "decode_common.cuh"

namespace ckv {

template <int D>
struct FDec : DecodeShape<D> {
  using Sh = DecodeShape<D>;
  static constexpr int THREADS = Sh::NCW * 32;
  static constexpr bool PSPLIT = D <= 128;  // P' as an fp16 hi + lo pair
  static constexpr int RED_BYTES = Sh::NP * Sh::RED_FLOATS * 4;
  static constexpr int OFF_XCHG = (RED_BYTES + 127) / 128 * 128;
  static constexpr int OFF_ML = OFF_XCHG + Sh::XCHG_BYTES;
  // D = 512, split form: each tile group's K and V tile (32 KB) staged here.
  static constexpr int OFF_STG = (OFF_ML + Sh::NP * 16 * 4 + 1023) / 1024 * 1024;
  static constexpr int SMEM = D == 512 ? OFF_STG + Sh::NP * 32768 : OFF_ML + Sh::NP * 16 * 4;
};

// Epilogue of the row-parallel form: group q holds the 8 rows of row group
// rg0 + q. Each group stores its accumulators and (m, l) as in the split
// epilogue; warp r < 8 then writes row r of every group, divided by its sum.
template <typename C>
__device__ __forceinline__ void rows_epilogue(const DecodeArgs& a, SoftmaxState st, float (&acc)[C::MT_W][4],
                                              float* red, float* mlbuf, int group, int wh, int warp, int lane, int b,
                                              int kvh, int rg0) {
  using Sh = typename C::Sh;
  constexpr int D = Sh::DIM;
  const int g = lane >> 2, t = lane & 3;
  st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 4);
  st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 8);
  st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 16);
  st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 4);
  st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 8);
  st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 16);
  if (wh == 0 && lane < 4) {
    mlbuf[group * 16 + (2 * t) * 2 + 0] = st.m0;
    mlbuf[group * 16 + (2 * t) * 2 + 1] = st.l0;
    mlbuf[group * 16 + (2 * t + 1) * 2 + 0] = st.m1;
    mlbuf[group * 16 + (2 * t + 1) * 2 + 1] = st.l1;
  }
  float* myred = red + group * Sh::RED_FLOATS;
#pragma unroll
  for (int i = 0; i < C::MT_W; ++i) {
    const int pd = Sh::GD * g + 2 * (wh * C::MT_W + i) + 2 * Sh::PS * g;
    *reinterpret_cast<float2*>(myred + (2 * t) * Sh::RP + pd) = make_float2(acc[i][0], acc[i][2]);
    *reinterpret_cast<float2*>(myred + (2 * t + 1) * Sh::RP + pd) = make_float2(acc[i][1], acc[i][3]);
  }
  named_bar(1, Sh::NCW * 32);
  if (warp >= 8) return;
  const int r = warp;
  for (int q = 0; q < Sh::NP; ++q) {
    float* orow;
    float* lrow;
    row_outputs(a, b, kvh, rg0 + q, r, &orow, &lrow);
    if (rg0 + q >= a.n_row_groups || !orow) continue;
    float m = mlbuf[q * 16 + r * 2], l = mlbuf[q * 16 + r * 2 + 1];
    // With a prior partial (normalised row, lse) over other keys, the two merge
    // exactly: weights 2^(m - M) for this row's sums and 2^(m_p - M) for the
    // prior, whose sum is 1.
    float w0 = 1.0f, w1 = 0.0f;
    const float2* p2 = nullptr;
    if (a.prior_o) {
      const float lp = __ldg(a.prior_lse + (lrow - a.lse));
      const float mp = lp == -INFINITY ? -INFINITY : lp * 1.4426950408889634f;
      const float M = fmaxf(m, mp);
      w0 = (m == -INFINITY) ? 0.0f : exp2f(m - M);
      w1 = (mp == -INFINITY) ? 0.0f : exp2f(mp - M);
      l = w0 * l + w1;
      m = M;
      p2 = reinterpret_cast<const float2*>(a.prior_o + (orow - a.out)) + lane;
    }
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    float2* o2 = reinterpret_cast<float2*>(orow) + lane;
#pragma unroll
    for (int e = 0; e < D / 64; ++e) {
      const int d = 64 * e + 2 * lane;
      float2 y = *reinterpret_cast<const float2*>(red + q * Sh::RED_FLOATS + r * Sh::RP + d +
                                                  2 * Sh::PS * (d / Sh::GD));
      if (p2) {
        const float2 pv = __ldg(p2 + 32 * e);
        y = make_float2(w0 * y.x + w1 * pv.x, w0 * y.y + w1 * pv.y);
      }
      o2[32 * e] = make_float2(y.x * inv, y.y * inv);
    }
    if (lane == 0) *lrow = l > 0.0f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
  }
}

// ROWS: the NP tile groups of a CTA take NP different row groups over the
// same tiles instead of splitting one row group's tiles (one split): each
// tile is then fetched from L2 once per CTA and served to the other groups
// from L1, which matters when many query rows share a short sequence (a
// prefill over a private fp16 tail). Each group writes its rows directly.
template <int D, bool ROWS>
__global__ void __launch_bounds__(FDec<D>::THREADS, 1) attn_decode_f16_kernel(DecodeArgs a) {
  using C = FDec<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int split = blockIdx.x, bh = blockIdx.z;
  const int rg = ROWS ? blockIdx.y * C::NP + warp / C::WT : blockIdx.y;
  const int b = bh / a.n_kv_heads, kvh = bh % a.n_kv_heads;
  const int group_q = a.n_q_heads / a.n_kv_heads;
  const int R = group_q * a.n_q;
  const int group = warp / C::WT, wh = warp % C::WT;
  const int g = lane >> 2, t = lane & 3;
  float4* xbuf = reinterpret_cast<float4*>(smem + C::OFF_XCHG);
  float* mlbuf = reinterpret_cast<float*>(smem + C::OFF_ML);

  // With a prior partial or another decode's slots to merge (written by the
  // previous grid: the shared prefix's decode) the wait moves to just before
  // the epilogue, so the tails stream while that grid finishes. Until then
  // the kernel only reads K, V, Q and seq_len, which no grid that can still be
  // running writes: the decode kernels start their dependents only after their
  // own wait, and the kernels that write caches or tails do not start them
  // early at all.
  const bool late_wait = a.prior_o || a.ext_part;
  griddep_launch_dependents();
  if (!late_wait) griddep_wait();
  int seqlen = a.seq_len[b];
  const int64_t lim = a.capacity < a.max_seq_len ? a.capacity : a.max_seq_len;
  if (seqlen < 0 || seqlen > lim) {
    if (tid == 0) raise_flag(a.flag, kFlagSeqLenRange);
    seqlen = 0;
  }
  int lo0, lim0, lo1, lim1;  // key ranges of this lane's rows 2t, 2t + 1
  row_key_range(a, rg * 8 + 2 * t, seqlen, lo0, lim0);
  row_key_range(a, rg * 8 + 2 * t + 1, seqlen, lo1, lim1);
  const int64_t n_tiles = (seqlen + kTile - 1) / kTile;
  int64_t tile_begin = split * n_tiles / a.n_split;
  int64_t tile_end = (split + 1) * n_tiles / a.n_split;
  int n_iters = static_cast<int>((tile_end - tile_begin + C::NP - 1) / C::NP);
  if constexpr (ROWS) {
    // Every tile up to the last one any row of this group sees, one per iteration.
    int hi = lim0 > lim1 ? lim0 : lim1;
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, 1));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, 2));
    tile_begin = 0;
    tile_end = (hi + kTile - 1) / kTile;
    if (tile_end > n_tiles) tile_end = n_tiles;
    n_iters = static_cast<int>(tile_end);
  }
  const __half* kb = a.k16 + (int64_t)(b * a.n_kv_heads + kvh) * a.capacity * D;
  const __half* vb = a.v16 + (int64_t)(b * a.n_kv_heads + kvh) * a.capacity * D;

  uint32_t qf[C::NB_W][4];
  {
    const int rr = rg * 8 + g;
    int qi = 0, h = 0;
    const bool ok = rr < R;
    if (ok) row_to_query(rr, group_q, kvh, qi, h);
    const __half* qrow = a.q + ((int64_t)(b * a.n_q + qi) * a.n_q_heads + h) * D;
    load_q_frags<C::NB_W>(qf, qrow, ok, wh * C::NB_W, t);
    if (a.q_bf16) {
      // bf16 queries: every bf16 value in the fp16 range converts exactly.
#pragma unroll
      for (int i = 0; i < C::NB_W; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qf[i][j]));
          const __half2 hq = __floats2half2_rn(f.x, f.y);
          qf[i][j] = *reinterpret_cast<const uint32_t*>(&hq);
        }
    }
  }
  float acc[C::MT_W][4];
#pragma unroll
  for (int i = 0; i < C::MT_W; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
  SoftmaxState st{-INFINITY, -INFINITY, 0.0f, 0.0f};
  const int dbase = C::GD * g + 2 * wh * C::MT_W;  // first output dim of this lane's m-tiles

  // ROWS at D = 512: the NP groups walk the same tiles, so the whole CTA
  // stages each tile in shared memory with cp.async, double-buffered, and the
  // groups read their fragments from there (one L2 round trip per tile, under
  // the previous tile's work, instead of one per fragment load). The 16-byte
  // chunk c of tile row r sits at chunk c ^ ((r & 7) << 2) of its 1 KB row for
  // K and c ^ (((c >> 3) + 2 ((r >> 1) & 3)) & 7) for V: the 8 lanes of each
  // phase of a fragment load then fall on 8 different bank groups. The loop
  // runs to the last tile of any group, so that every thread meets the
  // barriers; a group past its own last tile only helps to stage.
  constexpr bool STG = ROWS && D == 512;
  static_assert(!STG || (C::THREADS == 256 && C::MT_W == 16 && C::RED_BYTES >= 65536), "staging layout");
  const uint32_t stg0 = smem_u32(smem);
  // Split form at D = 512: the NP groups walk different tiles, so each group
  // stages its own: K of its next tile is copied (cp.async, by the group's 64
  // threads, same swizzles) as soon as both warps have read the current K (at
  // the S exchange), and V of its next tile once both have read the current V,
  // so the copies overlap the softmax and P.V of this tile and the S of the
  // next. Group barriers only: a group that has run out of tiles leaves the
  // loop on its own.
  constexpr bool STS = !ROWS && D == 512;
  const uint32_t sgk = smem_u32(smem) + C::OFF_STG + group * 32768, sgv = sgk + 16384;
  const int gtid = wh * 32 + lane;
  auto stage_rows = [&](const __half* src, uint32_t dst, bool is_v) {
#pragma unroll 4
    for (int r = 0; r < kTile; ++r) {
      const int c = gtid;  // chunk: 64 threads x 16 bytes = one 1 KB row
      const int cs = is_v ? (c ^ (((c >> 3) + 2 * ((r >> 1) & 3)) & 7)) : (c ^ ((r & 7) << 2));
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + r * 1024 + (cs << 4)),
                   "l"(src + r * D + c * 8) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  if constexpr (STS) {
    const int64_t t0 = tile_begin + group;
    if (n_iters > 0 && t0 < tile_end) {
      stage_rows(kb + t0 * kTile * D, sgk, false);
      stage_rows(vb + t0 * kTile * D, sgv, true);
    }
  }
  int cta_iters = n_iters;
  if constexpr (STG) {
    __shared__ int s_iters;
    if (tid == 0) s_iters = 0;
    __syncthreads();
    if (lane == 0) atomicMax(&s_iters, n_iters);
    __syncthreads();
    cta_iters = s_iters;
  }
  auto stage = [&](int64_t tile, int buf) {
    const __half* ks = kb + tile * kTile * D;
    const __half* vs = vb + tile * kTile * D;
    const uint32_t sk = stg0 + buf * 32768, sv = sk + 16384;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = tid + 256 * k;
      const int r = idx >> 6, c = idx & 63;
      const uint32_t dk = sk + r * 1024 + ((c ^ ((r & 7) << 2)) << 4);
      const uint32_t dv = sv + r * 1024 + ((c ^ (((c >> 3) + 2 * ((r >> 1) & 3)) & 7)) << 4);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dk), "l"(ks + r * D + c * 8) : "memory");
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dv), "l"(vs + r * D + c * 8) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  if constexpr (STG) {
    if (cta_iters > 0) stage(0, 0);
  }

  for (int it = 0; it < cta_iters; ++it) {
    if constexpr (STG) {
      if (it + 1 < cta_iters) {
        stage(it + 1, (it + 1) & 1);
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      } else {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
      }
      __syncthreads();  // tile it has landed for every thread's copies
    }
    const int64_t tile = ROWS ? (int64_t)it : tile_begin + (int64_t)it * C::NP + group;
    const bool active = tile < tile_end;  // uniform across the warps of a group
    if constexpr (!STG) {
      if (!active) break;
    }
    // STS: this tile's K and V are the group's two newest copy groups or older
    const int64_t next_tile = tile + C::NP;
    const bool next_active = STS && it + 1 < n_iters && next_tile < tile_end;
    if constexpr (STS) {
      asm volatile("cp.async.wait_group 1;" ::: "memory");  // K landed (V may still be in flight)
      named_bar(2 + group, 64);
    }
    if (active) {
      const int64_t tpos = tile * kTile;
      // ---- S^T = K Q^T ----
      float S[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const __half* k0p = kb + (tpos + g) * D + 8 * t;
      const __half* k1p = kb + (tpos + g + 8) * D + 8 * t;
#pragma unroll
      for (int i = 0; i < C::NB_W; ++i) {
        const int blk = wh * C::NB_W + i;
        uint4 k0, k1;
        if constexpr (STG || STS) {
          // rows g and g + 8 share the swizzle (r & 7 = g)
          const uint32_t off = (((blk * 4 + t) ^ (g << 2)) << 4) + (STG ? stg0 + (it & 1) * 32768 : sgk);
          k0 = lds128(off + g * 1024);
          k1 = lds128(off + (g + 8) * 1024);
        } else {
          k0 = __ldg(reinterpret_cast<const uint4*>(k0p + blk * 32));
          k1 = __ldg(reinterpret_cast<const uint4*>(k1p + blk * 32));
        }
        mma16816(S, k0.x, k1.x, k0.y, k1.y, qf[i][0], qf[i][1]);
        mma16816(S, k0.z, k1.z, k0.w, k1.w, qf[i][2], qf[i][3]);
      }
      if constexpr (C::WT >= 2) exchange_S<C::WT>(S, xbuf, group, wh, it & 1, lane);
      if constexpr (STS) {
        // both warps are past their K reads (the exchange's barrier): stage the next K
        if (next_active) stage_rows(kb + next_tile * kTile * D, sgk, false);
        else asm volatile("cp.async.commit_group;" ::: "memory");
      }
      uint32_t pb0, pb1, pl[2] = {0u, 0u};
      softmax_tile<C::MT_W, C::PSPLIT>(S, tpos, g, lo0, lim0, lo1, lim1, a.scale_log2, 1.0f, 1.0f, st, acc, pb0,
                                       pb1, pl);
      // ---- O^T += V^T P^T: lane reads positions 2t, 2t+1, 2t+8, 2t+9 ----
      const __half* vp = vb + tpos * D + dbase;
      // Rows at or past seq_len may hold any bytes (a NaN there would reach O
      // through P = 0): they enter as zero.
      const int64_t vrem = seqlen - tpos;
      const bool ve0 = 2 * t < vrem, vo0 = 2 * t + 1 < vrem, ve1 = 2 * t + 8 < vrem, vo1 = 2 * t + 9 < vrem;
      const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
      if constexpr (STS) {
        asm volatile("cp.async.wait_group 1;" ::: "memory");  // V landed (the next K may still be in flight)
        named_bar(2 + group, 64);
      }
#pragma unroll
      for (int c4 = 0; c4 < C::MT_W / 4; ++c4) {
        uint4 e0, o0, e1, o1;
        if constexpr (STG || STS) {
          // chunk 8 g + 4 wh + c4 of rows 2t, 2t+1, 2t+8, 2t+9: ((r >> 1) & 3) = t for all four
          const uint32_t sv = (STG ? stg0 + (it & 1) * 32768 + 16384 : sgv) +
                              (((8 * g + 4 * wh + c4) ^ ((g + 2 * t) & 7)) << 4);
          e0 = ve0 ? lds128(sv + (2 * t) * 1024) : z4;
          o0 = vo0 ? lds128(sv + (2 * t + 1) * 1024) : z4;
          e1 = ve1 ? lds128(sv + (2 * t + 8) * 1024) : z4;
          o1 = vo1 ? lds128(sv + (2 * t + 9) * 1024) : z4;
        } else {
          e0 = ve0 ? __ldg(reinterpret_cast<const uint4*>(vp + (2 * t) * D + c4 * 8)) : z4;
          o0 = vo0 ? __ldg(reinterpret_cast<const uint4*>(vp + (2 * t + 1) * D + c4 * 8)) : z4;
          e1 = ve1 ? __ldg(reinterpret_cast<const uint4*>(vp + (2 * t + 8) * D + c4 * 8)) : z4;
          o1 = vo1 ? __ldg(reinterpret_cast<const uint4*>(vp + (2 * t + 9) * D + c4 * 8)) : z4;
        }
        const uint32_t we[4] = {e0.x, e0.y, e0.z, e0.w}, wo[4] = {o0.x, o0.y, o0.z, o0.w};
        const uint32_t xe[4] = {e1.x, e1.y, e1.z, e1.w}, xo[4] = {o1.x, o1.y, o1.z, o1.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t a0, a1, a2, a3;
          asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(a0) : "r"(we[j]), "r"(wo[j]));
          asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(a1) : "r"(we[j]), "r"(wo[j]));
          asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(a2) : "r"(xe[j]), "r"(xo[j]));
          asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(a3) : "r"(xe[j]), "r"(xo[j]));
          mma16816(acc[c4 * 4 + j], a0, a1, a2, a3, pb0, pb1);
          if constexpr (C::PSPLIT) mma16816(acc[c4 * 4 + j], a0, a1, a2, a3, pl[0], pl[1]);
        }
      }
      if constexpr (STS) {
        named_bar(2 + group, 64);  // both warps are past their V reads: stage the next V
        if (next_active) stage_rows(vb + next_tile * kTile * D, sgv, true);
        else asm volatile("cp.async.commit_group;" ::: "memory");
      }
    }  // active
    if constexpr (STG) __syncthreads();  // the buffer of tile it is staged again at it + 2
  }
  if constexpr (STS) asm volatile("cp.async.wait_group 0;" ::: "memory");

  if (late_wait) griddep_wait();  // the prior partial (or the prefix's slots) is complete
  if constexpr (ROWS) {
    rows_epilogue<C>(a, st, acc, reinterpret_cast<float*>(smem), mlbuf, group, wh, warp, lane, b, kvh,
                     blockIdx.y * C::NP);
  } else {
    const int64_t gid = (int64_t)(b * a.n_kv_heads + kvh) * a.n_row_groups + rg;
    // One split and nothing to merge in: the rows go out directly.
    const bool direct = a.n_split == 1 && !a.prior_o && !a.ext_part;
    decode_epilogue<typename C::Sh, C::MT_W>(st, acc, reinterpret_cast<float*>(smem), mlbuf, group, wh, warp, lane,
                                             nullptr, a.part + (gid * a.n_split + split) * merge_slot_floats(D),
                                             kCentroidScale, nullptr, direct ? &a : nullptr, b, kvh, rg);
    if (direct) return;
    if (a.prior_o && split == 0) write_prior_slot<D>(a, gid, b, kvh, rg, tid, C::THREADS);
    decode_split_tail<D, C::RED_BYTES, C::THREADS>(a, split, gid, b, kvh, rg, tid, smem);
  }
}

template <int D>
static cudaError_t launch_f16_d(const DecodeArgs& a, cudaStream_t stream) {
  using C = FDec<D>;
  static bool configured = false;
  static ResidencyCache cap{};  // per device
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_f16_kernel<D, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_decode_f16_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (a.n_split == 1 && a.n_row_groups >= C::NP) {
    // Row-parallel CTAs: NP row groups each, no split merge.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, (a.n_row_groups + C::NP - 1) / C::NP, a.batch * a.n_kv_heads);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_decode_f16_kernel<D, true>, a);
  }
  return launch_split_decode(attn_decode_f16_kernel<D, false>, a, C::THREADS, C::SMEM, &cap, stream);
}

// Copy n_new rows per sequence into dense fp16 caches [batch][n_kv_heads]
// [capacity][D] at positions [seq_len[b] - n_new, seq_len[b]) (positions
// outside [0, capacity) are skipped). One CTA per (row, sequence), one 16-byte
// word per thread.
__global__ void f16_append_kernel(F16AppendArgs a) {
  const int j = blockIdx.x, b = blockIdx.y;
  const int64_t pos = (int64_t)a.seq_len[b] - a.n_new + j;
  if (pos < 0 || pos >= a.capacity) return;
  const int words = a.head_dim / 8;  // uint4 per (head) row
  for (int w = threadIdx.x; w < a.n_kv_heads * words; w += blockDim.x) {
    const int h = w / words, c = w % words;
    const int64_t src = b * a.batch_stride + (int64_t)j * a.token_stride + (int64_t)h * a.head_dim + 8 * c;
    const int64_t dst = (((int64_t)b * a.n_kv_heads + h) * a.capacity + pos) * a.head_dim + 8 * c;
    *reinterpret_cast<uint4*>(a.k + dst) = *reinterpret_cast<const uint4*>(a.k_new + src);
    *reinterpret_cast<uint4*>(a.v + dst) = *reinterpret_cast<const uint4*>(a.v_new + src);
  }
}

cudaError_t launch_f16_append(const F16AppendArgs& a, cudaStream_t stream) {
  if (a.n_new == 0 || a.batch == 0) return cudaSuccess;
  const int threads = a.n_kv_heads * a.head_dim / 8 < 256 ? a.n_kv_heads * a.head_dim / 8 : 256;
  f16_append_kernel<<<dim3(a.n_new, a.batch), (threads + 31) / 32 * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_attn_decode_f16(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.head_dim) {
    case 64: return launch_f16_d<64>(a, stream);
    case 128: return launch_f16_d<128>(a, stream);
    case 256: return launch_f16_d<256>(a, stream);
    case 512: return launch_f16_d<512>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ckv
