// pack_common.cuh — quantisation of one token position by one warp, shared by
// the packer and by the decode kernel's append of new tokens.
//
// K: q8_0 (PolyKV page, "F5 M6 — PolyKV (shared compressed KV pool)", section
// "What PolyKV is (reference)": K -> int8 q8_0, blocks of 32 with one fp16 scale).
// V: B-bit TurboQuant-MSE, B = 3 the method's TBQ3 (same section: FWHT rotation
// then Lloyd-Max; section "Phase-0 fork recon": the writer does the group
// transform with warp shuffles and bit-packs the codes; section "S2 — TurboQuant
// tier family": the same scheme at other bit widths, B = 2 and 4 here). Each lane holds D/32 consecutive values; the
// transform runs its first stages in registers and the rest across lanes with
// shuffles.
#pragma once

#include "ckv_device.cuh"

namespace ckv {
namespace pack {

// Lloyd-Max midpoints (nonnegative side) for the 8-level N(0,1) quantiser with
// centroids +/-0.2451, +/-0.7560, +/-1.3439, +/-2.1520.
__device__ __forceinline__ uint32_t tbq3_code(float u) {
  constexpr float t1 = 0.50055f, t2 = 1.04995f, t3 = 1.74795f;
  if (u >= 0.0f) {  // ties at a midpoint go to the smaller magnitude; u = 0 -> +0.2451
    return 4u + (u > t1) + (u > t2) + (u > t3);
  }
  return 3u - (u < -t1) - (u < -t2) - (u < -t3);
}

// Code of u at B bits: the index of the nearest centroid of the ascending
// B-bit table (tbq_centroid), comparing against the fp32 midpoints; ties go
// to the smaller magnitude and u = 0 to the smallest positive centroid.
template <int B>
__device__ __forceinline__ uint32_t tbq_code(float u) {
  if constexpr (B == 3) {
    return tbq3_code(u);
  } else if constexpr (B == 2) {
    constexpr float t1 = 0.9816f;  // (0.4528 + 1.5104) / 2
    if (u >= 0.0f) return 2u + (u > t1);
    return 1u - (u < -t1);
  } else {
    // (0.1284 + 0.3880) / 2, ..., (2.0690 + 2.7326) / 2
    constexpr float t1 = 0.2582f, t2 = 0.5224f, t3 = 0.79955f, t4 = 1.09925f, t5 = 1.4371f,
                    t6 = 1.8435f, t7 = 2.4008f;
    if (u >= 0.0f)
      return 8u + (u > t1) + (u > t2) + (u > t3) + (u > t4) + (u > t5) + (u > t6) + (u > t7);
    return 7u - (u < -t1) - (u < -t2) - (u < -t3) - (u < -t4) - (u < -t5) - (u < -t6) - (u < -t7);
  }
}

// Load E consecutive fp16 values as floats (16-byte loads where E allows).
template <int E>
__device__ __forceinline__ void load_row(const __half* p, float (&x)[E]) {
  if constexpr (E % 8 == 0) {
#pragma unroll
    for (int c = 0; c < E / 8; ++c) {
      const uint4 w = *reinterpret_cast<const uint4*>(p + 8 * c);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ws[j]));
        x[8 * c + 2 * j] = f.x;
        x[8 * c + 2 * j + 1] = f.y;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(p + e));
      x[e] = f.x;
      x[e + 1] = f.y;
    }
  }
}

// Stream word w of lane stream L: its byte offset inside a record.
template <int D, int B = 3>
__device__ __forceinline__ int v_word_offset(int L, int w) {
  constexpr int GR = v_granule(D, B);
  const int s = 4 * w;
  return v_code_offset(D) + ((s / GR) * 32 + L) * GR + (s % GR);
}

// Quantised forms of one position, per lane (values [E*lane, E*lane + E)).
template <int D, int B = 3>
struct PositionCodes {
  static constexpr int E = D / 32;
  // Window words: the compact bits span [0, 4BE - 5B), shifted by up to 31.
  static constexpr int NW = (4 * B * E - 5 * B + 31 + 31) / 32;
  uint8_t q[E];        // q8_0 codes, offset by 128
  __half d16;          // scale of this lane's block
  __half n16;          // fp16 norm (same in every lane)
  uint32_t val[NW];    // V code bits of the window, aligned to stream word w0
  uint32_t mask[NW];   // bits this position owns in those words
  int w0;              // first stream word of the window
  int L;               // lane stream
};

// This lane's values of one K row and one V row, and its sign entries.
template <int D>
struct PositionInput {
  static constexpr int E = D / 32;
  float kx[E], vx[E];
  int8_t sg[E];
};

template <int D>
__device__ __forceinline__ void load_position(const __half* krow, const __half* vrow, const int8_t* signs,
                                              int lane, PositionInput<D>& in) {
  constexpr int E = D / 32;
  load_row<E>(krow + lane * E, in.kx);
  load_row<E>(vrow + lane * E, in.vx);
#pragma unroll
  for (int e = 0; e < E; ++e) in.sg[e] = signs[lane * E + e];
}

// ROT = 1: the block-diagonal variant: each 128-dim group is transformed on
// its own (the butterfly stops at the group's lanes), the second sign diagonal
// `signs2` follows the transform, and each group has its own norm (every lane
// of a group holds it in n16).
template <int D, int B = 3, int ROT = 0>
__device__ __forceinline__ void quantise_loaded(const PositionInput<D>& in, int p, int lane,
                                                PositionCodes<D, B>& pc, const int8_t* signs2 = nullptr) {
  constexpr int E = D / 32;            // values per lane
  constexpr int LPB = 32 / E;          // lanes per q8_0 block
  using PC = PositionCodes<D, B>;
  const float (&kx)[E] = in.kx;
  const float (&vx)[E] = in.vx;

  // ---- K: q8_0 ----
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(kx[e]));
#pragma unroll
  for (int off = 1; off < LPB; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  pc.d16 = __float2half_rn(amax / 127.0f);  // IEEE division, then RNE to fp16
  const float d = __half2float(pc.d16);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    float q = 0.0f;
    if (d != 0.0f) {
      const float r = kx[e] / d;  // correctly rounded fp32 division
      q = copysignf(floorf(fabsf(r) + 0.5f), r);
      q = fminf(fmaxf(q, -127.0f), 127.0f);
    }
    // Stored offset by 128 (the byte q + 128): the readers then widen a code
    // to fp16 with byte permutes alone.
    pc.q[e] = static_cast<uint8_t>(static_cast<int8_t>(q)) ^ 0x80u;
  }

  // ---- V: B-bit TBQ ----
  float ss = 0.0f;
  float z[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    ss = fmaf(vx[e], vx[e], ss);
    z[e] = in.sg[e] < 0 ? -vx[e] : vx[e];
  }
  // Butterfly stages inside the lane (pairs closer than E apart).
#pragma unroll
  for (int hh = 1; hh < E; hh <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if ((e & hh) == 0) {
        const float x0 = z[e], x1 = z[e + hh];
        z[e] = x0 + x1;
        z[e + hh] = x0 - x1;
      }
    }
  }
  // Remaining stages across lanes: the partner lane differs in one lane bit.
  constexpr int LANES = ROT ? kRotGroup / E : 32;  // lanes per transform group
#pragma unroll
  for (int hl = 1; hl < LANES; hl <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, z[e], hl);
      z[e] = (lane & hl) ? (o - z[e]) : (z[e] + o);
    }
  }
  if constexpr (ROT) {
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (signs2[lane * E + e] < 0) z[e] = -z[e];
  }
#pragma unroll
  for (int off = LANES / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float r = sqrtf(ss);  // correctly rounded
  pc.n16 = __float2half_rn(r);

  // Bit positions. The lane's values i = E*lane + e all fall in the lane stream
  // L = 4 (i / G) + (p % 8) / 2 (G = D / 8 = 4 E), at pair field
  // k = 4 (u / 2) + u % 2 + 2 (p / 8) with u = i % G = E m + e (m = lane % 4),
  // bits [2B k + B (p % 2), +B). Relative to the lane's window start 4BE m:
  // 8B (e / 2) + 2B (e % 2) + 4B (p / 8) + B (p % 2).
  const int m = lane & 3;
  pc.L = 4 * (lane >> 2) + ((p & 7) >> 1);
  const int start = 4 * B * E * m + 4 * B * (p >> 3) + B * (p & 1);
  pc.w0 = start >> 5;
  const int sh = start & 31;
  // Compact form (shift 0), then one multiword shift by sh.
  uint32_t cv[PC::NW], cm[PC::NW];
#pragma unroll
  for (int w = 0; w < PC::NW; ++w) cv[w] = cm[w] = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    constexpr uint32_t kMask = (1u << B) - 1u;
    const uint32_t code = (r > 0.0f) ? tbq_code<B>(z[e] / r) : (1u << (B - 1));
    const int pos = 8 * B * (e >> 1) + 2 * B * (e & 1);  // compile-time
    const int wi = pos >> 5, bi = pos & 31;
    cv[wi] |= code << bi;
    cm[wi] |= kMask << bi;
    if (bi > 32 - B) {
      cv[wi + 1] |= code >> (32 - bi);
      cm[wi + 1] |= kMask >> (32 - bi);
    }
  }
#pragma unroll
  for (int w = PC::NW - 1; w >= 0; --w) {
    const uint32_t lo_v = (w > 0) ? cv[w - 1] : 0u, lo_m = (w > 0) ? cm[w - 1] : 0u;
    pc.val[w] = __funnelshift_l(lo_v, cv[w], sh);
    pc.mask[w] = __funnelshift_l(lo_m, cm[w], sh);
  }
}

template <int D, int B = 3, int ROT = 0>
__device__ __forceinline__ void quantise_position(const __half* krow, const __half* vrow, const int8_t* signs,
                                                  int p, int lane, PositionCodes<D, B>& pc,
                                                  const int8_t* signs2 = nullptr) {
  PositionInput<D> in;
  load_position<D>(krow, vrow, signs, lane, in);
  quantise_loaded<D, B, ROT>(in, p, lane, pc, signs2);
}

// Store a position's V norm(s) into a record: one per position, or (ROT) the
// first lane of every 128-dim group stores its group's norm at group-major
// offset 2 (16 j + p).
template <int D, int B, int ROT>
__device__ __forceinline__ void store_norm(uint8_t* rec, int p, int lane, __half n16) {
  if constexpr (ROT) {
    constexpr int LANES = kRotGroup / (D / 32);
    if (lane % LANES == 0) *reinterpret_cast<__half*>(rec + v_norm_offset(D, B) + 2 * (16 * (lane / LANES) + p)) = n16;
  } else {
    if (lane == 0) *reinterpret_cast<__half*>(rec + v_norm_offset(D, B) + 2 * p) = n16;
  }
}

// Byte offset inside a record of the 8-byte K-code chunk that holds dims
// [8c, 8c + 8) of position p.
__device__ __forceinline__ int k_chunk_byte(int p, int c) {
  const int lane = 4 * (p & 7) + (c & 3);
  return ((c >> 2) * 32 + lane) * 16 + (p >> 3) * 8;
}

// Store the lane's K codes (E bytes starting at dim E * lane) at `rec` (a record
// in shared or global memory).
template <int E>
__device__ __forceinline__ void store_k_codes(uint8_t* rec, int p, int lane, const uint8_t (&q)[E]) {
  if constexpr (E >= 8) {
#pragma unroll
    for (int c = 0; c < E / 8; ++c) {
      uint2 w;
      w.x = (uint32_t)q[8 * c] | ((uint32_t)q[8 * c + 1] << 8) | ((uint32_t)q[8 * c + 2] << 16) |
            ((uint32_t)q[8 * c + 3] << 24);
      w.y = (uint32_t)q[8 * c + 4] | ((uint32_t)q[8 * c + 5] << 8) | ((uint32_t)q[8 * c + 6] << 16) |
            ((uint32_t)q[8 * c + 7] << 24);
      *reinterpret_cast<uint2*>(rec + k_chunk_byte(p, (E * lane) / 8 + c)) = w;
    }
  } else {
    // E = 4 or 2: the lane's bytes sit inside one 8-byte chunk.
    const int i0 = E * lane;
    uint8_t* dst = rec + k_chunk_byte(p, i0 / 8) + (i0 % 8);
    if constexpr (E == 4) {
      *reinterpret_cast<uint32_t*>(dst) = (uint32_t)q[0] | ((uint32_t)q[1] << 8) | ((uint32_t)q[2] << 16) |
                                          ((uint32_t)q[3] << 24);
    } else {
      *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(q[0] | (q[1] << 8));
    }
  }
}


// Write a quantised position straight into a record in global memory: plain
// stores for its K codes, scale and norm; word-wide atomic AND then OR for its
// V fields, whose words it shares with the other positions of the record.
// Positions own disjoint bits, so concurrent writers of one record commute.
template <int D, int B = 3, int ROT = 0>
__device__ __forceinline__ void store_position_global(uint8_t* grec, int p, int lane,
                                                      const PositionCodes<D, B>& pc) {
  constexpr int E = D / 32;
  constexpr int LPB = 32 / E;
  using PC = PositionCodes<D, B>;
  store_k_codes<E>(grec, p, lane, pc.q);
  if (lane % LPB == 0)
    *reinterpret_cast<__half*>(grec + k_scale_offset(D) + 2 * (p * (D / 32) + lane / LPB)) = pc.d16;
  store_norm<D, B, ROT>(grec, p, lane, pc.n16);
#pragma unroll
  for (int w = 0; w < PC::NW; ++w) {
    if (pc.mask[w]) {
      uint32_t* word = reinterpret_cast<uint32_t*>(grec + v_word_offset<D, B>(pc.L, pc.w0 + w));
      atomicAnd(word, ~pc.mask[w]);
      atomicOr(word, pc.val[w]);
    }
  }
}

}  // namespace pack
}  // namespace ckv
