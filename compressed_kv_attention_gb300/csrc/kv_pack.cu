// kv_pack.cu — quantise new K/V rows into the packed cache.
//
// K: q8_0 (PolyKV page, "F5 M6 — PolyKV (shared compressed KV pool)", section
// "What PolyKV is (reference)": K -> int8 q8_0, blocks of 32 with one fp16 scale).
// V: 3-bit TurboQuant-MSE (same section: FWHT rotation then Lloyd-Max; section
// "Phase-0 fork recon": the writer does the group transform with warp shuffles
// and bit-packs the codes). Here one warp owns one token position: each lane
// holds D/32 consecutive values, the transform runs its first stages in
// registers and the rest across lanes with shuffles, and the 3-bit codes are
// OR-ed into the tile record in shared memory before one coalesced write-back.
#include "ckv_kernels.cuh"

namespace ckv {

namespace {

// Lloyd-Max midpoints (nonnegative side) for the 8-level N(0,1) quantiser with
// centroids +/-0.2451, +/-0.7560, +/-1.3439, +/-2.1520.
__device__ __forceinline__ uint32_t tbq3_code(float u) {
  constexpr float t1 = 0.50055f, t2 = 1.04995f, t3 = 1.74795f;
  if (u >= 0.0f) {  // ties at a midpoint go to the smaller magnitude; u = 0 -> +0.2451
    return 4u + (u > t1) + (u > t2) + (u > t3);
  }
  return 3u - (u < -t1) - (u < -t2) - (u < -t3);
}

// Byte offset inside a record of the K code of (position p, dim i).
__device__ __forceinline__ int k_code_byte(int p, int i) {
  const int lane = 4 * (p & 7) + ((i & 31) >> 3);
  return ((i >> 5) * 32 + lane) * 16 + (p >> 3) * 8 + (i & 7);
}

// Absolute bit index inside a record of bit k of the V code of (p, i).
template <int D>
__device__ __forceinline__ int v_code_bit(int p, int i, int k) {
  constexpr int G = D / 8;
  constexpr int GR = v_granule(D);
  const int g = i / G, u = i % G;
  const int lane = 4 * g + ((p & 7) >> 1);
  const int pair = 4 * (u >> 1) + (u & 1) + 2 * (p >> 3);
  const int sb = 6 * pair + 3 * (p & 1) + k;
  const int s = sb >> 3;
  const int byte = v_code_offset(D) + ((s / GR) * 32 + lane) * GR + (s % GR);
  return byte * 8 + (sb & 7);
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(512) kv_pack_kernel(PackArgs a) {
  constexpr int REC = record_bytes(D);
  constexpr int E = D / 32;            // values per lane
  constexpr int LPB = 32 / E;          // lanes per q8_0 block
  __shared__ __align__(16) uint8_t rec[REC];
  uint32_t* rec32 = reinterpret_cast<uint32_t*>(rec);

  const int bh = blockIdx.y;
  const int b = bh / a.n_kv_heads, h = bh % a.n_kv_heads;
  const int64_t tile = a.tok_offset / kTile + blockIdx.x;
  const int64_t pos0 = tile * kTile;
  const int64_t lo = a.tok_offset > pos0 ? a.tok_offset : pos0;
  const int64_t end = a.tok_offset + a.n_tok;
  const int64_t hi = end < pos0 + kTile ? end : pos0 + kTile;
  const bool full = (lo == pos0) && (hi == pos0 + kTile);
  uint8_t* grec = a.cache + ((int64_t)(b * a.n_kv_heads + h) * (a.capacity / kTile) + tile) * REC;

  // Start from the existing record when the tile is only partly rewritten;
  // otherwise every byte is overwritten except the V code bits, which are OR-ed.
  for (int ofs = threadIdx.x * 16; ofs < REC; ofs += blockDim.x * 16) {
    uint4 val = make_uint4(0, 0, 0, 0);
    if (!full) val = *reinterpret_cast<const uint4*>(grec + ofs);
    *reinterpret_cast<uint4*>(rec + ofs) = val;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p = warp;  // one warp per position
  const int64_t pos = pos0 + p;
  if (pos >= lo && pos < hi) {
    const int64_t j = pos - a.tok_offset;
    const __half* krow = a.k + b * a.batch_stride + j * a.token_stride + (int64_t)h * D + lane * E;
    const __half* vrow = a.v + b * a.batch_stride + j * a.token_stride + (int64_t)h * D + lane * E;
    float kx[E], vx[E];
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const __half2 k2 = *reinterpret_cast<const __half2*>(krow + e);
      const __half2 v2 = *reinterpret_cast<const __half2*>(vrow + e);
      kx[e] = __low2float(k2);
      kx[e + 1] = __high2float(k2);
      vx[e] = __low2float(v2);
      vx[e + 1] = __high2float(v2);
    }

    // ---- K: q8_0 ----
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(kx[e]));
#pragma unroll
    for (int off = 1; off < LPB; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const __half d16 = __float2half_rn(amax / 127.0f);  // IEEE division, then RNE to fp16
    const float d = __half2float(d16);
    uint8_t qb[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float q = 0.0f;
      if (d != 0.0f) {
        const float r = kx[e] / d;  // correctly rounded fp32 division
        q = copysignf(floorf(fabsf(r) + 0.5f), r);
        q = fminf(fmaxf(q, -127.0f), 127.0f);
      }
      qb[e] = static_cast<uint8_t>(static_cast<int8_t>(q));
    }
#pragma unroll
    for (int e = 0; e < E; ++e) rec[k_code_byte(p, lane * E + e)] = qb[e];
    if ((lane * E) % 32 == 0) {
      const int nb = (lane * E) / 32;
      *reinterpret_cast<__half*>(rec + k_scale_offset(D) + 2 * (p * (D / 32) + nb)) = d16;
    }

    // ---- V: TBQ3 ----
    float ss = 0.0f;
    float z[E];
    const int8_t* sg = a.signs + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      ss = fmaf(vx[e], vx[e], ss);
      z[e] = sg[e] < 0 ? -vx[e] : vx[e];
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
    // Remaining stages across lanes: partner lane differs in bit (hh / E).
#pragma unroll
    for (int hl = 1; hl < 32; hl <<= 1) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, z[e], hl);
        z[e] = (lane & hl) ? (o - z[e]) : (z[e] + o);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float r = sqrtf(ss);  // correctly rounded
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const uint32_t code = (r > 0.0f) ? tbq3_code(z[e] / r) : 4u;
      const int i = lane * E + e;
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int bit = v_code_bit<D>(p, i, k);
        const uint32_t m = 1u << (bit & 31);
        if ((code >> k) & 1u) atomicOr(&rec32[bit >> 5], m);
        else if (!full) atomicAnd(&rec32[bit >> 5], ~m);
      }
    }
    if (lane == 0) *reinterpret_cast<__half*>(rec + v_norm_offset(D) + 2 * p) = __float2half_rn(r);
  }
  __syncthreads();
  for (int ofs = threadIdx.x * 16; ofs < REC; ofs += blockDim.x * 16)
    *reinterpret_cast<uint4*>(grec + ofs) = *reinterpret_cast<const uint4*>(rec + ofs);
}

cudaError_t launch_kv_pack(const PackArgs& a, cudaStream_t stream) {
  if (a.n_tok == 0) return cudaSuccess;
  const int64_t t0 = a.tok_offset / kTile;
  const int64_t t1 = (a.tok_offset + a.n_tok - 1) / kTile;
  dim3 grid(static_cast<unsigned>(t1 - t0 + 1), static_cast<unsigned>(a.batch * a.n_kv_heads));
  // Same shared-memory carveout as the decode kernels, so that an SM does not
  // reconfigure its L1 / shared split between a pack and the decode after it.
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(kv_pack_kernel<64>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    cudaFuncSetAttribute(kv_pack_kernel<128>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    cudaFuncSetAttribute(kv_pack_kernel<256>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    cudaFuncSetAttribute(kv_pack_kernel<512>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    configured = true;
  }
  switch (a.head_dim) {
    case 64: kv_pack_kernel<64><<<grid, 512, 0, stream>>>(a); break;
    case 128: kv_pack_kernel<128><<<grid, 512, 0, stream>>>(a); break;
    case 256: kv_pack_kernel<256><<<grid, 512, 0, stream>>>(a); break;
    case 512: kv_pack_kernel<512><<<grid, 512, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ckv
