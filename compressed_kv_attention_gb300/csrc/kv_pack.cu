// kv_pack.cu — quantise new K/V rows into the packed cache.
//
// K: q8_0 (PolyKV page, "F5 M6 — PolyKV (shared compressed KV pool)", section
// "What PolyKV is (reference)": K -> int8 q8_0, blocks of 32 with one fp16 scale).
// V: B-bit TurboQuant-MSE, B = 3 by default and 2 or 4 for the other tiers
// (same section: FWHT rotation then Lloyd-Max; section "Phase-0 fork recon":
// the writer does the group transform with warp shuffles and bit-packs the
// codes). One warp owns one token position (pack_common.cuh).
//
// Two ways to write a position, chosen per tile record (CTA-uniform):
//  * a record whose 16 positions are all new is assembled in shared memory and
//    written back with coalesced 16-byte stores (bulk packing, prefill);
//  * a record that is only partly rewritten (the decode append of one token,
//    the ragged ends of a range) is updated in place: the position's K codes,
//    scale and norm are plain stores, and its B-bit V fields, which share
//    32-bit words with the other positions of the record, are cleared and set
//    with word-wide atomic AND / OR on global memory. Positions own disjoint
//    bits, so concurrent writers of one record cannot disturb each other.
#include "ckv_kernels.cuh"
#include "pack_common.cuh"

namespace ckv {

template <int D, int B, int ROT>
__global__ void __launch_bounds__(512) kv_pack_kernel(PackArgs a) {
  constexpr int REC = record_bytes(D, B, ROT ? D / kRotGroup : 1);
  constexpr int E = D / 32;
  constexpr int LPB = 32 / E;
  using PC = pack::PositionCodes<D, B>;
  __shared__ __align__(16) uint8_t rec[REC];

  const int bh = blockIdx.y;
  const int b = bh / a.n_kv_heads, h = bh % a.n_kv_heads;
  const int64_t tile = a.tok_offset / kTile + blockIdx.x;
  const int64_t pos0 = tile * kTile;
  const int64_t lo = a.tok_offset > pos0 ? a.tok_offset : pos0;
  const int64_t end = a.tok_offset + a.n_tok;
  const int64_t hi = end < pos0 + kTile ? end : pos0 + kTile;
  const bool full = (lo == pos0) && (hi == pos0 + kTile);
  uint8_t* grec = a.cache + ((int64_t)(b * a.n_kv_heads + h) * (a.capacity / kTile) + tile) * REC;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p = warp;  // one warp per position
  const int64_t pos = pos0 + p;

  if (full) {
    // Every byte of the record is rewritten: only the V code region, which is
    // OR-ed together from the 16 positions, starts from zero.
    for (int ofs = v_code_offset(D) + threadIdx.x * 16; ofs < v_norm_offset(D, B); ofs += blockDim.x * 16)
      *reinterpret_cast<uint4*>(rec + ofs) = make_uint4(0, 0, 0, 0);
    __syncthreads();
    {
      const int64_t j = pos - a.tok_offset;
      const __half* krow = a.k + b * a.batch_stride + j * a.token_stride + (int64_t)h * D;
      const __half* vrow = a.v + b * a.batch_stride + j * a.token_stride + (int64_t)h * D;
      PC pc;
      pack::quantise_position<D, B, ROT>(krow, vrow, a.signs, p, lane, pc, a.signs2);
      pack::store_k_codes<E>(rec, p, lane, pc.q);
      if (lane % LPB == 0)
        *reinterpret_cast<__half*>(rec + k_scale_offset(D) + 2 * (p * (D / 32) + lane / LPB)) = pc.d16;
      pack::store_norm<D, B, ROT>(rec, p, lane, pc.n16);
#pragma unroll
      for (int w = 0; w < PC::NW; ++w)
        if (pc.mask[w])
          atomicOr(reinterpret_cast<uint32_t*>(rec + pack::v_word_offset<D, B>(pc.L, pc.w0 + w)), pc.val[w]);
    }
    __syncthreads();
    for (int ofs = threadIdx.x * 16; ofs < REC; ofs += blockDim.x * 16)
      *reinterpret_cast<uint4*>(grec + ofs) = *reinterpret_cast<const uint4*>(rec + ofs);
    return;
  }

  // Partly rewritten record: update this position's bytes and bits in place.
  if (pos < lo || pos >= hi) return;
  const int64_t j = pos - a.tok_offset;
  const __half* krow = a.k + b * a.batch_stride + j * a.token_stride + (int64_t)h * D;
  const __half* vrow = a.v + b * a.batch_stride + j * a.token_stride + (int64_t)h * D;
  PC pc;
  pack::quantise_position<D, B, ROT>(krow, vrow, a.signs, p, lane, pc, a.signs2);
  pack::store_position_global<D, B, ROT>(grec, p, lane, pc);
}

template <int D, int B, int ROT>
static cudaError_t launch_pack_dbr(const PackArgs& a, dim3 grid, cudaStream_t stream) {
  // Same shared-memory carveout as the decode kernels, so that an SM does not
  // reconfigure its L1 / shared split between a pack and the decode after it.
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(kv_pack_kernel<D, B, ROT>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    configured = true;
  }
  kv_pack_kernel<D, B, ROT><<<grid, 512, 0, stream>>>(a);
  return cudaGetLastError();
}

template <int D, int B>
static cudaError_t launch_pack_db(const PackArgs& a, dim3 grid, cudaStream_t stream) {
  if constexpr (D >= kRotGroup) {
    if (a.rot) return launch_pack_dbr<D, B, 1>(a, grid, stream);
  } else {
    if (a.rot) return cudaErrorInvalidValue;
  }
  return launch_pack_dbr<D, B, 0>(a, grid, stream);
}

template <int D>
static cudaError_t launch_pack_d(const PackArgs& a, dim3 grid, cudaStream_t stream) {
  switch (a.v_bits) {
    case 2: return launch_pack_db<D, 2>(a, grid, stream);
    case 3: return launch_pack_db<D, 3>(a, grid, stream);
    case 4: return launch_pack_db<D, 4>(a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_kv_pack(const PackArgs& a, cudaStream_t stream) {
  if (a.n_tok == 0) return cudaSuccess;
  const int64_t t0 = a.tok_offset / kTile;
  const int64_t t1 = (a.tok_offset + a.n_tok - 1) / kTile;
  dim3 grid(static_cast<unsigned>(t1 - t0 + 1), static_cast<unsigned>(a.batch * a.n_kv_heads));
  switch (a.head_dim) {
    case 64: return launch_pack_d<64>(a, grid, stream);
    case 128: return launch_pack_d<128>(a, grid, stream);
    case 256: return launch_pack_d<256>(a, grid, stream);
    case 512: return launch_pack_d<512>(a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ckv
