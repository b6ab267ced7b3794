// ckv_device.cuh — device helpers shared by the kernels of the compressed-KV
// attention library (sm_103a): shared-memory addresses, mbarriers with bounded
// waits, bulk global->shared copies, warp-level tensor-core mma and movmatrix,
// and the cache-record geometry.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace ckv {

// ---------------------------------------------------------------- geometry --

constexpr int kTile = 16;  // token positions per tile record

// A record holds 16 positions: K codes [0, 16D), K scales [16D, 17D), V codes
// at B bits per value [17D, 17D + 2BD), V norms (32 bytes per norm group).
// B = 3 is TBQ3; 2 and 4 are the neighbouring tiers of the same quantiser.
// NG = 1 norm per position for the full D-point transform, D / 128 for the
// block-diagonal rotation; norm (p, j) at v_norm_offset + 2 (16 j + p).
__host__ __device__ constexpr int record_bytes(int D, int B = 3, int NG = 1) {
  return 17 * D + 2 * B * D + 32 * NG;
}
constexpr int kRotGroup = 128;  // dims per group of the block-diagonal rotation
__host__ __device__ constexpr int k_scale_offset(int D) { return 16 * D; }
__host__ __device__ constexpr int v_code_offset(int D) { return 17 * D; }
__host__ __device__ constexpr int v_norm_offset(int D, int B = 3) { return 17 * D + 2 * B * D; }
// Bytes of one lane's V-code stream in a record, and the granule in which it is interleaved.
__host__ __device__ constexpr int v_lane_bytes(int D, int B = 3) { return B * D / 16; }
__host__ __device__ constexpr int v_granule(int D, int B = 3) {
  return (v_lane_bytes(D, B) % 16 == 0) ? 16 : (v_lane_bytes(D, B) % 8 == 0) ? 8 : 4;
}

// The centroids enter the tensor cores as fp16 values of c / scale and the
// output is multiplied back by the scale. 3 bits: with 1.7475121 all four
// centroid magnitudes lie within 1.6e-5 (relative) of an fp16 value, where
// plain fp16 rounding of 0.7560 is off by 1.9e-4. 2 bits: 0.4528 / 1.6384 and
// 1.5104 / 1.6384 are exact fp16 values (283/1024, 944/1024). 4 bits: with
// 1.251395 the eight magnitudes lie within 9.3e-5 of fp16 values (plain
// rounding: 3.1e-4).
constexpr float kCentroidScale = 1.7475121f;
__host__ __device__ constexpr float centroid_scale(int B) {
  return B == 2 ? 1.6384f : B == 4 ? 1.251395f : kCentroidScale;
}

// Ascending Lloyd-Max centroids of N(0,1) for B-bit codes k (selects on
// immediates, no memory): 2 bits +/-0.4528, +/-1.5104; 3 bits +/-0.2451,
// +/-0.7560, +/-1.3439, +/-2.1520; 4 bits +/-0.1284, +/-0.3880, +/-0.6568,
// +/-0.9423, +/-1.2562, +/-1.6180, +/-2.0690, +/-2.7326.
template <int B>
__host__ __device__ __forceinline__ float tbq_centroid(int k) {
  constexpr int H = 1 << (B - 1);
  const int m = (k >= H) ? k - H : H - 1 - k;  // magnitude rank
  float mag;
  if constexpr (B == 2) {
    mag = (m == 0) ? 0.4528f : 1.5104f;
  } else if constexpr (B == 3) {
    mag = (m == 0) ? 0.2451f : (m == 1) ? 0.7560f : (m == 2) ? 1.3439f : 2.1520f;
  } else {
    mag = (m == 0) ? 0.1284f : (m == 1) ? 0.3880f : (m == 2) ? 0.6568f : (m == 3) ? 0.9423f
        : (m == 4) ? 1.2562f : (m == 5) ? 1.6180f : (m == 6) ? 2.0690f : 2.7326f;
  }
  return (k >= H) ? mag : -mag;
}

// Error codes written to the workspace flag word.
enum DeviceFlag : int32_t {
  kFlagNone = 0,
  kFlagWaitTimeout = 1,   // a bounded mbarrier wait ran out
  kFlagSeqLenRange = 2,   // seq_len[b] outside [0, min(capacity, max_seq_len)]
  kFlagInternal = 3,      // a work schedule the kernel cannot run (a library bug)
};

// ------------------------------------------------------------------- misc --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void raise_flag(int32_t* flag, int32_t code) {
  if (flag) atomicCAS(flag, 0, code);
}

// Bound for every wait on an asynchronous event: 2 s of wall time.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Barrier over `threads` threads (whole warps) of the CTA, id 1..15.
__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// --------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; gives up after
// kWaitLimitNs and returns false (the caller raises the device flag).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ------------------------------------------------------------ bulk copies --

// One bulk copy global -> shared (16-byte aligned addresses, size multiple of 16)
// completing on `bar` (transaction bytes).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------- programmatic launch --

// With programmatic stream serialisation a grid may start while the grid
// before it on the stream is still running. griddep_wait returns once that
// grid has completed and its memory operations are visible (at once when the
// launch had no such dependency); nothing before it may read or write global
// memory that another kernel touches. griddep_launch_dependents lets the next
// grid on the stream begin its own launch.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Order this thread's generic-proxy accesses (global data acquired from other
// CTAs, shared memory it used) before its later async-proxy (bulk copy) ones.
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

// ------------------------------------------------------------ shared loads --

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// --------------------------------------------------------- tensor-core mma --

// D = A(16x16, row) * B(16x8, col) + C, fp16 inputs, fp32 accumulate.
// Fragment ownership (lane = 4*g + t): a0 = A[g][2t..2t+1], a1 = A[g+8][2t..],
// a2 = A[g][2t+8..2t+9], a3 = A[g+8][2t+8..]; b0 = B[2t..2t+1][g], b1 = B[2t+8..][g];
// c0 = C[g][2t], c1 = C[g][2t+1], c2 = C[g+8][2t], c3 = C[g+8][2t+1].
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same with a zero accumulator input.
__device__ __forceinline__ void mma16816_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// Transpose an 8x8 matrix of 16-bit values held one row-pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Pack two fp32 into fp16x2 (round to nearest even): lo -> bits 0..15, hi -> 16..31.
// Lane-wise fp16 product of two packed fp16 pairs (one rounding per half).
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t x, uint32_t y) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
  return r;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four K codes (one 32-bit word, each the byte q + 128) -> two fp16x2 holding
// the integers q exactly: byte u becomes fp16 (1024 + u) - 1152 = q.
__device__ __forceinline__ void i8x4_to_half2x2(uint32_t u, uint32_t& lo, uint32_t& hi) {
  const uint32_t e = 0x64646464u;
  uint32_t x0, x1;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(x0) : "r"(u), "r"(e));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(x1) : "r"(u), "r"(e));
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 h0 = __hsub2(*reinterpret_cast<__half2*>(&x0), bias);
  __half2 h1 = __hsub2(*reinterpret_cast<__half2*>(&x1), bias);
  lo = *reinterpret_cast<uint32_t*>(&h0);
  hi = *reinterpret_cast<uint32_t*>(&h1);
}

// Four K codes (one 32-bit word, each the byte q + 128 in [1, 255]) -> two
// fp16x2 holding (q + 128) * 2^-24: a byte in the low half of an fp16 with a
// zero high half is exactly that many units of the smallest subnormal. The constant 128 * 2^-24 per code is removed by
// starting the accumulator at -2^-17 times the sum of the other operand.
__device__ __forceinline__ void i8x4_to_sub_half2x2(uint32_t u, uint32_t& lo, uint32_t& hi) {
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(u), "r"(0u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(u), "r"(0u));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace ckv

namespace ckv {

// ------------------------------------------------------------- tcgen05 --
// Fifth-generation tensor core (sm_100 family): single-thread MMA issue with
// operands in shared memory (described by 64-bit matrix descriptors) and the
// accumulator in tensor memory (TMEM), completion tracked by an mbarrier.

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzle layout: rows of 128 bytes (64 fp16), 8-row groups 1024 bytes apart
// (stride byte offset), 16-byte chunk c of row r stored at chunk c ^ (r % 8);
// the group base must be 1024-byte aligned. Fields: start address >> 4
// [0,14), leading byte offset >> 4 [16,30) (unused with this swizzle),
// stride byte offset >> 4 [32,46), descriptor version 1 [46,48), layout
// type 2 = 128-byte swizzle [61,64).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
  return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16 with fp16 A and B, fp32 accumulator, both
// operands K-major: c_format F32 at bit 4, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t umma_idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, one instruction (K = 16), issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u));
}

// Arrive on `bar` once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Make generic-proxy shared-memory writes visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 lanes x 32 consecutive columns of 32-bit TMEM words; lane i of the warp gets
// TMEM lane (quarter*32 + i). The caller waits with tmem_ld_wait().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Byte offset of element (row, k) of a K-major fp16 tile stored as 128-byte
// swizzled atoms: [k / 64 atoms][rows][128 B], atom stride rows * 128 bytes.
__device__ __forceinline__ uint32_t sw128_offset(int row, int k, int rows) {
  const int byte = (k & 63) * 2;
  return (uint32_t)((k >> 6) * rows * 128 + row * 128 + ((((byte >> 4) ^ (row & 7))) << 4) + (byte & 15));
}

}  // namespace ckv
