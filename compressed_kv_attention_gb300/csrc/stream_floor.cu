// stream_floor.cu — calibration: the decode's data movement with no compute.
//
// The split-K decode of a short cache (the Gemma-4 global-layer step: 48 MB
// of tile records over 152 CTAs) is bounded by fixed costs as much as by HBM
// bandwidth: the wait for the previous grid, the first stage's round trip,
// and the cross-CTA merge. This kernel streams the same records through the
// same staging (one CTA per (split, stream), a producer lane issuing one bulk
// copy of NP records per stage into a 4-stage shared-memory ring, the first
// two stages at once and each later first-round stage after the one two
// before it has landed; 8 consumer warps releasing each stage) with the same
// programmatic launch, and optionally ends with the same counter rendezvous of
// the CTAs of a stream. Its time per launch, back to back, is the floor that
// any kernel with this launch shape and staging can reach on the same bytes;
// it computes nothing from them.
#include <cuda_runtime.h>

#include "../../include/ckv.h"
#include "ckv_kernels.cuh"

namespace {

constexpr int kNP = 4;       // records per stage (one per consumer pair of the decode)
constexpr int kNStage = 4;   // ring depth
constexpr int kEarly = 2;    // stages issued at once at the start
constexpr int kNCW = 8;      // consumer warps

struct FloorArgs {
  const uint8_t* src;
  int64_t n_tiles;   // records per stream
  int rec;           // bytes per record
  int n_split;
  int rendezvous;
  int32_t* flag;
  uint32_t* counters;  // two per stream
};

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__global__ void __launch_bounds__((kNCW + 1) * 32, 1) stream_floor_kernel(FloorArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kNStage], empty[kNStage];
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, s_id = blockIdx.z;
  const int64_t t0 = split * a.n_tiles / a.n_split, t1 = (split + 1) * a.n_tiles / a.n_split;
  const int n_iters = static_cast<int>((t1 - t0 + kNP - 1) / kNP);
  const uint8_t* base = a.src + (s_id * a.n_tiles + t0) * a.rec;
  const int stage_bytes = kNP * a.rec;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNStage; ++s) {
      ckv::mbar_init(&full[s], 1);
      ckv::mbar_init(&empty[s], kNCW);
    }
    s_abort = 0;
    ckv::fence_barrier_init();
  }
  __syncthreads();
  ckv::griddep_wait();
  ckv::griddep_launch_dependents();

  if (warp == kNCW) {
    if (lane == 0) {
      int issued = 0;
      for (int it = 0; it < n_iters; ++it) {
        const int s = it % kNStage;
        bool ok = true;
        if (it >= kNStage) ok = ckv::mbar_wait(&empty[s], ((it / kNStage) - 1) & 1);
        else if (it >= kEarly) ok = ckv::mbar_wait(&full[it - kEarly], 0);
        if (!ok) {
          s_abort = 1;
          ckv::raise_flag(a.flag, ckv::kFlagWaitTimeout);
          break;
        }
        const int64_t left = t1 - (t0 + (int64_t)it * kNP);
        const uint32_t bytes = static_cast<uint32_t>(left < kNP ? left : kNP) * a.rec;
        ckv::mbar_arrive_expect_tx(&full[s], bytes);
        ckv::bulk_g2s(smem + s * stage_bytes, base + (int64_t)it * stage_bytes, bytes, &full[s]);
        ++issued;
      }
      // Do not leave while a copy may still be landing in this CTA's memory.
      for (int k = issued > kNStage ? issued - kNStage : 0; k < issued; ++k)
        if (!ckv::mbar_wait(&full[k % kNStage], (k / kNStage) & 1)) break;
    }
    return;
  }
  for (int it = 0; it < n_iters; ++it) {
    if (!*(volatile int*)&s_abort && !ckv::mbar_wait(&full[it % kNStage], (it / kNStage) & 1)) {
      *(volatile int*)&s_abort = 1;
      if (lane == 0) ckv::raise_flag(a.flag, ckv::kFlagWaitTimeout);
    }
    __syncwarp();
    if (lane == 0) ckv::mbar_arrive(&empty[it % kNStage]);
  }
  if (!a.rendezvous) return;
  // The decode's split rendezvous: arrive, wait (bounded) for the stream's
  // other CTAs, count departures; the last to leave resets both counters.
  __syncwarp();
  if (threadIdx.x == 0) {
    uint32_t* arrive = a.counters + 2 * s_id;
    uint32_t* depart = arrive + 1;
    const uint32_t n = static_cast<uint32_t>(a.n_split);
    __threadfence();
    atomicAdd(arrive, 1u);
    const uint64_t start = ckv::global_timer_ns();
    for (uint32_t k = 1; ld_acquire(arrive) < n; ++k) {
      if ((k & 255u) == 0 && ckv::global_timer_ns() - start > ckv::kWaitLimitNs) {
        ckv::raise_flag(a.flag, ckv::kFlagWaitTimeout);
        return;
      }
      __nanosleep(64);
    }
    if (atomicAdd(depart, 1u) + 1 == n) {
      *arrive = 0u;
      *depart = 0u;
    }
  }
}

}  // namespace

extern "C" CKV_API ckv_status ckv_calibrate_stream(const void* src, int64_t n_tiles, int32_t record_bytes,
                                                   int32_t n_streams, int32_t n_split, int32_t rendezvous,
                                                   void* workspace, size_t ws_bytes, void* stream) {
  const size_t need = 64 + 8 * static_cast<size_t>(n_streams > 0 ? n_streams : 0);
  if (!src || (reinterpret_cast<uintptr_t>(src) & 15) || n_tiles <= 0 || record_bytes <= 0 ||
      record_bytes % 16 || n_streams <= 0 || n_split <= 0 || n_split > 1024 ||
      static_cast<int64_t>(kNStage) * kNP * record_bytes > 200 * 1024)
    return static_cast<ckv_status>(ckv::set_last_error(CKV_ERR_INVALID_ARG, "calibrate_stream: bad arguments"));
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return static_cast<ckv_status>(
        ckv::set_last_error(CKV_ERR_WORKSPACE, "calibrate_stream: needs %zu zero-filled bytes, 256-aligned", need));
  FloorArgs a{};
  a.src = static_cast<const uint8_t*>(src);
  a.n_tiles = n_tiles;
  a.rec = record_bytes;
  a.n_split = n_split;
  a.rendezvous = rendezvous;
  a.flag = static_cast<int32_t*>(workspace);
  a.counters = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + 64);
  const int smem = kNStage * kNP * record_bytes;
  static int configured = 0;
  if (configured < smem) {
    const cudaError_t e = cudaFuncSetAttribute(stream_floor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               200 * 1024);
    if (e != cudaSuccess)
      return static_cast<ckv_status>(ckv::set_last_error(CKV_ERR_CUDA, "calibrate_stream: %s", cudaGetErrorString(e)));
    configured = 200 * 1024;
  }
  if (rendezvous) {
    // The rendezvous waits for every CTA of a stream: the grid must fit on the device at once.
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stream_floor_kernel, (kNCW + 1) * 32, smem) !=
            cudaSuccess ||
        static_cast<int64_t>(n_split) * n_streams > static_cast<int64_t>(sms) * per_sm)
      return static_cast<ckv_status>(
          ckv::set_last_error(CKV_ERR_UNSUPPORTED, "calibrate_stream: rendezvous grid does not fit at once"));
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_split, 1, n_streams);
  cfg.blockDim = dim3((kNCW + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, stream_floor_kernel, a);
  if (e != cudaSuccess)
    return static_cast<ckv_status>(ckv::set_last_error(CKV_ERR_CUDA, "calibrate_stream launch: %s", cudaGetErrorString(e)));
  return CKV_OK;
}
