// selftest.cu — check of the failure path every asynchronous wait takes.
//
// Every wait in the library's kernels (an mbarrier phase, a counter in global
// memory written by other CTAs) is bounded by kWaitLimitNs of wall time, after
// which the kernel raises kFlagWaitTimeout in the workspace's device flag and
// carries on, so a lost event turns into an error status on the host instead
// of a hung context. This entry point runs both forms of wait on events that
// never come and lets the caller check that the flag reports it and that the
// context still runs work afterwards.
#include <cuda_runtime.h>

#include "../../include/ckv.h"
#include "ckv_kernels.cuh"

namespace {

__device__ __forceinline__ uint32_t load_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__global__ void bounded_wait_selftest_kernel(int32_t* flag, const uint32_t* counter) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  // 1. An mbarrier phase nothing completes (the stage waits' form).
  ckv::mbar_init(&bar, 1);
  ckv::fence_barrier_init();
  if (!ckv::mbar_wait(&bar, 0)) ckv::raise_flag(flag, ckv::kFlagWaitTimeout);
  // 2. A global counter nothing raises (the split rendezvous' form).
  const uint64_t t0 = ckv::global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (load_acquire(counter) >= 1u) break;
    if ((it & 255u) == 0 && ckv::global_timer_ns() - t0 > ckv::kWaitLimitNs) {
      ckv::raise_flag(flag + 1, ckv::kFlagWaitTimeout);
      break;
    }
    __nanosleep(64);
  }
}

}  // namespace

extern "C" CKV_API ckv_status ckv_selftest_bounded_waits(void* workspace, size_t ws_bytes, void* stream) {
  if (!workspace || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return static_cast<ckv_status>(
        ckv::set_last_error(CKV_ERR_WORKSPACE, "selftest needs 256 zero-filled bytes, 256-byte aligned"));
  int32_t* flag = static_cast<int32_t*>(workspace);
  const uint32_t* counter = reinterpret_cast<const uint32_t*>(static_cast<uint8_t*>(workspace) + 64);
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(flag, counter);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return static_cast<ckv_status>(ckv::set_last_error(CKV_ERR_CUDA, "selftest launch: %s", cudaGetErrorString(e)));
  return CKV_OK;
}
