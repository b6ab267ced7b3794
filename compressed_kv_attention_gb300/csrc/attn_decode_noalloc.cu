// attn_decode_noalloc.cu — compressed decode for callers that cannot allocate
// device memory.
//
// ckv_attn_decode() needs a caller-provided workspace. Some callers have no way
// to provide one: a host framework that owns all device memory and gives a
// plug-in none of it, a latency-critical loop that must not call cudaMalloc
// (which can block and synchronise the device), or a process whose memory
// planner has already handed out the whole device. For them this entry point
// runs the same two kernels (split-K decode and split merge) with their scratch
// in a fixed array compiled into the library, so nothing is allocated at call
// time.
//
// Limits and sharing:
//  * The array holds kNoAllocScratchBytes (4 MiB) on every device that loads the
//    library, for the life of the process. A call whose scratch would not fit
//    (see ckv_attn_decode_workspace) is rejected with CKV_ERR_WORKSPACE.
//  * All calls share the one array and it keeps the previous call's contents.
//    Each call first clears, on its stream, the part of the array that holds
//    its split-merge counters (their size depends on the call's shape, and an
//    earlier call of another shape may have left partials or, after a timed-out
//    wait, counters there), then runs the decode, which rewrites every partial
//    it reads. Calls that overlap on the GPU (different streams, no ordering
//    between them) race on the array and give wrong results: order them on one
//    stream or with events.
//  * The device flag word (bounded-wait timeouts, out-of-range seq_len) sits at
//    the start of the array and is not cleared by a call: it keeps the first
//    error since it was last read. ckv_read_noalloc_flag() reads and clears it.
//  * The first call on a device (either entry point) looks up the array's
//    device address on that device (cudaGetSymbolAddress, with the device
//    current). Make that first call before any stream capture on the device.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/ckv.h"
#include "ckv_kernels.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" CKV_API ckv_status ckv_attn_decode_noalloc(const ckv_cache* cache, const int32_t* seq_len,
                                                      int64_t max_seq_len, const void* q_f16, int32_t n_q,
                                                      int32_t n_q_heads, float scale, int32_t n_split,
                                                      float* out, float* lse, void* stream) {
  // Size the scratch exactly as ckv_attn_decode would, and refuse what does not fit.
  size_t need = ckv_attn_decode_workspace(cache, max_seq_len, n_q, n_q_heads, n_split);
  if (need > kNoAllocScratchBytes && n_split == 0 && cache &&
      ckv::rows_decode_applies(cache->batch, cache->n_kv_heads, n_q_heads, n_q, n_split, max_seq_len)) {
    // The many-row tile path keeps one partial per tile and split; the
    // mma.sync path at its own automatic split count needs far less scratch.
    n_split = ckv::decode_auto_split(cache, max_seq_len, n_q, n_q_heads);
    need = ckv_attn_decode_workspace(cache, max_seq_len, n_q, n_q_heads, n_split);
  }
  if (need == 0) {
    // Invalid geometry: let the regular entry point produce the precise status and message.
    return ckv_attn_decode(cache, seq_len, max_seq_len, q_f16, n_q, n_q_heads, scale, n_split, out, lse,
                           nullptr, 0, stream);
  }
  if (need > kNoAllocScratchBytes)
    return static_cast<ckv_status>(ckv::set_last_error(
        CKV_ERR_WORKSPACE, "attn_decode_noalloc: needs %zu bytes of scratch, the built-in array holds %zu",
        need, kNoAllocScratchBytes));
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess)
    return static_cast<ckv_status>(ckv::set_last_error(
        CKV_ERR_CUDA, "attn_decode_noalloc: scratch address lookup: %s", cudaGetErrorString(e)));
  // Clear this call's counter words (bytes [4, header)); the flag word at 0 stays.
  const size_t header = ckv::decode_header_bytes(cache, max_seq_len, n_q, n_q_heads, n_split);
  if (header > kNoAllocScratchBytes)
    return static_cast<ckv_status>(ckv::set_last_error(
        CKV_ERR_WORKSPACE, "attn_decode_noalloc: header of %zu bytes exceeds the built-in array", header));
  e = cudaMemsetAsync(static_cast<unsigned char*>(scratch) + 4, 0, header - 4, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return static_cast<ckv_status>(ckv::set_last_error(
        CKV_ERR_CUDA, "attn_decode_noalloc: counter clear: %s", cudaGetErrorString(e)));
  return ckv_attn_decode(cache, seq_len, max_seq_len, q_f16, n_q, n_q_heads, scale, n_split, out, lse,
                         scratch, kNoAllocScratchBytes, stream);
}

extern "C" CKV_API ckv_status ckv_read_noalloc_flag(int32_t* flag, void* stream) {
  if (!flag)
    return static_cast<ckv_status>(ckv::set_last_error(CKV_ERR_INVALID_ARG, "read_noalloc_flag: flag is null"));
  void* scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess)
    return static_cast<ckv_status>(ckv::set_last_error(
        CKV_ERR_CUDA, "read_noalloc_flag: scratch address lookup: %s", cudaGetErrorString(e)));
  return ckv_read_device_flag(scratch, flag, stream);
}
