// paged_decode_attn_static: the decode call for callers that cannot
// allocate device memory.  Its split-KV scratch is a fixed array compiled
// into the library (file-scope, in device memory of every GPU that loads the
// library, for the life of the process) instead of a buffer the caller
// provides.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "paged_decode.h"

namespace {

constexpr size_t kStaticScratchBytes = PD_STATIC_SCRATCH_BYTES;
constexpr size_t kStaticCounterBytes = PD_STATIC_COUNTER_BYTES;
constexpr int kCountersPerPair = PD_COUNTERS_PER_PAIR;  // per (sequence, kv head)
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// device array, never a usable address: the device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the array on the current device (looked up on the first
// call made with that device current).
int static_scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return PD_ENODEV;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    // the array exists only in this library's sm_103a image: another
    // device is refused the way the other entry points refuse it
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        major != 10 || minor != 3) {
      cudaGetLastError();
      return PD_ENODEV;
    }
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver ||
                     e == cudaErrorNoKernelImageForDevice
                 ? PD_ENODEV
                 : PD_ECUDA;
    }
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return PD_OK;
}

}  // namespace

extern "C" PD_API int paged_decode_attn_static(
    const pd_tensor *q, const pd_tensor *k_cache, const pd_tensor *v_cache,
    const pd_tensor *block_table, const pd_tensor *seq_lens, pd_tensor *out, int num_q_heads,
    int num_kv_heads, int head_size, int page_size, int max_query_len, int window, float scale,
    int layout, void *stream) {
  if (!seq_lens || seq_lens->ndim != 1 || num_kv_heads <= 0) return PD_EINVAL;
  const int64_t S = seq_lens->shape[0];
  if (S < 0) return PD_EINVAL;
  if (S == 0) return PD_OK;
  // one set of counters per (sequence, kv head); the rest of the array holds
  // the partials, whose split the planner fits to what remains
  const int64_t counter_slots = S * (int64_t)num_kv_heads * kCountersPerPair;
  if (counter_slots * 4 > (int64_t)kStaticCounterBytes) return PD_ESCRATCH;
  void *base = nullptr;
  int rc = static_scratch_address(&base);
  if (rc != PD_OK) return rc;
  // The array keeps the previous call's contents: start this call's
  // counters at zero (partials are always written before they are read).
  if (cudaMemsetAsync(base, 0, (size_t)counter_slots * 4, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess) {
    cudaGetLastError();
    return PD_ECUDA;
  }
  pd_scratch scratch;
  scratch.data = base;
  scratch.bytes = kStaticScratchBytes;
  scratch.counter_slots = counter_slots;
  return paged_decode_attn(q, k_cache, v_cache, block_table, seq_lens, out, num_q_heads,
                           num_kv_heads, head_size, page_size, max_query_len, window, scale,
                           layout, &scratch, stream);
}
