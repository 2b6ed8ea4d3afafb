// ua_noalloc.cu -- ua_unified_attention_noalloc: the attention call for callers that may
// not allocate device memory.
//
// Who needs it: callers whose device memory is fixed up front (a serving runtime that
// hands all free memory to its own KV-cache pool at start-up, a process held to a
// memory budget) and callers on a latency-critical path where a cudaMalloc, which can
// block and synchronise the device, is not allowed.  ua_unified_attention itself
// allocates only when the split-KV path runs without a caller workspace; this entry
// point gives that path a fixed scratch array instead, so it never allocates.
//
// The scratch is one file-scope device array of UA_NOALLOC_SCRATCH_BYTES.  Every GPU
// that loads the library holds it until the process exits, and every call on a device
// shares it.  Its host-side name is only a stand-in for the device array: host code
// must not hand it to a kernel.  The device address comes from cudaGetSymbolAddress,
// looked up once per device, with that device current, by the first call made on it.
// The looked-up address is kept for the life of the process: it does not survive a
// cudaDeviceReset of that device (after one, this entry point must not be called again).
#include <mutex>

#include <cuda_runtime.h>

#include "ua.h"

namespace {

constexpr size_t kScratchBytes = UA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The split-KV path's fp32 max / sum / partial-output scratch for this entry point.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch on the current device (looked up on first use).
int scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return UA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return UA_ERR_CUDA;
    addr[dev] = ptr;
  }
  *out = addr[dev];
  return UA_OK;
}

}  // namespace

extern "C" int ua_unified_attention_noalloc(
    const void* q, const void* k_cache, const void* v_cache, void* out,
    const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, const int32_t* block_table,
    int block_size, int num_q_heads, int num_kv_heads, int head_dim, float scale, float softcap,
    int window_left, const float* alibi_slopes, const float* qq_bias, const float* sinks,
    int kv_dtype, const float* kv_scale, int backend, void* stream, const ua_shape_t* shape) {
  try {
    if (shape == nullptr) return UA_ERR_INVALID_ARG;
    ua_plan_t plan;
    int rc = ua_plan(shape, block_size, num_q_heads, num_kv_heads, head_dim, window_left,
                     kv_dtype, backend, 0, &plan);
    if (rc != UA_OK) return rc;
    if (plan.workspace_bytes > kScratchBytes) return UA_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if ((rc = scratch_address(&scratch)) != UA_OK) return rc;
    // The partition kernel writes every max, sum and partial-output entry the merge
    // kernel reads in the same call, so nothing in the scratch has to start at zero.
    ua_shape_t sh = *shape;
    sh.workspace = scratch;
    sh.workspace_bytes = kScratchBytes;
    rc = ua_unified_attention(q, k_cache, v_cache, out, cu_seqlens_q, seq_lens_k, block_table,
                              block_size, num_q_heads, num_kv_heads, head_dim, scale, softcap,
                              window_left, alibi_slopes, qq_bias, sinks, kv_dtype, kv_scale,
                              backend, stream, &sh);
    // The call plans again for another kernel when a tensor map cannot be encoded; if that
    // plan needs more scratch than the array, the inner call reports a short workspace,
    // which for this entry point means the fixed array is too small.
    return rc == UA_ERR_WORKSPACE ? UA_ERR_SCRATCH_LIMIT : rc;
  } catch (...) {
    return UA_ERR_CUDA;
  }
}
