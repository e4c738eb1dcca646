// pa_decode_static_workspace: paged decode whose split-K scratch is a fixed
// array inside this library instead of a buffer the caller allocates.
//
// It is for callers that cannot call cudaMalloc (or any allocator) to get a
// workspace: a host program whose device memory was reserved up front by
// another allocator, so a new allocation would fail or fragment that pool, or
// a serving loop that must not make calls that may synchronize the device,
// as cudaMalloc can.  Such a caller still passes its inputs and output; the
// partial results of long contexts go to the array below.
//
// The array is PA_STATIC_WORKSPACE_BYTES (16 MiB) of device memory that every
// GPU that loads this library holds until the process exits.  All calls
// share it, and it keeps whatever the last call wrote: nothing in it needs to
// start at zero, because a call reads only the partials it wrote itself, but
// two calls whose kernels overlap on the GPU (two streams, or two host
// threads) race on it and must be serialised by the caller.

#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// Device address of this device's copy of the array.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// with the device current: once per device, on the first call there, and
// again if the device's context was re-created since (cudaDeviceReset
// unloads the library's module; the old address would then dangle).
int scratch_address(void** out) {
  static void* addr[kMaxDevices] = {};
  static unsigned long long ctx_ids[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pa_fail(PA_ERR_CUDA, "pa_decode_static_workspace: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode_static_workspace: device ordinal");
  const unsigned long long ctx = pa_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || ctx == 0 || ctx != ctx_ids[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p) {
      static thread_local char buf[160];
      std::snprintf(buf, sizeof(buf), "pa_decode_static_workspace: cudaGetSymbolAddress failed: %s",
                    cudaGetErrorString(e));
      return pa_fail(PA_ERR_CUDA, buf);
    }
    addr[dev] = p;
    ctx_ids[dev] = pa_context_id();  // the lookup made the device's context current
  }
  *out = addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_static_workspace(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_tables, int max_blocks_per_seq,
                                          const int32_t* context_lens, int max_context_len, float scale, void* out,
                                          int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                          int block_size, int num_blocks, int partition_size, int dtype,
                                          void* stream) {
  const int P = pa_decode_partition_size(num_seqs, num_kv_heads, max_context_len, partition_size);
  if (P < 0) return P;
  const size_t need = pa_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, P);
  if (need > (size_t)PA_STATIC_WORKSPACE_BYTES) {
    static thread_local char buf[200];
    std::snprintf(buf, sizeof(buf),
                  "pa_decode_static_workspace: these sizes need %zu bytes of scratch, more than the fixed "
                  "%zu-byte array; use pa_decode with a caller workspace or a larger partition_size",
                  need, (size_t)PA_STATIC_WORKSPACE_BYTES);
    return pa_fail(PA_ERR_INVALID, buf);
  }
  void* ws = nullptr;
  if (need > 0) {
    const int rc = scratch_address(&ws);
    if (rc) return rc;
  }
  return pa_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, max_context_len, scale,
                   out, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, P, ws,
                   need > 0 ? (size_t)PA_STATIC_WORKSPACE_BYTES : 0, dtype, stream);
}
