// KV append (scatter of new tokens into their slots) and whole-block copy
// (copy-on-write), both plain 16-byte-vector copies.
//
// Append: "Day 6/90 of Inference Engineering", PagedAttention notes,
// paragraph 2 (each new token goes into the current cache block; a new block
// when it is full) -- the slot comes from the host allocator.  Block copy:
// paragraph 5 (a sequence that diverges from a shared prefix writes into a
// new block, which first receives the shared block's rows).
//
// Both are bandwidth-trivial (a few MB per decode step) and launch-latency
// bound; each thread moves one 16-byte vector of K and one of V.
//
// FP8 append: the same scatter into an E4M3 cache; each stored byte is the
// bf16 input divided by the cache's scale (IEEE fp32 division) and rounded
// to the nearest E4M3 value, saturating at ±448 -- FP8 storage being this
// library's reading of the pages' call for fewer bytes moved (memory notes,
// "Core Ideas" 1).

#include <cuda_fp8.h>

#include "device_common.cuh"
#include "kernels.h"

namespace pa {
namespace {

// One thread per (token, KV head, 16-byte vector of the head's row).
__global__ void cache_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                    const int64_t* __restrict__ slots, int T, uint4* k_cache, uint4* v_cache,
                                    long long num_slots, int Hkv, int B, int vpr, unsigned* status) {
  // A decode launched right after this kernel (programmatic dependent
  // launch) may start its prologue now; it reads the cache only after
  // griddepcontrol.wait, i.e. after this kernel has completed.
  pdl_launch_dependents();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long per_tok = (long long)Hkv * vpr;
  if (idx >= (long long)T * per_tok) return;
  const int i = (int)(idx / per_tok);
  const int rem = (int)(idx - (long long)i * per_tok);
  const int h = rem / vpr;
  const int c = rem - h * vpr;
  const int64_t slot = __ldg(slots + i);
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (rem == 0) raise_status(status, PA_STATUS_BAD_SLOT);
    return;
  }
  const int64_t blk = slot / B;
  const int64_t row = slot - blk * B;
  const size_t dst = (((size_t)blk * Hkv + h) * B + row) * vpr + c;
  const size_t src = (size_t)idx;  // k, v are [T][Hkv][vpr] vectors
  k_cache[dst] = __ldg(k + src);
  v_cache[dst] = __ldg(v + src);
}

// One thread per (token, KV head, 16 elements of the head's row): 32 bytes of
// bf16 in, 16 bytes of E4M3 codes out, for K and for V.
__global__ void cache_append_fp8_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                        const int64_t* __restrict__ slots, int T, uint4* k_cache, uint4* v_cache,
                                        long long num_slots, int Hkv, int B, int vpr, float k_scale, float v_scale,
                                        unsigned* status) {
  pdl_launch_dependents();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long per_tok = (long long)Hkv * vpr;
  if (idx >= (long long)T * per_tok) return;
  const int i = (int)(idx / per_tok);
  const int rem = (int)(idx - (long long)i * per_tok);
  const int h = rem / vpr;
  const int c = rem - h * vpr;
  const int64_t slot = __ldg(slots + i);
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (rem == 0) raise_status(status, PA_STATUS_BAD_SLOT);
    return;
  }
  const int64_t blk = slot / B;
  const int64_t row = slot - blk * B;
  const size_t dst = (((size_t)blk * Hkv + h) * B + row) * vpr + c;
  auto quantize16 = [](const uint4* src, float scale) {
    const uint4 a = __ldg(src), b = __ldg(src + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t packed = 0;
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const uint32_t pair = w[2 * j + hlf];  // two bf16: low half first
        float2 f;
        f.x = __fdiv_rn(__uint_as_float(pair << 16), scale);
        f.y = __fdiv_rn(__uint_as_float(pair & 0xffff0000u), scale);
        const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
        packed |= (uint32_t)q << (16 * hlf);
      }
      o[j] = packed;
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  };
  const size_t src = (size_t)idx * 2;  // k, v are [T][Hkv][vpr] pairs of 16-byte vectors
  k_cache[dst] = quantize16(k + src, k_scale);
  v_cache[dst] = quantize16(v + src, v_scale);
}

// grid.y = pair index; threads stride over the block's 16-byte vectors.
__global__ void copy_blocks_kernel(uint4* k_cache, uint4* v_cache, const int32_t* __restrict__ pairs,
                                   int num_blocks, long long vpb, unsigned* status) {
  const int pi = blockIdx.y;
  const int src = __ldg(pairs + 2 * pi);
  const int dst = __ldg(pairs + 2 * pi + 1);
  if ((unsigned)src >= (unsigned)num_blocks || (unsigned)dst >= (unsigned)num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_status(status, PA_STATUS_BAD_BLOCK);
    return;
  }
  const size_t so = (size_t)src * vpb, d = (size_t)dst * vpb;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < vpb;
       e += (long long)gridDim.x * blockDim.x) {
    k_cache[d + e] = k_cache[so + e];
    v_cache[d + e] = v_cache[so + e];
  }
}

}  // namespace

cudaError_t launch_cache_append(const void* k, const void* v, const int64_t* slots, int T, void* k_cache,
                                void* v_cache, int num_blocks, int Hkv, int D, int B, int elem_bytes,
                                unsigned* status, cudaStream_t stream) {
  const int vpr = D * elem_bytes / 16;
  const long long n = (long long)T * Hkv * vpr;
  if (n <= 0) return cudaSuccess;
  const int threads = 256;
  const long long grid = (n + threads - 1) / threads;
  cache_append_kernel<<<(unsigned)grid, threads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots, T, static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), (long long)num_blocks * B, Hkv, B, vpr, status);
  return cudaGetLastError();
}

cudaError_t launch_cache_append_fp8(const void* k, const void* v, const int64_t* slots, int T, void* k_cache,
                                    void* v_cache, int num_blocks, int Hkv, int D, int B, float k_scale,
                                    float v_scale, unsigned* status, cudaStream_t stream) {
  const int vpr = D / 16;  // 16-byte vectors of codes per row
  const long long n = (long long)T * Hkv * vpr;
  if (n <= 0) return cudaSuccess;
  const int threads = 256;
  const long long grid = (n + threads - 1) / threads;
  cache_append_fp8_kernel<<<(unsigned)grid, threads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots, T, static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), (long long)num_blocks * B, Hkv, B, vpr, k_scale, v_scale, status);
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs, int num_blocks,
                               size_t block_bytes, unsigned* status, cudaStream_t stream) {
  if (num_pairs <= 0) return cudaSuccess;
  const long long vpb = (long long)(block_bytes / 16);
  const int threads = 256;
  const long long gx = std::min<long long>((vpb + threads - 1) / threads, 64);
  copy_blocks_kernel<<<dim3((unsigned)gx, (unsigned)num_pairs), threads, 0, stream>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), pairs, num_blocks, vpb, status);
  return cudaGetLastError();
}

}  // namespace pa
