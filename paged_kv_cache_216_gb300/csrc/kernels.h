// Host-side launch interface of the library's kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {

// Head of the decode workspace: the work counter of the persistent kernel
// and the length of the work list that follows it.
struct PlanHeader {
  unsigned counter;
  int num_pairs;  // (sequence, partition) pairs in the list; items = pairs * Hkv
  int pad[62];
};

// Everything a decode launch needs besides the cache tensor maps.
struct DecodeArgs {
  const void* q;                // [S][H][D]
  const void* k_cache;          // [N][Hkv][B][D] (fp32 path reads it directly)
  const void* v_cache;
  void* out;                    // [S][H][D]
  const int32_t* block_tables;  // [S][max_blocks_per_seq]
  const int32_t* context_lens;  // [S]
  float* ws_o;                  // [S][max_parts][H][D] split-K partial outputs
  float2* ws_ml;                // [S][max_parts][H] (max, sum), log2 domain
  PlanHeader* hdr;              // work counter + list length
  const int2* plan;             // [S * max_parts] {s | part << 16, clamped ctx}; ctx 0 = empty context
  unsigned* status;             // device status word
  int S, H, Hkv, g, D, B;
  int num_blocks, max_blocks_per_seq, max_ctx;
  int P;                        // partition size in tokens (multiple of 32)
  int max_parts;                // ceil(max_ctx / P)
  float scale_log2;             // scale * log2(e)
};

constexpr int kMaxGroup = 8;

// bf16, tensor cores; grid = persistent CTAs.
cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream);
// Dynamic shared memory of the tensor-core kernel for this head_dim.
size_t decode_tc_smem_bytes(int D);
// Whether the tensor-core kernel loads whole [B x D] slabs as one TMA box
// of 2B lines of 128 bytes (true) or one box per 64-dim half (false); the
// cache tensor maps must be made to match.
bool decode_tc_interleaved(int D, int B);

// Work list (longest items first) for the tensor-core kernel, built on the
// device from a.context_lens into a.hdr / a.plan.  Must precede
// launch_decode_tc on the stream.
cudaError_t launch_decode_plan(const DecodeArgs& a, cudaStream_t stream);

// fp32, CUDA cores; one CTA per (sequence, partition, KV head).
cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t stream);

// Log-sum-exp merge of split-K partials into `out` (dtype PA_F32/PA_BF16).
cudaError_t launch_lse_merge(const DecodeArgs& a, int dtype, cudaStream_t stream);

cudaError_t launch_cache_append(const void* k, const void* v, const int64_t* slots, int T, void* k_cache,
                                void* v_cache, int num_blocks, int Hkv, int D, int B, int elem_bytes,
                                unsigned* status, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                               int num_blocks, size_t block_bytes, unsigned* status, cudaStream_t stream);

}  // namespace pa
