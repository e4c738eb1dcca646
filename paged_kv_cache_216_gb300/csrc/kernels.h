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

// Bound of a pipeline wait of the decode kernels unless a call says
// otherwise (a wait this long means the pipeline is broken).
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;  // 2 s

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
  const int2* plan;             // [S * max_parts] {s | part << 16, clamped ctx}; ctx 0 = empty context;
                                // shared-prefix items: prefix_entry()
  unsigned* status;             // device status word
  int S, H, Hkv, g, D, B;
  int num_blocks, max_blocks_per_seq, max_ctx;
  int P;                        // partition size in tokens (multiple of 32)
  int max_parts;                // ceil(max_ctx / P)
  float scale_log2;             // scale * log2(e)
  int shared_items;             // the work list may hold shared-prefix items
  float v_scale;                // FP8 caches: value of a V code = e4m3(code) * v_scale (1 otherwise)
  // Bound of every pipeline wait of the bf16 kernel (2 s normally), and a
  // test hook: the producer of each CTA never issues the CTA's chunk number
  // `withhold_chunk` (-1: none), so that the wait for it runs out.
  unsigned long long wait_limit_ns;
  int withhold_chunk;
};

constexpr int kMaxGroup = 8;   // query rows of an ordinary decode work item (heads of one KV head)
constexpr int kGroupRows = 128;  // query rows of a shared-prefix work item (one tensor-core tile)

// Groups of sequences whose contexts start with the same tokens in the same
// cache blocks (prefix sharing, "Day 6/90 of Inference Engineering",
// PagedAttention notes, paragraph 5).  Group i is sequences
// first[i] .. first[i] + count[i] - 1; its first parts[i] partitions
// (parts[i] * P tokens) are shared.  The work list attends each shared
// partition, per KV head, with shared-prefix items that each cover the
// query rows of up to kGroupRows / g members -- one item per partition and
// KV head for a group of up to 128 / g members, so each shared block is read
// once per group -- and leaves the members' own items for those partitions
// out.
constexpr int kMaxPrefixGroups = 64;

struct PrefixGroups {
  int n;                         // groups with at least one shared partition
  int first[kMaxPrefixGroups];   // ascending, ranges disjoint
  int count[kMaxPrefixGroups];
  int parts[kMaxPrefixGroups];
};

// Members per shared-prefix item: their g query rows each fill the
// kGroupRows rows (tensor-memory lanes) of the item's tile.
__host__ __device__ inline int prefix_members_per_item(int g) { return kGroupRows / g; }

// Work-list entry of a shared-prefix item: the table of sequence `table_seq`
// (the group's first), partition `part`, query rows of sequences s0 .. s0 +
// nm - 1 (nm <= 128).  The second word is negative, which tells it from an
// ordinary entry {s | part << 16, context length}.
__host__ __device__ inline int2 prefix_entry(int table_seq, int part, int s0, int nm) {
  return make_int2(table_seq | (part << 16), (int)(0x80000000u | ((unsigned)s0 << 8) | (unsigned)nm));
}

// Shared partitions of sequence s (0 if it is in no group).
__host__ __device__ inline int prefix_parts_of(const PrefixGroups& pg, int s) {
  int lo = 0, hi = pg.n - 1, at = -1;
  while (lo <= hi) {  // last group whose first sequence is <= s
    const int mid = (lo + hi) >> 1;
    if (pg.first[mid] <= s) {
      at = mid;
      lo = mid + 1;
    } else {
      hi = mid - 1;
    }
  }
  return (at >= 0 && s < pg.first[at] + pg.count[at]) ? pg.parts[at] : 0;
}

// bf16, tensor cores; grid = persistent CTAs.  kmap/vmap: the bf16 caches
// as 4D block maps (one box per block of one KV head, block_layout.cuh).
cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream);
// Dynamic shared memory of the tensor-core kernel for this head_dim.
size_t decode_tc_smem_bytes(int D);

// FP8 (E4M3) caches, head_dim 128, bf16 q/out; same work list, workspace and
// merge as the bf16 kernel.  scale_log2 must include the K scale.
cudaError_t launch_decode_fp8(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                              cudaStream_t stream);
size_t decode_fp8_smem_bytes();

// Work list (longest items first) for the tensor-core kernel, built on the
// device from a.context_lens into a.hdr / a.plan.  Must precede
// launch_decode_tc on the stream.
cudaError_t launch_decode_plan(const DecodeArgs& a, const PrefixGroups& pg, cudaStream_t stream);

// Shared-prefix entries of the work list (the same on host and device):
// for each group, partition p < parts and chunk of prefix_members_per_item(g)
// consecutive members.
__host__ __device__ inline int prefix_entries(const PrefixGroups& pg, int g) {
  const int nm = prefix_members_per_item(g);
  int n = 0;
  for (int i = 0; i < pg.n; ++i) n += pg.parts[i] * ((pg.count[i] + nm - 1) / nm);
  return n;
}
__host__ __device__ inline int2 prefix_entry_at(const PrefixGroups& pg, int g, int e) {
  const int nm = prefix_members_per_item(g);
  for (int i = 0;; ++i) {
    const int chunks = (pg.count[i] + nm - 1) / nm;
    if (e < pg.parts[i] * chunks) {
      const int part = e / chunks, s0 = pg.first[i] + (e % chunks) * nm;
      const int left = pg.first[i] + pg.count[i] - s0;
      return prefix_entry(pg.first[i], part, s0, left < nm ? left : nm);
    }
    e -= pg.parts[i] * chunks;
  }
}

// fp32, CUDA cores; one CTA per (sequence, partition, KV head).
cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t stream);

// Log-sum-exp merge of split-K partials into `out` (dtype PA_F32/PA_BF16).
// Members of a prefix group always go through the merge (their shared
// partitions were written as partials).
cudaError_t launch_lse_merge(const DecodeArgs& a, const PrefixGroups& pg, int dtype, cudaStream_t stream);

// Prefill: causal attention of the new tokens of each sequence.
struct PrefillArgs {
  const void* q;                // [T][H][D] bf16, the new tokens of all sequences one after another
  const void* k_cache;          // [N][Hkv][B][D] bf16, the new tokens already appended
  const void* v_cache;
  void* out;                    // [T][H][D] bf16
  const int32_t* block_tables;  // [S][max_blocks_per_seq]
  const int32_t* query_start;   // [S + 1] rows of q owned by each sequence
  const int32_t* context_lens;  // [S] tokens after the append
  unsigned* status;
  int S, T, H, Hkv, g, D, B;
  int num_blocks, max_blocks_per_seq, max_ctx, max_query_len;
  float scale_log2;
};
// Prefill on tcgen05, head_dim 64 or 128: persistent CTAs, one per SM; kmap/vmap: the bf16 caches as
// 4D (64 dims, 8 rows, 64-dim half, 8-row group) with boxes of one block (64, 8, D / 64, B / 8); qmap:
// q as (dims, head, token) with boxes of [64 dims x g heads x 128 / g tokens]; omap: out, the same.
cudaError_t launch_prefill_tc(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                              const CUtensorMap& qmap, const CUtensorMap& omap, cudaStream_t stream);

cudaError_t launch_cache_append(const void* k, const void* v, const int64_t* slots, int T, void* k_cache,
                                void* v_cache, int num_blocks, int Hkv, int D, int B, int elem_bytes,
                                unsigned* status, cudaStream_t stream);

// bf16 tokens quantized into an E4M3 cache (codes = RNE(x / scale), saturating).
cudaError_t launch_cache_append_fp8(const void* k, const void* v, const int64_t* slots, int T, void* k_cache,
                                    void* v_cache, int num_blocks, int Hkv, int D, int B, float k_scale,
                                    float v_scale, unsigned* status, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                               int num_blocks, size_t block_bytes, unsigned* status, cudaStream_t stream);

}  // namespace pa
