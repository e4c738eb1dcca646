// C ABI entry points (include/pa.h): argument validation, partition and
// workspace sizing, TMA descriptor set-up and kernel dispatch.  No device
// memory is allocated here; every buffer is the caller's.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "kernels.h"
#include "pa.h"
#include "pa_internal.h"

namespace {

// Device status word: OR of PA_STATUS_* bits raised by kernels.  Each device
// that loads the library has its own copy.
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;

int cuda_fail(cudaError_t e, const char* what) {
  static thread_local char buf[256];
  std::snprintf(buf, sizeof(buf), "%s: %s", what, cudaGetErrorString(e));
  return pa_fail(PA_ERR_CUDA, buf);
}

// Address of this device's status word, looked up once per device and
// context (again if the device's context was re-created since).
int status_ptr(unsigned** out) {
  static unsigned* ptrs[kMaxDevices] = {};
  static unsigned long long ctx_ids[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return pa_fail(PA_ERR_UNSUPPORTED, "device ordinal too large");
  const unsigned long long ctx = pa_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev] || ctx == 0 || ctx != ctx_ids[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    ptrs[dev] = static_cast<unsigned*>(p);
    ctx_ids[dev] = pa_context_id();  // the lookup made the device's context current
  }
  *out = ptrs[dev];
  return PA_OK;
}

template <typename Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(p);
  return nullptr;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map over an E4M3 cache (head_dim 128): [N*Hkv*B rows][128 bytes],
// one box of B rows per (block, head) slab, 128-byte swizzle.
int make_cache_map_fp8(CUtensorMap* map, const void* base, int num_blocks, int Hkv, int B) {
  auto fn = encode_fn();
  if (!fn) return pa_fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {128u, (cuuint64_t)num_blocks * Hkv * B};
  cuuint64_t strides[1] = {128u};
  cuuint32_t box[2] = {128u, (cuuint32_t)B};
  cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return pa_fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  return PA_OK;
}

// The cache [N_blk][Hkv][B][D] bf16 for the tensor-core kernels (decode and
// prefill), as 4D (64 dims, 8 rows, 64-dim half, group of 8 rows): a box of
// (64, 8, D / 64, B / 8) brings one block of one head in one copy and lands
// as groups of 8 rows, each group holding its halves 1 KB apart ([group]
// [half][8 rows][128 B], 128-byte swizzle), so 8-row groups are a uniform
// D / 64 KB apart: the layout of a K-major operand of the tensor cores
// (keys) and of an MN-major one (values), and for ldmatrix eight rows of a
// half in eight different bank groups.  Two 2D boxes per block (one per
// half) were half as large: for the prefill a chunk of 128 keys and values
// was 32 boxes, more than the TMA unit issues in the time the tensor cores
// take for the chunk.
int make_block_map(CUtensorMap* map, const void* base, int num_blocks, int Hkv, int B, int D) {
  auto fn = encode_fn();
  if (!fn) return pa_fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t groups = (cuuint64_t)num_blocks * Hkv * B / 8;
  const cuuint32_t halves = (cuuint32_t)(D / 64);
  cuuint64_t dims[4] = {64u, 8u, halves, groups};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2u, 128u, (cuuint64_t)D * 16u};
  cuuint32_t box[4] = {64u, 8u, halves, (cuuint32_t)(B / 8)};
  cuuint32_t elem_strides[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                  elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return pa_fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (block map)");
  return PA_OK;
}

// Query rows of one KV head for the tcgen05 prefill: q [T][H][D] bf16 as a
// 3D tensor (dims, head, token); a box of 64 dims x g heads x 128 / g tokens
// lands as 128 rows of 128 bytes, row = token * g + head, 128-byte swizzle.
int make_query_map(CUtensorMap* map, const void* q, int T, int H, int g, int D) {
  auto fn = encode_fn();
  if (!fn) return pa_fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2u, (cuuint64_t)H * D * 2u};
  cuuint32_t box[3] = {64u, (cuuint32_t)g, (cuuint32_t)(128 / g)};
  cuuint32_t elem_strides[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, elem_strides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return pa_fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  return PA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool supported_shape(int D, int B) { return (D == 64 || D == 128) && (B == 8 || B == 16 || B == 32); }

int elem_bytes(int dtype) { return dtype == PA_BF16 ? 2 : dtype == PA_F32 ? 4 : dtype == PA_FP8_E4M3 ? 1 : 0; }

bool good_scale(float s) { return std::isfinite(s) && s > 0.f; }

// Work items (sequence x partition x KV head) below which the library
// splits contexts into smaller partitions; about four per resident CTA.
constexpr long long kMinItems = 1216;
constexpr int kDefaultPartition = 512;
constexpr int kMinPartition = 64;
// A batch with this many (sequence, KV head) pairs keeps every CTA busy
// without splitting: contexts up to kWholeContext tokens are then one
// partition each (no partials, no merge), longer ones split in partitions of
// that size.  On the 32-sequence MHA batch and the 256-sequence serving
// batches this took the decode call from 96 to 93 us and from 177-184 to
// 173-176 us; narrower batches keep the split for balance.
constexpr long long kWideBatch = 1024;
constexpr int kWholeContext = 4096;
// Calls with prefix groups lengthen the partitions up to this many tokens
// while each group's prefix still holds a whole partition.
constexpr int kMaxSharedPartition = 1024;

long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace of pa_decode: [header 256 B][work list][split-K partial outputs]
// [split-K (max, sum) pairs]; the last two only when a context can span more
// than one partition.
struct WsLayout {
  size_t plan, o, ml, total;
  long long parts;
};

bool ws_layout(int S, int H, int D, int max_ctx, int P, WsLayout* l) {
  if (S <= 0 || H <= 0 || D <= 0 || max_ctx < 1 || P < 32) return false;
  l->parts = cdiv(max_ctx, P);
  const size_t pairs = (size_t)S * l->parts;
  l->plan = sizeof(pa::PlanHeader);
  l->o = l->plan + align256(pairs * sizeof(int2));
  if (l->parts > 1) {
    const size_t rows = pairs * H;
    l->ml = l->o + align256(rows * D * 4);
    l->total = l->ml + rows * 8;
  } else {
    l->ml = l->o;
    l->total = l->o;
  }
  return true;
}

}  // namespace

unsigned long long pa_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_current = driver_fn<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent");
    get_id = driver_fn<PFN_cuCtxGetId_v12000>("cuCtxGetId");
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

extern "C" {

int pa_get_status(void* stream, uint32_t* status) {
  if (!status) return pa_fail(PA_ERR_INVALID, "pa_get_status: null status");
  unsigned* dptr = nullptr;
  int rc = status_ptr(&dptr);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, dptr, sizeof(unsigned), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dptr, 0, sizeof(unsigned), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "pa_get_status");
  *status = host;
  return PA_OK;
}

int pa_cache_append(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens, void* k_cache,
                    void* v_cache, int num_blocks, int num_kv_heads, int head_dim, int block_size, int dtype,
                    void* stream) {
  const int es = elem_bytes(dtype);
  if (es == 0 || dtype == PA_FP8_E4M3)
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_cache_append: dtype (FP8 caches: pa_cache_append_fp8)");
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0)
    return pa_fail(PA_ERR_INVALID, "pa_cache_append: sizes");
  if (!supported_shape(head_dim, block_size)) return pa_fail(PA_ERR_UNSUPPORTED, "pa_cache_append: head_dim/block_size");
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return pa_fail(PA_ERR_INVALID, "pa_cache_append: null pointer");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return pa_fail(PA_ERR_INVALID, "pa_cache_append: misaligned pointer");
  unsigned* status = nullptr;
  int rc = status_ptr(&status);
  if (rc) return rc;
  cudaError_t e = pa::launch_cache_append(k, v, slot_mapping, num_tokens, k_cache, v_cache, num_blocks,
                                          num_kv_heads, head_dim, block_size, es, status,
                                          static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "pa_cache_append launch");
  return PA_OK;
}

int pa_cache_append_fp8(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens, void* k_cache,
                        void* v_cache, int num_blocks, int num_kv_heads, int head_dim, int block_size,
                        float k_scale, float v_scale, void* stream) {
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0)
    return pa_fail(PA_ERR_INVALID, "pa_cache_append_fp8: sizes");
  if (!supported_shape(head_dim, block_size))
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_cache_append_fp8: head_dim/block_size");
  if (!good_scale(k_scale) || !good_scale(v_scale))
    return pa_fail(PA_ERR_INVALID, "pa_cache_append_fp8: scales must be finite and > 0");
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return pa_fail(PA_ERR_INVALID, "pa_cache_append_fp8: null pointer");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return pa_fail(PA_ERR_INVALID, "pa_cache_append_fp8: misaligned pointer");
  unsigned* status = nullptr;
  int rc = status_ptr(&status);
  if (rc) return rc;
  cudaError_t e = pa::launch_cache_append_fp8(k, v, slot_mapping, num_tokens, k_cache, v_cache, num_blocks,
                                              num_kv_heads, head_dim, block_size, k_scale, v_scale, status,
                                              static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "pa_cache_append_fp8 launch");
  return PA_OK;
}

int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs, int num_blocks,
                   int num_kv_heads, int head_dim, int block_size, int dtype, void* stream) {
  const int es = elem_bytes(dtype);
  if (es == 0) return pa_fail(PA_ERR_UNSUPPORTED, "pa_copy_blocks: dtype");
  if (num_pairs < 0 || num_blocks <= 0 || num_kv_heads <= 0) return pa_fail(PA_ERR_INVALID, "pa_copy_blocks: sizes");
  if (!supported_shape(head_dim, block_size)) return pa_fail(PA_ERR_UNSUPPORTED, "pa_copy_blocks: head_dim/block_size");
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !pairs) return pa_fail(PA_ERR_INVALID, "pa_copy_blocks: null pointer");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(pairs, 4))
    return pa_fail(PA_ERR_INVALID, "pa_copy_blocks: misaligned pointer");
  unsigned* status = nullptr;
  int rc = status_ptr(&status);
  if (rc) return rc;
  const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * es;
  for (int off = 0; off < num_pairs; off += 65535) {
    const int n = std::min(65535, num_pairs - off);
    cudaError_t e = pa::launch_copy_blocks(k_cache, v_cache, pairs + 2 * (size_t)off, n, num_blocks, block_bytes,
                                           status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_copy_blocks launch");
  }
  return PA_OK;
}

int pa_decode_partition_size(int num_seqs, int num_kv_heads, int max_context_len, int partition_size) {
  if (num_seqs < 0 || num_kv_heads <= 0 || max_context_len < 1)
    return pa_fail(PA_ERR_INVALID, "pa_decode_partition_size: sizes");
  if (partition_size > 0) {
    if (partition_size % 32) return pa_fail(PA_ERR_INVALID, "partition_size must be a multiple of 32");
    return partition_size;
  }
  if (partition_size < 0) return pa_fail(PA_ERR_INVALID, "partition_size < 0");
  if ((long long)num_seqs * num_kv_heads >= kWideBatch)
    return max_context_len <= kWholeContext ? (int)(cdiv(max_context_len, 32) * 32) : kWholeContext;
  int P = kDefaultPartition;
  while (P > kMinPartition && (long long)num_seqs * num_kv_heads * cdiv(max_context_len, P) < kMinItems) P /= 2;
  return P;
}

int pa_decode_partition_size_shared_prefix(int num_seqs, int num_kv_heads, int max_context_len, int partition_size,
                                           const int32_t* groups, int num_groups) {
  int P = pa_decode_partition_size(num_seqs, num_kv_heads, max_context_len, partition_size);
  if (P < 0 || partition_size > 0 || num_groups <= 0) return P;
  if (!groups) return pa_fail(PA_ERR_INVALID, "pa_decode_partition_size_shared_prefix: null groups");
  // Longer partitions while every group's prefix still holds a whole one:
  // fewer shared items and partials per group (on a 64-sequence GQA batch
  // with a 1024-token prefix, 1024 gave 115.6 us against 118.4 us at 512).
  int shortest = max_context_len;
  for (int i = 0; i < num_groups; ++i) shortest = std::min(shortest, std::max(groups[3 * i + 2], 0));
  while (P < kMaxSharedPartition && 2 * P <= shortest) P *= 2;
  return P;
}

size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                 int partition_size) {
  WsLayout l;
  if (!ws_layout(num_seqs, num_heads, head_dim, max_context_len, partition_size, &l)) return 0;
  return l.total;
}

}  // extern "C"

// pa_decode and pa_decode_planned: `plan` (device) is a work list built by
// pa_decode_plan_host, or NULL to build it on the device.
static int decode_impl(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                       int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, float scale,
                       void* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                       int num_blocks, int partition_size, const void* plan, const int32_t* groups,
                       int num_groups, void* workspace, size_t workspace_bytes, int dtype, void* stream,
                       float k_scale = 1.f, float v_scale = 1.f,
                       unsigned long long wait_limit_ns = pa::kDefaultWaitLimitNs, int withhold_chunk = -1) {
  // dtype is the caches' type; with PA_FP8_E4M3 q and out are bf16.
  const int es = elem_bytes(dtype);
  if (es == 0) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: dtype");
  const bool fp8 = dtype == PA_FP8_E4M3;
  if (fp8 && head_dim != 128) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode_fp8: head_dim 128 only");
  if (fp8 && (!good_scale(k_scale) || !good_scale(v_scale)))
    return pa_fail(PA_ERR_INVALID, "pa_decode_fp8: scales must be finite and > 0");
  if (fp8 && num_groups != 0) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode_fp8: no prefix groups");
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 || max_context_len < 1 ||
      max_blocks_per_seq <= 0 || !std::isfinite(scale))
    return pa_fail(PA_ERR_INVALID, "pa_decode: sizes");
  if (num_heads % num_kv_heads) return pa_fail(PA_ERR_INVALID, "pa_decode: num_heads % num_kv_heads != 0");
  const int g = num_heads / num_kv_heads;
  if (!(g == 1 || g == 2 || g == 4 || g == 8)) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: heads per KV head");
  if (!supported_shape(head_dim, block_size)) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: head_dim/block_size");
  if (cdiv(max_context_len, block_size) > max_blocks_per_seq)
    return pa_fail(PA_ERR_INVALID, "pa_decode: max_blocks_per_seq < ceil(max_context_len / block_size)");
  if ((long long)num_blocks * num_kv_heads * block_size * 2 >= (1LL << 31))
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: pool rows exceed 2^30 (TMA coordinates are 32-bit)");
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return pa_fail(PA_ERR_INVALID, "pa_decode: null pointer");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return pa_fail(PA_ERR_INVALID, "pa_decode: misaligned pointer");
  const int P = num_groups ? pa_decode_partition_size_shared_prefix(num_seqs, num_kv_heads, max_context_len,
                                                                     partition_size, groups, num_groups)
                           : pa_decode_partition_size(num_seqs, num_kv_heads, max_context_len, partition_size);
  if (P < 0) return P;
  const long long parts = cdiv(max_context_len, P);
  if (parts * num_seqs * num_kv_heads >= (1LL << 31)) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: too many work items");
  if (num_seqs > 65535 || parts > 32767)
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: more than 65535 sequences or 32767 partitions per context");
  WsLayout wl;
  ws_layout(num_seqs, num_heads, head_dim, max_context_len, P, &wl);
  if (!workspace || workspace_bytes < wl.total) return pa_fail(PA_ERR_INVALID, "pa_decode: workspace too small");
  if (!aligned(workspace, 256)) return pa_fail(PA_ERR_INVALID, "pa_decode: workspace not 256-byte aligned");
  if (plan && dtype == PA_F32) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode_planned: bf16 or FP8 caches only");
  if (plan && !aligned(plan, 256)) return pa_fail(PA_ERR_INVALID, "pa_decode_planned: plan not 256-byte aligned");
  if (num_groups != 0 && dtype != PA_BF16) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode_shared_prefix: bf16 only");
  pa::PrefixGroups pg;
  int rc = pa_prefix_groups(groups, num_groups, num_seqs, max_context_len, P, &pg, "pa_decode_shared_prefix");
  if (rc) return rc;

  pa::DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.out = out;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  char* ws = static_cast<char*>(workspace);
  char* pl = plan ? static_cast<char*>(const_cast<void*>(plan)) : ws;
  a.hdr = reinterpret_cast<pa::PlanHeader*>(pl);
  a.plan = reinterpret_cast<const int2*>(pl + wl.plan);
  if (parts > 1) {
    a.ws_o = reinterpret_cast<float*>(ws + wl.o);
    a.ws_ml = reinterpret_cast<float2*>(ws + wl.ml);
  }
  rc = status_ptr(&a.status);
  if (rc) return rc;
  a.S = num_seqs;
  a.H = num_heads;
  a.Hkv = num_kv_heads;
  a.g = g;
  a.D = head_dim;
  a.B = block_size;
  a.num_blocks = num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_ctx = max_context_len;
  a.P = P;
  a.max_parts = (int)parts;
  a.scale_log2 = (float)((double)scale * (fp8 ? (double)k_scale : 1.0) * 1.4426950408889634);  // log2(e)
  a.shared_items = pg.n > 0;
  a.v_scale = fp8 ? v_scale : 1.f;
  a.wait_limit_ns = wait_limit_ns;
  a.withhold_chunk = withhold_chunk;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  cudaError_t e;
  if (dtype == PA_BF16) {
    CUtensorMap kmap, vmap;
    rc = make_block_map(&kmap, k_cache, num_blocks, num_kv_heads, block_size, head_dim);
    if (rc) return rc;
    rc = make_block_map(&vmap, v_cache, num_blocks, num_kv_heads, block_size, head_dim);
    if (rc) return rc;
    if (!plan) {
      e = pa::launch_decode_plan(a, pg, st);
      if (e != cudaSuccess) return cuda_fail(e, "pa_decode plan launch");
    }
    e = pa::launch_decode_tc(a, kmap, vmap, st);
  } else if (fp8) {
    CUtensorMap kmap, vmap;
    rc = make_cache_map_fp8(&kmap, k_cache, num_blocks, num_kv_heads, block_size);
    if (rc) return rc;
    rc = make_cache_map_fp8(&vmap, v_cache, num_blocks, num_kv_heads, block_size);
    if (rc) return rc;
    if (!plan) {
      e = pa::launch_decode_plan(a, pg, st);
      if (e != cudaSuccess) return cuda_fail(e, "pa_decode plan launch");
    }
    e = pa::launch_decode_fp8(a, kmap, vmap, st);
  } else {
    e = pa::launch_decode_simt(a, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "pa_decode launch");
  if (parts > 1) {
    e = pa::launch_lse_merge(a, pg, fp8 ? PA_BF16 : dtype, st);
    if (e != cudaSuccess) return cuda_fail(e, "pa_decode merge launch");
  }
  return PA_OK;
}


extern "C" {

int pa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, float scale, void* out,
              int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
              int partition_size, void* workspace, size_t workspace_bytes, int dtype, void* stream) {
  if (dtype == PA_FP8_E4M3) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: FP8 caches need pa_decode_fp8");
  return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, max_context_len, scale,
                     out, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, partition_size,
                     nullptr, nullptr, 0, workspace, workspace_bytes, dtype, stream);
}

int pa_decode_test_withhold(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                            int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, float scale,
                            void* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                            int num_blocks, int partition_size, void* workspace, size_t workspace_bytes,
                            int withheld_chunk, int wait_limit_us, void* stream) {
  if (withheld_chunk < 0) return pa_fail(PA_ERR_INVALID, "pa_decode_test_withhold: withheld_chunk < 0");
  if (wait_limit_us < 1 || wait_limit_us > 2000000)
    return pa_fail(PA_ERR_INVALID, "pa_decode_test_withhold: wait_limit_us outside [1, 2000000]");
  return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, max_context_len, scale,
                     out, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, partition_size,
                     nullptr, nullptr, 0, workspace, workspace_bytes, PA_BF16, stream, 1.f, 1.f,
                     1000ull * (unsigned long long)wait_limit_us, withheld_chunk);
}

int pa_decode_planned(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                      int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, float scale,
                      void* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                      int num_blocks, int partition_size, const void* plan, void* workspace,
                      size_t workspace_bytes, int dtype, void* stream) {
  if (!plan) return pa_fail(PA_ERR_INVALID, "pa_decode_planned: null plan");
  if (dtype == PA_FP8_E4M3) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode_planned: FP8 caches need pa_decode_fp8");
  return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, max_context_len, scale,
                     out, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, partition_size,
                     plan, nullptr, 0, workspace, workspace_bytes, dtype, stream);
}

int pa_prefill(const void* q, const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
               const int32_t* query_start, const int32_t* context_lens, const int32_t* block_tables,
               int max_blocks_per_seq, int max_query_len, int max_context_len, float scale, void* k_cache,
               void* v_cache, void* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
               int block_size, int num_blocks, int dtype, void* stream) {
  if (dtype != PA_BF16) return pa_fail(PA_ERR_UNSUPPORTED, "pa_prefill: bf16 only");
  if (num_seqs < 0 || num_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0 || max_query_len < 0 || max_context_len < 1 || !std::isfinite(scale))
    return pa_fail(PA_ERR_INVALID, "pa_prefill: sizes");
  if (num_heads % num_kv_heads) return pa_fail(PA_ERR_INVALID, "pa_prefill: num_heads % num_kv_heads != 0");
  const int g = num_heads / num_kv_heads;
  if (!(g == 1 || g == 2 || g == 4 || g == 8)) return pa_fail(PA_ERR_UNSUPPORTED, "pa_prefill: heads per KV head");
  if (!supported_shape(head_dim, block_size)) return pa_fail(PA_ERR_UNSUPPORTED, "pa_prefill: head_dim/block_size");
  if (cdiv(max_context_len, block_size) > max_blocks_per_seq)
    return pa_fail(PA_ERR_INVALID, "pa_prefill: max_blocks_per_seq < ceil(max_context_len / block_size)");
  if (max_query_len > max_context_len) return pa_fail(PA_ERR_INVALID, "pa_prefill: max_query_len > max_context_len");
  if (num_seqs > 65535 || num_kv_heads > 65535) return pa_fail(PA_ERR_UNSUPPORTED, "pa_prefill: more than 65535 sequences");
  if ((long long)num_blocks * num_kv_heads * block_size >= (1LL << 31))
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_prefill: pool rows exceed 2^31 (TMA coordinates are 32-bit)");
  if ((long long)max_query_len * g > (1LL << 30)) return pa_fail(PA_ERR_UNSUPPORTED, "pa_prefill: prompt too long");
  if (cdiv(max_query_len * g, 128) > 65535)
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_prefill: more than 65535 query tiles of 128 rows");
  if (num_seqs == 0 || num_tokens == 0) return PA_OK;
  if (!q || !k || !v || !slot_mapping || !query_start || !context_lens || !block_tables || !k_cache || !v_cache ||
      !out)
    return pa_fail(PA_ERR_INVALID, "pa_prefill: null pointer");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(out, 16) || !aligned(slot_mapping, 8) || !aligned(query_start, 4) || !aligned(context_lens, 4) ||
      !aligned(block_tables, 4))
    return pa_fail(PA_ERR_INVALID, "pa_prefill: misaligned pointer");
  pa::PrefillArgs a{};
  int rc = status_ptr(&a.status);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The prompt's keys and values first; the attention kernel waits for them.
  cudaError_t e = pa::launch_cache_append(k, v, slot_mapping, num_tokens, k_cache, v_cache, num_blocks,
                                          num_kv_heads, head_dim, block_size, 2, a.status, st);
  if (e != cudaSuccess) return cuda_fail(e, "pa_prefill append launch");
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.out = out;
  a.block_tables = block_tables;
  a.query_start = query_start;
  a.context_lens = context_lens;
  a.S = num_seqs;
  a.T = num_tokens;
  a.H = num_heads;
  a.Hkv = num_kv_heads;
  a.g = g;
  a.D = head_dim;
  a.B = block_size;
  a.num_blocks = num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_ctx = max_context_len;
  a.max_query_len = max_query_len;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  // 5th-generation tensor cores (tcgen05) for head_dim 64 and 128
  CUtensorMap kmap, vmap, qmap, omap;
  rc = make_block_map(&kmap, k_cache, num_blocks, num_kv_heads, block_size, head_dim);
  if (rc) return rc;
  rc = make_block_map(&vmap, v_cache, num_blocks, num_kv_heads, block_size, head_dim);
  if (rc) return rc;
  rc = make_query_map(&qmap, q, num_tokens, num_heads, g, head_dim);
  if (rc) return rc;
  rc = make_query_map(&omap, out, num_tokens, num_heads, g, head_dim);  // full tiles of output rows are stored by TMA
  if (rc) return rc;
  e = pa::launch_prefill_tc(a, kmap, vmap, qmap, omap, st);
  if (e != cudaSuccess) return cuda_fail(e, "pa_prefill launch");
  return PA_OK;
}

int pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                  int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, float scale,
                  float k_scale, float v_scale, void* out, int num_seqs, int num_heads, int num_kv_heads,
                  int head_dim, int block_size, int num_blocks, int partition_size, const void* plan,
                  void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, max_context_len, scale,
                     out, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, partition_size, plan,
                     nullptr, 0, workspace, workspace_bytes, PA_FP8_E4M3, stream, k_scale, v_scale);
}

int pa_decode_shared_prefix(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                            int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, float scale,
                            void* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                            int num_blocks, int partition_size, const int32_t* groups, int num_groups,
                            void* workspace, size_t workspace_bytes, int dtype, void* stream) {
  return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, max_context_len, scale,
                     out, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, partition_size,
                     nullptr, groups, num_groups, workspace, workspace_bytes, dtype, stream);
}

int pa_decode_planned_shared_prefix(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, int max_blocks_per_seq,
                                    const int32_t* context_lens, int max_context_len, float scale, void* out,
                                    int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, int partition_size, const int32_t* groups, int num_groups,
                                    const void* plan, void* workspace, size_t workspace_bytes, int dtype,
                                    void* stream) {
  if (!plan) return pa_fail(PA_ERR_INVALID, "pa_decode_planned_shared_prefix: null plan");
  return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, max_context_len, scale,
                     out, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, partition_size,
                     plan, groups, num_groups, workspace, workspace_bytes, dtype, stream);
}

}  // extern "C"
