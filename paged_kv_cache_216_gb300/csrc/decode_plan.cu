// Work list for the persistent decode kernel, longest items first.
//
// The decode work is one item per (sequence, partition, KV head).  All
// partitions of a context are `P` tokens except its last one.  Persistent
// CTAs take items from this list through an atomic counter (the dynamic work
// queue of "PagedAttention Kernel：大模型推理优化的显存管理革新" section 3.2),
// and in this order: every full partition first, then the partial ones from
// the longest to the shortest, so that the last items handed out are the
// shortest and no CTA is left with a long item at the end.
//
// Shared partitions of prefix groups (kernels.h) come first, as
// shared-prefix items that each cover several members; the members' own
// items for those partitions are left out.
//
// One CTA of 1024 threads.  It also validates the context lengths (status
// bit, clamping); an empty context gets one entry of length 0 at the end of
// the list, for which the decode kernel writes a zero output row.  It lets
// the decode kernel launch right away (programmatic dependent launch); the
// decode kernel waits for it before its first read of the list.

#include "device_common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kBuckets = 1024;

// Exclusive prefix sum of one value per thread over the CTA; *total gets the
// sum.  Uses `scratch` (32 ints) in shared memory.
__device__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    scratch[lane] = w;  // inclusive sums of the warps
  }
  __syncthreads();
  const int before = (warp ? scratch[warp - 1] : 0) + x - v;
  *total = scratch[31];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const int32_t* __restrict__ context_lens, int S,
                                                                   int P, int max_ctx, PlanHeader* hdr, int2* plan,
                                                                   unsigned* status, int g,
                                                                   const __grid_constant__ PrefixGroups pg) {
  pdl_launch_dependents();
  __shared__ int scratch[32];
  __shared__ int bucket_count[kBuckets];
  __shared__ int bucket_cursor[kBuckets];
  const int tid = threadIdx.x;
  for (int b = tid; b < kBuckets; b += kPlanThreads) bucket_count[b] = 0;
  __syncthreads();
  // Each thread owns a contiguous range of sequences.
  const int per = (S + kPlanThreads - 1) / kPlanThreads;
  const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
  int nfull = 0, nempty = 0;
  for (int s = s0; s < s1; ++s) {
    int c = context_lens[s];
    if (c < 1 || c > max_ctx) {
      raise_status(status, PA_STATUS_BAD_CONTEXT);
      c = c < 1 ? 0 : max_ctx;
    }
    const int skip = prefix_parts_of(pg, s);
    nfull += max(0, c / P - skip);
    nempty += c == 0;
    const int rem = c % P;
    if (rem && c / P >= skip) atomicAdd(&bucket_count[(int)((long long)(rem - 1) * kBuckets / P)], 1);
  }
  // Shared-prefix items: full partitions, at the head of the list.
  const int npre = prefix_entries(pg, g);
  for (int e = tid; e < npre; e += kPlanThreads) plan[e] = prefix_entry_at(pg, g, e);
  int total_full = 0;
  int pos = npre + block_exclusive_scan(nfull, scratch, &total_full);
  total_full += npre;
  for (int s = s0; s < s1; ++s) {
    int c = min(max(context_lens[s], 0), max_ctx);
    for (int p = prefix_parts_of(pg, s); p < c / P; ++p) plan[pos++] = make_int2(s | (p << 16), c);
  }
  // Partial partitions: buckets from the longest remainder down.
  int total_partial = 0;
  const int rb = kBuckets - 1 - tid;  // thread t scans bucket (kBuckets-1-t)
  const int cnt = rb >= 0 ? bucket_count[rb] : 0;
  const int start = block_exclusive_scan(cnt, scratch, &total_partial);
  if (rb >= 0) bucket_cursor[rb] = total_full + start;
  int total_empty = 0;
  int epos = total_full + total_partial + block_exclusive_scan(nempty, scratch, &total_empty);
  for (int s = s0; s < s1; ++s) {
    int c = min(max(context_lens[s], 0), max_ctx);
    if (c == 0) {
      plan[epos++] = make_int2(s, 0);
      continue;
    }
    const int rem = c % P;
    if (!rem || c / P < prefix_parts_of(pg, s)) continue;
    const int at = atomicAdd(&bucket_cursor[(int)((long long)(rem - 1) * kBuckets / P)], 1);
    plan[at] = make_int2(s | ((c / P) << 16), c);
  }
  if (tid == 0) {
    hdr->counter = 0u;
    hdr->num_pairs = total_full + total_partial + total_empty;
  }
}

}  // namespace

cudaError_t launch_decode_plan(const DecodeArgs& a, const PrefixGroups& pg, cudaStream_t stream) {
  decode_plan_kernel<<<1, kPlanThreads, 0, stream>>>(a.context_lens, a.S, a.P, a.max_ctx, a.hdr,
                                                     const_cast<int2*>(a.plan), a.status, a.g, pg);
  return cudaGetLastError();
}

}  // namespace pa
