// Log-sum-exp merge of split-K partials.
//
// A context longer than one partition is decoded as independent partitions
// p, each leaving an un-normalised output O_p (weights exp2(s - M_p)), its
// max M_p and its weight sum L_p (all in the log2 domain).  The exact
// softmax over the whole context is then
//     out = sum_p 2^(M_p - M) O_p / sum_p 2^(M_p - M) L_p,   M = max_p M_p,
// the same value the unsplit softmax(q Kᵀ) V of "PagedAttention Kernel：
// 大模型推理优化的显存管理革新" section 3.1 gives, up to rounding.
//
// Each (sequence, query head) gets `wpr` warps (8 for contexts of 32 or more
// partitions, else 1) and a CTA of eight warps serves 8 / wpr of them; warp
// w of a group takes partitions w, w + wpr, ...  Up to 32 of them, lane i
// reads partition i's (max, sum) once; the warp reduces the max and the
// weighted sum with shuffles and hands each partition's weight to the other
// lanes, which then sum the weighted partial rows, lane L holding D/32
// consecutive dims (each row one coalesced 4*D-byte line, no row's load
// waiting for another's, 16 rows in flight).  When no context has more than
// 16 partitions, a variant issues a warp's (max, sum) and row loads all
// together, one round trip to L2 instead of two.  The group's warps are combined
// through shared memory.  Sequences that fit one partition were written by
// the decode kernel and are skipped, unless they belong to a prefix group:
// there even a single partition is a partial written by the shared-prefix
// items.  Launched with programmatic dependent launch: the CTAs start while
// the decode kernel drains, read the context lengths (inputs) and only then
// wait for the decode kernel's results with griddepcontrol.wait.

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "device_common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kMaxWarps = 8;
// Calls whose contexts have at most this many partitions run a variant in
// which each warp (one per row) issues all its loads at once.
constexpr int kBatch = 16;

template <typename T, int D, bool kAllAtOnce>
__global__ void __launch_bounds__(kMaxWarps * 32) lse_merge_kernel(const DecodeArgs p, int wpr,
                                                                    const __grid_constant__ PrefixGroups pg) {
  constexpr int E = D / 32;
  __shared__ float s_m[kMaxWarps], s_l[kMaxWarps];
  __shared__ __align__(16) float s_o[kMaxWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long sh = (long long)blockIdx.x * (kMaxWarps / wpr) + warp / wpr;
  const int wg = warp % wpr;  // warp within its (sequence, head) group
  // The row's partition count comes from the inputs, not from the decode
  // kernel's results: it is known before the wait for them.
  int s = 0, h = 0, np = 0, first = 2;  // merge when np >= first
  if (sh < (long long)p.S * p.H) {
    s = (int)(sh / p.H);
    h = (int)(sh - (long long)s * p.H);
    const int ctx = min(max(p.context_lens[s], 0), p.max_ctx);
    np = (ctx + p.P - 1) / p.P;
    if (pg.n > 0 && prefix_parts_of(pg, s) > 0) first = 1;
  }
  pdl_wait_primary();
  float m = -INFINITY, l = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  if (np >= first) {
    const size_t base = (size_t)s * p.max_parts * p.H + h;  // row of partition 0
    const int cnt = np > wg ? (np - wg + wpr - 1) / wpr : 0;  // this warp's partitions wg, wg + wpr, ...
    // Their max and weight sum first, the lanes taking partitions: then the
    // weight of every partial row is known and the rows' loads below do not
    // wait on one another (a running max would chain them).
    if (kAllAtOnce) {
      // every load at once (cnt <= kBatch): lane i < cnt reads partition i's (max, sum),
      // and each lane its dims of all cnt partial rows; the weights follow
      float2 ml = make_float2(-INFINITY, 0.f);
      if (lane < cnt) ml = p.ws_ml[base + (size_t)(wg + lane * wpr) * p.H];
      float x[kBatch][E];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (i < cnt) {
          const float* src = p.ws_o + (base + (size_t)(wg + i * wpr) * p.H) * D + lane * E;
          if constexpr (E == 4) {
            const float4 v = *reinterpret_cast<const float4*>(src);
            x[i][0] = v.x, x[i][1] = v.y, x[i][2] = v.z, x[i][3] = v.w;
          } else {
            const float2 v = *reinterpret_cast<const float2*>(src);
            x[i][0] = v.x, x[i][1] = v.y;
          }
        }
      }
      m = ml.x;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      const float w = lane < cnt ? exp2f(ml.x - m) : 0.f;
      l = w * ml.y;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const float b = __shfl_sync(0xffffffffu, w, i);
        if (i < cnt) {
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] += x[i][e] * b;
        }
      }
    } else if (cnt <= 32) {
      // one partition per lane: its (max, sum) is read once and its weight
      // handed to the other lanes
      float2 ml = make_float2(-INFINITY, 0.f);
      if (lane < cnt) ml = p.ws_ml[base + (size_t)(wg + lane * wpr) * p.H];
      m = ml.x;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      const float w = lane < cnt ? exp2f(ml.x - m) : 0.f;
      l = w * ml.y;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll 16
      for (int i = 0; i < cnt; ++i) {
        const float b = __shfl_sync(0xffffffffu, w, i);
        const float* src = p.ws_o + (base + (size_t)(wg + i * wpr) * p.H) * D + lane * E;
        float x[E];
        if constexpr (E == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          x[0] = v.x, x[1] = v.y;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += x[e] * b;
      }
    } else {
      for (int i = lane; i < cnt; i += 32) m = fmaxf(m, p.ws_ml[base + (size_t)(wg + i * wpr) * p.H].x);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      for (int i = lane; i < cnt; i += 32) {
        const float2 ml = p.ws_ml[base + (size_t)(wg + i * wpr) * p.H];
        l += exp2f(ml.x - m) * ml.y;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll 8
      for (int i = 0; i < cnt; ++i) {
        const size_t wi = base + (size_t)(wg + i * wpr) * p.H;
        const float b = exp2f(p.ws_ml[wi].x - m);
        float x[E];
        if constexpr (E == 4) {
          const float4 v = *reinterpret_cast<const float4*>(p.ws_o + wi * D + lane * E);
          x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(p.ws_o + wi * D + lane * E);
          x[0] = v.x, x[1] = v.y;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += x[e] * b;
      }
    }
  }
  if (wpr > 1) {  // combine the group's warps through shared memory
    if (lane == 0) {
      s_m[warp] = m;
      s_l[warp] = l;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) s_o[warp][lane * E + e] = acc[e];
    __syncthreads();
    if (wg != 0 || np < first) return;
    float M = -INFINITY;
    for (int w = warp; w < warp + wpr; ++w) M = fmaxf(M, s_m[w]);
    l = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int w = warp; w < warp + wpr; ++w) {
      const float wt = exp2f(s_m[w] - M);  // a warp without partitions has max -inf: weight 0
      l += wt * s_l[w];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] += wt * s_o[w][lane * E + e];
    }
  } else if (np < first) {
    return;
  }
  const float inv = 1.f / l;
  T* dst = static_cast<T*>(p.out) + ((size_t)s * p.H + h) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if constexpr (sizeof(T) == 2)
      dst[e] = __float2bfloat16(acc[e] * inv);
    else
      dst[e] = acc[e] * inv;
  }
}

template <typename T, int D>
cudaError_t launch_typed(const DecodeArgs& a, const PrefixGroups& pg, cudaStream_t stream) {
  // Warps per (sequence, head): one while every context has at most kBatch
  // partitions (all loads at once), else enough to keep several partial rows
  // in flight for the longest context without idling warps on short ones.
  const bool all_at_once = a.max_parts <= kBatch;
  const int wpr = a.max_parts >= 32 ? 8 : 1;
  const long long pairs = (long long)a.S * a.H;
  const int per_cta = kMaxWarps / wpr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((pairs + per_cta - 1) / per_cta));
  cfg.blockDim = dim3(kMaxWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (all_at_once) return cudaLaunchKernelEx(&cfg, lse_merge_kernel<T, D, true>, a, wpr, pg);
  return cudaLaunchKernelEx(&cfg, lse_merge_kernel<T, D, false>, a, wpr, pg);
}

}  // namespace

cudaError_t launch_lse_merge(const DecodeArgs& a, const PrefixGroups& pg, int dtype, cudaStream_t stream) {
  if ((long long)a.S * a.H <= 0) return cudaSuccess;
  if (dtype == PA_BF16)
    return a.D == 128 ? launch_typed<__nv_bfloat16, 128>(a, pg, stream)
                      : launch_typed<__nv_bfloat16, 64>(a, pg, stream);
  return a.D == 128 ? launch_typed<float, 128>(a, pg, stream) : launch_typed<float, 64>(a, pg, stream);
}

}  // namespace pa
