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
// One warp per (sequence, query head); lanes hold D/32 consecutive dims, so
// each partial row is read as one coalesced 4*D-byte line.  Sequences that
// fit one partition were written by the decode kernel and are skipped.
// Launched with programmatic dependent launch: the CTAs may start while the
// decode kernel drains and wait for its results with griddepcontrol.wait.

#include <cuda_bf16.h>

#include <cmath>

#include "device_common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kWarps = 4;

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) lse_merge_kernel(const DecodeArgs p) {
  constexpr int E = D / 32;
  pdl_wait_primary();
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (wid >= (long long)p.S * p.H) return;
  const int s = (int)(wid / p.H);
  const int h = (int)(wid - (long long)s * p.H);
  const int ctx = min(max(p.context_lens[s], 0), p.max_ctx);
  const int np = (ctx + p.P - 1) / p.P;
  if (np <= 1) return;
  const size_t base = (size_t)s * p.max_parts * p.H + h;  // index of partition 0
  float M = -INFINITY;
  for (int pp = lane; pp < np; pp += 32) M = fmaxf(M, p.ws_ml[base + (size_t)pp * p.H].x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float L = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int pp = 0; pp < np; ++pp) {
    const size_t wi = base + (size_t)pp * p.H;
    const float2 ml = p.ws_ml[wi];
    const float wt = exp2f(ml.x - M);
    L += wt * ml.y;
    const float* src = p.ws_o + wi * D + lane * E;
    if constexpr (E == 4) {
      const float4 x = *reinterpret_cast<const float4*>(src);
      acc[0] += wt * x.x;
      acc[1] += wt * x.y;
      acc[2] += wt * x.z;
      acc[3] += wt * x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(src);
      acc[0] += wt * x.x;
      acc[1] += wt * x.y;
    }
  }
  const float inv = 1.f / L;
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
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t stream) {
  const long long warps = (long long)a.S * a.H;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((warps + kWarps - 1) / kWarps));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lse_merge_kernel<T, D>, a);
}

}  // namespace

cudaError_t launch_lse_merge(const DecodeArgs& a, int dtype, cudaStream_t stream) {
  if ((long long)a.S * a.H <= 0) return cudaSuccess;
  if (dtype == PA_BF16)
    return a.D == 128 ? launch_typed<__nv_bfloat16, 128>(a, stream) : launch_typed<__nv_bfloat16, 64>(a, stream);
  return a.D == 128 ? launch_typed<float, 128>(a, stream) : launch_typed<float, 64>(a, stream);
}

}  // namespace pa
