// Paged decode attention in fp32 on CUDA cores (fp32 storage, fp32 math).
//
// Same computation as the tensor-core path ("PagedAttention Kernel：
// 大模型推理优化的显存管理革新", section 3.1: Q·Kᵀ, softmax, P·V over the
// sequence's cache blocks), for caches stored in fp32 where bf16 tensor-core
// inputs would lose precision.  One CTA per (sequence, partition, KV head);
// each warp walks every fourth token of the partition: the lanes hold D/32
// consecutive dims of each of the g query heads, a token's key row is read
// coalesced (one row per warp load), the dot products are reduced with warp
// shuffles, and every lane keeps the same online-softmax state.  The four
// warps' states are merged through shared memory at the end.

#include <cmath>

#include "device_common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kWarps = 4;

template <int D>
__global__ void __launch_bounds__(kWarps * 32) paged_decode_simt_kernel(const DecodeArgs p) {
  constexpr int E = D / 32;  // dims per lane
  __shared__ float sO[kWarps][kMaxGroup][D];
  __shared__ float2 sML[kWarps][kMaxGroup];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x;
  const int per_seq = p.max_parts * p.Hkv;
  const int s = item / per_seq;
  const int part = (item - s * per_seq) / p.Hkv;
  const int kvh = item - s * per_seq - part * p.Hkv;
  int ctx = p.context_lens[s];
  if (ctx < 1 || ctx > p.max_ctx) {
    if (part == 0 && kvh == 0 && threadIdx.x == 0) raise_status(p.status, PA_STATUS_BAD_CONTEXT);
    ctx = ctx < 1 ? 0 : p.max_ctx;
  }
  const float* q = static_cast<const float*>(p.q);
  const float* kc = static_cast<const float*>(p.k_cache);
  const float* vc = static_cast<const float*>(p.v_cache);
  float* out = static_cast<float*>(p.out);
  if (ctx == 0) {
    if (part == 0)
      for (int e = threadIdx.x; e < p.g * D; e += blockDim.x)
        out[((size_t)s * p.H + kvh * p.g) * D + e] = 0.f;
    return;
  }
  const int t0 = part * p.P;
  if (t0 >= ctx) return;
  const int t1 = min(ctx, t0 + p.P);
  const int g = p.g;

  float qr[kMaxGroup][E], o[kMaxGroup][E], m[kMaxGroup], l[kMaxGroup];
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      o[h][e] = 0.f;
      qr[h][e] = h < g ? q[((size_t)s * p.H + kvh * g + h) * D + lane * E + e] : 0.f;
    }
  }
  const int32_t* table = p.block_tables + (size_t)s * p.max_blocks_per_seq;
  for (int t = t0 + warp; t < t1; t += kWarps) {
    int blk = table[t / p.B];
    if ((unsigned)blk >= (unsigned)p.num_blocks) {
      raise_status(p.status, PA_STATUS_BAD_BLOCK);
      blk = 0;
    }
    const size_t rowoff = (((size_t)blk * p.Hkv + kvh) * p.B + (t % p.B)) * D + lane * E;
    float kr[E], vr[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      kr[e] = kc[rowoff + e];
      vr[e] = vc[rowoff + e];
    }
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      if (h >= g) break;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) dot = fmaf(qr[h][e], kr[e], dot);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      const float sc = dot * p.scale_log2;
      const float mn = fmaxf(m[h], sc);
      const float alpha = exp2f(m[h] - mn);
      const float pw = exp2f(sc - mn);
      l[h] = l[h] * alpha + pw;
#pragma unroll
      for (int e = 0; e < E; ++e) o[h][e] = fmaf(pw, vr[e], o[h][e] * alpha);
      m[h] = mn;
    }
  }
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    if (h >= g) break;
    if (lane == 0) sML[warp][h] = make_float2(m[h], l[h]);
#pragma unroll
    for (int e = 0; e < E; ++e) sO[warp][h][lane * E + e] = o[h][e];
  }
  __syncthreads();
  const int np = (ctx + p.P - 1) / p.P;
  for (int u = threadIdx.x; u < g * D; u += blockDim.x) {
    const int h = u / D, d = u - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sML[w][h].x);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float wt = exp2f(sML[w][h].x - M);
      L += wt * sML[w][h].y;
      acc += wt * sO[w][h][d];
    }
    const int qh = kvh * g + h;
    if (np == 1) {
      out[((size_t)s * p.H + qh) * D + d] = acc / L;
    } else {
      const size_t wi = ((size_t)s * p.max_parts + part) * p.H + qh;
      p.ws_o[wi * D + d] = acc;
      if (d == 0) p.ws_ml[wi] = make_float2(M, L);
    }
  }
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t stream) {
  const long long grid = (long long)a.S * a.max_parts * a.Hkv;
  if (grid <= 0) return cudaSuccess;
  if (a.D == 128)
    paged_decode_simt_kernel<128><<<(unsigned)grid, kWarps * 32, 0, stream>>>(a);
  else
    paged_decode_simt_kernel<64><<<(unsigned)grid, kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pa
