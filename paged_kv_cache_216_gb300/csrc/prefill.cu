// Prefill: causal attention of a prompt's tokens over a paged cache (bf16
// storage, fp32 accumulation, tensor cores).
//
// The step before decode: a prompt's keys and values are written into their
// slots like any appended token ("Day 6/90 of Inference Engineering",
// PagedAttention notes, paragraph 2), then every new token attends the
// sequence's tokens up to and including itself -- the softmax(scale·Q·Kᵀ)·V
// of "PagedAttention Kernel：大模型推理优化的显存管理革新" section 3.1 with a
// causal limit per query.  For sequence s with n_s new tokens and a context
// of ctx_s tokens after the append, new token i sits at position
// ctx_s - n_s + i.
//
// One CTA per (sequence, KV head, tile of 64 rows), the rows being (new
// token, query head) pairs of that KV head, token-major; tiles are taken
// longest first (the last tile of a prompt attends the most keys).  Four
// warps of 16 rows.  Keys and values stream through a 4-stage shared-memory
// ring 32 tokens at a time (cp.async, 16-byte pieces, rows XOR-swizzled so
// ldmatrix is conflict-free) up to the tile's last position; S = Q·Kᵀ and
// P·V use mma.m16n8k16 with the query rows as the 16 rows of A and the
// score accumulators repacked in registers as the A operand of P·V; each row
// is masked at its own position.  Launched after the append kernel with
// programmatic dependent launch: the query tile is loaded first, the cache
// only after griddepcontrol.wait.

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "device_common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kRows = 64;                   // query rows per CTA
constexpr int kChunk = 32;                  // keys per stage
constexpr int kStages = 4;
constexpr int kWarps = kRows / 16;
constexpr int kThreads = kWarps * 32;
constexpr unsigned kAll = 0xffffffffu;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int D>
struct PreCfg {
  static constexpr int kUnits = D / 8;                 // 16-byte pieces per row
  static constexpr int kQBytes = kRows * D * 2;
  static constexpr int kTileBytes = kChunk * D * 2;    // keys (or values) of a stage
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kOffRing = kQBytes;
  static constexpr int kBytes = kOffRing + kStages * kStageBytes;
};

// Byte offset of 16-byte piece u of row r (pieces XOR-permuted by the row's
// low three bits: the 8 rows of an ldmatrix phase hit 8 bank groups).
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int u) {
  return (uint32_t)(r * (D * 2) + ((u ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const PrefillArgs p) {
  using C = PreCfg<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int s = blockIdx.z, kvh = blockIdx.y;
  const int tile = (int)gridDim.x - 1 - (int)blockIdx.x;  // longest first

  const int q0 = __ldg(p.query_start + s), q1 = __ldg(p.query_start + s + 1);
  const int ctx = __ldg(p.context_lens + s);
  const int n_new = q1 - q0;
  const int rows = n_new * p.g;
  if (q0 < 0 || n_new < 0 || n_new > p.max_query_len || ctx < n_new || ctx > p.max_ctx || q1 > p.T) {
    if (tile == 0 && kvh == 0 && tid == 0) raise_status(p.status, PA_STATUS_BAD_CONTEXT);
    return;
  }
  const int row0 = tile * kRows;
  if (row0 >= rows) return;
  const int first_pos = ctx - n_new;             // position of new token 0
  const int last_row = min(rows, row0 + kRows) - 1;
  const int t_end = first_pos + last_row / p.g + 1;  // keys the tile attends
  const int nch = (t_end + kChunk - 1) / kChunk;

  const uint32_t sbase = smem_addr(smem);
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
  const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(p.k_cache);
  const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(p.v_cache);
  const int32_t* table = p.block_tables + (size_t)s * p.max_blocks_per_seq;

  // Query tile (an input, not written by the append).
  for (int i = tid; i < kRows * C::kUnits; i += kThreads) {
    const int r = i / C::kUnits, u = i % C::kUnits;
    const int gr = row0 + r;
    if (gr < rows) {
      const int h = kvh * p.g + gr % p.g;
      cp_async16(sbase + swz<D>(r, u), q + ((size_t)(q0 + gr / p.g) * p.H + h) * D + u * 8);
    } else {
      *reinterpret_cast<uint4*>(smem + swz<D>(r, u)) = make_uint4(0, 0, 0, 0);
    }
  }
  pdl_wait_primary();  // the prompt's keys and values are in the cache from here on

  auto load_chunk = [&](int c) {
    const uint32_t koff = C::kOffRing + (c % kStages) * C::kStageBytes;
    for (int i = tid; i < kChunk * C::kUnits; i += kThreads) {
      const int j = i / C::kUnits, u = i % C::kUnits;
      const uint32_t off = koff + swz<D>(j, u);
      const int t = c * kChunk + j;
      if (t < t_end) {
        int blk = __ldg(table + t / p.B);
        if ((unsigned)blk >= (unsigned)p.num_blocks) {
          raise_status(p.status, PA_STATUS_BAD_BLOCK);
          blk = 0;
        }
        const size_t row = ((size_t)blk * p.Hkv + kvh) * p.B + t % p.B;
        cp_async16(sbase + off, kc + row * D + u * 8);
        cp_async16(sbase + off + C::kTileBytes, vc + row * D + u * 8);
      } else {  // past the tile's last position: zeros, never stale NaN
        *reinterpret_cast<uint4*>(smem + off) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(smem + off + C::kTileBytes) = make_uint4(0, 0, 0, 0);
      }
    }
  };
  // The query tile joins the first chunk's group; one group per chunk.
#pragma unroll
  for (int c = 0; c < kStages - 1; ++c) {
    if (c < nch) load_chunk(c);
    cp_async_commit();
  }

  // Positions of this thread's two rows (a: gq, b: gq + 8 of the warp's 16).
  const int ra = row0 + warp * 16 + gq, rb = ra + 8;
  const int lim_a = ra < rows ? first_pos + ra / p.g + 1 : 0;  // keys 0 .. lim - 1
  const int lim_b = rb < rows ? first_pos + rb / p.g + 1 : 0;

  constexpr int KS = D / 16;
  constexpr int NT = D / 8;
  uint32_t qa[KS][4];
  float o[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

  for (int c = 0; c < nch; ++c) {
    if (c + kStages - 1 < nch) load_chunk(c + kStages - 1);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncthreads();
    if (c == 0) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        ldmatrix_x4(sbase + swz<D>(r, 2 * ks + (lane >> 4)), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
      }
    }
    const uint32_t kb = sbase + C::kOffRing + (c % kStages) * C::kStageBytes;
    const uint32_t vb = kb + C::kTileBytes;
    const int tc = c * kChunk;
    // A warp whose rows all end before this chunk skips it.
    const int warp_lim = min(rows - 1, row0 + warp * 16 + 15);
    if (row0 + warp * 16 < rows && tc < first_pos + warp_lim / p.g + 1) {
      float sc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 32; ++kk) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kb + swz<D>(nt * 8 + (lane & 7), 4 * kk + (lane >> 3)), b0, b1, b2, b3);
          mma_bf16_16816(sc[nt], qa[2 * kk][0], qa[2 * kk][1], qa[2 * kk][2], qa[2 * kk][3], b0, b1);
          mma_bf16_16816(sc[nt], qa[2 * kk + 1][0], qa[2 * kk + 1][1], qa[2 * kk + 1][2], qa[2 * kk + 1][3], b2,
                         b3);
        }
      }
      float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = tc + nt * 8 + 2 * tq + e;
          const float va = tok < lim_a ? sc[nt][e] * p.scale_log2 : -INFINITY;
          const float vb2 = tok < lim_b ? sc[nt][2 + e] * p.scale_log2 : -INFINITY;
          sc[nt][e] = va;
          sc[nt][2 + e] = vb2;
          mx_a = fmaxf(mx_a, va);
          mx_b = fmaxf(mx_b, vb2);
        }
      }
      mx_a = fmaxf(mx_a, __shfl_xor_sync(kAll, mx_a, 1));
      mx_a = fmaxf(mx_a, __shfl_xor_sync(kAll, mx_a, 2));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(kAll, mx_b, 1));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(kAll, mx_b, 2));
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      // A row with no key yet (a padding row) keeps weight 0, not NaN.
      const float base_a = mn_a == -INFINITY ? 0.f : mn_a;
      const float base_b = mn_b == -INFINITY ? 0.f : mn_b;
      const float al_a = exp2f(m_a - base_a), al_b = exp2f(m_b - base_b);
      float ls_a = 0.f, ls_b = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sc[nt][0] = exp2f(sc[nt][0] - base_a);
        sc[nt][1] = exp2f(sc[nt][1] - base_a);
        sc[nt][2] = exp2f(sc[nt][2] - base_b);
        sc[nt][3] = exp2f(sc[nt][3] - base_b);
        ls_a += sc[nt][0] + sc[nt][1];
        ls_b += sc[nt][2] + sc[nt][3];
      }
      l_a = l_a * al_a + ls_a;
      l_b = l_b * al_b + ls_b;
      m_a = mn_a;
      m_b = mn_b;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        o[nt][0] *= al_a;
        o[nt][1] *= al_a;
        o[nt][2] *= al_b;
        o[nt][3] *= al_b;
      }
#pragma unroll
      for (int kt = 0; kt < 2; ++kt) {
        const uint32_t a0 = pack_bf16x2(sc[2 * kt][0], sc[2 * kt][1]);
        const uint32_t a1 = pack_bf16x2(sc[2 * kt][2], sc[2 * kt][3]);
        const uint32_t a2 = pack_bf16x2(sc[2 * kt + 1][0], sc[2 * kt + 1][1]);
        const uint32_t a3 = pack_bf16x2(sc[2 * kt + 1][2], sc[2 * kt + 1][3]);
        const int mi = lane >> 3;
        const int t = kt * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(vb + swz<D>(t, 2 * np + (mi >> 1)), b0, b1, b2, b3);
          mma_bf16_16816(o[2 * np], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();  // the stage is refilled by a later iteration's load
  }
  cp_async_wait<0>();

  l_a += __shfl_xor_sync(kAll, l_a, 1);
  l_a += __shfl_xor_sync(kAll, l_a, 2);
  l_b += __shfl_xor_sync(kAll, l_b, 1);
  l_b += __shfl_xor_sync(kAll, l_b, 2);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? rb : ra;
    if (r >= rows) continue;
    const float inv = 1.f / (half ? l_b : l_a);
    const int h = kvh * p.g + r % p.g;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + ((size_t)(q0 + r / p.g) * p.H + h) * D + 2 * tq;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float x = half ? o[nt][2] : o[nt][0], y = half ? o[nt][3] : o[nt][1];
      *reinterpret_cast<uint32_t*>(dst + nt * 8) = pack_bf16x2(x * inv, y * inv);
    }
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  const int tiles = (a.max_query_len * a.g + kRows - 1) / kRows;
  if (tiles <= 0 || a.S <= 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::once_flag once[64];
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t init_err = cudaSuccess;
  std::call_once(once[dev], [&] {
    init_err = cudaFuncSetAttribute(prefill_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)PreCfg<128>::kBytes);
    if (init_err == cudaSuccess)
      init_err = cudaFuncSetAttribute(prefill_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)PreCfg<64>::kBytes);
  });
  if (init_err != cudaSuccess) return init_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tiles, (unsigned)a.Hkv, (unsigned)a.S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = a.D == 128 ? PreCfg<128>::kBytes : PreCfg<64>::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.D == 128 ? cudaLaunchKernelEx(&cfg, prefill_kernel<128>, a) : cudaLaunchKernelEx(&cfg, prefill_kernel<64>, a);
}

}  // namespace pa
