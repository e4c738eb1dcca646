// Paged decode attention, bf16 storage, fp32 accumulation, on tensor cores.
//
// What it computes ("PagedAttention Kernel：大模型推理优化的显存管理革新",
// section 3.1): for each sequence and query head, Q·Kᵀ over the sequence's
// cache blocks, a softmax, and P·V over the same blocks.  Blocks are reached
// through the block table ("Day 6/90 of Inference Engineering", PagedAttention
// notes, paragraph 6).  The softmax is computed online (running max and sum),
// and a context is split into partitions whose partial results are merged by
// log-sum-exp (lse_merge.cu) when it spans more than one.
//
// Structure (sm_103a):
//  * Persistent CTAs, one or two per SM.  Work items are (partition,
//    sequence, KV head) triples taken round-robin.
//  * Warp 4 is the producer.  For each item it bulk-copies the item's g
//    query rows into a 2-slot Q ring, then streams the item's keys and values
//    32 tokens at a time into a ring of shared-memory stages: per cache block
//    of the chunk, one 2D TMA box of [B rows x 64 dims] per 64-dim half, for
//    K and for V, with 128-byte swizzle.  Block ids are read 32 at a time
//    (one per lane) one window ahead.  This is the prefetch of the same
//    page's section 2.2, done by the copy engine.
//  * Warps 0-3 are consumers; warp w takes the item's chunks w, w+4, ...
//    For a chunk, S = Q Kᵀ uses mma.m16n8k16 with the g query heads as the
//    16 rows of A (rows >= g are zero) and 8 tokens per B tile (ldmatrix
//    from the swizzled stage, conflict-free).  The accumulator layout of S
//    is exactly the B-operand layout of the P·V product computed as
//    Oᵀ = Vᵀ Pᵀ (ldmatrix.trans of V), so P never leaves registers.
//  * At the end of an item the four warps' (max, sum, O) states are merged
//    through shared memory; the result is written as bf16 output, or as an
//    fp32 partial for the merge kernel.
// Every wait is bounded (device_common.cuh); on time-out the kernel raises
// PA_STATUS_TIMEOUT and winds down without touching global memory further.

#include <cuda_bf16.h>

#include <cmath>

#include "device_common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kChunk = 32;  // tokens per pipeline stage
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kHalfBytes = kChunk * 128;  // one 64-dim half of 32 rows

template <int D>
struct TcCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kRegion = kHalves * kHalfBytes;  // K (or V) of a stage
  static constexpr int kStage = 2 * kRegion;
  // A multiple of the consumer-warp count: chunk k goes to warp k % 4 and
  // stage k % kStages, so every stage is always consumed by the same warp.
  // Otherwise a warp running ahead could test a stage's barrier while it is
  // still two phases behind, and the parity wait would pass on the wrong
  // phase.
  static constexpr int kStages = (D == 128) ? 4 : 8;
  static_assert(kStages % kConsumerWarps == 0, "each stage must belong to one consumer warp");
  static constexpr int kQSlot = kMaxGroup * D * 2;
  static constexpr int kOStride = D + 4;  // floats per (warp, head) row; +4 spreads banks
  static constexpr int kOBuf = kConsumerWarps * kMaxGroup * kOStride * 4;
  static constexpr int kML = kConsumerWarps * kMaxGroup * 8;
  static constexpr int kBars = (2 * kStages + 4) * 8;
  // byte offsets from the 1024-aligned base
  static constexpr int kOffQ = kStages * kStage;
  static constexpr int kOffO = kOffQ + 2 * kQSlot;
  static constexpr int kOffML = kOffO + kOBuf;
  static constexpr int kOffBar = kOffML + kML;
  static constexpr int kOffAbort = kOffBar + kBars;
  static constexpr int kOffCtx = kOffAbort + 16;
  static size_t bytes(int S) { return 1024 + kOffCtx + (size_t)S * 4; }
};

struct Item {
  int s, part, kvh, t0, t1;
};

// Item i of the round-robin order: partition-major, then sequence, then KV
// head.  Returns false for an empty slot (partition past the context).
__device__ __forceinline__ bool item_at(const DecodeArgs& p, const int* sctx, int i, Item& it) {
  const int per_part = p.S * p.Hkv;
  it.part = i / per_part;
  const int r = i - it.part * per_part;
  it.s = r / p.Hkv;
  it.kvh = r - it.s * p.Hkv;
  const int ctx = sctx[it.s];
  it.t0 = it.part * p.P;
  if (it.t0 >= ctx) return false;
  it.t1 = min(ctx, it.t0 + p.P);
  return true;
}

__device__ __forceinline__ int load_block_id(const int32_t* row, int rel, int nblk) {
  return rel < nblk ? __ldg(row + rel) : 0;
}

template <int D>
__device__ void producer(const CUtensorMap* kmap, const CUtensorMap* vmap, const DecodeArgs& p, uint8_t* base,
                         const int* sctx, volatile int* abort) {
  using C = TcCfg<D>;
  const int lane = threadIdx.x & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + C::kOffBar);
  uint64_t* empty = full + C::kStages;
  uint64_t* qfull = empty + C::kStages;
  uint64_t* qempty = qfull + 2;
  const uint64_t policy = policy_evict_first();
  const int total = p.max_parts * p.S * p.Hkv;
  const int bpc = kChunk / p.B;  // cache blocks per chunk
  const uint32_t qbytes = (uint32_t)(p.g * D * 2);
  const uint32_t chunk_block_bytes = (uint32_t)(p.B * D * 2 * 2);  // K + V of one block
  uint32_t kseq = 0, n = 0;
  bool ok = true;
  for (int i = blockIdx.x; i < total && ok; i += gridDim.x) {
    Item it;
    if (!item_at(p, sctx, i, it)) continue;
    const int slot = n & 1;
    if (!mbar_wait(&qempty[slot], ((n >> 1) & 1) ^ 1, abort)) {
      ok = false;
      break;
    }
    if (lane == 0) {
      mbar_arrive_expect_tx(&qfull[slot], qbytes);
      const __nv_bfloat16* src =
          static_cast<const __nv_bfloat16*>(p.q) + ((size_t)it.s * p.H + (size_t)it.kvh * p.g) * D;
      bulk_load(base + C::kOffQ + slot * C::kQSlot, src, qbytes, &qfull[slot]);
    }
    ++n;  // items whose Q copy has been issued
    const int32_t* row = p.block_tables + (size_t)it.s * p.max_blocks_per_seq + it.t0 / p.B;
    const int nblk = (it.t1 - it.t0 + p.B - 1) / p.B;
    int cur = load_block_id(row, lane, nblk);
    int nxt = load_block_id(row, 32 + lane, nblk);
    int wbase = 0;
    const int nch = (it.t1 - it.t0 + kChunk - 1) / kChunk;
    for (int ch = 0; ch < nch; ++ch, ++kseq) {
      const int jb = ch * bpc;
      if (jb >= wbase + 32) {
        cur = nxt;
        wbase += 32;
        nxt = load_block_id(row, wbase + 32 + lane, nblk);
      }
      const int nv = min(kChunk, it.t1 - (it.t0 + ch * kChunk));
      const int nb = (nv + p.B - 1) / p.B;
      int id = __shfl_sync(0xffffffffu, cur, (jb - wbase + lane) & 31);
      if (lane < nb && (unsigned)id >= (unsigned)p.num_blocks) {
        raise_status(p.status, PA_STATUS_BAD_BLOCK);
        id = 0;
      }
      const int stage = kseq % C::kStages;
      if (!mbar_wait(&empty[stage], ((kseq / C::kStages) & 1) ^ 1, abort)) {
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], (uint32_t)nb * chunk_block_bytes);
      __syncwarp();
      if (lane < nb) {
        const int y = (id * p.Hkv + it.kvh) * p.B;
        uint8_t* sk = base + stage * C::kStage + lane * p.B * 128;
        uint8_t* sv = sk + C::kRegion;
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf) {
          tma_load_2d(sk + hf * kHalfBytes, kmap, &full[stage], hf * 64, y, policy);
          tma_load_2d(sv + hf * kHalfBytes, vmap, &full[stage], hf * 64, y, policy);
        }
      }
    }
  }
  if (!ok) {
    raise_status(p.status, PA_STATUS_TIMEOUT);
    *abort = 1;
    // Let copies already issued land before the CTA's shared memory goes away.
    const volatile int never = 0;
    for (uint32_t k = (kseq > (uint32_t)C::kStages ? kseq - C::kStages : 0); k < kseq; ++k)
      mbar_wait(&full[k % C::kStages], (k / C::kStages) & 1, &never);
    for (uint32_t k = (n > 2 ? n - 2 : 0); k < n; ++k) mbar_wait(&qfull[k & 1], (k >> 1) & 1, &never);
  }
}

template <int D>
__device__ void consumer(const DecodeArgs& p, uint8_t* base, const int* sctx, volatile int* abort) {
  using C = TcCfg<D>;
  constexpr int KS = D / 16;  // k-steps of the Q·Kᵀ product
  constexpr int MT = D / 16;  // m-tiles of the Oᵀ = Vᵀ Pᵀ product
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2;  // mma group id: head row of S, token row of K tiles
  const int tq = lane & 3;   // thread in group
  uint64_t* full = reinterpret_cast<uint64_t*>(base + C::kOffBar);
  uint64_t* empty = full + C::kStages;
  uint64_t* qfull = empty + C::kStages;
  uint64_t* qempty = qfull + 2;
  float* sO = reinterpret_cast<float*>(base + C::kOffO);
  float2* sML = reinterpret_cast<float2*>(base + C::kOffML);
  const int total = p.max_parts * p.S * p.Hkv;
  const uint32_t base_addr = smem_addr(base);
  bool alive = true;
  uint32_t kseq = 0, n = 0;

  for (int i = blockIdx.x; i < total; i += gridDim.x) {
    Item it;
    if (!item_at(p, sctx, i, it)) continue;
    const int nch = (it.t1 - it.t0 + kChunk - 1) / kChunk;
    const int slot = n & 1;
    uint32_t qa[KS][2];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) qa[ks][0] = qa[ks][1] = 0u;
    if (alive && !mbar_wait(&qfull[slot], (n >> 1) & 1, abort)) {
      alive = false;
      *abort = 1;
      raise_status(p.status, PA_STATUS_TIMEOUT);
    }
    if (alive) {
      const __nv_bfloat16* sq = reinterpret_cast<const __nv_bfloat16*>(base + C::kOffQ + slot * C::kQSlot);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa[ks][0] = gq < p.g ? *reinterpret_cast<const uint32_t*>(sq + gq * D + ks * 16 + 2 * tq) : 0u;
        qa[ks][1] = gq < p.g ? *reinterpret_cast<const uint32_t*>(sq + gq * D + ks * 16 + 8 + 2 * tq) : 0u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[slot]);
    }
    float m_run = -INFINITY, l_run = 0.f;
    float o[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    for (int ch = 0; ch < nch; ++ch, ++kseq) {
      if ((int)(kseq & (kConsumerWarps - 1)) != warp || !alive) continue;
      const int stage = kseq % C::kStages;
      if (!mbar_wait(&full[stage], (kseq / C::kStages) & 1, abort)) {
        alive = false;
        *abort = 1;
        raise_status(p.status, PA_STATUS_TIMEOUT);
        continue;
      }
      const int nv = min(kChunk, it.t1 - (it.t0 + ch * kChunk));
      const uint32_t sk = base_addr + stage * C::kStage;
      const uint32_t sv = sk + C::kRegion;
      if (nv < kChunk) {
        // Rows past the context hold stale or unwritten data: zero their V
        // (their scores are masked below, but 0 * NaN would still be NaN).
        uint8_t* vrow = base + stage * C::kStage + C::kRegion;
        const int units = (kChunk - nv) * C::kHalves * 8;
        for (int u = lane; u < units; u += 32) {
          const int r = nv + u / (C::kHalves * 8);
          const int rem = u % (C::kHalves * 8);
          *reinterpret_cast<uint4*>(vrow + (rem >> 3) * kHalfBytes + r * 128 + (rem & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      // S = Q Kᵀ : 4 tiles of 8 tokens; rows = heads (only c0, c1 are real).
      float sc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 32; ++kk) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int t = nt * 8 + (lane & 7);
          const int cidx = 4 * kk + (lane >> 3);
          const uint32_t addr = sk + (cidx >> 3) * kHalfBytes + t * 128 + (((cidx & 7) ^ (t & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(addr, b0, b1, b2, b3);
          mma_bf16_16816(sc[nt], qa[2 * kk][0], 0u, qa[2 * kk][1], 0u, b0, b1);
          mma_bf16_16816(sc[nt], qa[2 * kk + 1][0], 0u, qa[2 * kk + 1][1], 0u, b2, b3);
        }
      }
      // Online softmax (log2 domain) for head row gq over this chunk.
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = nt * 8 + 2 * tq + e;
          const float v = tok < nv ? sc[nt][e] * p.scale_log2 : -INFINITY;
          sc[nt][e] = v;
          mx = fmaxf(mx, v);
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = exp2f(m_run - m_new);
      float ls = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sc[nt][0] = exp2f(sc[nt][0] - m_new);
        sc[nt][1] = exp2f(sc[nt][1] - m_new);
        ls += sc[nt][0] + sc[nt][1];
      }
      l_run = l_run * alpha + ls;
      m_run = m_new;
      const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * tq);
      const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * tq + 4);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        o[mt][0] *= a_lo;
        o[mt][1] *= a_hi;
        o[mt][2] *= a_lo;
        o[mt][3] *= a_hi;
      }
      // Oᵀ += Vᵀ Pᵀ : k = 16 tokens per step, m = 16 dims per tile.
#pragma unroll
      for (int kt = 0; kt < 2; ++kt) {
        const uint32_t pb0 = pack_bf16x2(sc[2 * kt][0], sc[2 * kt][1]);
        const uint32_t pb1 = pack_bf16x2(sc[2 * kt + 1][0], sc[2 * kt + 1][1]);
        const int t = 16 * kt + ((lane >> 4) << 3) + (lane & 7);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int cidx = 2 * mt + ((lane >> 3) & 1);
          const uint32_t addr = sv + (cidx >> 3) * kHalfBytes + t * 128 + (((cidx & 7) ^ (t & 7)) << 4);
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4_trans(addr, a0, a1, a2, a3);
          mma_bf16_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }

    // ---- item epilogue: merge the four warps' states ----
    float l = l_run;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (tq == 0 && gq < p.g) sML[warp * kMaxGroup + gq] = make_float2(m_run, l);
    float* ob = sO + warp * kMaxGroup * C::kOStride;
    const int h0 = 2 * tq, h1 = 2 * tq + 1;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int d = 16 * mt + gq;
      if (h0 < p.g) {
        ob[h0 * C::kOStride + d] = o[mt][0];
        ob[h0 * C::kOStride + d + 8] = o[mt][2];
      }
      if (h1 < p.g) {
        ob[h1 * C::kOStride + d] = o[mt][1];
        ob[h1 * C::kOStride + d + 8] = o[mt][3];
      }
    }
    named_barrier_sync(1, kConsumerWarps * 32);
    const bool live = alive && !*abort;
    const int tid = threadIdx.x;
    const int units = p.g * (D / 8);
    const int np = (sctx[it.s] + p.P - 1) / p.P;
    for (int u = tid; u < units && live; u += kConsumerWarps * 32) {
      const int h = u / (D / 8);
      const int d0 = (u % (D / 8)) * 8;
      float mw[kConsumerWarps];
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        mw[w] = sML[w * kMaxGroup + h].x;
        M = fmaxf(M, mw[w]);
      }
      float L = 0.f, acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float wt = exp2f(mw[w] - M);
        L += wt * sML[w * kMaxGroup + h].y;
        const float4* src = reinterpret_cast<const float4*>(sO + (w * kMaxGroup + h) * C::kOStride + d0);
        const float4 x0 = src[0], x1 = src[1];
        acc[0] += wt * x0.x;
        acc[1] += wt * x0.y;
        acc[2] += wt * x0.z;
        acc[3] += wt * x0.w;
        acc[4] += wt * x1.x;
        acc[5] += wt * x1.y;
        acc[6] += wt * x1.z;
        acc[7] += wt * x1.w;
      }
      const int qh = it.kvh * p.g + h;
      if (np == 1) {
        const float inv = 1.f / L;
        uint4 pk;
        pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
        pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + ((size_t)it.s * p.H + qh) * D + d0;
        *reinterpret_cast<uint4*>(dst) = pk;
      } else {
        const size_t wi = ((size_t)it.s * p.max_parts + it.part) * p.H + qh;
        float4* dst = reinterpret_cast<float4*>(p.ws_o + wi * D + d0);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        if (d0 == 0) p.ws_ml[wi] = make_float2(M, L);
      }
    }
    named_barrier_sync(1, kConsumerWarps * 32);
    ++n;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const DecodeArgs p) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int* sctx = reinterpret_cast<int*>(base + C::kOffCtx);
  volatile int* abort = reinterpret_cast<volatile int*>(base + C::kOffAbort);

  for (int s = threadIdx.x; s < p.S; s += blockDim.x) {
    int c = p.context_lens[s];
    if (c < 1 || c > p.max_ctx) {
      if (blockIdx.x == 0) raise_status(p.status, PA_STATUS_BAD_CONTEXT);
      c = c < 1 ? 0 : p.max_ctx;
    }
    sctx[s] = c;
  }
  if (threadIdx.x == 0) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kOffBar);
    for (int k = 0; k < C::kStages; ++k) {
      mbar_init(&bars[k], 1);                            // full: producer arrival + TMA bytes
      mbar_init(&bars[C::kStages + k], 1);               // empty: the consuming warp
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bars[2 * C::kStages + k], 1);               // Q full
      mbar_init(&bars[2 * C::kStages + 2 + k], kConsumerWarps);  // Q empty
    }
    *abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  // Sequences with an empty context get a zero output row.
  if (blockIdx.x == 0) {
    for (int s = 0; s < p.S; ++s) {
      if (sctx[s] != 0) continue;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + (size_t)s * p.H * D;
      for (int e = threadIdx.x; e < p.H * D; e += blockDim.x) dst[e] = __float2bfloat16(0.f);
    }
  }

  if ((threadIdx.x >> 5) == kConsumerWarps) {
    if ((threadIdx.x & 31) == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    producer<D>(&kmap, &vmap, p, base, sctx, abort);
  } else {
    consumer<D>(p, base, sctx, abort);
  }
}

}  // namespace

size_t decode_tc_smem_bytes(int D, int S) {
  return D == 128 ? TcCfg<128>::bytes(S) : TcCfg<64>::bytes(S);
}

cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream) {
  const size_t smem = decode_tc_smem_bytes(a.D, a.S);
  auto kern = a.D == 128 ? paged_decode_tc_kernel<128> : paged_decode_tc_kernel<64>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static thread_local int cached_dev = -1;
  static thread_local int sms = 0;
  if (cached_dev != dev) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cached_dev = dev;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const long long total = (long long)a.max_parts * a.S * a.Hkv;
  const int grid = (int)std::min<long long>(total, (long long)sms * per_sm);
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, kThreads, smem, stream>>>(kmap, vmap, a);
  return cudaGetLastError();
}

}  // namespace pa
