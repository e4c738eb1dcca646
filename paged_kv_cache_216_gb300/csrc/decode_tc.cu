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
//  * Persistent CTAs, two per SM.  Work items are (sequence, partition, KV
//    head) triples taken from a longest-first work list (decode_plan.cu)
//    through an atomic counter, the dynamic work queue of the same page's
//    section 3.2; the producer claims the next item as it starts one.
//  * Warp 4 is the producer.  For each item it writes the item's descriptor
//    and bulk-copies its g query rows into a 2-slot Q ring, then streams the item's keys and values
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
//    through shared memory (two mbarriers order the exchange); the result is
//    written as bf16 output, or as an fp32 partial for the merge kernel.
// Every wait is bounded (device_common.cuh); on time-out the kernel raises
// PA_STATUS_TIMEOUT and winds down without touching global memory further.

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "device_common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kChunk = 32;  // tokens per pipeline stage
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kHalfBytes = kChunk * 128;  // one 64-dim half of 32 rows
constexpr unsigned kFull = 0xffffffffu;

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
  // mbarriers: full[kStages], empty[kStages], qfull[2], qempty[2], epi_full, epi_done
  static constexpr int kBars = (2 * kStages + 6) * 8;
  // byte offsets from the 1024-aligned base
  static constexpr int kOffQ = kStages * kStage;
  static constexpr int kOffO = kOffQ + 2 * kQSlot;
  static constexpr int kOffML = kOffO + kOBuf;
  static constexpr int kOffDesc = kOffML + kML;  // int4 per Q slot: {s, part, kvh, ctx or -1}
  static constexpr int kOffBar = kOffDesc + 2 * 16;
  static constexpr int kOffAbort = kOffBar + kBars;
  static constexpr size_t kBytes = 1024 + kOffAbort + 16;
};

struct Bars {
  uint64_t *full, *empty, *qfull, *qempty, *epi_full, *epi_done;
};

template <int D>
__device__ __forceinline__ Bars bars_at(uint8_t* base) {
  using C = TcCfg<D>;
  Bars b;
  b.full = reinterpret_cast<uint64_t*>(base + C::kOffBar);
  b.empty = b.full + C::kStages;
  b.qfull = b.empty + C::kStages;
  b.qempty = b.qfull + 2;
  b.epi_full = b.qempty + 2;
  b.epi_done = b.epi_full + 1;
  return b;
}

__device__ __forceinline__ void give_up(const DecodeArgs& p, volatile int* abort) {
  *abort = 1;
  raise_status(p.status, PA_STATUS_TIMEOUT);
}

// kInter: each 256-byte token row is two 128-byte lines of the stage
// (line 2t + half) and one TMA box brings a whole [B x D] slab; otherwise
// the two 64-dim halves of a chunk are separate 32-line regions (line
// half*32 + t) filled by one box per half.  The first halves the number of
// TMA requests (used for 8-token blocks, whose per-half boxes are only
// 1 KB); the second keeps ldmatrix free of bank conflicts.
template <int D, bool kInter>
__device__ __forceinline__ int stage_line(int t, int half) {
  return kInter ? 2 * t + half : half * kChunk + t;
}

template <int D, bool kInter, bool kShared>
__device__ void producer(const CUtensorMap* kmap, const CUtensorMap* vmap, const DecodeArgs& p, uint8_t* base,
                         volatile int* abort) {
  using C = TcCfg<D>;
  const int lane = threadIdx.x & 31;
  const Bars bar = bars_at<D>(base);
  int4* desc = reinterpret_cast<int4*>(base + C::kOffDesc);
  const uint64_t policy = policy_evict_first();
  const int bpc = kChunk / p.B;  // cache blocks per chunk
  const uint32_t qbytes = (uint32_t)(p.g * D * 2);
  const uint32_t chunk_block_bytes = (uint32_t)(p.B * D * 2 * 2);  // K + V of one block

  pdl_wait_primary();  // the work list is complete and visible from here on
  const int total = __ldcg(&p.hdr->num_pairs) * p.Hkv;
  unsigned* counter = &p.hdr->counter;
  // Lane 0 claims the next work item when it starts the current one and
  // reads that item's list entry once the current item's first chunk is on
  // its way, so the atomic and the read overlap the copies.  Holding only
  // one item ahead keeps the tail of the queue balanced across CTAs.
  int cur_idx = total;
  int2 cur_pr = make_int2(0, -1);
  if (lane == 0) {
    cur_idx = (int)atomicAdd(counter, 1u);
    if (cur_idx < total) cur_pr = __ldcg(p.plan + cur_idx / p.Hkv);
  }
  uint32_t kseq = 0, nq = 0;
  bool ok = true;
  for (uint32_t n = 0;; ++n) {
    int2 nxt_pr = make_int2(0, -1);
    int nxt_idx = total;
    if (lane == 0 && cur_idx < total) nxt_idx = (int)atomicAdd(counter, 1u);
    const int idx = __shfl_sync(kFull, cur_idx, 0);
    const int prx = __shfl_sync(kFull, cur_pr.x, 0);
    const int ctx = __shfl_sync(kFull, cur_pr.y, 0);  // < 0: a shared-prefix item
    const int slot = n & 1;
    if (!mbar_wait(&bar.qempty[slot], ((n >> 1) & 1) ^ 1, abort, p.wait_limit_ns)) {
      ok = false;
      break;
    }
    if (idx >= total) {  // no work left: tell the consumers
      if (lane == 0) {
        desc[slot] = make_int4(0, 0, 0, -1);
        mbar_arrive(&bar.qfull[slot]);
      }
      break;
    }
    // Table row ts; query rows of nm sequences s0 .. s0 + nm - 1 (one for
    // ordinary items; a shared-prefix item covers a whole partition).
    const bool shared = kShared && ctx < 0;
    const int ts = prx & 0xffff, part = prx >> 16, kvh = idx % p.Hkv;
    const int s0 = shared ? (ctx >> 4) & 0xffff : ts;
    const int nm = shared ? ctx & 15 : 1;
    const int t0 = part * p.P, t1 = shared ? t0 + p.P : min(ctx, t0 + p.P);
    if (lane == 0) {
      // a shared item's descriptor also carries its member count and a flag
      const int dy = kShared ? part | (nm << 16) | (shared ? 1 << 20 : 0) : part;
      desc[slot] = make_int4(s0, dy, kvh, shared ? t1 : ctx);
      mbar_arrive_expect_tx(&bar.qfull[slot], (uint32_t)nm * qbytes);
      for (int i = 0; i < nm; ++i) {
        const __nv_bfloat16* src =
            static_cast<const __nv_bfloat16*>(p.q) + ((size_t)(s0 + i) * p.H + (size_t)kvh * p.g) * D;
        bulk_load(base + C::kOffQ + slot * C::kQSlot + i * qbytes, src, qbytes, &bar.qfull[slot]);
      }
    }
    ++nq;
    const int32_t* row = p.block_tables + (size_t)ts * p.max_blocks_per_seq + t0 / p.B;
    const int nblk = (t1 - t0 + p.B - 1) / p.B;
    int cur = load_block_id(row, lane, nblk);
    int nxt = load_block_id(row, 32 + lane, nblk);
    int wbase = 0;
    const int nch = (t1 - t0 + kChunk - 1) / kChunk;
    for (int ch = 0; ch < nch; ++ch, ++kseq) {
      const int jb = ch * bpc;
      if (jb >= wbase + 32) {
        cur = nxt;
        wbase += 32;
        nxt = load_block_id(row, wbase + 32 + lane, nblk);
      }
      const int nv = min(kChunk, t1 - (t0 + ch * kChunk));
      const int nb = (nv + p.B - 1) / p.B;
      int id = __shfl_sync(kFull, cur, (jb - wbase + lane) & 31);
      if (lane < nb && (unsigned)id >= (unsigned)p.num_blocks) {
        raise_status(p.status, PA_STATUS_BAD_BLOCK);
        id = 0;
      }
      const int stage = kseq % C::kStages;
      // Test hook: a withheld chunk is never issued (no copy in flight, no
      // arrival), so the consumer's wait for it runs out.
      const bool issue = kseq != (uint32_t)p.withhold_chunk;
      if (issue && !mbar_wait(&bar.empty[stage], ((kseq / C::kStages) & 1) ^ 1, abort, p.wait_limit_ns)) {
        ok = false;
        break;
      }
      if (issue && lane == 0) mbar_arrive_expect_tx(&bar.full[stage], (uint32_t)nb * chunk_block_bytes);
      __syncwarp();
      if (issue && lane < nb) {
        const int y = (id * p.Hkv + kvh) * p.B;
        if constexpr (kInter) {
          uint8_t* sk = base + stage * C::kStage + lane * p.B * 256;
          tma_load_2d(sk, kmap, &bar.full[stage], 0, 2 * y, policy);
          tma_load_2d(sk + C::kRegion, vmap, &bar.full[stage], 0, 2 * y, policy);
        } else {
          uint8_t* sk = base + stage * C::kStage + lane * p.B * 128;
          uint8_t* sv = sk + C::kRegion;
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf) {
            tma_load_2d(sk + hf * kHalfBytes, kmap, &bar.full[stage], hf * 64, y, policy);
            tma_load_2d(sv + hf * kHalfBytes, vmap, &bar.full[stage], hf * 64, y, policy);
          }
        }
      }
      if (ch == 0 && lane == 0 && nxt_idx < total) nxt_pr = __ldcg(p.plan + nxt_idx / p.Hkv);
    }
    if (!ok) break;
    if (nch == 0 && lane == 0 && nxt_idx < total) nxt_pr = __ldcg(p.plan + nxt_idx / p.Hkv);
    cur_idx = nxt_idx;
    cur_pr = nxt_pr;
  }
  if (!ok) {
    give_up(p, abort);
    // Let copies already issued land before the CTA's shared memory goes away.
    const volatile int never = 0;
    for (uint32_t k = (kseq > (uint32_t)C::kStages ? kseq - C::kStages : 0); k < kseq; ++k)
      mbar_wait(&bar.full[k % C::kStages], (k / C::kStages) & 1, &never, p.wait_limit_ns);
    for (uint32_t k = (nq > 2 ? nq - 2 : 0); k < nq; ++k) mbar_wait(&bar.qfull[k & 1], (k >> 1) & 1, &never, p.wait_limit_ns);
  }
}

template <int D, bool kInter, bool kShared>
__device__ void consumer(const DecodeArgs& p, uint8_t* base, volatile int* abort) {
  using C = TcCfg<D>;
  constexpr int KS = D / 16;  // k-steps of the Q·Kᵀ product
  constexpr int MT = D / 16;  // m-tiles of the Oᵀ = Vᵀ Pᵀ product
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2;  // mma group id: head row of S, token row of K tiles
  const int tq = lane & 3;   // thread in group
  const Bars bar = bars_at<D>(base);
  const int4* desc = reinterpret_cast<const int4*>(base + C::kOffDesc);
  float* sO = reinterpret_cast<float*>(base + C::kOffO);
  float2* sML = reinterpret_cast<float2*>(base + C::kOffML);
  const uint32_t base_addr = smem_addr(base);
  uint32_t kseq = 0;

  for (uint32_t n = 0;; ++n) {
    const int slot = n & 1;
    if (!mbar_wait(&bar.qfull[slot], (n >> 1) & 1, abort, p.wait_limit_ns)) {
      give_up(p, abort);
      return;
    }
    const int4 d = desc[slot];
    if (d.w < 0) return;  // no work left
    const int s0 = d.x, kvh = d.z, ctx = d.w;
    const int part = kShared ? d.y & 0xffff : d.y, nm = kShared ? (d.y >> 16) & 15 : 1;
    const bool shared = kShared && ((d.y >> 20) & 1);
    const int t0 = part * p.P, t1 = min(ctx, t0 + p.P);
    const int nch = (t1 - t0 + kChunk - 1) / kChunk;
    const int np = shared ? 2 : (ctx + p.P - 1) / p.P;  // a shared item always leaves a partial
    const int nrow = nm * p.g;                           // rows of S: (sequence, query head) pairs
    // Tokens row gq attends: its own sequence's length on a shared item.
    const int lim = !shared ? ctx : gq < nrow ? min(max(__ldg(p.context_lens + s0 + gq / p.g), 0), p.max_ctx) : 0;
    uint32_t qa[KS][2];
    {
      const __nv_bfloat16* sq = reinterpret_cast<const __nv_bfloat16*>(base + C::kOffQ + slot * C::kQSlot);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa[ks][0] = gq < nrow ? *reinterpret_cast<const uint32_t*>(sq + gq * D + ks * 16 + 2 * tq) : 0u;
        qa[ks][1] = gq < nrow ? *reinterpret_cast<const uint32_t*>(sq + gq * D + ks * 16 + 8 + 2 * tq) : 0u;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar.qempty[slot]);

    float m_run = -INFINITY, l_run = 0.f;
    float o[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    for (int ch = 0; ch < nch; ++ch, ++kseq) {
      if ((int)(kseq & (kConsumerWarps - 1)) != warp) continue;
      const int stage = kseq % C::kStages;
      if (!mbar_wait(&bar.full[stage], (kseq / C::kStages) & 1, abort, p.wait_limit_ns)) {
        give_up(p, abort);
        return;
      }
      const int nv = min(kChunk, t1 - (t0 + ch * kChunk));
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
          *reinterpret_cast<uint4*>(vrow + stage_line<D, kInter>(r, rem >> 3) * 128 + (rem & 7) * 16) =
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
          const int line = stage_line<D, kInter>(t, cidx >> 3);
          const uint32_t addr = sk + line * 128 + (((cidx & 7) ^ (line & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(addr, b0, b1, b2, b3);
          mma_bf16_16816(sc[nt], qa[2 * kk][0], 0u, qa[2 * kk][1], 0u, b0, b1);
          mma_bf16_16816(sc[nt], qa[2 * kk + 1][0], 0u, qa[2 * kk + 1][1], 0u, b2, b3);
        }
      }
      // Online softmax (log2 domain) for head row gq over this chunk.
      // tokens of the chunk row gq may attend
      const int left = kShared ? min(nv, lim - (t0 + ch * kChunk)) : nv;
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = nt * 8 + 2 * tq + e;
          const float v = tok < left ? sc[nt][e] * p.scale_log2 : -INFINITY;
          sc[nt][e] = v;
          mx = fmaxf(mx, v);
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      // A row with no token yet (shared items only) keeps weight 0.
      const float m_use = (kShared && m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f(m_run - m_use);
      float ls = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sc[nt][0] = exp2f(sc[nt][0] - m_use);
        sc[nt][1] = exp2f(sc[nt][1] - m_use);
        ls += sc[nt][0] + sc[nt][1];
      }
      l_run = l_run * alpha + ls;
      m_run = m_new;
      const float a_lo = __shfl_sync(kFull, alpha, 8 * tq);
      const float a_hi = __shfl_sync(kFull, alpha, 8 * tq + 4);
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
          const int line = stage_line<D, kInter>(t, cidx >> 3);
          const uint32_t addr = sv + line * 128 + (((cidx & 7) ^ (line & 7)) << 4);
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4_trans(addr, a0, a1, a2, a3);
          mma_bf16_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.empty[stage]);
    }

    // ---- item epilogue: merge the four warps' states ----
    // The previous item's combine must be over before its buffers are reused.
    if (n > 0 && !mbar_wait(bar.epi_done, (n - 1) & 1, abort, p.wait_limit_ns)) {
      give_up(p, abort);
      return;
    }
    float l = l_run;
    l += __shfl_xor_sync(kFull, l, 1);
    l += __shfl_xor_sync(kFull, l, 2);
    if (tq == 0 && gq < nrow) sML[warp * kMaxGroup + gq] = make_float2(m_run, l);
    float* ob = sO + warp * kMaxGroup * C::kOStride;
    const int h0 = 2 * tq, h1 = 2 * tq + 1;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int dd = 16 * mt + gq;
      if (h0 < nrow) {
        ob[h0 * C::kOStride + dd] = o[mt][0];
        ob[h0 * C::kOStride + dd + 8] = o[mt][2];
      }
      if (h1 < nrow) {
        ob[h1 * C::kOStride + dd] = o[mt][1];
        ob[h1 * C::kOStride + dd + 8] = o[mt][3];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar.epi_full);
    if (!mbar_wait(bar.epi_full, n & 1, abort, p.wait_limit_ns)) {
      give_up(p, abort);
      return;
    }
    const int units = nrow * (D / 8);
    for (int u = threadIdx.x; u < units; u += kConsumerWarps * 32) {
      const int h = u / (D / 8);
      const int d0 = (u % (D / 8)) * 8;
      float mw[kConsumerWarps];
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        mw[w] = sML[w * kMaxGroup + h].x;
        M = fmaxf(M, mw[w]);
      }
      if (kShared && M == -INFINITY) M = 0.f;  // a shared-item row without tokens here: all weights 0
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
      const int s = kShared ? s0 + h / p.g : s0;
      const int qh = kShared ? kvh * p.g + h % p.g : kvh * p.g + h;
      if (np <= 1) {  // one partition, or an empty context (zero row)
        uint4 pk = make_uint4(0, 0, 0, 0);
        if (np == 1) {
          const float inv = 1.f / L;
          pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
          pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
          pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
          pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
        }
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + ((size_t)s * p.H + qh) * D + d0;
        *reinterpret_cast<uint4*>(dst) = pk;
      } else {
        const size_t wi = ((size_t)s * p.max_parts + part) * p.H + qh;
        float4* dst = reinterpret_cast<float4*>(p.ws_o + wi * D + d0);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        if (d0 == 0) p.ws_ml[wi] = make_float2(M, L);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar.epi_done);
  }
}

template <int D, bool kInter, bool kShared>
__global__ void __launch_bounds__(kThreads, 2)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const DecodeArgs p) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile int* abort = reinterpret_cast<volatile int*>(base + C::kOffAbort);
  if (threadIdx.x == 0) {
    const Bars b = bars_at<D>(base);
    for (int k = 0; k < C::kStages; ++k) {
      mbar_init(&b.full[k], 1);   // producer arrival + TMA bytes
      mbar_init(&b.empty[k], 1);  // the consuming warp
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&b.qfull[k], 1);                // producer arrival + Q bytes
      mbar_init(&b.qempty[k], kConsumerWarps);  // every consumer warp has read Q
    }
    mbar_init(b.epi_full, kConsumerWarps);  // every warp's state is in shared memory
    mbar_init(b.epi_done, kConsumerWarps);  // every warp has finished the combine
    *abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  if ((threadIdx.x >> 5) == kConsumerWarps) {
    if ((threadIdx.x & 31) == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    producer<D, kInter, kShared>(&kmap, &vmap, p, base, abort);
  } else {
    consumer<D, kInter, kShared>(p, base, abort);
  }
}

}  // namespace

size_t decode_tc_smem_bytes(int D) { return D == 128 ? TcCfg<128>::kBytes : TcCfg<64>::kBytes; }

bool decode_tc_interleaved(int D, int B) { return D == 128 && B == 8; }

cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream) {
  const size_t smem = decode_tc_smem_bytes(a.D);
  const bool inter = decode_tc_interleaved(a.D, a.B);
  using Kern = void (*)(const CUtensorMap, const CUtensorMap, const DecodeArgs);
  // [shared items][D == 128 ? (inter ? 2 : 1) : 0]
  static const Kern kernels[2][3] = {
      {paged_decode_tc_kernel<64, false, false>, paged_decode_tc_kernel<128, false, false>,
       paged_decode_tc_kernel<128, true, false>},
      {paged_decode_tc_kernel<64, false, true>, paged_decode_tc_kernel<128, false, true>,
       paged_decode_tc_kernel<128, true, true>}};
  const Kern kern = kernels[a.shared_items ? 1 : 0][a.D == 128 ? (inter ? 2 : 1) : 0];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // Per-device launch shape, computed once (threads of one process share it).
  struct Shape {
    int sms = 0, per_sm128 = 0, per_sm64 = 0;
  };
  static Shape shapes[64];
  static std::once_flag once[64];
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t init_err = cudaSuccess;
  std::call_once(once[dev], [&] {
    Shape sh;
    init_err = cudaDeviceGetAttribute(&sh.sms, cudaDevAttrMultiProcessorCount, dev);
    for (int v = 0; v < 2 && init_err == cudaSuccess; ++v)
      for (int k = 0; k < 3 && init_err == cudaSuccess; ++k)
        init_err = cudaFuncSetAttribute(kernels[v][k], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)(k ? TcCfg<128>::kBytes : TcCfg<64>::kBytes));
    // The variants share one launch shape; take the smallest occupancy.
    sh.per_sm128 = sh.per_sm64 = 1 << 30;
    for (int v = 0; v < 2 && init_err == cudaSuccess; ++v)
      for (int k = 0; k < 3 && init_err == cudaSuccess; ++k) {
        int n = 0;
        init_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernels[v][k], kThreads,
                                                                 k ? TcCfg<128>::kBytes : TcCfg<64>::kBytes);
        int& per = k ? sh.per_sm128 : sh.per_sm64;
        per = std::min(per, n);
      }
    shapes[dev] = sh;
  });
  if (init_err != cudaSuccess) return init_err;
  const Shape& sh = shapes[dev];
  const int per_sm = a.D == 128 ? sh.per_sm128 : sh.per_sm64;
  if (per_sm < 1 || sh.sms < 1) return cudaErrorInvalidConfiguration;
  const long long total = (long long)a.max_parts * a.S * a.Hkv;  // upper bound of the work items
  const int grid = (int)std::min<long long>(total, (long long)sh.sms * per_sm);
  if (grid <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, a);
}

}  // namespace pa
