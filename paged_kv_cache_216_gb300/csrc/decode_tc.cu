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
//    and bulk-copies its g query rows into a 2-slot Q ring, then streams
//    the item's keys and values 32 tokens at a time into a ring of
//    shared-memory stages: one TMA box per cache block of the chunk for K
//    and one for V (the 4D block view of block_layout.cuh: 8-row groups
//    holding both 64-dim halves, 128-byte swizzle).  Block ids are read 32
//    at a time (one per lane) one window ahead.  This is the prefetch of the
//    same page's section 2.2, done by the copy engine.
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

#include "block_layout.cuh"
#include "device_common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pa {
namespace {

constexpr int kChunk = 32;  // tokens per pipeline stage
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kHalfBytes = kChunk * 128;  // one 64-dim half of a chunk's 32 rows
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
  // mbarriers: full[kStages], empty[kStages], qfull[2], qempty[2], epi_full, epi_done, and for
  // shared-prefix items q_ready, s_ready, p_ready, o_done, drained
  static constexpr int kBars = (2 * kStages + 6 + 5) * 8;
  // byte offsets from the 1024-aligned base
  static constexpr int kOffQ = kStages * kStage;
  static constexpr int kOffO = kOffQ + 2 * kQSlot;
  static constexpr int kOffML = kOffO + kOBuf;
  static constexpr int kOffDesc = kOffML + kML;  // int4 per Q slot: {s, part, kvh, ctx or -1}
  static constexpr int kOffBar = kOffDesc + 2 * 16;
  static constexpr int kOffAbort = kOffBar + kBars;  // abort flag, then the tensor-memory address
  static constexpr size_t kBytes = 1024 + kOffAbort + 16;
  // Tensor memory of a shared-prefix item (kGroupRows lanes): O (fp32, D
  // columns), S of a chunk (fp32, kChunk columns; P as bf16 pairs over its
  // first half), the query rows (bf16 pairs, D / 2 columns).
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kColO = 0, kColS = 128, kColQ = 192;
  static_assert(D <= 128 && kColS + kChunk <= kColQ && kColQ + D / 2 <= kTmemCols, "tensor-memory columns");
};

struct Bars {
  uint64_t *full, *empty, *qfull, *qempty, *epi_full, *epi_done;
  // shared-prefix items: every warp's query rows are in tensor memory; S of
  // a chunk is in; every warp's P of a chunk is in; the item's last P·V is
  // done; every MMA issued is done
  uint64_t *q_ready, *s_ready, *p_ready, *o_done, *drained;
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
  b.q_ready = b.epi_done + 1;
  b.s_ready = b.q_ready + 1;
  b.p_ready = b.s_ready + 1;
  b.o_done = b.p_ready + 1;
  b.drained = b.o_done + 1;
  return b;
}

__device__ __forceinline__ void give_up(const DecodeArgs& p, volatile int* abort) {
  *abort = 1;
  raise_status(p.status, PA_STATUS_TIMEOUT);
}

template <int D, bool kShared>
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
    const int s0 = shared ? (ctx >> 8) & 0xffff : ts;
    const int nm = shared ? ctx & 0xff : 1;
    const int t0 = part * p.P, t1 = shared ? t0 + p.P : min(ctx, t0 + p.P);
    if (lane == 0) {
      if (shared) {
        // A shared item's descriptor carries its member count and a flag; the
        // consumers load its query rows into tensor memory themselves.
        desc[slot] = make_int4(s0, part | (nm << 16) | (1 << 24), kvh, t1);
        mbar_arrive(&bar.qfull[slot]);
      } else {
        desc[slot] = make_int4(s0, part, kvh, ctx);
        mbar_arrive_expect_tx(&bar.qfull[slot], qbytes);
        const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(p.q) + ((size_t)s0 * p.H + (size_t)kvh * p.g) * D;
        bulk_load(base + C::kOffQ + slot * C::kQSlot, src, qbytes, &bar.qfull[slot]);
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
        // one box per block: both halves of its B rows, 8-row groups
        uint8_t* sk = base + stage * C::kStage + lane * p.B * D * 2;
        const int grp = (id * p.Hkv + kvh) * (p.B >> 3);
        tma_load_4d(sk, kmap, &bar.full[stage], 0, 0, 0, grp, policy);
        tma_load_4d(sk + C::kRegion, vmap, &bar.full[stage], 0, 0, 0, grp, policy);
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

// A shared-prefix item: one partition of a group's shared prefix, one KV
// head, the query rows of up to kGroupRows / g members (row r = member
// r / g, head r % g) -- a dense tile, so it runs on the 5th-generation tensor
// cores with its accumulators in tensor memory, and every block of the
// partition is read once for the whole tile.  All four consumer warps take
// part: thread r owns row r (tensor-memory lane r) and thread 0 issues the
// MMAs.  Per 32-token chunk of the ring: S = Q Kᵀ (M 128, N 32, K = D: A the
// query rows in tensor memory, B the keys in the stage), the online softmax
// of each row masked to its own sequence's length (a member may end inside
// the shared part), P as bf16 over S, then O += P V (A = P in tensor memory,
// B the values, an MN-major operand) and a commit that frees the stage.  O
// is rescaled only when a row's max grows by more than 2^8 (the stale max
// serves O and the sum alike).  The result of each row is its member's
// split-K partial for this partition; the log-sum-exp merge combines it with
// the member's other partitions.  Returns false after a time-out.
template <int D>
__device__ bool group_item(const DecodeArgs& p, uint8_t* base, const Bars& bar, uint32_t tmem, int s0, int nm,
                           int part, int kvh, int t1, uint32_t& kseq, uint32_t& gi, uint32_t& gch,
                           volatile int* abort) {
  using C = TcCfg<D>;
  constexpr float kRescaleLog2 = 8.f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, r = threadIdx.x;
  const bool issuer = threadIdx.x == 0;
  const int rows = nm * p.g;
  const int t0 = part * p.P;
  const int nch = (t1 - t0) / kChunk;  // a shared partition is whole, P a multiple of kChunk
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  int s = 0, qh = 0, lim = 0;  // the row's sequence, query head, and tokens it attends
  if (r < rows) {
    s = s0 + r / p.g;
    qh = kvh * p.g + r % p.g;
    lim = min(max(__ldg(p.context_lens + s), 0), p.max_ctx);
  }
  // The row's query into tensor memory (bf16 pairs; rows past the members: zeros).
  {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + ((size_t)s * p.H + qh) * D);
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 x = r < rows ? __ldg(src + 4 * i + j) : make_uint4(0, 0, 0, 0);
        w[4 * j] = x.x;
        w[4 * j + 1] = x.y;
        w[4 * j + 2] = x.z;
        w[4 * j + 3] = x.w;
      }
      tmem_st16(lane_base + C::kColQ + 16 * i, w);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar.q_ready);
  }
  const uint32_t id_s = instr_desc(kGroupRows, kChunk, false);
  const uint32_t id_o = instr_desc(kGroupRows, D, true);
  const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;
  for (int ch = 0; ch < nch; ++ch, ++kseq, ++gch) {
    const int stage = kseq % C::kStages;
    const uint32_t sk = smem_addr(base + stage * C::kStage);
    if (issuer) {
      // the keys of the chunk (and, first, every warp's query rows) are in
      bool okm = mbar_spin(&bar.full[stage], (kseq / C::kStages) & 1, abort, p.wait_limit_ns);
      if (okm && ch == 0) okm = mbar_spin(bar.q_ready, gi & 1, abort, p.wait_limit_ns);
      if (okm) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ts(tmem + C::kColS, tmem + C::kColQ + kk * 8,
                 smem_desc(sk, 16, C::kHalves * 1024) + (uint64_t)(((kk >> 2) * 1024 + (kk & 3) * 32) >> 4), id_s,
                 kk > 0);
        mma_commit(bar.s_ready);
      } else {
        give_up(p, abort);
      }
    }
    if (!__all_sync(kFull, mbar_wait(bar.s_ready, gch & 1, abort, p.wait_limit_ns))) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t raw[kChunk];
    tmem_ld16_nowait(lane_base + C::kColS, raw);
    tmem_ld16_nowait(lane_base + C::kColS + 16, raw + 16);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    // tokens of the chunk this row attends (none for a row past the members)
    const int nvalid = min(kChunk, lim - (t0 + ch * kChunk));
    float sc[kChunk];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) sc[j] = j < nvalid ? __uint_as_float(raw[j]) : -INFINITY;
    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < kChunk / 2; ++j) m4[j & 3] = fmax3(m4[j & 3], sc[2 * j], sc[2 * j + 1]);
    const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
    const bool grow = mx > m_run + kRescaleLog2 || (m_run == -INFINITY && mx != -INFINITY);
    const float m_new = grow ? mx : m_run;
    const float alpha = grow ? exp2f(m_run - m_new) : 1.f;  // m_run = -inf: alpha 0
    if (ch > 0 && __any_sync(kFull, grow && m_run != -INFINITY)) {
      // O holds P·V of the chunks before: the commit that released S covers them
#pragma unroll 1
      for (int i = 0; i < D / 16; ++i) {
        float v[16];
        tmem_ld16(lane_base + C::kColO + 16 * i, v);
        uint32_t w[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) w[q] = __float_as_uint(v[q] * alpha);
        tmem_st16(lane_base + C::kColO + 16 * i, w);
      }
    }
    l_run *= alpha;
    m_run = m_new;
    const float base_m = m_run == -INFINITY ? 0.f : m_run;
    const float2 nb2 = make_float2(-base_m, -base_m);
    float2 l2 = make_float2(0.f, 0.f);
    uint32_t w[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float2 x = __ffma2_rn(make_float2(sc[2 * q], sc[2 * q + 1]), sl2, nb2);
      const float2 e = make_float2(ex2_ftz(x.x), ex2_ftz(x.y));
      l2 = __fadd2_rn(l2, e);
      w[q] = pack_bf16x2(e.x, e.y);
    }
    l_run += l2.x + l2.y;
    tmem_st16(lane_base + C::kColS, w);  // P over the first 16 columns of S
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar.p_ready);
    if (issuer) {
      if (mbar_spin(bar.p_ready, gch & 1, abort, p.wait_limit_ns)) {
        tc_fence_after();
        const uint32_t sv = sk + C::kRegion;
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk)
          mma_ts(tmem + C::kColO, tmem + C::kColS + kk * 8,
                 smem_desc(sv, 1024, C::kHalves * 1024) + (uint64_t)((kk * 2 * C::kHalves * 1024) >> 4), id_o,
                 ch > 0 || kk > 0);
        mma_commit(&bar.empty[stage]);  // the stage is free once this chunk's products are done
        if (ch + 1 == nch) mma_commit(bar.o_done);
      } else {
        give_up(p, abort);
      }
    }
  }
  // the row's partial: un-normalised O, running max and sum
  if (ok) ok = __all_sync(kFull, mbar_wait(bar.o_done, gi & 1, abort, p.wait_limit_ns));
  if (ok) {
    tc_fence_after();
    uint32_t o[D];
#pragma unroll
    for (int i = 0; i < D / 16; ++i) tmem_ld16_nowait(lane_base + C::kColO + 16 * i, o + 16 * i);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    tc_fence_before();
    // a row whose sequence ends before this partition has no partial here
    // (the merge does not read it)
    if (r < rows && lim > t0) {
      const size_t wi = ((size_t)s * p.max_parts + part) * p.H + qh;
      float4* dst = reinterpret_cast<float4*>(p.ws_o + wi * D);
#pragma unroll
      for (int u = 0; u < D / 4; ++u)
        dst[u] = make_float4(__uint_as_float(o[4 * u]), __uint_as_float(o[4 * u + 1]), __uint_as_float(o[4 * u + 2]),
                             __uint_as_float(o[4 * u + 3]));
      p.ws_ml[wi] = make_float2(m_run, l_run);
    }
  }
  ++gi;
  return ok;
}

template <int D, bool kShared>
__device__ void consumer(const DecodeArgs& p, uint8_t* base, volatile int* abort, uint32_t tmem) {
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
  uint32_t gi = 0, gch = 0;  // shared-prefix items and their chunks so far

  for (uint32_t n = 0;; ++n) {
    const int slot = n & 1;
    if (!mbar_wait(&bar.qfull[slot], (n >> 1) & 1, abort, p.wait_limit_ns)) {
      give_up(p, abort);
      return;
    }
    const int4 d = desc[slot];
    if (d.w < 0) return;  // no work left
    if (kShared && ((d.y >> 24) & 1)) {
      // a shared-prefix item: every warp works on it (the query slot is not used)
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.qempty[slot]);
      if (!group_item<D>(p, base, bar, tmem, d.x, (d.y >> 16) & 0xff, d.y & 0xffff, d.z, d.w, kseq, gi, gch, abort)) {
        give_up(p, abort);
        return;
      }
      // the item epilogue's handshake, which keeps its phases one per item
      if (n > 0 && !mbar_wait(bar.epi_done, (n - 1) & 1, abort, p.wait_limit_ns)) {
        give_up(p, abort);
        return;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.epi_full);
      if (!mbar_wait(bar.epi_full, n & 1, abort, p.wait_limit_ns)) {
        give_up(p, abort);
        return;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.epi_done);
      continue;
    }
    const int s0 = d.x, kvh = d.z, ctx = d.w;
    const int part = d.y;
    const int t0 = part * p.P, t1 = min(ctx, t0 + p.P);
    const int nch = (t1 - t0 + kChunk - 1) / kChunk;
    const int np = (ctx + p.P - 1) / p.P;
    const int nrow = p.g;  // rows of S: the query heads of the KV head
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
          *reinterpret_cast<uint4*>(vrow + kv_row_offset<C::kHalves>(r, rem >> 3) + (rem & 7) * 16) =
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
          const uint32_t addr = sk + kv_row_offset<C::kHalves>(t, cidx >> 3) + (((cidx & 7) ^ (t & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(addr, b0, b1, b2, b3);
          mma_bf16_16816(sc[nt], qa[2 * kk][0], 0u, qa[2 * kk][1], 0u, b0, b1);
          mma_bf16_16816(sc[nt], qa[2 * kk + 1][0], 0u, qa[2 * kk + 1][1], 0u, b2, b3);
        }
      }
      // Online softmax (log2 domain) for head row gq over this chunk.
      // tokens of the chunk row gq may attend
      const int left = nv;
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
      const float m_use = m_new;
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
          const uint32_t addr = sv + kv_row_offset<C::kHalves>(t, cidx >> 3) + (((cidx & 7) ^ (t & 7)) << 4);
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
      const int s = s0;
      const int qh = kvh * p.g + h;
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

template <int D, bool kShared>
__global__ void __launch_bounds__(kThreads, 2)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const DecodeArgs p) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile int* abort = reinterpret_cast<volatile int*>(base + C::kOffAbort);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(base + C::kOffAbort + 4);
  const Bars b = bars_at<D>(base);
  if (threadIdx.x == 0) {
    for (int k = 0; k < C::kStages; ++k) {
      mbar_init(&b.full[k], 1);   // producer arrival + TMA bytes
      mbar_init(&b.empty[k], 1);  // the consuming warp (or the commit of a shared item's products)
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&b.qfull[k], 1);                // producer arrival + Q bytes
      mbar_init(&b.qempty[k], kConsumerWarps);  // every consumer warp has read Q
    }
    mbar_init(b.epi_full, kConsumerWarps);  // every warp's state is in shared memory
    mbar_init(b.epi_done, kConsumerWarps);  // every warp has finished the combine
    mbar_init(b.q_ready, kConsumerWarps);
    mbar_init(b.s_ready, 1);
    mbar_init(b.p_ready, kConsumerWarps);
    mbar_init(b.o_done, 1);
    mbar_init(b.drained, 1);
    *abort = 0;
    fence_barrier_init();
  }
  // Shared-prefix items keep their tiles in tensor memory: 256 columns per
  // CTA, two CTAs per SM.
  if (kShared && (threadIdx.x >> 5) == 0) tmem_alloc(tslot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = kShared ? *tslot : 0u;
  pdl_launch_dependents();
  if ((threadIdx.x >> 5) == kConsumerWarps) {
    if ((threadIdx.x & 31) == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    producer<D, kShared>(&kmap, &vmap, p, base, abort);
  } else {
    consumer<D, kShared>(p, base, abort, tmem);
  }
  if (kShared) {
    // Every MMA issued has completed before tensor memory is released.
    if (threadIdx.x == 0) {
      mma_commit(b.drained);
      const volatile int never = 0;
      mbar_wait(b.drained, 0, &never, p.wait_limit_ns);
    }
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
      tc_fence_after();
      tmem_free(tmem, C::kTmemCols);
    }
  }
}

}  // namespace

size_t decode_tc_smem_bytes(int D) { return D == 128 ? TcCfg<128>::kBytes : TcCfg<64>::kBytes; }

cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream) {
  const size_t smem = decode_tc_smem_bytes(a.D);
  using Kern = void (*)(const CUtensorMap, const CUtensorMap, const DecodeArgs);
  // [shared items][D == 128]
  static const Kern kernels[2][2] = {
      {paged_decode_tc_kernel<64, false>, paged_decode_tc_kernel<128, false>},
      {paged_decode_tc_kernel<64, true>, paged_decode_tc_kernel<128, true>}};
  const int v = a.shared_items ? 1 : 0, k = a.D == 128 ? 1 : 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // Per-device launch shape of each variant, computed once (threads of one
  // process share it).
  struct Shape {
    int sms = 0, per_sm[2][2] = {};
  };
  static Shape shapes[64];
  static std::once_flag once[64];
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t init_err = cudaSuccess;
  std::call_once(once[dev], [&] {
    Shape sh;
    init_err = cudaDeviceGetAttribute(&sh.sms, cudaDevAttrMultiProcessorCount, dev);
    for (int vi = 0; vi < 2 && init_err == cudaSuccess; ++vi)
      for (int ki = 0; ki < 2 && init_err == cudaSuccess; ++ki) {
        const size_t bytes = ki ? TcCfg<128>::kBytes : TcCfg<64>::kBytes;
        init_err = cudaFuncSetAttribute(kernels[vi][ki], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (init_err == cudaSuccess)
          init_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&sh.per_sm[vi][ki], kernels[vi][ki], kThreads,
                                                                   bytes);
      }
    shapes[dev] = sh;
  });
  if (init_err != cudaSuccess) return init_err;
  const Shape& sh = shapes[dev];
  const Kern kern = kernels[v][k];
  int per_sm = sh.per_sm[v][k];
  if (a.shared_items) {
    // The occupancy query counts a kernel that allocates tensor memory as
    // one CTA per SM.  This one holds 256 of the SM's 512 columns, so two
    // fit, as registers and shared memory allow (the same as the plain
    // variant's); a CTA that does not fit waits for one to finish.
    per_sm = std::min(sh.per_sm[0][k], (int)(512 / TcCfg<128>::kTmemCols));
  }
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
