// Prefill on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory), head_dim 64 or 128, bf16 storage, fp32 accumulation.
//
// Every new token of a sequence attends the sequence's tokens up to its own
// position ("PagedAttention Kernel：大模型推理优化的显存管理革新" section 3.1
// with a causal limit; the prompt's keys and values were appended into their
// blocks first, "Day 6/90 of Inference Engineering", PagedAttention notes,
// paragraph 2).
//
// One CTA per (sequence, KV head, pair of adjacent tiles of 128 query rows),
// the rows being (new token, query head) pairs, token-major; pairs with the
// most keys first.  Both tiles read every stage of keys and values, so each
// TMA box feeds 256 rows.  Roles (352 threads, one CTA per SM):
//  * warps 8 and 9 (producers): stream the keys (warp 8) and values (warp 9)
//    the pair attends, 128 tokens per stage, into rings of their own (3
//    stages of keys, 2 of values), as 2D TMA boxes of [B tokens x 64 dims]
//    with 128-byte swizzle (the K-major UMMA layout), after
//    griddepcontrol.wait; lane b issues block b of a chunk from block-table
//    entries fetched 32 at a time.  Warp 8 first loads both query tiles,
//    one 3D box per 64-dim half, so they land with the first keys;
//  * warp 10 (MMA): one thread issues, per tile, S = Q Kᵀ (M 128, N 128,
//    K = head_dim: head_dim / 16 tcgen05.mma kind::f16 from shared-memory
//    descriptors) into the tile's S and O += P V (M 128, N = head_dim,
//    K 128: eight MMAs, P read from tensor memory, V an MN-major operand in
//    shared memory), in a fixed order -- per chunk c and tile, P·V(c) and
//    then S(c + 1) -- spinning on one barrier at a time, so the tensor cores
//    work for one tile while the other tile's softmax runs (ping-pong);
//    tcgen05.commit signals the mbarriers and releases each stage after the
//    last MMA that reads it;
//  * warps 0-3 and 4-7 (softmax, one warpgroup per tile): thread t of a
//    warpgroup owns query row t of its tile (tensor-memory lane t): it
//    reads its 128 scores (tcgen05.ld), masks keys past its position, keeps
//    the running max and sum, writes P as bf16 back to tensor memory
//    (tcgen05.st) and rescales its row of O only when its max grows by more
//    than 2^8 (otherwise the stale max stays: exp2 values up to 256 are
//    exact enough and O and the sum use the same max); at the end it reads
//    its row of O, divides by the sum and stores it (a full tile through
//    its query buffer and one TMA box per 64-dim half, the sequence's last
//    tile row by row).
// Tensor memory (512 columns allocated): O of tile t at columns DH·t ..
// DH·t + DH - 1 and its S at 2·DH + 128t (DH = head_dim); P is written over
// the first half of its S.  Value rows past the pair's keys are zeroed in
// shared memory before the first P·V of that stage so stale cache rows
// cannot turn 0 x NaN into NaN.  Every wait is bounded; on a time-out the
// kernel raises PA_STATUS_TIMEOUT and stops issuing work.

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "device_common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kM = 128;                 // query rows per tile (one tensor-memory lane each)
constexpr int kTiles = 2;               // query tiles per CTA, sharing every stage
constexpr int kN = 128;                 // keys per stage (the N of S = Q Kᵀ)
constexpr int kStagesK = 3;             // stages in the key ring
constexpr int kStagesV = 2;             // stages in the value ring
constexpr int kSoftWarps = 4;           // per tile
constexpr int kProducerWarp = kTiles * kSoftWarps;  // keys; the next warp streams values
constexpr int kMmaWarp = kProducerWarp + 2;
constexpr int kThreadsT = (kTiles * kSoftWarps + 3) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kQHalf = kM * 128;         // bytes of one 64-dim half of a query tile
constexpr int kKVHalf = kN * 128;        // bytes of one 64-dim half of a stage of K (or V)
// full_k[], empty_k[], full_v[], empty_v[]; per tile s_full, p_full,
// o_final, q_full
constexpr int kTileBars = 4;

// Layout for head_dim DH (64 or 128): tiles and stages hold DH / 64 halves
// of 64 dims; O of tile t at columns DH·t .. DH·t + DH - 1, S of tile t at
// 2·DH + 128t (128 columns), P (bf16 pairs) over the first 64 columns of S.
template <int DH>
struct PfCfg {
  static constexpr int kHalves = DH / 64;
  static constexpr int kQTile = kHalves * kQHalf;
  static constexpr int kKVStage = kHalves * kKVHalf;
  static constexpr int kOffK = kTiles * kQTile;
  static constexpr int kOffV = kOffK + kStagesK * kKVStage;
  static constexpr int kOffBars = kOffV + kStagesV * kKVStage;
  static constexpr int kOffMisc = kOffBars + (2 * (kStagesK + kStagesV) + kTiles * kTileBars) * 8;  // tensor-memory address, abort flag
  static constexpr size_t kBytes = 1024 + kOffMisc + 16;
  static constexpr uint32_t kColO = 0, kColS = 2 * DH;
  static_assert(DH == 64 || DH == 128, "head_dim 64 or 128");
  static_assert(kBytes <= 227 * 1024, "shared memory of one CTA");
  static_assert(kColS + kTiles * 128 <= kTmemCols, "tensor-memory columns");
};
constexpr float kRescaleLog2 = 8.f;      // rescale O only when a row's max grows by more than 2^8

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version of this architecture
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B.
__device__ __forceinline__ uint32_t instr_desc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)acc));
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"((uint32_t)acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t addr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Same without waiting: several loads in flight, then one tcgen05.wait::ld.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t addr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
}

__device__ __forceinline__ void tmem_st16(uint32_t addr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          addr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for a phase by spinning on test_wait (bounded like mbar_wait): a
// thread suspended in try_wait resumed several hundred cycles after the
// phase completed, which the MMA thread cannot afford on its critical path.
__device__ __forceinline__ bool mbar_spin(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (unsigned i = 0; i < kWaitLimitIters; ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 255u) == 255u && (*abort || global_timer_ns() - t0 > kWaitLimitNs)) return false;
  }
  return false;
}

template <int DH>
__global__ void __launch_bounds__(kThreadsT, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                      const PrefillArgs p) {
  using C = PfCfg<DH>;
  constexpr int kQTile = C::kQTile, kKVStage = C::kKVStage, kOffK = C::kOffK, kOffV = C::kOffV;
  constexpr uint32_t kColO = C::kColO, kColS = C::kColS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The pair index is the slowest grid dimension and runs backwards, so the
  // pairs with the most keys start first across all sequences and heads.
  const int kvh = blockIdx.x, s = blockIdx.y;
  const int pair = (int)gridDim.z - 1 - (int)blockIdx.z;

  const int q0 = __ldg(p.query_start + s), q1 = __ldg(p.query_start + s + 1);
  const int ctx = __ldg(p.context_lens + s);
  const int n_new = q1 - q0;
  const int rows = n_new * p.g;
  if (q0 < 0 || n_new < 0 || n_new > p.max_query_len || ctx < n_new || ctx > p.max_ctx || q1 > p.T) {
    if (pair == 0 && kvh == 0 && tid == 0) raise_status(p.status, PA_STATUS_BAD_CONTEXT);
    return;
  }
  const int first_pos = ctx - n_new;
  // Keys each tile attends (0 for a tile past the sequence's rows) and the
  // 64-key chunks that hold them; tile 1 is the later one, so it attends
  // at least as many keys as tile 0.
  const int row00 = pair * kTiles * kM, row01 = row00 + kM;
  if (row00 >= rows) return;
  const int t_end0 = first_pos + (min(rows, row00 + kM) - 1) / p.g + 1;
  const int t_end1 = row01 < rows ? first_pos + (min(rows, row01 + kM) - 1) / p.g + 1 : 0;
  const int nch0 = (t_end0 + kN - 1) / kN, nch1 = (t_end1 + kN - 1) / kN;
  const int t_end = max(t_end0, t_end1);
  const int nch = max(nch0, nch1);

  uint64_t* full_k = reinterpret_cast<uint64_t*>(base + C::kOffBars);
  uint64_t* empty_k = full_k + kStagesK;
  uint64_t* full_v = empty_k + kStagesK;
  uint64_t* empty_v = full_v + kStagesV;
  uint64_t* tile_bars = empty_v + kStagesV;  // kTileBars per tile
  // per tile: [0] S of a chunk is in, [1] P of a chunk is in, [2] the last
  // P·V is done, [3] the query tile is in
  auto s_full = [&](int t) { return tile_bars + t * kTileBars; };
  auto p_full = [&](int t) { return tile_bars + t * kTileBars + 1; };
  auto o_final = [&](int t) { return tile_bars + t * kTileBars + 2; };
  auto q_full = [&](int t) { return tile_bars + t * kTileBars + 3; };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(base + C::kOffMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(base + C::kOffMisc + 4);
  const uint32_t sbase = smem_addr(base);

  if (tid == 0) {
    for (int k = 0; k < kStagesK; ++k) {
      mbar_init(&full_k[k], 1);
      mbar_init(&empty_k[k], 1);
    }
    for (int k = 0; k < kStagesV; ++k) {
      mbar_init(&full_v[k], 1);
      mbar_init(&empty_v[k], 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), kSoftWarps * 32);
      mbar_init(o_final(t), 1);
      mbar_init(q_full(t), 1);
    }
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tslot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == kProducerWarp || warp == kProducerWarp + 1) {
    // One warp streams the keys, the next the values, each into its own
    // ring, so neither waits behind the other's release.  Lane b loads
    // block b of a chunk; block-table entries are fetched 32 at a time, one
    // per lane, a window ahead, so no TMA issue waits on a dependent load.
    const int kv = warp - kProducerWarp;  // 0 keys, 1 values
    if (kv == 0 && lane == 0) {
      // The query tiles (an input the append does not write), one box per
      // 64-dim half: 128 / g tokens x g heads of this KV head.  Rows past the
      // sequence read the next sequence's queries (or zeros past the last
      // token); their scores are all masked and their rows never stored.
      const uint64_t qpol = policy_evict_first();
#pragma unroll 1
      for (int t = 0; t < kTiles; ++t) {
        if ((t == 0 ? nch0 : nch1) == 0) continue;
        const int z = q0 + (row00 + t * kM) / p.g;
        mbar_arrive_expect_tx(q_full(t), (uint32_t)kQTile);
#pragma unroll
        for (int h = 0; h < C::kHalves; ++h)
          tma_load_3d(base + t * kQTile + h * kQHalf, &qmap, q_full(t), 64 * h, kvh * p.g, z, qpol);
      }
    }
    pdl_wait_primary();  // the prompt's keys and values are in the cache from here on
    const int32_t* row = p.block_tables + (size_t)s * p.max_blocks_per_seq;
    const int nblk = (t_end + p.B - 1) / p.B;
    const int bpc = kN / p.B;  // blocks per chunk (block sizes 8, 16, 32: 16, 8 or 4, dividing 32)
    const uint64_t policy = policy_evict_first();
    const CUtensorMap* map = kv == 0 ? &kmap : &vmap;
    uint64_t* fulls = kv == 0 ? full_k : full_v;
    uint64_t* empties = kv == 0 ? empty_k : empty_v;
    const int stages = kv == 0 ? kStagesK : kStagesV;
    int cur = load_block_id(row, lane, nblk);
    int nxt = load_block_id(row, 32 + lane, nblk);
    int wbase = 0;
    for (int c = 0; c < nch; ++c) {
      const int jb = c * bpc;
      if (jb >= wbase + 32) {
        cur = nxt;
        wbase += 32;
        nxt = load_block_id(row, wbase + 32 + lane, nblk);
      }
      int id = __shfl_sync(0xffffffffu, cur, (jb - wbase + lane) & 31);
      const int nb = (min(kN, t_end - c * kN) + p.B - 1) / p.B;
      if (lane < nb && (unsigned)id >= (unsigned)p.num_blocks) {
        raise_status(p.status, PA_STATUS_BAD_BLOCK);
        id = 0;
      }
      const int st = c % stages;
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(&empties[st], ((c / stages) & 1) ^ 1, abort);
        if (ok) {
          mbar_arrive_expect_tx(&fulls[st], (uint32_t)(nb * p.B * 128 * C::kHalves));
        } else {
          *abort = 1;
          raise_status(p.status, PA_STATUS_TIMEOUT);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      __syncwarp();  // the expected byte count is set before any copy can land
      if (lane < nb) {
        const int y = (id * p.Hkv + kvh) * p.B;
        uint8_t* d = base + (kv == 0 ? kOffK : kOffV) + st * kKVStage + lane * p.B * 128;
#pragma unroll
        for (int h = 0; h < C::kHalves; ++h) tma_load_2d(d + h * kKVHalf, map, &fulls[st], 64 * h, y, policy);
      }
    }
  } else if (warp == kMmaWarp) {
    // One thread issues every MMA in a fixed order, waiting (bounded
    // try_wait) for one barrier at a time: S of both tiles for chunk 0,
    // then per chunk c and tile t: P·V(c) as soon as the tile's P(c) is in,
    // and right behind it S(c + 1) of that tile.  Each tile has one S
    // buffer, so its softmax and its products alternate, and the tensor
    // cores work for one tile while the other tile's softmax runs.  The
    // tensor cores run one thread's MMAs in order: S(c + 1) overwrites P(c)
    // only after P·V(c) has read it, and the commit that releases S(c + 1)
    // to the softmax also covers P·V(c), so the softmax may rescale O at
    // once.  A stage is released by a commit after the last MMA that reads
    // it.
    const uint32_t id_s = instr_desc(kM, kN, false);
    const uint32_t id_o = instr_desc(kM, DH, true);
    bool ok = true;
    auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
      int r = 1;
      if (lane == 0) r = mbar_spin(bar, parity, abort);
      ok = ok && __shfl_sync(0xffffffffu, r, 0);
      return ok;
    };
    // Descriptors are built once per group; a k-step adds its byte offset
    // / 16 to the address field (every shared address is below 256 KB, so
    // the 14-bit field never carries).  This thread shares its scheduler
    // with two softmax warps, so fewer instructions per MMA matter.
    auto issue_s = [&](int t, int c) {  // lane 0; the keys of chunk c have landed
      tc_fence_after();
      const uint64_t a0 = smem_desc(sbase + t * kQTile, 16, 1024);
      const uint64_t b0 = smem_desc(sbase + kOffK + (c % kStagesK) * kKVStage, 16, 1024);
      const uint32_t d = tmem + kColS + (uint32_t)t * 128;
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        const int hlf = kk >> 2, w = kk & 3;
        mma_ss(d, a0 + (uint64_t)((hlf * kQHalf + w * 32) >> 4), b0 + (uint64_t)((hlf * kKVHalf + w * 32) >> 4), id_s,
               kk > 0);
      }
      mma_commit(s_full(t));
    };
    auto issue_pv = [&](int t, int c) {  // lane 0; P(c) and the values of chunk c are in
      tc_fence_after();
      const uint64_t b0 = smem_desc(sbase + kOffV + (c % kStagesV) * kKVStage, kKVHalf, 1024);
      const uint32_t p_cols = tmem + kColS + (uint32_t)t * 128;
      const uint32_t d = tmem + kColO + (uint32_t)t * DH;
#pragma unroll
      for (int kk = 0; kk < kN / 16; ++kk) mma_ts(d, p_cols + kk * 8, b0 + (uint64_t)((kk * 16 * 128) >> 4), id_o, c > 0 || kk > 0);
      if (c + 1 == (t == 0 ? nch0 : nch1)) mma_commit(o_final(t));
    };
    if (wait_bar(q_full(0), 0) && (nch1 == 0 || wait_bar(q_full(1), 0)) && wait_bar(&full_k[0], 0)) {
      if (lane == 0) {
        issue_s(0, 0);
        if (nch1 > 0) issue_s(1, 0);
        mma_commit(&empty_k[0]);
      }
      __syncwarp();
    }
    for (int c = 0; c < nch && ok; ++c) {
      if (!wait_bar(&full_v[c % kStagesV], (c / kStagesV) & 1)) break;
      const int nv = min(kN, t_end - c * kN);
      if (nv < kN) {  // value rows past the pair's keys: zeros (their keys are masked)
        uint8_t* vs = base + kOffV + (c % kStagesV) * kKVStage;
        for (int u = lane; u < (kN - nv) * 8 * C::kHalves; u += 32) {
          const int hlf = u / ((kN - nv) * 8), rem = u % ((kN - nv) * 8);
          *reinterpret_cast<uint4*>(vs + hlf * kKVHalf + (nv + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      bool k_next = false;  // the keys of chunk c + 1 have landed
#pragma unroll 1
      for (int t = 0; t < kTiles; ++t) {
        const int nch_t = t == 0 ? nch0 : nch1;
        if (c >= nch_t) continue;
        if (!wait_bar(p_full(t), c & 1)) break;
        if (lane == 0) issue_pv(t, c);
        __syncwarp();
        if (c + 1 < nch_t) {
          if (!k_next && !(k_next = wait_bar(&full_k[(c + 1) % kStagesK], ((c + 1) / kStagesK) & 1))) break;
          if (lane == 0) {
            issue_s(t, c + 1);
            // the last tile that reads the keys of chunk c + 1
            if (t == kTiles - 1 || c + 1 >= nch1) mma_commit(&empty_k[(c + 1) % kStagesK]);
          }
          __syncwarp();
        }
      }
      if (ok && lane == 0) mma_commit(&empty_v[c % kStagesV]);
      __syncwarp();
    }
    if (!ok) {
      *abort = 1;
      raise_status(p.status, PA_STATUS_TIMEOUT);
    }
  } else if (warp < kProducerWarp) {
    // softmax warpgroup t: thread lt owns row lt of tile t (tensor-memory lane lt)
    const int t = warp / kSoftWarps, lt = tid - t * kM;
    const int row0 = row00 + t * kM;
    const int nch_t = t == 0 ? nch0 : nch1;
    if (nch_t > 0) {
      const int r = row0 + lt;
      const int pos = r < rows ? first_pos + r / p.g : -1;  // keys 0 .. pos
      const uint32_t lane_base = tmem + ((uint32_t)((warp % kSoftWarps) * 32) << 16);
      const uint32_t o_cols = lane_base + kColO + (uint32_t)t * DH;
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int c = 0; c < nch_t; ++c) {
        // the warp leaves together (warp-wide votes follow)
        if (!__all_sync(0xffffffffu, mbar_wait(s_full(t), c & 1, abort))) {
          ok = false;
          break;
        }
        const uint32_t s_cols = lane_base + kColS + (uint32_t)t * 128;
        tc_fence_after();
        uint32_t raw[kN];
#pragma unroll
        for (int i = 0; i < kN / 16; ++i) tmem_ld16_nowait(s_cols + 16 * i, raw + 16 * i);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        float sc[kN];
#pragma unroll
        for (int j = 0; j < kN; ++j) sc[j] = __uint_as_float(raw[j]);
        // Keys t0 .. t0 + nvalid - 1 of this chunk are at or before the row's
        // position; masking is needed only in chunks that cross it.
        const int t0 = c * kN;
        const int nvalid = min(kN, pos - t0 + 1);
        // max of the raw (unscaled) valid scores, four chains at a time
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (nvalid >= kN) {
#pragma unroll
          for (int j = 0; j < kN; ++j) m4[j & 3] = fmaxf(m4[j & 3], sc[j]);
        } else {
#pragma unroll
          for (int j = 0; j < kN; ++j) {
            sc[j] = j < nvalid ? sc[j] : -INFINITY;
            m4[j & 3] = fmaxf(m4[j & 3], sc[j]);
          }
        }
        const float mxr = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        const float mx = mxr * p.scale_log2;  // scale > 0: the max of the scaled scores
        // Raise the running max (and rescale O) only when it grows past the
        // threshold; the decision is made per warp because tensor-memory
        // loads and stores are warp-wide.
        const bool grow = mx > m_run + kRescaleLog2 || (m_run == -INFINITY && mx != -INFINITY);
        const float m_new = grow ? mx : m_run;
        const float alpha = grow ? exp2f(m_run - m_new) : 1.f;  // m_run = -inf: alpha 0
        if (c > 0 && __any_sync(0xffffffffu, grow && m_run != -INFINITY)) {
          // O holds P·V(c - 1): the commit that released S(c) covers it
#pragma unroll 1
          for (int i = 0; i < DH / 16; ++i) {
            float v[16];
            tmem_ld16(o_cols + 16 * i, v);
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = __float_as_uint(v[j] * alpha);
            tmem_st16(o_cols + 16 * i, w);
          }
        }
        l_run *= alpha;
        m_run = m_new;
        const float base_m = m_run == -INFINITY ? 0.f : m_run;
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kN / 32; ++i) {  // exp2(s * scale - max): one FMA per score
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float e0 = exp2f(fmaf(sc[32 * i + 2 * j], p.scale_log2, -base_m));
            const float e1 = exp2f(fmaf(sc[32 * i + 2 * j + 1], p.scale_log2, -base_m));
            l4[j & 3] += e0 + e1;
            w[j] = pack_bf16x2(e0, e1);
          }
          tmem_st16(s_cols + 16 * i, w);  // P over the first 64 columns of its S
        }
        l_run += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        mbar_arrive(p_full(t));
      }
      // One outcome for the whole warpgroup: the full-tile store below syncs it.
      if (named_barrier_and(1 + t, kSoftWarps * 32, ok && mbar_wait(o_final(t), 0, abort))) {
        tc_fence_after();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        uint32_t o[DH];  // the row of O, all loads in flight at once
#pragma unroll
        for (int i = 0; i < DH / 16; ++i) tmem_ld16_nowait(o_cols + 16 * i, o + 16 * i);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        auto piece = [&](int u) {  // dims 8u .. 8u + 7 of the row, normalized, as bf16
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o[8 * u]) * inv, __uint_as_float(o[8 * u + 1]) * inv);
          w.y = pack_bf16x2(__uint_as_float(o[8 * u + 2]) * inv, __uint_as_float(o[8 * u + 3]) * inv);
          w.z = pack_bf16x2(__uint_as_float(o[8 * u + 4]) * inv, __uint_as_float(o[8 * u + 5]) * inv);
          w.w = pack_bf16x2(__uint_as_float(o[8 * u + 6]) * inv, __uint_as_float(o[8 * u + 7]) * inv);
          return w;
        };
        if (row0 + kM <= rows) {
          // A full tile: stage the rows in this tile's query buffer (its last
          // S has completed) in the layout the query boxes arrived in, then
          // store them with two TMA boxes through the same geometry.
          uint8_t* qt = base + t * kQTile;
#pragma unroll
          for (int u = 0; u < DH / 8; ++u)
            *reinterpret_cast<uint4*>(qt + (u >> 3) * kQHalf + lt * 128 + (((u & 7) ^ (lt & 7)) << 4)) = piece(u);
          fence_proxy_async_smem();
          named_barrier_sync(1 + t, kSoftWarps * 32);
          if (lt == 0) {
            const int z = q0 + row0 / p.g;
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h) tma_store_3d(&omap, qt + h * kQHalf, 64 * h, kvh * p.g, z);
            bulk_store_drain();
          }
        } else if (r < rows) {  // the sequence's last tile: only its own rows
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                ((size_t)(q0 + r / p.g) * p.H + kvh * p.g + r % p.g) * DH);
#pragma unroll
          for (int u = 0; u < DH / 8; ++u) dst[u] = piece(u);
        }
      } else {
        *abort = 1;
        raise_status(p.status, PA_STATUS_TIMEOUT);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

template <int DH>
cudaError_t launch_prefill_tc_dh(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const CUtensorMap& qmap, const CUtensorMap& omap, int pairs, cudaStream_t stream) {
  constexpr size_t kBytes = PfCfg<DH>::kBytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::once_flag once[64];
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t init_err = cudaSuccess;
  std::call_once(once[dev], [&] {
    init_err = cudaFuncSetAttribute(prefill_tc_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBytes);
  });
  if (init_err != cudaSuccess) return init_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.Hkv, (unsigned)a.S, (unsigned)pairs);
  cfg.blockDim = dim3(kThreadsT);
  cfg.dynamicSmemBytes = kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<DH>, kmap, vmap, qmap, omap, a);
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                              const CUtensorMap& qmap, const CUtensorMap& omap, cudaStream_t stream) {
  const int tiles = (a.max_query_len * a.g + kM - 1) / kM;
  const int pairs = (tiles + kTiles - 1) / kTiles;
  if (tiles <= 0 || a.S <= 0) return cudaSuccess;
  if (pairs > 65535 || a.S > 65535 || a.Hkv > 65535) return cudaErrorInvalidConfiguration;
  if (a.D == 128) return launch_prefill_tc_dh<128>(a, kmap, vmap, qmap, omap, pairs, stream);
  if (a.D == 64) return launch_prefill_tc_dh<64>(a, kmap, vmap, qmap, omap, pairs, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
