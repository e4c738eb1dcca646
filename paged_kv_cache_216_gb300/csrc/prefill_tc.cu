// Prefill on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory), head_dim 128, bf16 storage, fp32 accumulation.
//
// Same result as prefill.cu: every new token of a sequence attends the
// sequence's tokens up to its own position ("PagedAttention Kernel：大模型
// 推理优化的显存管理革新" section 3.1 with a causal limit; the prompt's keys
// and values were appended into their blocks first, "Day 6/90 of Inference
// Engineering", PagedAttention notes, paragraph 2).
//
// One CTA per (sequence, KV head, tile of 128 query rows), the rows being
// (new token, query head) pairs, token-major; tiles longest first.  Roles:
//  * warp 4 (producer): after griddepcontrol.wait, streams the keys and
//    values a tile attends, 64 tokens per stage of a 2-stage ring, as 2D TMA
//    boxes of [B tokens x 64 dims] with 128-byte swizzle (the K-major UMMA
//    layout), lane b issuing block b of a chunk from block-table entries
//    fetched 32 at a time; keys and values have separate barriers and keys
//    run a chunk ahead, released as soon as S has read them;
//  * warp 5 (MMA): S = Q Kᵀ (M 128, N 64, K 128: eight tcgen05.mma
//    kind::f16 from shared-memory descriptors) into one of two S buffers in
//    tensor memory as soon as a stage's keys have landed, and O += P V
//    (M 128, N 128, K 64: P read from tensor memory, V an MN-major operand
//    in shared memory) as soon as the softmax warps have written P, polling
//    both conditions without blocking; S of the next chunk thus overlaps the
//    softmax of this one; tcgen05.commit signals the mbarriers;
//  * warps 0-3 (softmax): thread t owns query row t (tensor-memory lane t):
//    it reads its 64 scores (tcgen05.ld), masks keys past its position,
//    keeps the running max and sum, writes P as bf16 back to tensor memory
//    (tcgen05.st) and rescales its row of O only when its max grows by more
//    than 2^8 (otherwise the stale max stays: exp2 values up to 256 are
//    exact enough and O and the sum use the same max); at the end it reads
//    its row of O, divides by the sum and stores it.
// Tensor memory: O at columns 0-127 and two S buffers (128-191, 192-255)
// so that S of the next chunk is computed while the softmax works on this
// one; P is written over the first half of its own S buffer (256 columns
// allocated; two CTAs per SM).  Rows past the tile's valid keys are zeroed
// in shared memory before P·V so stale cache rows cannot turn 0 x NaN into
// NaN.  Every wait is bounded; on a time-out the kernel raises
// PA_STATUS_TIMEOUT and stops issuing work.

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "device_common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kM = 128;                 // query rows per CTA (one tensor-memory lane each)
constexpr int kN = 64;                  // keys per stage
constexpr int kDh = 128;                // head_dim
// Two stages of 64 keys (four of 32 in the same shared memory measured
// slower: the per-stage barrier round trips cost more than the deeper ring
// saves).
constexpr int kStagesT = 2;
constexpr int kSoftWarps = 4;
constexpr int kProducerWarp = kSoftWarps;
constexpr int kMmaWarp = kSoftWarps + 1;
constexpr int kThreadsT = (kSoftWarps + 2) * 32;
constexpr uint32_t kTmemCols = 256;
// O at columns 0-127; S of chunk c in buffer c % 2 (columns 128-191 or
// 192-255), and P of chunk c written over the first 32 columns of that buffer.
constexpr uint32_t kColO = 0, kColS = 128;
constexpr int kQHalf = kM * 128;         // bytes of one 64-dim half of the query tile
constexpr int kKVHalf = kN * 128;        // bytes of one 64-dim half of K (or V) of a stage
constexpr int kStageT = 4 * kKVHalf;     // K half 0, K half 1, V half 0, V half 1
constexpr int kOffStages = 2 * kQHalf;
// full_k[], full_v[], empty_k[], empty_v[], s_full[2], p_full[2], o_done, o_final, q_full
constexpr int kOffBars = kOffStages + kStagesT * kStageT;
constexpr int kOffMisc = kOffBars + (4 * kStagesT + 7) * 8; // tensor-memory address, abort flag
constexpr size_t kBytesT = 1024 + kOffMisc + 16;
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

// Non-blocking test of an mbarrier phase (try_wait may suspend the thread;
// the MMA warp polls two barriers and must not sleep on either).
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Byte offset of 16-byte piece u (0..15) of row r in a K-major tile of
// `rows` rows stored as two 64-dim halves with 128-byte swizzle.
__device__ __forceinline__ uint32_t kmajor_off(int r, int u, int rows) {
  return (uint32_t)((u >> 3) * rows * 128 + r * 128 + (((u & 7) ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kThreadsT, 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const PrefillArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The tile index is the slowest grid dimension and runs backwards, so the
  // tiles with the most keys start first across all sequences and heads.
  const int kvh = blockIdx.x, s = blockIdx.y;
  const int tile = (int)gridDim.z - 1 - (int)blockIdx.z;

  const int q0 = __ldg(p.query_start + s), q1 = __ldg(p.query_start + s + 1);
  const int ctx = __ldg(p.context_lens + s);
  const int n_new = q1 - q0;
  const int rows = n_new * p.g;
  if (q0 < 0 || n_new < 0 || n_new > p.max_query_len || ctx < n_new || ctx > p.max_ctx || q1 > p.T) {
    if (tile == 0 && kvh == 0 && tid == 0) raise_status(p.status, PA_STATUS_BAD_CONTEXT);
    return;
  }
  const int row0 = tile * kM;
  if (row0 >= rows) return;
  const int first_pos = ctx - n_new;
  const int last_row = min(rows, row0 + kM) - 1;
  const int t_end = first_pos + last_row / p.g + 1;  // keys the tile attends
  const int nch = (t_end + kN - 1) / kN;

  // Keys and values of a stage have their own barriers: the keys of chunk c
  // are released when S(c) completes, the values when P·V(c) does.
  uint64_t* full_k = reinterpret_cast<uint64_t*>(base + kOffBars);
  uint64_t* full_v = full_k + kStagesT;
  uint64_t* empty_k = full_v + kStagesT;
  uint64_t* empty_v = empty_k + kStagesT;
  uint64_t* s_full = empty_v + kStagesT;  // [2]: S of chunk c is in buffer c % 2
  uint64_t* p_full = s_full + 2;          // [2]: P of chunk c is in S buffer c % 2
  uint64_t* o_done = p_full + 2;          // one phase per P·V
  uint64_t* o_final = o_done + 1;
  uint64_t* q_full = o_final + 1;         // the query tile is in shared memory
  uint32_t* tslot = reinterpret_cast<uint32_t*>(base + kOffMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(base + kOffMisc + 4);
  const uint32_t sbase = smem_addr(base);

  if (tid == 0) {
    for (int k = 0; k < kStagesT; ++k) {
      mbar_init(&full_k[k], 1);
      mbar_init(&full_v[k], 1);
      mbar_init(&empty_k[k], 1);
      mbar_init(&empty_v[k], 1);
    }
    mbar_init(q_full, kSoftWarps * 32);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&p_full[0], kSoftWarps * 32);
    mbar_init(&p_full[1], kSoftWarps * 32);
    mbar_init(o_done, 1);
    mbar_init(o_final, 1);
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

  if (warp == kProducerWarp) {
    // The whole warp: lane b loads block b of a chunk.  Block-table entries
    // are fetched 32 at a time, one per lane, a window ahead, so no TMA
    // issue waits on a dependent table load.
    pdl_wait_primary();  // the prompt's keys and values are in the cache from here on
    const int32_t* row = p.block_tables + (size_t)s * p.max_blocks_per_seq;
    const int nblk = (t_end + p.B - 1) / p.B;
    const int bpc = kN / p.B;  // blocks per chunk (block sizes 8, 16, 32)
    const uint64_t policy = policy_evict_first();
    int cur = load_block_id(row, lane, nblk);
    int nxt = load_block_id(row, 32 + lane, nblk);
    int wbase = 0, id_prev = 0;
    bool alive = true;
    // Keys run one chunk ahead of values: K(j) waits for S(j - 2) and
    // V(j - 1) for P·V(j - 3), and the tensor pipe completes S(j - 2),
    // P·V(j - 3), S(j - 1), ... in that order, so neither wait holds the
    // other back.
    for (int j = 0; j <= nch && alive; ++j) {
      int id = 0;
      if (j < nch) {
        const int jb = j * bpc;
        if (jb >= wbase + 32) {
          cur = nxt;
          wbase += 32;
          nxt = load_block_id(row, wbase + 32 + lane, nblk);
        }
        id = __shfl_sync(0xffffffffu, cur, (jb - wbase + lane) & 31);
        const int nb = (min(kN, t_end - j * kN) + p.B - 1) / p.B;
        if (lane < nb && (unsigned)id >= (unsigned)p.num_blocks) {
          raise_status(p.status, PA_STATUS_BAD_BLOCK);
          id = 0;
        }
      }
#pragma unroll 1
      for (int kv = 0; kv < 2; ++kv) {
        const int c = j - kv;
        if (c < 0 || c >= nch) continue;
        const int st = c % kStagesT;
        const int nb = (min(kN, t_end - c * kN) + p.B - 1) / p.B;
        uint64_t* fb = kv == 0 ? &full_k[st] : &full_v[st];
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait(kv == 0 ? &empty_k[st] : &empty_v[st], ((c / kStagesT) & 1) ^ 1, abort);
          if (ok) {
            mbar_arrive_expect_tx(fb, (uint32_t)(nb * p.B * 128 * 2));
          } else {
            *abort = 1;
            raise_status(p.status, PA_STATUS_TIMEOUT);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          alive = false;
          break;
        }
        __syncwarp();  // the expected byte count is set before any copy can land
        if (lane < nb) {
          const int y = ((kv == 0 ? id : id_prev) * p.Hkv + kvh) * p.B;
          uint8_t* d = base + kOffStages + st * kStageT + kv * 2 * kKVHalf + lane * p.B * 128;
          const CUtensorMap* map = kv == 0 ? &kmap : &vmap;
          tma_load_2d(d, map, fb, 0, y, policy);
          tma_load_2d(d + kKVHalf, map, fb, 64, y, policy);
        }
      }
      id_prev = id;
    }
  } else if (warp == kMmaWarp) {
    // S(c) and P·V(c) are issued as soon as each is ready -- S(c) when its
    // keys have landed and its buffer is free (P·V(c - 2) issued), P·V(c)
    // when the softmax has written P(c) -- so S of the next chunk overlaps
    // the softmax of this one without holding P·V back.  The tensor cores
    // run one thread's MMAs in order: S(c + 2) overwrites buffer c % 2 only
    // after P·V(c) has read P(c) from it, and the commit that releases
    // S(c + 1) to the softmax also covers P·V(c - 1).  P(c) is signalled on
    // p_full[c % 2]: the softmax can finish P(c + 1) before this warp has
    // seen P(c), but not P(c + 2), which needs S(c + 2), so neither barrier
    // runs a phase ahead of the poll.
    const uint32_t id_s = instr_desc(kM, kN, false);
    const uint32_t id_o = instr_desc(kM, kDh, true);
    int ns = 0, npv = 0;  // next S and next P·V to issue
    bool ok = true, q_ready = false;
    const unsigned long long t_start = global_timer_ns();
    unsigned spins = 0;
    while (npv < nch) {
      int what = 0;  // 1: issue S(ns), 2: issue P·V(npv)
      if (lane == 0) {
        if (npv < ns && mbar_test(&p_full[npv & 1], (npv >> 1) & 1) &&
            mbar_test(&full_v[npv % kStagesT], (npv / kStagesT) & 1))
          what = 2;
        else if (ns < nch && ns <= npv + 1 && (q_ready || (q_ready = mbar_test(q_full, 0))) &&
                 mbar_test(&full_k[ns % kStagesT], (ns / kStagesT) & 1))
          what = 1;
      }
      what = __shfl_sync(0xffffffffu, what, 0);
      if (what == 1) {
        const int c = ns++;
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sst = sbase + kOffStages + (c % kStagesT) * kStageT;
#pragma unroll
          for (int kk = 0; kk < kDh / 16; ++kk) {
            const int hlf = kk >> 2, w = kk & 3;
            const uint64_t a = smem_desc(sbase + hlf * kQHalf + w * 32, 16, 1024);
            const uint64_t b = smem_desc(sst + hlf * kKVHalf + w * 32, 16, 1024);
            mma_ss(tmem + kColS + (uint32_t)(c & 1) * kN, a, b, id_s, kk > 0);
          }
          mma_commit(&s_full[c & 1]);
          mma_commit(&empty_k[c % kStagesT]);
        }
        __syncwarp();
        spins = 0;
      } else if (what == 2) {
        const int c = npv++;
        uint8_t* stage = base + kOffStages + (c % kStagesT) * kStageT;
        const int nv = min(kN, t_end - c * kN);
        if (nv < kN) {  // value rows past the tile's keys: zeros (their keys are masked)
          for (int u = lane; u < (kN - nv) * 8 * 2; u += 32) {
            const int hlf = u / ((kN - nv) * 8), rem = u % ((kN - nv) * 8);
            *reinterpret_cast<uint4*>(stage + (2 + hlf) * kKVHalf + (nv + rem / 8) * 128 + (rem % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sst = sbase + kOffStages + (c % kStagesT) * kStageT;
          const uint32_t p_cols = tmem + kColS + (uint32_t)(c & 1) * kN;
#pragma unroll
          for (int kk = 0; kk < kN / 16; ++kk) {
            const uint64_t b = smem_desc(sst + 2 * kKVHalf + kk * 16 * 128, kKVHalf, 1024);
            mma_ts(tmem + kColO, p_cols + kk * 8, b, id_o, c > 0 || kk > 0);
          }
          mma_commit(o_done);
          mma_commit(&empty_v[c % kStagesT]);
        }
        __syncwarp();
        spins = 0;
      } else if ((++spins & 63u) == 0) {
        if (*abort || global_timer_ns() - t_start > kWaitLimitNs * 8) {
          ok = false;
          break;
        }
      }
    }
    if (!ok) {
      *abort = 1;
      raise_status(p.status, PA_STATUS_TIMEOUT);
    }
    if (lane == 0) mma_commit(o_final);
  } else {
    // Query tile (an input, not written by the append), K-major with
    // 128-byte swizzle; loaded here so that it overlaps the first stages.
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    for (int i = tid; i < kM * 16; i += kSoftWarps * 32) {
      const int rr = i >> 4, u = i & 15;
      const int gr = row0 + rr;
      const uint32_t off = kmajor_off(rr, u, kM);
      if (gr < rows) {
        const int h = kvh * p.g + gr % p.g;
        cp_async16(sbase + off, q + ((size_t)(q0 + gr / p.g) * p.H + h) * kDh + u * 8);
      } else {
        *reinterpret_cast<uint4*>(base + off) = make_uint4(0, 0, 0, 0);
      }
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    fence_proxy_async_smem();  // the query tile is read by the tensor cores (async proxy)
    mbar_arrive(q_full);
    // softmax: thread tid owns row tid (tensor-memory lane tid)
    const int r = row0 + tid;
    const int pos = r < rows ? first_pos + r / p.g : -1;  // keys 0 .. pos
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int c = 0; c < nch; ++c) {
      if (!mbar_wait(&s_full[c & 1], (c >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      const uint32_t s_cols = lane_base + kColS + (uint32_t)(c & 1) * kN;
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
      float mxr = -INFINITY;  // max of the raw (unscaled) valid scores
      if (nvalid >= kN) {
#pragma unroll
        for (int j = 0; j < kN; ++j) mxr = fmaxf(mxr, sc[j]);
      } else {
#pragma unroll
        for (int j = 0; j < kN; ++j) {
          sc[j] = j < nvalid ? sc[j] : -INFINITY;
          mxr = fmaxf(mxr, sc[j]);
        }
      }
      const float mx = mxr * p.scale_log2;  // scale > 0: the max of the scaled scores
      // Raise the running max (and rescale O) only when it grows past the
      // threshold; the decision is made per warp because tensor-memory
      // loads and stores are warp-wide.
      const bool grow = mx > m_run + kRescaleLog2 || (m_run == -INFINITY && mx != -INFINITY);
      const float m_new = grow ? mx : m_run;
      const float alpha = grow ? exp2f(m_run - m_new) : 1.f;  // m_run = -inf: alpha 0
      if (c > 0 && __any_sync(0xffffffffu, grow && m_run != -INFINITY)) {
        // O must hold P·V(c - 1) before it is rescaled
        if (!mbar_wait(o_done, (c - 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int i = 0; i < kDh / 16; ++i) {
          float v[16];
          tmem_ld16(lane_base + kColO + 16 * i, v);
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) w[j] = __float_as_uint(v[j] * alpha);
          tmem_st16(lane_base + kColO + 16 * i, w);
        }
      }
      l_run *= alpha;
      m_run = m_new;
      const float base_m = m_run == -INFINITY ? 0.f : m_run;
      uint32_t pk[kN / 2];
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < kN / 2; ++j) {  // exp2(s * scale - max): one FMA per score
        const float e0 = exp2f(fmaf(sc[2 * j], p.scale_log2, -base_m));
        const float e1 = exp2f(fmaf(sc[2 * j + 1], p.scale_log2, -base_m));
        ls += e0 + e1;
        pk[j] = pack_bf16x2(e0, e1);
      }
      l_run += ls;
#pragma unroll
      for (int i = 0; i < kN / 32; ++i) {
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = pk[16 * i + j];
        tmem_st16(s_cols + 16 * i, w);  // P over the first 32 columns of its S buffer
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      mbar_arrive(&p_full[c & 1]);
    }
    if (ok && mbar_wait(o_final, 0, abort)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      __nv_bfloat16* dst =
          r < rows ? static_cast<__nv_bfloat16*>(p.out) + ((size_t)(q0 + r / p.g) * p.H + kvh * p.g + r % p.g) * kDh
                   : nullptr;
#pragma unroll 1
      for (int i = 0; i < kDh / 16; ++i) {
        float v[16];
        tmem_ld16(lane_base + kColO + 16 * i, v);
        if (dst) {
          uint4 a, b2;
          a.x = pack_bf16x2(v[0] * inv, v[1] * inv);
          a.y = pack_bf16x2(v[2] * inv, v[3] * inv);
          a.z = pack_bf16x2(v[4] * inv, v[5] * inv);
          a.w = pack_bf16x2(v[6] * inv, v[7] * inv);
          b2.x = pack_bf16x2(v[8] * inv, v[9] * inv);
          b2.y = pack_bf16x2(v[10] * inv, v[11] * inv);
          b2.z = pack_bf16x2(v[12] * inv, v[13] * inv);
          b2.w = pack_bf16x2(v[14] * inv, v[15] * inv);
          reinterpret_cast<uint4*>(dst + 16 * i)[0] = a;
          reinterpret_cast<uint4*>(dst + 16 * i)[1] = b2;
        }
      }
    } else {
      *abort = 1;
      raise_status(p.status, PA_STATUS_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                              cudaStream_t stream) {
  const int tiles = (a.max_query_len * a.g + kM - 1) / kM;
  if (tiles <= 0 || a.S <= 0) return cudaSuccess;
  if (tiles > 65535 || a.S > 65535 || a.Hkv > 65535) return cudaErrorInvalidConfiguration;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::once_flag once[64];
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t init_err = cudaSuccess;
  std::call_once(once[dev], [&] {
    init_err = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBytesT);
  });
  if (init_err != cudaSuccess) return init_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.Hkv, (unsigned)a.S, (unsigned)tiles);
  cfg.blockDim = dim3(kThreadsT);
  cfg.dynamicSmemBytes = kBytesT;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel, kmap, vmap, a);
}

}  // namespace pa
