// Paged decode attention over an FP8 (E4M3) KV cache: bf16 queries and
// output, FP16 tensor-core products, FP32 accumulation (the mixed-precision
// recipe of "PagedAttention Kernel：大模型推理优化的显存管理革新" section 6:
// compute in FP16, accumulate in FP32), on keys and values stored as one
// byte each -- half the bytes of bf16 to move, the memory notes' measure
// ("Core Ideas" 1).  Stored code c of a cache with scale s reads as
// e4m3(c) * s.
//
// The schedule of the bf16 kernel (decode_tc.cu): persistent CTAs, two per
// SM, take (sequence, partition, KV head) items from the longest-first work
// list through an atomic counter; warp 5 loads each item's g query rows and
// streams its blocks by TMA into a 5-stage shared-memory ring (one box of
// [B tokens x 128 bytes] per block for keys and one for values, 128-byte
// swizzle; blocks of 8 tokens, 1 KB, by 16-byte cp.async into the same
// layout instead, one TMA box per KB being beyond the TMA unit's rate of
// boxes), 64 tokens per stage; warps 0-4 take the chunks in turn (one
// more consumer warp than the bf16 kernel: this consumer does about three
// times the work per byte) and merge their (max, sum, O) states at the end
// of the item.  Head dim 128.
//
// The consumer never widens a whole stage: it reads codes with ldmatrix and
// converts them in registers (cvt e4m3x2 -> f16x2, exact), so each code
// crosses shared memory once.
//  * Sᵀ = K Qᵀ (mma.m16n8k16 f16): 16 tokens of a step as the rows of A,
//    the query heads as the 8 columns of B (g of them real), so one MMA
//    covers twice the tokens that Q Kᵀ with the heads as rows would.  A
//    16-bit ldmatrix of key rows gives a lane four consecutive dims of one
//    token, so each 16-dim step uses a permuted k order -- k 2t, 2t+1 are
//    dims 4t, 4t+1 and k 2t+8, 2t+9 are dims 4t+2, 4t+3 -- and Q's fragments
//    are built in the same order (a dot product does not depend on it).
//  * Oᵀ = Vᵀ Pᵀ: the 8-bit transposing ldmatrix (m16n16) of a 16-token x
//    16-dim V tile gives a lane one dim of four consecutive tile rows, so the
//    token order of each 16-token step is permuted the same way (k 2t, 2t+1
//    are tile rows 4t, 4t+1 and k 2t+8, 2t+9 tile rows 4t+2, 4t+3; tile row
//    i is token pf8_row(i)).  The rows of each step's Sᵀ are gathered in the
//    matching order -- tokens {0,1,4,5,10,11,14,15} then {2,3,6,7,8,9,12,13}
//    -- so that a transposing movmatrix of each 8 x 8 half of P gives exactly
//    the B operand, and the eight key rows of each 8 x 8 matrix lie in eight
//    different bank groups.
//  * The online softmax keeps, per lane, heads 2t and 2t+1; their maxima
//    are reduced over the eight lanes holding the other tokens, and O (held
//    as Oᵀ, heads as columns) is rescaled without shuffles.
// Every wait is bounded (device_common.cuh); a time-out raises
// PA_STATUS_TIMEOUT and the CTA winds down.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "device_common.cuh"
#include "kernels.h"

namespace pa {
namespace {

// 16 bytes global -> shared by the load/store unit (not the TMA unit),
// cached in L2 only, with an L2 eviction policy.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "l"(policy)
               : "memory");
}

// The barrier's current phase also waits for every cp.async this thread has
// issued so far (its pending count is raised now and lowered when they land).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

constexpr int kD = 128;                      // head_dim
constexpr int kChunk = 64;                   // tokens per pipeline stage
constexpr int kRegion = kChunk * kD;         // 8 KB: the keys (or values) of a stage
constexpr int kStage = 2 * kRegion;
// Five stages (80 KB) fit two CTAs per SM.  Chunk k goes to stage k mod S
// and consumer warp k mod W; when S is not a multiple of W a stage passes
// from warp to warp, so a warp waits for the release of its stage's
// previous chunk before testing the stage's full barrier (which could
// otherwise be two phases behind and pass the parity test on the wrong
// phase).  That wait is itself exact only while there are no more consumer
// warps than stages: a warp at chunk k knows that chunk k - W - S was
// released (its previous chunk, k - W, was filled after it), and its parity
// tests need chunk k - 2S released.  (With W = S = 5 each stage belongs to
// one warp; the wait stays for other counts.)
constexpr int kStages = 5;
constexpr int KSTEPS = kChunk / 16;          // 16-token steps of P·V per stage
constexpr int kConsumerWarps = 5;
static_assert(kConsumerWarps <= kStages, "the stage hand-off between warps needs W <= S");
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kQSlot = kMaxGroup * kD * 2;   // bf16 query rows of one item
constexpr int kOStride = kD + 4;
constexpr int kOBuf = kConsumerWarps * kMaxGroup * kOStride * 4;
constexpr int kML = kConsumerWarps * kMaxGroup * 8;
constexpr int kBars = (2 * kStages + 6) * 8;  // full, empty, qfull[2], qempty[2], epi_full, epi_done
constexpr int kOffQ = kStages * kStage;
constexpr int kOffO = kOffQ + 2 * kQSlot;
constexpr int kOffML = kOffO + kOBuf;
constexpr int kOffDesc = kOffML + kML;
constexpr int kOffBar = kOffDesc + 2 * 16;
constexpr int kOffAbort = kOffBar + kBars;
constexpr size_t kBytes = 1024 + kOffAbort + 16;

struct Bars {
  uint64_t *full, *empty, *qfull, *qempty, *epi_full, *epi_done;
};

__device__ __forceinline__ Bars bars_at(uint8_t* base) {
  Bars b;
  b.full = reinterpret_cast<uint64_t*>(base + kOffBar);
  b.empty = b.full + kStages;
  b.qfull = b.empty + kStages;
  b.qempty = b.qfull + 2;
  b.epi_full = b.qempty + 2;
  b.epi_done = b.epi_full + 1;
  return b;
}

// Thread (g, t) of the warp receives bytes [4t .. 4t+3] of row g (tokens
// 4t..4t+3) at column g and g + 8 of a 16 x 16 byte tile, transposed:
// d0 byte j = tile[4t + j][g], d1 byte j = tile[4t + j][g + 8].  Lanes 0-15
// give the addresses of rows 0-15.
__device__ __forceinline__ void ldmatrix_b8_trans(uint32_t addr, uint32_t& d0, uint32_t& d1) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x1.trans.shared.b8 {%0, %1}, [%2];" : "=r"(d0), "=r"(d1) : "r"(addr));
}

// Token of tile row i (0-15) of a 16-token step of values: rows 0-7 are
// tokens 0-7, rows 8-15 tokens 10, 11, 8, 9, 14, 15, 12, 13.  Any order
// serves (the key rows follow it); this one makes the rows that one 8 x 8
// matrix of the keys' ldmatrix reads fall in eight different 16-byte bank
// groups of the 128-byte swizzle (the plain order put tokens t and t + 8
// in the same one).
__device__ __forceinline__ int pf8_row(int i) { return i ^ ((i & 8) >> 2); }

// Two E4M3 codes (low byte first) -> two f16 (low half first); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((unsigned short)two));
  return r;
}

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Transpose of an 8 x 8 matrix of 16-bit values held one row pair per lane
// (lane 4r + c holds row r, columns 2c, 2c + 1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// Two bf16 (one 32-bit word) -> two f16; exact for |x| in [2^-14, 65504].
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ void give_up(const DecodeArgs& p, volatile int* abort) {
  *abort = 1;
  raise_status(p.status, PA_STATUS_TIMEOUT);
}

__device__ void producer(const CUtensorMap* kmap, const CUtensorMap* vmap, const DecodeArgs& p, uint8_t* base,
                         volatile int* abort) {
  const int lane = threadIdx.x & 31;
  const Bars bar = bars_at(base);
  int4* desc = reinterpret_cast<int4*>(base + kOffDesc);
  const uint64_t policy = policy_evict_first();
  const int bpc = kChunk / p.B;  // cache blocks per chunk
  const uint32_t qbytes = (uint32_t)(p.g * kD * 2);
  const uint32_t block_bytes = (uint32_t)(p.B * kD * 2);  // keys + values of one block

  pdl_wait_primary();  // the work list is complete and visible from here on
  const int total = __ldcg(&p.hdr->num_pairs) * p.Hkv;
  unsigned* counter = &p.hdr->counter;
  // The next item is claimed when the current one starts and its list
  // entry read once the current item's first chunk is issued.
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
    const int ctx = __shfl_sync(kFull, cur_pr.y, 0);
    const int slot = n & 1;
    if (!mbar_wait(&bar.qempty[slot], ((n >> 1) & 1) ^ 1, abort)) {
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
    const int s = prx & 0xffff, part = prx >> 16, kvh = idx % p.Hkv;
    const int t0 = part * p.P, t1 = min(ctx, t0 + p.P);
    if (lane == 0) {
      desc[slot] = make_int4(s, part, kvh, ctx);
      mbar_arrive_expect_tx(&bar.qfull[slot], qbytes);
      const __nv_bfloat16* src =
          static_cast<const __nv_bfloat16*>(p.q) + ((size_t)s * p.H + (size_t)kvh * p.g) * kD;
      bulk_load(base + kOffQ + slot * kQSlot, src, qbytes, &bar.qfull[slot]);
    }
    ++nq;
    const int32_t* row = p.block_tables + (size_t)s * p.max_blocks_per_seq + t0 / p.B;
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
      const int stage = kseq % kStages;
      if (!mbar_wait(&bar.empty[stage], ((kseq / kStages) & 1) ^ 1, abort)) {
        ok = false;
        break;
      }
      if (p.B == 8) {
        // Blocks of 8 tokens are 1 KB: one TMA box each would cap the
        // stream at the TMA unit's rate of boxes.  The warp copies them in
        // 16-byte pieces instead (lane: piece u of rows rp and rp + 4 of
        // each block, 512 contiguous bytes per instruction), into the
        // layout the boxes would have left (128-byte swizzle: piece u of
        // stage row r at r * 128 + ((u ^ (r & 7)) << 4)); the stage's
        // barrier completes once lane 0 has arrived and every lane's copies
        // have landed.
        const int u = lane & 7, rp = lane >> 3;
        uint8_t* sk = base + stage * kStage;
        const uint8_t* kc = static_cast<const uint8_t*>(p.k_cache);
        const uint8_t* vc = static_cast<const uint8_t*>(p.v_cache);
        for (int b = 0; b < nb; ++b) {
          const size_t row0 = ((size_t)__shfl_sync(kFull, id, b) * p.Hkv + kvh) * 8;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int i = rp + 4 * h;  // row of the block
            const uint32_t off = (uint32_t)((8 * b + i) * kD + ((u ^ i) << 4));
            const size_t src = (row0 + i) * kD + u * 16;
            cp_async16(sk + off, kc + src, policy);
            cp_async16(sk + kRegion + off, vc + src, policy);
          }
        }
        cp_async_mbar_arrive(&bar.full[stage]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.full[stage]);
      } else {
        if (lane == 0) mbar_arrive_expect_tx(&bar.full[stage], (uint32_t)nb * block_bytes);
        __syncwarp();
        if (lane < nb) {
          const int y = (id * p.Hkv + kvh) * p.B;
          uint8_t* sk = base + stage * kStage + lane * p.B * kD;
          tma_load_2d(sk, kmap, &bar.full[stage], 0, y, policy);
          tma_load_2d(sk + kRegion, vmap, &bar.full[stage], 0, y, policy);
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
    for (uint32_t k = (kseq > (uint32_t)kStages ? kseq - kStages : 0); k < kseq; ++k)
      mbar_wait(&bar.full[k % kStages], (k / kStages) & 1, &never);
    for (uint32_t k = (nq > 2 ? nq - 2 : 0); k < nq; ++k) mbar_wait(&bar.qfull[k & 1], (k >> 1) & 1, &never);
  }
}

// Byte offset of 16-byte piece c of token row r of a stage region (TMA's
// 128-byte swizzle: pieces XOR-permuted by the row's low three bits).
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * kD + ((c ^ (r & 7)) << 4)); }

__device__ void consumer(const DecodeArgs& p, uint8_t* base, volatile int* abort) {
  constexpr int KS = kD / 16;  // 16-dim steps of Q·Kᵀ
  constexpr int MT = kD / 16;  // 16-dim tiles of Oᵀ = Vᵀ Pᵀ
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2;  // mma group id
  const int tq = lane & 3;   // thread in group
  const Bars bar = bars_at(base);
  const int4* desc = reinterpret_cast<const int4*>(base + kOffDesc);
  float* sO = reinterpret_cast<float*>(base + kOffO);
  float2* sML = reinterpret_cast<float2*>(base + kOffML);
  const uint32_t base_addr = smem_addr(base);
  // Key row of this lane's ldmatrix address within a 16-token step: rows
  // 0-7 of the step's Sᵀ tile are tokens {0,1,4,5,10,11,14,15}, rows 8-15
  // tokens {2,3,6,7,8,9,12,13} (lane L addresses row L % 8 of matrix L / 8;
  // odd matrices hold rows 8-15): the order of the values' tile rows
  // (pf8_row), each half eight different rows modulo 8, i.e. eight different
  // 16-byte bank groups of the swizzled stage.
  const int krow = pf8_row(4 * ((lane & 7) >> 1) + (lane & 1) + 2 * ((lane >> 3) & 1));
  uint32_t kseq = 0;

  for (uint32_t n = 0;; ++n) {
    const int slot = n & 1;
    if (!mbar_wait(&bar.qfull[slot], (n >> 1) & 1, abort)) {
      give_up(p, abort);
      return;
    }
    const int4 d = desc[slot];
    if (d.w < 0) return;  // no work left
    const int s = d.x, part = d.y, kvh = d.z, ctx = d.w;
    const int t0 = part * p.P, t1 = min(ctx, t0 + p.P);
    const int nch = (t1 - t0 + kChunk - 1) / kChunk;
    const int np = (ctx + p.P - 1) / p.P;
    // Q fragments in f16, dims of each 16-dim step in the permuted order.
    uint32_t qa[KS][2];
    {
      const __nv_bfloat16* sq = reinterpret_cast<const __nv_bfloat16*>(base + kOffQ + slot * kQSlot);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const __nv_bfloat16* r = sq + gq * kD + ks * 16 + 4 * tq;
        qa[ks][0] = gq < p.g ? bf16x2_to_f16x2(*reinterpret_cast<const uint32_t*>(r)) : 0u;
        qa[ks][1] = gq < p.g ? bf16x2_to_f16x2(*reinterpret_cast<const uint32_t*>(r + 2)) : 0u;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar.qempty[slot]);

    // running max and (this lane's share of the) sum of heads 2tq, 2tq + 1
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    for (int ch = 0; ch < nch; ++ch, ++kseq) {
      if ((int)(kseq % kConsumerWarps) != warp) continue;
      const int stage = kseq % kStages;
      if (kseq >= (uint32_t)kStages && !mbar_wait(&bar.empty[stage], ((kseq - kStages) / kStages) & 1, abort)) {
        give_up(p, abort);
        return;
      }
      if (!mbar_wait(&bar.full[stage], (kseq / kStages) & 1, abort)) {
        give_up(p, abort);
        return;
      }
      const int nv = min(kChunk, t1 - (t0 + ch * kChunk));
      const uint32_t sk = base_addr + stage * kStage;
      const uint32_t sv = sk + kRegion;
      if (nv < kChunk) {
        // Rows past the context hold stale or unwritten codes (possibly
        // NaN): zero their values; their scores are masked below.
        uint8_t* vrow = base + stage * kStage + kRegion;
        for (int u = lane; u < (kChunk - nv) * 8; u += 32)
          *reinterpret_cast<uint4*>(vrow + (nv + u / 8) * kD + (u % 8) * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncwarp();
      }
      // Sᵀ = K Qᵀ per 16-token step j: rows = the step's tokens in the
      // order above, columns = query heads (g of the 8 are real), k = dims in
      // the permuted order of each 16-dim step.  A = keys from a 16-bit
      // ldmatrix of the codes (a lane gets four consecutive dims of a token,
      // converted to two f16 pairs), B = the query rows.
      float st[KSTEPS][4];
#pragma unroll
      for (int jj = 0; jj < KSTEPS; ++jj) {
        st[jj][0] = st[jj][1] = st[jj][2] = st[jj][3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < KS / 2; ++kb) {
          uint32_t w[4];
          ldmatrix_x4(sk + swz(16 * jj + krow, 2 * kb + (lane >> 4)), w[0], w[1], w[2], w[3]);
          mma_f16_16816(st[jj], e4m3x2_to_f16x2(w[0]), e4m3x2_to_f16x2(w[1]), e4m3x2_to_f16x2(w[0] >> 16),
                        e4m3x2_to_f16x2(w[1] >> 16), qa[2 * kb][0], qa[2 * kb][1]);
          mma_f16_16816(st[jj], e4m3x2_to_f16x2(w[2]), e4m3x2_to_f16x2(w[3]), e4m3x2_to_f16x2(w[2] >> 16),
                        e4m3x2_to_f16x2(w[3] >> 16), qa[2 * kb + 1][0], qa[2 * kb + 1][1]);
        }
      }
      // Online softmax (log2 domain) of heads 2tq, 2tq + 1 over this chunk:
      // this lane holds tokens pf8_row(4(gq / 2) + (gq % 2)) and
      // pf8_row(that + 2) of each step; the other seven of each head are on
      // the lanes with the same tq.
      const int tok_lo = 4 * (gq >> 1) + (gq & 1);
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int jj = 0; jj < KSTEPS; ++jj) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int tok = 16 * jj + pf8_row(tok_lo + 2 * (c >> 1));
          const float v = tok < nv ? st[jj][c] * p.scale_log2 : -INFINITY;
          st[jj][c] = v;
          mx[c & 1] = fmaxf(mx[c & 1], v);
        }
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx[0] = fmaxf(mx[0], __shfl_xor_sync(kFull, mx[0], off));
        mx[1] = fmaxf(mx[1], __shfl_xor_sync(kFull, mx[1], off));
      }
      float alpha[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float m_new = fmaxf(m_run[e], mx[e]);
        alpha[e] = exp2f(m_run[e] - m_new);
        m_run[e] = m_new;
        l_run[e] *= alpha[e];
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        o[mt][0] *= alpha[0];
        o[mt][1] *= alpha[1];
        o[mt][2] *= alpha[0];
        o[mt][3] *= alpha[1];
      }
      // P in f16; a transposing movmatrix of each 8 x 8 half of a step turns
      // (token row, head pair) into (head gq, tokens 4tq, 4tq + 1) and
      // (head gq, tokens 4tq + 2, 4tq + 3): the B operand of Oᵀ = Vᵀ Pᵀ in the
      // token order of the values' transposing ldmatrix.
      uint32_t pb[KSTEPS][2];
#pragma unroll
      for (int jj = 0; jj < KSTEPS; ++jj) {
        const float e0 = exp2f(st[jj][0] - m_run[0]), e1 = exp2f(st[jj][1] - m_run[1]);
        const float e2 = exp2f(st[jj][2] - m_run[0]), e3 = exp2f(st[jj][3] - m_run[1]);
        l_run[0] += e0 + e2;
        l_run[1] += e1 + e3;
        pb[jj][0] = movmatrix_trans(pack_f16x2(e0, e1));
        pb[jj][1] = movmatrix_trans(pack_f16x2(e2, e3));
      }
      // Oᵀ += Vᵀ Pᵀ : 16 tokens per step, 16 dims per tile; lane i < 16
      // addresses tile row i, token pf8_row(i) of the step.
#pragma unroll
      for (int kt = 0; kt < KSTEPS; ++kt) {
        const uint32_t pb0 = pb[kt][0];  // tile rows 4tq, 4tq+1 of the step, head gq
        const uint32_t pb1 = pb[kt][1];  // tile rows 4tq+2, 4tq+3
        const int r = 16 * kt + pf8_row(lane & 15);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t d0, d1;
          ldmatrix_b8_trans(sv + swz(r, mt), d0, d1);
          mma_f16_16816(o[mt], e4m3x2_to_f16x2(d0), e4m3x2_to_f16x2(d1), e4m3x2_to_f16x2(d0 >> 16),
                        e4m3x2_to_f16x2(d1 >> 16), pb0, pb1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.empty[stage]);
    }

    // ---- item epilogue: merge the four warps' states ----
    if (n > 0 && !mbar_wait(bar.epi_done, (n - 1) & 1, abort)) {
      give_up(p, abort);
      return;
    }
    float l0 = l_run[0], l1 = l_run[1];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, off);
      l1 += __shfl_xor_sync(kFull, l1, off);
    }
    if (gq == 0) {
      if (2 * tq < p.g) sML[warp * kMaxGroup + 2 * tq] = make_float2(m_run[0], l0);
      if (2 * tq + 1 < p.g) sML[warp * kMaxGroup + 2 * tq + 1] = make_float2(m_run[1], l1);
    }
    float* ob = sO + warp * kMaxGroup * kOStride;
    const int h0 = 2 * tq, h1 = 2 * tq + 1;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int dd = 16 * mt + gq;
      if (h0 < p.g) {
        ob[h0 * kOStride + dd] = o[mt][0];
        ob[h0 * kOStride + dd + 8] = o[mt][2];
      }
      if (h1 < p.g) {
        ob[h1 * kOStride + dd] = o[mt][1];
        ob[h1 * kOStride + dd + 8] = o[mt][3];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar.epi_full);
    if (!mbar_wait(bar.epi_full, n & 1, abort)) {
      give_up(p, abort);
      return;
    }
    const int units = p.g * (kD / 8);
    for (int u = threadIdx.x; u < units; u += kConsumerWarps * 32) {
      const int h = u / (kD / 8);
      const int d0 = (u % (kD / 8)) * 8;
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
        const float4* src = reinterpret_cast<const float4*>(sO + (w * kMaxGroup + h) * kOStride + d0);
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
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] *= p.v_scale;  // codes -> values
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
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + ((size_t)s * p.H + qh) * kD + d0;
        *reinterpret_cast<uint4*>(dst) = pk;
      } else {
        const size_t wi = ((size_t)s * p.max_parts + part) * p.H + qh;
        float4* dst = reinterpret_cast<float4*>(p.ws_o + wi * kD + d0);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        if (d0 == 0) p.ws_ml[wi] = make_float2(M, L);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar.epi_done);
  }
}

__global__ void __launch_bounds__(kThreads, 2)
    paged_decode_fp8_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                            const DecodeArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile int* abort = reinterpret_cast<volatile int*>(base + kOffAbort);
  if (threadIdx.x == 0) {
    const Bars b = bars_at(base);
    for (int k = 0; k < kStages; ++k) {
      mbar_init(&b.full[k], 1);
      mbar_init(&b.empty[k], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&b.qfull[k], 1);
      mbar_init(&b.qempty[k], kConsumerWarps);
    }
    mbar_init(b.epi_full, kConsumerWarps);
    mbar_init(b.epi_done, kConsumerWarps);
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
    producer(&kmap, &vmap, p, base, abort);
  } else {
    consumer(p, base, abort);
  }
}

}  // namespace

size_t decode_fp8_smem_bytes() { return kBytes; }

cudaError_t launch_decode_fp8(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                              cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  struct Shape {
    int sms = 0, per_sm = 0;
  };
  static Shape shapes[64];
  static std::once_flag once[64];
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t init_err = cudaSuccess;
  std::call_once(once[dev], [&] {
    Shape sh;
    init_err = cudaDeviceGetAttribute(&sh.sms, cudaDevAttrMultiProcessorCount, dev);
    if (init_err == cudaSuccess)
      init_err = cudaFuncSetAttribute(paged_decode_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kBytes);
    if (init_err == cudaSuccess)
      init_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&sh.per_sm, paged_decode_fp8_kernel, kThreads, kBytes);
    shapes[dev] = sh;
  });
  if (init_err != cudaSuccess) return init_err;
  const Shape& sh = shapes[dev];
  if (sh.per_sm < 1 || sh.sms < 1) return cudaErrorInvalidConfiguration;
  const long long total = (long long)a.max_parts * a.S * a.Hkv;  // upper bound of the work items
  const int grid = (int)std::min<long long>(total, (long long)sh.sms * sh.per_sm);
  if (grid <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_decode_fp8_kernel, kmap, vmap, a);
}

}  // namespace pa
