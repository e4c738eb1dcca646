// Prefill on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory), head_dim 64 or 128, bf16 storage, fp32 accumulation.
//
// Every new token of a sequence attends the sequence's tokens up to its own
// position ("PagedAttention Kernel：大模型推理优化的显存管理革新" section 3.1
// with a causal limit; the prompt's keys and values were appended into their
// blocks first, "Day 6/90 of Inference Engineering", PagedAttention notes,
// paragraph 2).
//
// Work items are (sequence, KV head, pair of adjacent tiles of 128 query
// rows), the rows being (new token, query head) pairs, token-major; the
// pairs with the most keys come first.  Both tiles of an item read every
// stage of keys and values, so each TMA box feeds 256 rows.  The kernel is
// persistent: one CTA per SM (384 threads) walks a fixed list of items that
// it computes in its prologue (the items sorted by cost when the prompts are
// ragged; a snake over the CTAs, or the costliest items to the CTAs that
// take one item fewer, whichever leaves the busiest CTA less work), so the
// set-up (barriers, tensor memory) is paid once per SM, there is no tail of
// whole waves, and the next item's loads overlap the current item's last
// products and epilogue.  The keys are taken in steps of 64: per tile two
// S buffers in tensor memory, so that S of the next step is ready when the
// softmax finishes a step.  Roles:
//  * warps 8 and 9 (producers): stream the keys (warp 8) and values (warp 9)
//    of each item, 128 tokens (two steps) per stage, into rings of their
//    own (2 stages each) that run on across items, with an L2 policy that
//    keeps them for the other pairs of the same sequence and head, one TMA
//    box per block (a 4D view of the cache: groups of 8 rows with both
//    64-dim halves, 128-byte swizzle, which is the layout of a K-major
//    operand of the tensor cores for keys and of an MN-major one for
//    values); chunks of cached tokens go out while the append kernel may
//    still run, the first chunk that holds a new token after
//    griddepcontrol.wait (the append writes only the new tokens' slots);
//    lane b issues block b of a chunk from block-table entries fetched 32
//    at a time.  Warp 8 first loads the
//    item's query tiles, one 3D box per 64-dim half, once the previous
//    item's last S has completed.  Value rows past a sequence's end (in its
//    last block) are cleared by warp 9 once their copy has landed, and the
//    value ring starts as zeros, so every value row a P·V reads is finite
//    (masked keys get exact zero weights, and 0 x NaN would still be NaN);
//  * warps 10 and 11 (MMA, one per tile): lane 0 alone issues the tile's
//    S = Q Kᵀ (M 128, N 64, K = head_dim: head_dim / 16 tcgen05.mma
//    kind::f16 from shared-memory descriptors) and O += P V (M 128,
//    N = head_dim, K 64: four MMAs, P read from tensor memory, V an
//    MN-major operand in shared memory): per item S(0) and S(1) into the
//    two buffers, then per step u, once P(u) is in, P·V(u) and S(u + 2)
//    into the buffer P·V(u) has just read, and one commit into that
//    buffer's barrier; the other lanes idle, since a warp-wide
//    synchronisation after a group of MMAs waits for the tensor cores to
//    take the group.  With one issuing thread per tile the tensor cores
//    interleave the two tiles' products;
//  * warps 0-3 and 4-7 (softmax, one warpgroup per tile, both running at
//    once): thread t of a warpgroup owns query row t of its tile
//    (tensor-memory lane t).  Per step it takes the commit that follows
//    S(u) (it also covers P·V(u - 2)) and releases, as far as its tile is
//    concerned, the keys after the second step of a chunk, the values
//    after the second P·V of a chunk, and the query tile after the item's
//    last S: one arrival per tile, so the MMA thread spends no commits on
//    releases.  It reads its 64 scores (tcgen05.ld), masks keys past its
//    position, keeps the running max and sum, writes P as bf16 over S
//    (tcgen05.st; one arrival per warp on the buffer's P barrier) and
//    rescales its row of O only when its max grows by more than 2^8
//    (otherwise the stale max stays: exp2 values up to 256 are exact
//    enough and O and the sum use the same max), after taking the next
//    commit, which covers P·V(u - 1).  The exponentials are one packed FMA
//    per two scores (scale and max) and one ex2 each; the max is taken
//    three operands at a time.  At the end of the item it takes the
//    commits that cover the last P·V, reads its row of O and divides by
//    the sum; a tile of 128 query rows is staged in shared memory (one
//    buffer, the two tiles' in turns) and stored by TMA, the rows of a
//    sequence's last tile directly, the four lanes of each quad trading
//    32-byte pieces so that every store writes whole 128-byte lines.
// The softmax warpgroups run with 224 registers a thread and the producer
// and MMA warps with 56 (setmaxnreg).  Both tiles attend all of the item's
// steps (the earlier tile's keys past its rows' positions are masked),
// which keeps the two tiles' releases symmetric.  Tensor memory (512
// columns allocated once per CTA): O of tile t at columns DH·t .. DH·t +
// DH - 1 and its S buffers at 2·DH + 128t and 2·DH + 128t + 64 (DH =
// head_dim); P is written over the first half of its buffer.  Every wait
// is bounded; on a time-out the kernel raises PA_STATUS_TIMEOUT, stops
// issuing work, lets its copies and products in flight finish, and exits.

#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "block_layout.cuh"
#include "device_common.cuh"
#include "kernels.h"
#include "pa.h"
#include "pa_internal.h"
#include "tcgen05.cuh"

namespace pa {
namespace {

// One 32-byte store of eight 32-bit words (dst 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

constexpr int kM = 128;                 // query rows per tile (one tensor-memory lane each)
constexpr int kTiles = 2;               // query tiles per CTA, sharing every stage
constexpr int kN = 128;                 // keys per stage of the rings
constexpr int kSub = 64;                // keys per softmax step (the N of S = Q Kᵀ)
constexpr int kStagesK = 2;             // stages in the key ring
constexpr int kStagesV = 2;             // stages in the value ring
constexpr int kSoftWarps = 4;           // per tile
constexpr int kProducerWarp = kTiles * kSoftWarps;  // keys; the next warp streams values
constexpr int kMmaWarp = kProducerWarp + 2;         // tile 0's MMAs; the next warp issues tile 1's
constexpr int kThreadsT = (kTiles * kSoftWarps + 2 + kTiles) * 32;
// Registers per thread: the launch gets kRegsLaunch (what 384 threads at one
// CTA per SM compile to); then the softmax warpgroups raise theirs to
// kRegsSoft and the warpgroup of producers and MMA warps lowers its own to
// kRegsAux.  The split must fit in what the launch reserved, or the raise
// would wait forever; the host checks the compiled count before launching.
constexpr int kRegsLaunch = 168, kRegsSoft = 224, kRegsAux = 56;
static_assert(kTiles * kSoftWarps * 32 * kRegsSoft + (kThreadsT - kTiles * kSoftWarps * 32) * kRegsAux <=
                  kThreadsT * kRegsLaunch,
              "register split exceeds the launch's registers");
static_assert(kProducerWarp % 4 == 0 && kThreadsT - kProducerWarp * 32 == 128,
              "producers and MMA warps form one warpgroup");
constexpr uint32_t kTmemCols = 512;
constexpr int kQHalf = kM * 128;         // bytes of one 64-dim half of a query tile
constexpr int kKVHalf = kN * 128;        // bytes of one 64-dim half of a stage of K (or V)
// A stage holds its keys (or values) in groups of 8 rows, each group both
// 64-dim halves, 1 KB apart ([group][half][8 rows][128 B]), so that one TMA
// box brings a whole block (see kv_row_offset).
// full_k[], empty_k[], full_v[], empty_v[]; per tile s_full and p_full of
// each S buffer, q_full
constexpr int kTileBars = 5;
// Items a CTA can list in shared memory; launches hold at most kListCap
// items per CTA (the host splits larger batches over several launches).
constexpr int kListCap = 440;

// Layout for head_dim DH (64 or 128): tiles and stages hold DH / 64 halves
// of 64 dims; O of tile t at columns DH·t .. DH·t + DH - 1, its two S
// buffers (64 columns each) at 2·DH + 128t and 2·DH + 128t + 64, the P
// (bf16 pairs) of a buffer over its first 32 columns.
template <int DH>
struct PfCfg {
  static constexpr int kHalves = DH / 64;
  static constexpr int kQTile = kHalves * kQHalf;
  static constexpr int kKVStage = kHalves * kKVHalf;
  static constexpr int kOffK = kTiles * kQTile;
  static constexpr int kOffV = kOffK + kStagesK * kKVStage;
  static constexpr int kOffOut = kOffV + kStagesV * kKVStage;  // one tile's output rows, staged for a TMA store
  static constexpr int kOffBars = kOffOut + kQTile;
  // barriers: the rings, kTileBars per tile, q_empty, drained and staged per tile, v_land, out_free
  static constexpr int kOffMisc = kOffBars + (2 * (kStagesK + kStagesV) + kTiles * kTileBars + 3 * kTiles + 2) * 8;
  // misc: tensor-memory address, abort flag, the busiest CTA's load of each
  // candidate list (4), the CTA's item count; then its items
  static constexpr int kOffList = kOffMisc + 32;
  static constexpr size_t kBytes = 1024 + kOffList + 4 * kListCap;
  static constexpr uint32_t kColO = 0, kColS = 2 * DH;
  static_assert(DH == 64 || DH == 128, "head_dim 64 or 128");
  static_assert(kBytes <= 227 * 1024, "shared memory of one CTA");
  static_assert(kColS + kTiles * 128 <= kTmemCols, "tensor-memory columns");
};
constexpr float kRescaleLog2 = 8.f;      // rescale O only when a row's max grows by more than 2^8

// Work item j of S * Hkv * pairs: pair of query tiles pairs - 1 - j / (S * Hkv)
// (the pairs with the most keys first), sequence (j / Hkv) % S, KV head
// j % Hkv.  Every role of a CTA walks the same items in the same order and
// derives the same chunk counts from them, so they need no messages beyond
// the pipeline's barriers.
struct PfItem {
  int s, kvh, pair, q0, rows, first_pos, row00, ctx;
  int nch, nsub, t_end;        // stages (128 keys) and steps (64 keys) the pair attends, and its keys
  int state;                   // 0: work; 1: no rows of the sequence in this pair; 2: inconsistent lengths
};

// The lengths' fields the items are derived from, by value: the item-list
// builder (a function of its own) reads them from registers rather than
// through a reference to the kernel's arguments.
struct PfLens {
  const int32_t* query_start;
  const int32_t* context_lens;
  int S, T, Hkv, g, max_ctx, max_query_len;
};

template <class A>
__device__ __forceinline__ PfItem pf_item(const A& p, int j, int pairs) {
  PfItem it{};
  const int per = p.S * p.Hkv;
  it.pair = pairs - 1 - j / per;
  it.s = (j % per) / p.Hkv;
  it.kvh = j % p.Hkv;
  const int q0 = __ldg(p.query_start + it.s), q1 = __ldg(p.query_start + it.s + 1);
  const int ctx = __ldg(p.context_lens + it.s);
  const int n_new = q1 - q0;
  if (q0 < 0 || n_new < 0 || n_new > p.max_query_len || ctx < n_new || ctx > p.max_ctx || q1 > p.T) {
    it.state = 2;
    return it;
  }
  it.q0 = q0;
  it.ctx = ctx;
  it.rows = n_new * p.g;
  it.first_pos = ctx - n_new;
  it.row00 = it.pair * kTiles * kM;
  if (it.row00 >= it.rows) {
    it.state = 1;
    return it;
  }
  // Keys the pair attends: up to the position of its last row (tile 1 is
  // the later one).  Both tiles run over all of them; a tile's rows mask
  // the keys past their positions.
  it.t_end = it.first_pos + (min(it.rows, it.row00 + kTiles * kM) - 1) / p.g + 1;
  it.nch = (it.t_end + kN - 1) / kN;
  it.nsub = (it.t_end + kSub - 1) / kSub;
  return it;
}

// The items of one CTA in a list of n items: item r (r < count) is list
// position base + r * stride + (r even ? slot : stride - 1 - slot), i.e.
// rounds of `stride` items over `stride` CTAs, alternately in and against
// CTA order, so that a CTA given one of the costliest items of a round gets
// one of the cheapest of the next.  Two orders on G CTAs (n = q·G + e):
//  * plain: one snake over all G CTAs;
//  * count-aware: the first G - e CTAs take q items each and the last e take
//    q + 1; the costliest q·(G - e) items go to the CTAs with fewer items and
//    the rest to the others, each group a snake of its own.
// On 512 items of 5-8 chunks (128 of each) on 152 CTAs the count-aware order
// gives the busiest CTA 22 chunks, the least possible, against 25 in the
// plain one; on ragged batches it can do worse.
struct PfOrder {
  int base, stride, slot, count;
};

__device__ __forceinline__ PfOrder pf_order(int b, int G, int n, int q, bool aware) {  // q = n / G
  const int e = n - q * G, ga = G - e;
  if (!aware) return PfOrder{0, G, b, q + ((q & 1) ? (b >= ga ? 1 : 0) : (b < e ? 1 : 0))};
  if (b < ga) return PfOrder{0, ga, b, q};
  return PfOrder{q * ga, e, b - ga, q + 1};
}

__device__ __forceinline__ int pf_list_pos(const PfOrder& o, int r) {
  return o.base + r * o.stride + ((r & 1) ? o.stride - 1 - o.slot : o.slot);
}

// Cost of an item for balancing: its chunks of keys plus one for its start
// and end (0 for a pair without rows).
template <class A>
__device__ __forceinline__ int pf_item_cost(const A& p, int j, int pairs) {
  const PfItem it = pf_item(p, j, pairs);
  return it.state ? 0 : it.nch + 1;
}

// The candidate lists are compared when every CTA has at most this many
// items, and the items sorted when the batch has at most this many (pair,
// sequence) entries and cost levels.
constexpr int kMaxCheckedItemsPerCta = 16;
constexpr int kMaxSortedEntries = 2048;
constexpr int kMaxCostLevels = 1024;

// The CTA's list of items.  Every CTA computes the same assignment from
// the same inputs (the lengths, which the append kernel does not write:
// no wait for it is needed), in the value ring before it is cleared.
// Items are (pair, sequence, KV head), the KV heads of an entry (pair,
// sequence) consecutive; entries are listed pair-major, the pairs with the
// most keys first, or -- when that is not already from the costliest to
// the cheapest, as it is not for ragged prompts -- sorted by cost, most
// first, stably (a counting sort; warp 0 places the entries in order).
// Of the lists {pair-major, sorted} x orders {plain, count-aware}, the one
// whose busiest CTA has the least cost is taken.  A launch of a batch
// split over several launches (first_item > 0, or more items than fit the
// comparison) takes the pair-major list in the plain order.
// Called by every thread of the CTA, before the value ring is cleared:
// `cost` is the ring (ring_ints ints of scratch), `busiest` 4 ints, the
// CTA's item count and items go to *my_count and my_items.
__device__ __noinline__ void pf_build_list(const PfLens p, int pairs, int first_item, int num_items,
                                           int* cost, int ring_ints, int* busiest, int* my_count, int* my_items) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = (int)gridDim.x, b = (int)blockIdx.x;
  const int E = pairs * p.S;
  const int levels = (p.max_ctx + kN - 1) / kN + 2;  // costs are below this
  const bool check = first_item == 0 && num_items == E * p.Hkv && num_items <= kMaxCheckedItemsPerCta * G &&
                     E <= ring_ints / 2;
  bool sorting = check && E <= kMaxSortedEntries && levels <= kMaxCostLevels && 2 * E + levels <= ring_ints;
  const int q_all = num_items / G;
  // j / Hkv without a division chain per item: a float estimate (j < 2^24)
  // corrected by one either way
  const float inv_hkv = 1.f / (float)p.Hkv;
  auto div_hkv = [&](int j) {
    int e = (int)((float)j * inv_hkv);
    e -= e * p.Hkv > j ? 1 : 0;
    e += (e + 1) * p.Hkv <= j ? 1 : 0;
    return e;
  };
  int* sorted = cost + E;            // [E] entries by cost, most first
  int* next = sorted + E;            // [levels] per cost level: the next free position
  if (check)
    for (int i = tid; i < E; i += kThreadsT) cost[i] = pf_item_cost(p, i * p.Hkv, pairs);
  if (tid < 4) busiest[tid] = 0;
  if (sorting)
    for (int i = tid; i < levels; i += kThreadsT) next[i] = 0;
  __syncthreads();
  if (sorting) {
    bool in_order = true;
    for (int i = tid; i + 1 < E; i += kThreadsT) in_order = in_order && cost[i] >= cost[i + 1];
    sorting = !__syncthreads_and(in_order);
  }
  if (sorting) {
    for (int i = tid; i < E; i += kThreadsT) atomicAdd(&next[cost[i]], 1);
    __syncthreads();
    if (tid == 0) {  // positions of the levels, costliest first
      int at = 0;
      for (int c = levels - 1; c >= 0; --c) {
        const int k = next[c];
        next[c] = at;
        at += k;
      }
    }
    __syncthreads();
    if (warp == 0)
      for (int i0 = 0; i0 < E; i0 += 32) {
        const int i = i0 + lane;
        const int c = i < E ? cost[i] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, c);
        const int before = __popc(peers & ((1u << lane) - 1u));
        const int pos = c >= 0 ? next[c] + before : 0;
        __syncwarp();
        if (c >= 0) {
          sorted[pos] = i;
          if (before == 0) next[c] += __popc(peers);
        }
        __syncwarp();
      }
    __syncthreads();
  }
  if (check)
    for (int c0 = 0; c0 < G; c0 += kThreadsT) {
      const int c = c0 + tid;
      int load[4] = {0, 0, 0, 0};
      if (c < G)
        for (int k = 0; k < (sorting ? 4 : 2); ++k) {
          const PfOrder o = pf_order(c, G, num_items, q_all, k & 1);
          for (int r = 0; r < o.count; ++r) {
            const int e = div_hkv(pf_list_pos(o, r));
            load[k] += cost[k >= 2 ? sorted[e] : e];
          }
        }
#pragma unroll
      for (int k = 0; k < 4; ++k) load[k] = __reduce_max_sync(0xffffffffu, load[k]);
      if (lane == 0)
#pragma unroll
        for (int k = 0; k < 4; ++k) atomicMax(&busiest[k], load[k]);
    }
  __syncthreads();
  {
    int pick = 0;  // pair-major, plain
    if (check)
      for (int k = 1; k < (sorting ? 4 : 2); ++k)
        if (busiest[k] < busiest[pick]) pick = k;
    const PfOrder o = pf_order(b, G, num_items, q_all, pick & 1);
    if (warp == 0)
      for (int r = lane; r < o.count; r += 32) {
        const int j = pf_list_pos(o, r);
        my_items[r] = first_item + (pick >= 2 ? sorted[j / p.Hkv] * p.Hkv + j % p.Hkv : j);
      }
    if (tid == 0) *my_count = o.count;
  }
}

template <int DH>
__global__ void __launch_bounds__(kThreadsT, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                      const __grid_constant__ PrefillArgs p, int pairs, int first_item, int num_items,
                      int withhold) {
  using C = PfCfg<DH>;
  constexpr int kQTile = C::kQTile, kKVStage = C::kKVStage, kOffK = C::kOffK, kOffV = C::kOffV;
  constexpr uint32_t kColO = C::kColO, kColS = C::kColS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint64_t* full_k = reinterpret_cast<uint64_t*>(base + C::kOffBars);
  uint64_t* empty_k = full_k + kStagesK;
  uint64_t* full_v = empty_k + kStagesK;
  uint64_t* empty_v = full_v + kStagesV;
  uint64_t* tile_bars = empty_v + kStagesV;  // kTileBars per tile
  // per tile: [0], [1] the MMAs issued before a commit into buffer 0 or 1
  // are done, [2], [3] P of a step is in buffer 0 or 1, [4] the item's
  // query tile is in
  auto s_full = [&](int t, int buf) { return tile_bars + t * kTileBars + buf; };
  auto p_full = [&](int t, int buf) { return tile_bars + t * kTileBars + 2 + buf; };
  auto q_full = [&](int t) { return tile_bars + t * kTileBars + 4; };
  uint64_t* q_empty = tile_bars + kTiles * kTileBars;  // per tile: the item's last S is done, the query tile is free
  uint64_t* drained = q_empty + kTiles;                // per MMA warp: every MMA it issued is done
  uint64_t* staged = drained + kTiles;                 // per tile: its warps have staged their output rows
  uint64_t* v_land = staged + kTiles;                  // the values of a chunk that holds rows past its sequence have landed
  uint64_t* out_free = v_land + 1;                     // a tile's turn on the output staging buffer has ended
  uint32_t* tslot = reinterpret_cast<uint32_t*>(base + C::kOffMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(base + C::kOffMisc + 4);
  const uint32_t sbase = smem_addr(base);

  if (tid == 0) {
    // a stage (and the query tiles) is free once both tiles' softmax
    // warpgroups have released it
    for (int k = 0; k < kStagesK; ++k) {
      mbar_init(&full_k[k], 1);
      mbar_init(&empty_k[k], kTiles);
    }
    for (int k = 0; k < kStagesV; ++k) {
      mbar_init(&full_v[k], 1);
      mbar_init(&empty_v[k], kTiles);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(s_full(t, 0), 1);
      mbar_init(s_full(t, 1), 1);
      mbar_init(p_full(t, 0), kSoftWarps);  // one arrival per warp
      mbar_init(p_full(t, 1), kSoftWarps);
      mbar_init(q_full(t), 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(q_empty + t, 1);
      mbar_init(drained + t, 1);
      mbar_init(staged + t, kSoftWarps);  // one arrival per warp
    }
    mbar_init(v_land, 1);
    mbar_init(out_free, 1);
    *abort = 0;
    fence_barrier_init();
  }
  int* my_count = reinterpret_cast<int*>(base + C::kOffMisc + 24);
  int* my_items = reinterpret_cast<int*>(base + C::kOffList);
  const PfLens lens{p.query_start, p.context_lens, p.S, p.T, p.Hkv, p.g, p.max_ctx, p.max_query_len};
  pf_build_list(lens, pairs, first_item, num_items, reinterpret_cast<int*>(base + kOffV), kStagesV * kKVStage / 4,
                reinterpret_cast<int*>(base + C::kOffMisc + 8), my_count, my_items);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tslot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp >= kProducerWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsAux));
    if (warp < kMmaWarp) {
      // One warp streams the keys, the next the values, each into its own
      // ring, so neither waits behind the other's release.  Lane b loads
      // block b of a chunk; block-table entries are fetched 32 at a time, one
      // per lane, a window ahead, so no TMA issue waits on a dependent load.
      // The key warp also loads each item's query tiles, once the previous
      // item's last S has completed.
      const int kv = warp - kProducerWarp;  // 0 keys, 1 values
      const int bpc = kN / p.B;             // blocks per chunk (block sizes 8, 16, 32: 16, 8 or 4, dividing 32)
      // The other pairs of the same sequence and KV head read the same keys
      // and values: keep them in L2.
      const uint64_t policy = policy_evict_last();
      const CUtensorMap* map = kv == 0 ? &kmap : &vmap;
      uint64_t* fulls = kv == 0 ? full_k : full_v;
      uint64_t* empties = kv == 0 ? empty_k : empty_v;
      const int stages = kv == 0 ? kStagesK : kStagesV;
      if (kv == 1) {
        // Value rows that no copy writes must still be finite (their weights
        // are exact zeros, and 0 x NaN is NaN): the value ring starts as
        // zeros (it held the item lists' scratch until the set-up's barrier),
        // and rows past a sequence's end are cleared after their copy lands.
        for (int u = lane; u < kStagesV * kKVStage / 16; u += 32)
          reinterpret_cast<uint4*>(base + kOffV)[u] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();  // before any copy into the ring
        __syncwarp();
      }
      uint32_t k = 0;                // chunks issued into this ring over the CTA's items
      uint32_t qn[kTiles] = {0, 0};  // query-tile loads per tile
      uint32_t vl = 0;               // chunks of values cleared past their sequence's end
      bool waited = false, ok = true, landing = false;
      for (int r = 0; ok; ++r) {
        const int j = (r < *my_count ? my_items[r] : -1);
        if (j < 0) break;
        const PfItem it = pf_item(p, j, pairs);
        if (it.state) continue;
        // The query tiles (an input the append does not write), one box per
        // 64-dim half: 128 / g tokens x g heads of this KV head.  Rows past
        // the sequence read the next sequence's queries (or zeros past the
        // last token); their scores are all masked and their rows never
        // stored.  Tile t's is loaded once the tile's last S of the previous
        // item has completed: tile 0's first, then the item's first keys,
        // then tile 1's.
        auto load_q = [&](int t) {
          int okq = 1;
          if (lane == 0) {
            if (qn[t] > 0) okq = mbar_wait(q_empty + t, (qn[t] - 1) & 1, abort);
            if (okq) {
              const int z = it.q0 + (it.row00 + t * kM) / p.g;
              mbar_arrive_expect_tx(q_full(t), (uint32_t)kQTile);
#pragma unroll
              for (int h = 0; h < C::kHalves; ++h)
                tma_load_3d(base + t * kQTile + h * kQHalf, &qmap, q_full(t), 64 * h, it.kvh * p.g, z,
                            policy_evict_first());
              ++qn[t];
            }
          }
          return __shfl_sync(0xffffffffu, okq, 0) != 0;
        };
        if (kv == 0) {
          if (!load_q(0)) {
            ok = false;
            break;
          }
        }
        const int32_t* row = p.block_tables + (size_t)it.s * p.max_blocks_per_seq;
        const int nblk = (it.t_end + p.B - 1) / p.B;
        int cur = load_block_id(row, lane, nblk);
        int nxt = load_block_id(row, 32 + lane, nblk);
        int wbase = 0;
        for (int c = 0; c < it.nch; ++c, ++k) {
          const int jb = c * bpc;
          if (jb >= wbase + 32) {
            cur = nxt;
            wbase += 32;
            nxt = load_block_id(row, wbase + 32 + lane, nblk);
          }
          int id = __shfl_sync(0xffffffffu, cur, (jb - wbase + lane) & 31);
          const int nb = (min(kN, it.t_end - c * kN) + p.B - 1) / p.B;
          if (lane < nb && (unsigned)id >= (unsigned)p.num_blocks) {
            raise_status(p.status, PA_STATUS_BAD_BLOCK);
            id = 0;
          }
          // The append kernel writes only the slots of the new tokens
          // (positions first_pos and later): chunks of older tokens are
          // read before waiting for it, the first chunk that holds a new
          // token after (griddepcontrol.wait).
          if (!waited && (c + 1) * kN > it.first_pos) {
            pdl_wait_primary();
            waited = true;
          }
          const int st = (int)(k % (uint32_t)stages);
          // A chunk of values whose last block runs past the sequence's end
          // (stage rows z0 .. z1 - 1): its copies signal v_land instead, the
          // rows past the end are cleared once they have landed, and a plain
          // arrival then releases the chunk to the MMA warps.
          const int z0 = it.ctx - c * kN, z1 = nb * p.B;
          const bool clear = kv == 1 && z0 < z1;
          uint64_t* land = clear ? v_land : &fulls[st];
          int okc = 1;
          // (test hook: the key warp never issues its CTA's chunk number
          // `withhold`, so that the waits for it run out)
          const bool issue = !(kv == 0 && k == (uint32_t)withhold);
          if (lane == 0) {
            okc = mbar_wait(&empties[st], ((k / stages) & 1) ^ 1, abort);
            if (okc && issue) mbar_arrive_expect_tx(land, (uint32_t)(nb * p.B * 128 * C::kHalves));
          }
          if (!__shfl_sync(0xffffffffu, okc, 0)) {
            ok = false;
            break;
          }
          __syncwarp();  // the expected byte count is set before any copy can land
          if (issue && lane < nb) {  // block `lane` of the chunk: one box of B rows, both halves
            const int grp = (id * p.Hkv + it.kvh) * (p.B / 8);
            uint8_t* d = base + (kv == 0 ? kOffK : kOffV) + st * kKVStage + lane * p.B * 128 * C::kHalves;
            tma_load_4d(d, map, land, 0, 0, 0, grp, policy);
          }
          if (kv == 0 && c == 0 && !load_q(1)) {
            ok = false;
            ++k;  // chunk 0's keys were issued
            break;
          }
          if (clear) {
            int okl = 1;
            if (lane == 0) okl = mbar_wait(v_land, vl & 1, abort);
            ++vl;
            if (!__shfl_sync(0xffffffffu, okl, 0)) {
              ok = false;
              landing = true;
              break;
            }
            uint8_t* vs = base + kOffV + st * kKVStage;
            const int units = (z1 - z0) * 8;  // 16-byte units past the end, per 64-dim half
            for (int u = lane; u < units * C::kHalves; u += 32) {
              const int h = u / units, rem = u % units;
              *reinterpret_cast<uint4*>(vs + kv_row_offset<C::kHalves>(z0 + rem / 8, h) + (rem % 8) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();  // the zeros before the tensor cores' reads
            __syncwarp();
            if (lane == 0) mbar_arrive(&fulls[st]);
          }
        }
      }
      if (!ok) {
        if (lane == 0) {
          *abort = 1;
          raise_status(p.status, PA_STATUS_TIMEOUT);
          // Let copies already issued land before the CTA's shared memory goes away.
          const volatile int never = 0;
          for (uint32_t c = (k > (uint32_t)stages ? k - stages : 0); c < k; ++c)
            mbar_wait(&fulls[c % stages], (c / stages) & 1, &never);
          if (landing) mbar_wait(v_land, (vl - 1) & 1, &never);
          for (int t = 0; t < kTiles; ++t)
            if (qn[t] > 0) mbar_wait(q_full(t), (qn[t] - 1) & 1, &never);
        }
        __syncwarp();
      }
      // Every CTA waits for the append before it completes, even one whose
      // items held no new token: a batch split over several launches makes
      // each launch the next one's primary, and that launch's
      // griddepcontrol.wait stands for the append only if this one's
      // completion implies the append's.
      if (!waited) pdl_wait_primary();
    } else {
      // MMA warp of tile t: its lane 0 alone issues the tile's MMAs in a
      // fixed order, waiting for one barrier at a time: per item S(0) and
      // S(1) into the two buffers, then per step u P·V(u) as soon as P(u)
      // is in and right behind it S(u + 2) into the same buffer.  The other
      // lanes have nothing to do: a warp-wide synchronisation right after a
      // group of MMAs waited for the group to be taken by the tensor cores,
      // several hundred cycles on the tile's critical path.  Each tile has
      // its own issuing thread and the tensor cores interleave the two
      // tiles' work.  The tile's MMAs run in issue order: S(u + 2)
      // overwrites P(u) only after P·V(u) has read it.  The commit after
      // P·V(u) and S(u + 2) goes to the buffer's barrier: the softmax takes
      // it before step u + 2 (or, to rescale O, at step u + 1).  Each buffer
      // has its own P barrier: P(u + 2) can only arrive after this commit,
      // which the thread issues after it has taken P(u), so no barrier runs
      // two phases ahead of its waiter.  The first P·V of an item
      // overwrites O without a barrier of its own: it waits for P(0), which
      // the warpgroup writes only after it has read the previous item's O.
      // Value rows past the pair's keys need no clearing here: their
      // weights are exact zeros and the rows hold finite values (see the
      // value producer).
      if (lane == 0) {
        const int t = warp - kMmaWarp;
        const uint32_t id_s = instr_desc(kM, kSub, false);
        const uint32_t id_o = instr_desc(kM, DH, true);
        bool ok = true;
        auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
          ok = ok && mbar_spin(bar, parity, abort);
          return ok;
        };
        // Descriptors are built once per group; a k-step adds its byte offset
        // / 16 to the address field (every shared address is below 256 KB, so
        // the 14-bit field never carries).
        const uint64_t a_q = smem_desc(sbase + t * kQTile, 16, 1024);
        const uint32_t s_base = tmem + kColS + (uint32_t)t * 128;  // S buffer b at s_base + kSub·b
        const uint32_t o_cols = tmem + kColO + (uint32_t)t * DH;
        // S of keys kSub·h .. kSub·h + kSub - 1 of the stage kst into buffer b
        auto issue_s = [&](int kst, int h, int b) {
          tc_fence_after();
          // keys: K-major, 8-row groups kHalves KB apart, halves 1 KB apart
          const uint64_t b0 = smem_desc(sbase + kOffK + kst * kKVStage + h * (kSub / 8) * C::kHalves * 1024, 16,
                                        C::kHalves * 1024);
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk) {
            const int hlf = kk >> 2, w = kk & 3;
            mma_ss(s_base + kSub * b, a_q + (uint64_t)((hlf * kQHalf + w * 32) >> 4),
                   b0 + (uint64_t)((hlf * 1024 + w * 32) >> 4), id_s, kk > 0);
          }
        };
        // O += P(buffer b) · (values kSub·h .. of the stage vst)
        auto issue_pv = [&](int vst, int h, int b, bool acc) {
          tc_fence_after();
          // values: MN-major, the dims' halves 1 KB apart, 8-key groups
          // kHalves KB apart; a K-step of 16 keys is two groups
          const uint64_t b0 = smem_desc(sbase + kOffV + vst * kKVStage, 1024, C::kHalves * 1024);
#pragma unroll
          for (int kk = 0; kk < kSub / 16; ++kk)
            mma_ts(o_cols, s_base + kSub * b + kk * 8,
                   b0 + (uint64_t)((((kSub / 16) * h + kk) * 2 * C::kHalves * 1024) >> 4), id_o, acc || kk > 0);
        };
        uint32_t kq = 0, spc[2] = {0, 0}, nit = 0;  // chunks of keys (and values) before the item, P phases per buffer, items
        for (int r = 0; ok; ++r) {
          const int j = (r < *my_count ? my_items[r] : -1);
          if (j < 0) break;
          const PfItem it = pf_item(p, j, pairs);
          if (it.state) continue;
          const int ns = it.nsub;
          if (!wait_bar(q_full(t), nit & 1)) break;
          if (!wait_bar(&full_k[kq % kStagesK], (kq / kStagesK) & 1)) break;
          issue_s((int)(kq % kStagesK), 0, 0);
          mma_commit(s_full(t, 0));
          if (ns > 1) {
            issue_s((int)(kq % kStagesK), 1, 1);
            mma_commit(s_full(t, 1));
          }
          for (int u = 0; u < ns; ++u) {
            const int b = u & 1;
            const uint32_t vc = kq + (u >> 1);        // chunk of values of step u
            const uint32_t kc = kq + ((u + 2) >> 1);  // chunk of keys of step u + 2
            const bool more = u + 2 < ns;
            if (b == 0 && !wait_bar(&full_v[vc % kStagesV], (vc / kStagesV) & 1)) break;
            // The keys S(u + 2) reads are awaited before P(u) and before any
            // MMA: P·V(u) and S(u + 2) then go out back to back (a barrier
            // test right after a group of MMAs waits for the group to be
            // taken).
            if (more && b == 0 && !wait_bar(&full_k[kc % kStagesK], (kc / kStagesK) & 1)) break;
            if (!wait_bar(p_full(t, b), spc[b] & 1)) break;
            ++spc[b];
            issue_pv((int)(vc % kStagesV), b, b, u > 0);
            if (more) issue_s((int)(kc % kStagesK), b, b);  // into the buffer P·V(u) has just read
            mma_commit(s_full(t, b));  // P·V(u) and S(u + 2) are done
          }
          kq += (uint32_t)it.nch;
          ++nit;
        }
        if (!ok) {
          *abort = 1;
          raise_status(p.status, PA_STATUS_TIMEOUT);
        }
        // Every MMA this thread issued has completed before tensor memory is released.
        mma_commit(drained + t);
        const volatile int never = 0;
        mbar_wait(drained + t, 0, &never);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoft));
    // softmax warpgroup t: thread lt owns row lt of its tile (tensor-memory lane lt)
    const int t = warp / kSoftWarps, lt = tid - t * kM;
    const uint32_t lane_base = tmem + ((uint32_t)((warp % kSoftWarps) * 32) << 16);
    const uint32_t o_cols = lane_base + kColO + (uint32_t)t * DH;
    const uint32_t s_base = lane_base + kColS + (uint32_t)t * 128;  // S buffer b at s_base + kSub·b
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    // Phases consumed per S buffer, chunks of keys (and values) before the
    // item, items finished, tiles staged for a TMA store.
    uint32_t sfc[2] = {0, 0}, ch = 0, done = 0, nstaged = 0;
    bool ok = true;
    // Commit C(v) of an item of ns steps is the MMA thread's commit into
    // buffer v % 2 that follows S(v) (v = 0, 1) or P·V(v - 2) and, for
    // v < ns, S(v); once it is taken, every MMA issued before it is done.
    // The warp waits together (warp-wide tensor-memory accesses follow).
    // After P·V of the second step of a chunk (or the item's last) the
    // chunk's values are free as far as this tile is concerned.
    auto take = [&](int v, int ns) {
      const bool w = __all_sync(0xffffffffu, mbar_wait(s_full(t, v & 1), sfc[v & 1] & 1, abort));
      ++sfc[v & 1];
      tc_fence_after();
      const int pw = v - 2;
      if (lt == 0 && pw >= 0 && ((pw & 1) || pw == ns - 1)) mbar_arrive(&empty_v[(ch + (pw >> 1)) % kStagesV]);
      return w;
    };
    for (int r = 0; ok; ++r) {
      const int j = (r < *my_count ? my_items[r] : -1);
      if (j < 0) break;
      const PfItem it = pf_item(p, j, pairs);
      if (it.state == 2) {
        if (t == 0 && lt == 0 && it.pair == 0 && it.kvh == 0) raise_status(p.status, PA_STATUS_BAD_CONTEXT);
        continue;
      }
      if (it.state) continue;
      const int ns = it.nsub;  // both tiles attend every step of the item
      const int row0 = it.row00 + t * kM;
      const int rr = row0 + lt;
      const int pos = rr < it.rows ? it.first_pos + rr / p.g : -1;  // keys 0 .. pos
      float m_run = -INFINITY, l_run = 0.f;
      bool ahead = false;  // the previous step has taken this step's commit
      for (int u = 0; u < ns; ++u) {
        const int b = u & 1;
        if (!ahead && !take(u, ns)) {  // S(u) is in
          ok = false;
          break;
        }
        ahead = false;
        // S(u) is done: after the second step of a chunk (or the item's
        // last) its keys are free as far as this tile is concerned, and
        // after the item's last S its query tile.
        if (lt == 0) {
          if (b == 1 || u + 1 == ns) mbar_arrive(&empty_k[(ch + (u >> 1)) % kStagesK]);
          if (u + 1 == ns) mbar_arrive(q_empty + t);
        }
        const uint32_t s_cols = s_base + kSub * b;
        uint32_t raw[kSub];
#pragma unroll
        for (int i = 0; i < kSub / 16; ++i) tmem_ld16_nowait(s_cols + 16 * i, raw + 16 * i);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        float sc[kSub];
#pragma unroll
        for (int q = 0; q < kSub; ++q) sc[q] = __uint_as_float(raw[q]);
        // Keys t0 .. t0 + nvalid - 1 of this step are at or before the row's
        // position; masking is needed only in steps that cross it.
        const int t0 = u * kSub;
        const int nvalid = min(kSub, pos - t0 + 1);
        if (nvalid < kSub) {
#pragma unroll
          for (int q = 0; q < kSub; ++q) sc[q] = q < nvalid ? sc[q] : -INFINITY;
        }
        // max of the raw (unscaled) scores: three-input max, four chains
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < kSub / 2; ++q) m4[q & 3] = fmax3(m4[q & 3], sc[2 * q], sc[2 * q + 1]);
        const float mxr = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        const float mx = mxr * p.scale_log2;  // scale > 0: the max of the scaled scores
        // Raise the running max (and rescale O) only when it grows past the
        // threshold; the decision is made per warp because tensor-memory
        // loads and stores are warp-wide.
        const bool grow = mx > m_run + kRescaleLog2 || (m_run == -INFINITY && mx != -INFINITY);
        const bool rescale = grow && m_run != -INFINITY;  // O holds products to scale
        const float m_new = grow ? mx : m_run;
        const float alpha = grow ? exp2f(m_run - m_new) : 1.f;  // m_run = -inf: alpha 0
        const float base_m = m_new == -INFINITY ? 0.f : m_new;
        const float2 nb2 = make_float2(-base_m, -base_m);
        float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < kSub / 32; ++i) {  // exp2(s * scale - max): one packed FMA per two scores
          uint32_t w[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float2 x = __ffma2_rn(make_float2(sc[32 * i + 2 * q], sc[32 * i + 2 * q + 1]), sl2, nb2);
            const float2 e = make_float2(ex2_ftz(x.x), ex2_ftz(x.y));
            l2[q & 1] = __fadd2_rn(l2[q & 1], e);
            w[q] = pack_bf16x2(e.x, e.y);
          }
          tmem_st16(s_cols + 16 * i, w);  // P over the first kSub / 2 columns of its buffer
        }
        l_run = l_run * alpha + ((l2[0].x + l2[0].y) + (l2[1].x + l2[1].y));
        m_run = m_new;
        // tcgen05.st and its wait are warp-wide: once the wait returns, the
        // warp's P is in tensor memory.
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        if (u > 0 && __any_sync(0xffffffffu, rescale)) {
          // O must hold every product before this step's before it is
          // rescaled: P·V(u - 1) is covered by C(u + 1), which the next step
          // would wait for anyway.  The next P·V waits for this step's P.
          if (!take(u + 1, ns)) {
            ok = false;
            break;
          }
          ahead = true;
#pragma unroll 1
          for (int i = 0; i < DH / 16; ++i) {
            float v[16];
            tmem_ld16(o_cols + 16 * i, v);
            uint32_t w[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) w[q] = __float_as_uint(v[q] * alpha);
            tmem_st16(o_cols + 16 * i, w);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(p_full(t, b));  // one arrival speaks for the warp
        }
      }
      if (!ok) break;
      // The item's last P·V is covered by C(ns + 1), which follows C(ns)
      // (there is none for a single step).
      if ((ns > 1 && !ahead && !take(ns, ns)) || !take(ns + 1, ns)) {
        ok = false;
        break;
      }
      ch += (uint32_t)it.nch;
      // Read the row of O (all loads in flight at once).  The next item's
      // first P·V overwrites it only after this warpgroup's next P(0),
      // which comes after these loads have completed.
      uint32_t o[DH];
#pragma unroll
      for (int i = 0; i < DH / 16; ++i) tmem_ld16_nowait(o_cols + 16 * i, o + 16 * i);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      tc_fence_before();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      uint32_t w[DH / 2];  // the row normalized, as bf16 pairs; piece k (32 bytes) is w[8k .. 8k + 7]
#pragma unroll
      for (int q = 0; q < DH / 2; ++q)
        w[q] = pack_bf16x2(__uint_as_float(o[2 * q]) * inv, __uint_as_float(o[2 * q + 1]) * inv);
      auto row_out = [&](int row) {  // the output row of query row `row` of the pair
        return static_cast<__nv_bfloat16*>(p.out) +
               ((size_t)(it.q0 + row / p.g) * p.H + it.kvh * p.g + row % p.g) * DH;
      };
      // A tile whose 128 rows are all query rows is staged in shared memory
      // (the layout its query tile had) and written by two TMA stores, one
      // per 64-dim half, so that the warpgroup is free within a few hundred
      // cycles; the two tiles have one staging buffer and take turns
      // (tile 0 of an item, tile 1, tile 0 of the next item, ...), turn k
      // waiting for the end of turn k - 1.  Other tiles (a sequence's last)
      // store their rows directly.
      // Every wait here is a bounded mbarrier wait, each warp its own: a
      // warp that gave up earlier (a time-out) never leaves the others
      // waiting without a limit.  They spin rather than suspend in
      // try_wait, which resumed several hundred cycles late here.  The
      // turn passes on only once all four warps have taken it (their
      // arrivals on `staged`), so no warp's parity test can meet a later
      // turn's phase.
      const uint32_t turn = 2 * done + (uint32_t)t;
      ++done;
      if (!__all_sync(0xffffffffu, turn == 0 || mbar_spin(out_free, (turn - 1) & 1, abort))) {
        ok = false;
        break;
      }
      const bool full = row0 + kM <= it.rows;
      uint8_t* stage = base + C::kOffOut;
      if (full) {
#pragma unroll
        for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(stage + h * kQHalf + lt * 128 + ((u ^ (lt & 7)) << 4)) =
                make_uint4(w[32 * h + 4 * u], w[32 * h + 4 * u + 1], w[32 * h + 4 * u + 2], w[32 * h + 4 * u + 3]);
        fence_proxy_async_smem();  // the rows before the TMA unit reads them
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(staged + t);  // one arrival speaks for the warp
      int staged_ok = 1;
      if (lt == 0) {
        staged_ok = mbar_spin(staged + t, nstaged & 1, abort);
        if (staged_ok) {
          if (full) {
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h)
              tma_store_3d(&omap, stage + h * kQHalf, 64 * h, it.kvh * p.g, it.q0 + row0 / p.g);
            bulk_store_drain();  // the buffer has been read
          }
          mbar_arrive(out_free);
        }
      }
      // the first warp of the tile leaves together (warp-wide shuffles follow)
      if (warp % kSoftWarps == 0 && !__shfl_sync(0xffffffffu, staged_ok, 0)) {
        ok = false;
        break;
      }
      ++nstaged;
      if (!full) {
        if ((reinterpret_cast<uintptr_t>(p.out) & 31) == 0) {
          // The four lanes of a quad trade pieces (a 4 x 4 transpose of
          // 32-byte pieces per 128 bytes of row, two rounds of xor shuffles):
          // lane j then holds piece 4h + j of each of the quad's four rows,
          // so that each store of the warp writes eight whole 128-byte lines
          // instead of 32 pieces of 32 lines.
          const int jq = lane & 3;
#pragma unroll
          for (int h = 0; h < DH / 64; ++h) {
            uint32_t* x = w + 32 * h;
#pragma unroll
            for (int m = 1; m <= 2; m <<= 1) {
              const bool hi = (jq & m) != 0;
#pragma unroll
              for (int sl = 0; sl < 4; ++sl) {
                if (sl & m) continue;  // the pair of pieces (sl, sl + m)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const uint32_t got = __shfl_xor_sync(0xffffffffu, hi ? x[8 * sl + e] : x[8 * (sl + m) + e], m);
                  if (hi)
                    x[8 * sl + e] = got;
                  else
                    x[8 * (sl + m) + e] = got;
                }
              }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rq = rr - jq + i;  // row i of the quad
              if (rq < it.rows) st_global_v8(row_out(rq) + 16 * (4 * h + jq), x + 8 * i);
            }
          }
        } else if (rr < it.rows) {  // 16-byte stores of the thread's own row
          __nv_bfloat16* dst = row_out(rr);
#pragma unroll
          for (int u = 0; u < DH / 8; ++u)
            reinterpret_cast<uint4*>(dst)[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
    }
    // The stores issued by TMA are complete before the kernel ends.
    if (lt == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    if (!ok) {
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

// Test hooks: a smaller bound on the items of one launch, 0 for none
// (pa_prefill_test_items_per_launch); the key chunk every CTA withholds,
// -1 for none (pa_prefill_test_withhold).
std::atomic<int> g_items_per_launch{0};
std::atomic<int> g_withhold{-1};

template <int DH>
cudaError_t launch_prefill_tc_dh(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const CUtensorMap& qmap, const CUtensorMap& omap, int pairs, cudaStream_t stream) {
  constexpr size_t kBytes = PfCfg<DH>::kBytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static int sms[64];
  static std::once_flag once[64];
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t init_err = cudaSuccess;
  std::call_once(once[dev], [&] {
    init_err = cudaFuncSetAttribute(prefill_tc_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBytes);
    if (init_err == cudaSuccess) init_err = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    // The kernel's register split assumes kRegsLaunch registers a thread at
    // launch: with fewer, its setmaxnreg.inc could never be granted.
    cudaFuncAttributes fa{};
    if (init_err == cudaSuccess) init_err = cudaFuncGetAttributes(&fa, prefill_tc_kernel<DH>);
    if (init_err == cudaSuccess && fa.numRegs != kRegsLaunch) init_err = cudaErrorInvalidConfiguration;
  });
  if (init_err != cudaSuccess) return init_err;
  if (sms[dev] < 1) return cudaErrorInvalidConfiguration;
  // Persistent CTAs, one per SM (the shared memory allows no more), each
  // listing at most kListCap items: a larger batch takes several launches,
  // each over a contiguous range of the items.
  const long long items = (long long)a.S * a.Hkv * pairs;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  long long per_launch = (long long)kListCap * sms[dev];
  const int cap = g_items_per_launch.load(std::memory_order_relaxed);
  const int withhold = g_withhold.load(std::memory_order_relaxed);
  if (cap > 0) per_launch = std::min<long long>(per_launch, cap);
  for (long long first = 0; first < items; first += per_launch) {
    const long long n = std::min(per_launch, items - first);
    const int grid = (int)std::min<long long>(n, sms[dev]);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreadsT);
    cfg.dynamicSmemBytes = kBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel<DH>, kmap, vmap, qmap, omap, a, pairs, (int)first, (int)n,
                           withhold);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                              const CUtensorMap& qmap, const CUtensorMap& omap, cudaStream_t stream) {
  const int tiles = (a.max_query_len * a.g + kM - 1) / kM;
  const int pairs = (tiles + kTiles - 1) / kTiles;
  if (tiles <= 0 || a.S <= 0) return cudaSuccess;
  if (a.D == 128) return launch_prefill_tc_dh<128>(a, kmap, vmap, qmap, omap, pairs, stream);
  if (a.D == 64) return launch_prefill_tc_dh<64>(a, kmap, vmap, qmap, omap, pairs, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa

extern "C" int pa_prefill_test_items_per_launch(int items_per_launch) {
  if (items_per_launch < 0) return pa_fail(PA_ERR_INVALID, "pa_prefill_test_items_per_launch: negative");
  pa::g_items_per_launch.store(items_per_launch, std::memory_order_relaxed);
  return PA_OK;
}

extern "C" int pa_prefill_test_withhold(int chunk) {
  if (chunk < -1) return pa_fail(PA_ERR_INVALID, "pa_prefill_test_withhold: chunk < -1");
  pa::g_withhold.store(chunk, std::memory_order_relaxed);
  return PA_OK;
}
