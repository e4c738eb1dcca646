// Host block allocator of the paged KV cache: free list, ref-counted prefix
// sharing and copy-on-write at the divergence block.
//
// "Day 6/90 of Inference Engineering" (bittide.aicompass.dev), notes on
// PagedAttention: paragraph 2 (one block at a time; a new block only when the
// last is full), paragraph 5 (shared prefix blocks; a new block where the
// sequences diverge), paragraph 6 (per-sequence block table).  The free list
// is a stack (first pop = free_order[0]; freed blocks pushed on top, in table
// order); every failing call leaves the state unchanged.

#include <cstdint>
#include <cstring>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "pa.h"
#include "pa_internal.h"

struct pa_alloc {
  struct Seq {
    std::vector<int32_t> blocks;
    int64_t tokens = 0;
    uint64_t stamp = 0;  // batch that last touched the sequence
  };
  uint64_t batch = 0;
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> free_stack;  // top = back()
  std::vector<int32_t> ref;
  std::unordered_map<int64_t, Seq> seqs;

  int32_t pop() {
    int32_t b = free_stack.back();
    free_stack.pop_back();
    ref[b] = 1;
    return b;
  }
  // Blocks an append to `s` would take: a new one if the last is full (or
  // there is none), a copy if the last is partly filled and shared.
  int append_needs(const Seq& s) const {
    if (s.tokens % block_size == 0) return 1;
    return ref[s.blocks.back()] > 1 ? 1 : 0;
  }
  // Caller has checked append_needs() <= free blocks.
  void append(Seq& s, int64_t* slot, int32_t* src, int32_t* dst, bool* table_changed) {
    int64_t r = s.tokens % block_size;
    *src = -1;
    *dst = -1;
    *table_changed = false;
    if (r == 0) {
      s.blocks.push_back(pop());
      *table_changed = true;
    } else {
      int32_t last = s.blocks.back();
      if (ref[last] > 1) {
        int32_t fresh = pop();
        ref[last] -= 1;
        s.blocks.back() = fresh;
        *src = last;
        *dst = fresh;
        *table_changed = true;
      }
    }
    s.tokens += 1;
    *slot = (int64_t)s.blocks.back() * block_size + r;
  }
};

extern "C" {

int pa_alloc_create(int num_blocks, int block_size, const int32_t* free_order, pa_alloc** out) {
  if (!out || num_blocks < 0 || block_size <= 0) return pa_fail(PA_ERR_INVALID, "pa_alloc_create: bad arguments");
  pa_alloc* a = new (std::nothrow) pa_alloc();
  if (!a) return pa_fail(PA_ERR_OOM, "pa_alloc_create: host allocation failed");
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->ref.assign(num_blocks, 0);
  a->free_stack.resize(num_blocks);
  std::vector<char> seen(num_blocks, 0);
  for (int i = 0; i < num_blocks; ++i) {
    int32_t b = free_order ? free_order[i] : i;
    if (b < 0 || b >= num_blocks || seen[b]) {
      delete a;
      return pa_fail(PA_ERR_INVALID, "pa_alloc_create: free_order is not a permutation");
    }
    seen[b] = 1;
    a->free_stack[num_blocks - 1 - i] = b;  // first pop returns free_order[0]
  }
  *out = a;
  return PA_OK;
}

void pa_alloc_destroy(pa_alloc* a) { delete a; }

int pa_alloc_num_free(const pa_alloc* a) {
  if (!a) return pa_fail(PA_ERR_INVALID, "null allocator");
  return (int)a->free_stack.size();
}

int pa_seq_add(pa_alloc* a, int64_t seq_id, int num_tokens) {
  if (!a || num_tokens < 0) return pa_fail(PA_ERR_INVALID, "pa_seq_add: bad arguments");
  if (a->seqs.count(seq_id)) return pa_fail(PA_ERR_STATE, "pa_seq_add: sequence exists");
  int64_t need = ((int64_t)num_tokens + a->block_size - 1) / a->block_size;
  if (need > (int64_t)a->free_stack.size()) return pa_fail(PA_ERR_OOM, "pa_seq_add: out of blocks");
  pa_alloc::Seq s;
  s.tokens = num_tokens;
  s.blocks.reserve(need);
  for (int64_t i = 0; i < need; ++i) s.blocks.push_back(a->pop());
  a->seqs.emplace(seq_id, std::move(s));
  return PA_OK;
}

int pa_seq_fork(pa_alloc* a, int64_t parent_id, int64_t child_id) {
  if (!a) return pa_fail(PA_ERR_INVALID, "null allocator");
  auto it = a->seqs.find(parent_id);
  if (it == a->seqs.end()) return pa_fail(PA_ERR_STATE, "pa_seq_fork: unknown parent");
  if (a->seqs.count(child_id)) return pa_fail(PA_ERR_STATE, "pa_seq_fork: child exists");
  pa_alloc::Seq child = it->second;
  for (int32_t b : child.blocks) a->ref[b] += 1;
  a->seqs.emplace(child_id, std::move(child));
  return PA_OK;
}

int pa_seq_append_slot(pa_alloc* a, int64_t seq_id, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
  if (!a || !slot || !cow_src || !cow_dst) return pa_fail(PA_ERR_INVALID, "pa_seq_append_slot: null argument");
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return pa_fail(PA_ERR_STATE, "pa_seq_append_slot: unknown sequence");
  if (a->append_needs(it->second) > (int)a->free_stack.size())
    return pa_fail(PA_ERR_OOM, "pa_seq_append_slot: out of blocks");
  bool changed;
  a->append(it->second, slot, cow_src, cow_dst, &changed);
  return PA_OK;
}

int pa_seq_free(pa_alloc* a, int64_t seq_id) {
  if (!a) return pa_fail(PA_ERR_INVALID, "null allocator");
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return pa_fail(PA_ERR_STATE, "pa_seq_free: unknown sequence");
  for (int32_t b : it->second.blocks) {
    if (a->ref[b] <= 0) return pa_fail(PA_ERR_STATE, "pa_seq_free: refcount underflow");
  }
  for (int32_t b : it->second.blocks) {
    if (--a->ref[b] == 0) a->free_stack.push_back(b);
  }
  a->seqs.erase(it);
  return PA_OK;
}

int pa_seq_num_tokens(const pa_alloc* a, int64_t seq_id) {
  if (!a) return pa_fail(PA_ERR_INVALID, "null allocator");
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return pa_fail(PA_ERR_STATE, "pa_seq_num_tokens: unknown sequence");
  return (int)it->second.tokens;
}

int pa_seq_block_table(const pa_alloc* a, int64_t seq_id, int32_t* out, int cap, int* n_out) {
  if (!a || !n_out || cap < 0 || (cap > 0 && !out)) return pa_fail(PA_ERR_INVALID, "pa_seq_block_table: bad arguments");
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return pa_fail(PA_ERR_STATE, "pa_seq_block_table: unknown sequence");
  const auto& t = it->second.blocks;
  *n_out = (int)t.size();
  if ((int)t.size() > cap) return pa_fail(PA_ERR_INVALID, "pa_seq_block_table: capacity too small");
  if (!t.empty()) std::memcpy(out, t.data(), t.size() * sizeof(int32_t));
  return PA_OK;
}

int pa_block_refcount(const pa_alloc* a, int block_id) {
  if (!a || block_id < 0 || block_id >= a->num_blocks) return pa_fail(PA_ERR_INVALID, "pa_block_refcount: bad block");
  return a->ref[block_id];
}

int pa_seqs_append_slots(pa_alloc* a, const int64_t* seq_ids, int n, int64_t* slot_mapping,
                         int32_t* cow_pairs, int* num_cow, int32_t* block_tables, int width,
                         int32_t* context_lens) {
  if (!a || n < 0 || (n > 0 && (!seq_ids || !slot_mapping || !cow_pairs)) || !num_cow ||
      (block_tables && width <= 0))
    return pa_fail(PA_ERR_INVALID, "pa_seqs_append_slots: bad arguments");
  // Validate the whole batch first so that a failure changes nothing.
  std::vector<pa_alloc::Seq*> ss(n);
  int64_t need = 0;
  for (int i = 0; i < n; ++i) {
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end()) return pa_fail(PA_ERR_STATE, "pa_seqs_append_slots: unknown sequence");
    ss[i] = &it->second;
    if (block_tables) {
      int64_t nb = (it->second.tokens + 1 + a->block_size - 1) / a->block_size;
      if (nb > width) return pa_fail(PA_ERR_INVALID, "pa_seqs_append_slots: table width too small");
    }
  }
  const uint64_t stamp = ++a->batch;
  for (int i = 0; i < n; ++i) {
    if (ss[i]->stamp == stamp) return pa_fail(PA_ERR_INVALID, "pa_seqs_append_slots: repeated sequence");
    ss[i]->stamp = stamp;
  }
  for (int i = 0; i < n; ++i) need += a->append_needs(*ss[i]);
  if (need > (int64_t)a->free_stack.size()) return pa_fail(PA_ERR_OOM, "pa_seqs_append_slots: out of blocks");
  // A copy-on-write inside the batch can only lower later needs (it drops a
  // reference), so the check above covers the whole batch.
  int nc = 0;
  for (int i = 0; i < n; ++i) {
    int32_t src, dst;
    bool changed;
    a->append(*ss[i], &slot_mapping[i], &src, &dst, &changed);
    if (src >= 0) {
      cow_pairs[2 * nc] = src;
      cow_pairs[2 * nc + 1] = dst;
      ++nc;
    }
    if (block_tables && changed) {
      size_t j = ss[i]->blocks.size() - 1;
      block_tables[(size_t)i * width + j] = ss[i]->blocks[j];
    }
    if (context_lens) context_lens[i] = (int32_t)ss[i]->tokens;
  }
  *num_cow = nc;
  return PA_OK;
}

int pa_seqs_block_tables(const pa_alloc* a, const int64_t* seq_ids, int n, int32_t* block_tables,
                         int width, int32_t* context_lens) {
  if (!a || n < 0 || width <= 0 || (n > 0 && (!seq_ids || !block_tables)))
    return pa_fail(PA_ERR_INVALID, "pa_seqs_block_tables: bad arguments");
  std::vector<const pa_alloc::Seq*> ss(n);
  for (int i = 0; i < n; ++i) {
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end()) return pa_fail(PA_ERR_STATE, "pa_seqs_block_tables: unknown sequence");
    if ((int64_t)it->second.blocks.size() > width) return pa_fail(PA_ERR_INVALID, "pa_seqs_block_tables: table width too small");
    ss[i] = &it->second;
  }
  for (int i = 0; i < n; ++i) {
    int32_t* row = block_tables + (size_t)i * width;
    const auto& t = ss[i]->blocks;
    for (int j = 0; j < width; ++j) row[j] = j < (int)t.size() ? t[j] : -1;
    if (context_lens) context_lens[i] = (int32_t)ss[i]->tokens;
  }
  return PA_OK;
}

}  // extern "C"
