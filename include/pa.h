/*
 * pa.h -- C ABI of the paged KV cache library (libpa.so): KV append, paged
 * decode attention with split-K and log-sum-exp merge, block copy for
 * copy-on-write, and a host-side block allocator.
 *
 * Sources (web pages on paged KV caches):
 *   [Day6]  "Day 6/90 of Inference Engineering" (post on
 *           bittide.aicompass.dev), notes on PagedAttention: paragraph 2
 *           (the cache manager hands out one fixed-size block at a time, a
 *           new one when the last is full), paragraph 5 (a shared prefix
 *           shares blocks; a diverging sequence writes to a new block),
 *           paragraph 6 (the block table makes scattered blocks read as a
 *           contiguous KV cache).
 *   [PAK]   "PagedAttention Kernel：大模型推理优化的显存管理革新"
 *           (intelliparadigm.com), section 3.1 (Q·Kᵀ by blocks, softmax,
 *           P·V by blocks) and section 2.2 (prefetch the next page while
 *           computing the current one).
 *
 * Conventions for every entry point
 *   - Pointers named "device" are CUDA device pointers owned by the caller;
 *     the library never allocates, frees or retains them.  Pointers named
 *     "host" are ordinary host memory, also caller-owned.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and is asynchronous: the call returns once the kernels are
 *     launched.  Buffers must stay valid until the stream reaches that point.
 *   - Return value: PA_OK (0) or a negative PA_ERR_* code.  On error nothing
 *     was launched and no buffer was touched; pa_last_error() describes it.
 *   - Host-visible arguments are validated before any launch.  Arguments
 *     that live on the device (slots, block ids, context lengths) are
 *     checked in the kernels: an out-of-range value skips the access and
 *     sets a bit in the device status word (pa_get_status), never faults.
 *
 * Cache layout (the pages give none; this library's choice):
 *   k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim],
 *   row-major, element type `dtype`.  Token t of a sequence lives in
 *   physical block block_tables[seq][t / block_size], row t % block_size.
 *   Slot s = block * block_size + row.
 *
 * Supported set: dtype PA_BF16 or PA_F32 (PA_FP8_E4M3 caches through the
 * _fp8 entry points, head_dim 128); head_dim 64 or 128; block_size 8,
 * 16 or 32; g = num_heads / num_kv_heads in {1, 2, 4, 8}.  Anything else
 * returns PA_ERR_UNSUPPORTED.  Decode in bf16 runs on tensor cores with fp32
 * accumulation; fp32 decode runs on CUDA cores in fp32.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define PA_OK 0
#define PA_ERR_INVALID (-1)     /* bad argument (null pointer, size, range) */
#define PA_ERR_UNSUPPORTED (-2) /* valid but outside the supported set */
#define PA_ERR_OOM (-3)         /* allocator: not enough free blocks */
#define PA_ERR_STATE (-4)       /* allocator: unknown or duplicate sequence */
#define PA_ERR_CUDA (-5)        /* a CUDA runtime call failed */

/* Element types of q, k, v, caches and out (all the same in one call). */
#define PA_F32 0
#define PA_BF16 1
/* E4M3 8-bit floats (caches only; q, k, v inputs and out are then bf16). */
#define PA_FP8_E4M3 2

/* Bits of the device status word. */
#define PA_STATUS_BAD_SLOT 1u    /* append: slot >= num_blocks*block_size */
#define PA_STATUS_BAD_BLOCK 2u   /* block id outside [0, num_blocks) */
#define PA_STATUS_BAD_CONTEXT 4u /* context_len < 1 or > max_context_len */
#define PA_STATUS_TIMEOUT 8u     /* a pipeline wait gave up (kernel aborted) */

/* Message for the last error on the calling thread ("" if none). */
const char* pa_last_error(void);

/* Library ABI version (increments on any signature change). */
int pa_version(void);

/*
 * Read and clear the device status word of the current device (a bitwise OR
 * of PA_STATUS_* raised by kernels since the last call).  Synchronizes
 * `stream`.  *status (host) receives the word.
 */
int pa_get_status(void* stream, uint32_t* status);

/*
 * KV append [Day6 paragraph 2]: write each new token's key and value into
 * its slot of the paged cache.
 *   k, v          device, [num_tokens][num_kv_heads][head_dim], dtype
 *   slot_mapping  device, [num_tokens] int64; slot = block*block_size + row;
 *                 a negative slot skips the token; slots must be distinct
 *                 (two tokens writing one slot leave either value)
 *   k_cache, v_cache  device, cache layout above, written in place
 * A slot >= num_blocks*block_size is skipped and sets PA_STATUS_BAD_SLOT.
 * The copy is bitwise.
 */
int pa_cache_append(const void* k, const void* v, const int64_t* slot_mapping,
                    int num_tokens, void* k_cache, void* v_cache, int num_blocks,
                    int num_kv_heads, int head_dim, int block_size, int dtype,
                    void* stream);

/*
 * KV append into an FP8 cache: the same scatter as pa_cache_append, of the
 * bf16 tokens k, v ([num_tokens][num_kv_heads][head_dim]) stored as E4M3
 * codes: code = round-to-nearest-even(x / scale) in E4M3 (bias 7, largest
 * finite 448; no infinities), the quotient an IEEE fp32 division; finite
 * quotients beyond ±448 and infinities store ±448, NaN stores a NaN code.
 * k_scale, v_scale: finite, > 0, one per cache.  The pages ask for fewer
 * bytes moved (memory notes, "Core Ideas" 1; [PAK section 6]: FP16
 * compute, FP32 accumulation); one byte per element is this library's
 * reading.  k_cache, v_cache: cache layout above with 1-byte elements.
 */
int pa_cache_append_fp8(const void* k, const void* v,
                        const int64_t* slot_mapping, int num_tokens,
                        void* k_cache, void* v_cache, int num_blocks,
                        int num_kv_heads, int head_dim, int block_size,
                        float k_scale, float v_scale, void* stream);

/*
 * Block copy for copy-on-write [Day6 paragraph 5]: for each pair
 * (src, dst) in `pairs` (device, [num_pairs][2] int32) copy the whole block
 * src of k_cache and of v_cache (every KV head, every row) to block dst.
 * dst blocks must be distinct and must not appear as a src in the same call.
 * An id outside [0, num_blocks) skips the pair and sets PA_STATUS_BAD_BLOCK.
 */
int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs,
                   int num_pairs, int num_blocks, int num_kv_heads,
                   int head_dim, int block_size, int dtype, void* stream);

/*
 * Partition size (tokens) that pa_decode uses for these sizes: the given
 * `partition_size` if > 0 (it must be a positive multiple of 32), else the
 * library's choice (a multiple of 32).  Returns the size, or a negative
 * PA_ERR_* code.
 */
int pa_decode_partition_size(int num_seqs, int num_kv_heads,
                             int max_context_len, int partition_size);

/*
 * Bytes of device workspace pa_decode needs for these sizes (0 only for
 * invalid sizes).  The workspace holds a 256-byte header and the work list
 * of the persistent decode kernel (8 bytes per sequence and partition) and,
 * when a context can span more than one partition, the split-K partials:
 * per (sequence, partition, query head) head_dim fp32 un-normalised outputs
 * and a (max, sum) pair.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                 int max_context_len, int partition_size);

/*
 * Paged decode attention [PAK section 3.1; Day6 paragraph 6]: for every
 * sequence s and query head h, with n = context_lens[s] and kv = h / g,
 *     out[s][h] = softmax(scale * K_s q[s][h]) V_s
 * where K_s, V_s are the sequence's first n key/value rows of KV head kv,
 * gathered through block_tables[s].  Contexts are split into partitions of
 * partition_size tokens (0 = library choice) processed in parallel and
 * merged by log-sum-exp.
 *   q             device, [num_seqs][num_heads][head_dim], dtype
 *   k_cache, v_cache  device, cache layout above
 *   block_tables  device, [num_seqs][max_blocks_per_seq] int32; entries past
 *                 a sequence's last block are not read
 *   context_lens  device, [num_seqs] int32, each in [1, max_context_len]
 *   max_context_len  host upper bound of context_lens;
 *                 ceil(max_context_len / block_size) <= max_blocks_per_seq
 *   out           device, [num_seqs][num_heads][head_dim], dtype
 *   workspace     device, >= pa_decode_workspace_bytes(...) bytes, 256-byte
 *                 aligned; contents on entry do not matter; calls whose
 *                 kernels overlap on the GPU need separate workspaces
 * Up to 65535 sequences and 32767 partitions per context.
 * q and the caches must be 16-byte aligned.  A context length outside
 * [1, max_context_len] sets PA_STATUS_BAD_CONTEXT (length 0 gives a zero
 * output row; longer ones are cut to max_context_len).
 */
int pa_decode(const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, int max_blocks_per_seq,
              const int32_t* context_lens, int max_context_len, float scale,
              void* out, int num_seqs, int num_heads, int num_kv_heads,
              int head_dim, int block_size, int num_blocks, int partition_size,
              void* workspace, size_t workspace_bytes, int dtype, void* stream);

/*
 * Test hook for the decode kernel's time-out path; not for production use.
 * The pages recommend defensive checks in the kernel [PAK section 5.1]:
 * every pipeline wait of the bf16 decode kernel is bounded, and one that
 * runs out raises PA_STATUS_TIMEOUT and stops the CTA instead of hanging.
 * This call is pa_decode (bf16 caches, same arguments and workspace) with
 * two changes that make such a wait run out on purpose, with no fault:
 *   - every pipeline wait gives up after wait_limit_us microseconds
 *     (1 .. 2000000) instead of 2 s;
 *   - the copy warp of every persistent CTA never issues that CTA's chunk
 *     number withheld_chunk (>= 0, counted over the CTA's work from 0): no
 *     copy is in flight for it and its barrier is never armed, so the
 *     consumer waiting for it runs out of time.
 * A CTA that gives up raises PA_STATUS_TIMEOUT, waits (bounded the same
 * way) for its own copies in flight, and exits; the other CTAs follow once
 * they reach the chunk.  `out` is then undefined; the context stays usable
 * and later calls are unaffected.  Read the status with pa_get_status.
 */
int pa_decode_test_withhold(const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables,
                            int max_blocks_per_seq,
                            const int32_t* context_lens, int max_context_len,
                            float scale, void* out, int num_seqs,
                            int num_heads, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, int partition_size,
                            void* workspace, size_t workspace_bytes,
                            int withheld_chunk, int wait_limit_us,
                            void* stream);

/*
 * Work list of the decode kernel built on the host, for callers that know
 * their context lengths there (a serving loop's allocator does) and can
 * upload it with their block tables, so that no planning kernel runs in the
 * step.  Same list as pa_decode builds on the device [PAK section 3.2: a
 * dynamic work queue]: every full partition, then partial ones from the
 * longest to the shortest, then one entry per empty context.
 *   context_lens  host, [num_seqs] int32, each in [0, max_context_len]
 *   plan          host, pa_decode_plan_bytes(...) bytes; a 256-byte header
 *                 (work counter = 0, list length) and 8 bytes per entry
 * partition_size must be the value pa_decode_partition_size returns for the
 * decode call (a positive multiple of 32).
 */
size_t pa_decode_plan_bytes(int num_seqs, int max_context_len,
                            int partition_size);
int pa_decode_plan_host(const int32_t* context_lens, int num_seqs,
                        int max_context_len, int partition_size, void* plan);

/*
 * pa_decode with a work list from pa_decode_plan_host, copied to the device
 * (`plan`, 256-byte aligned).  bf16 only.  The call consumes the list's work
 * counter: every call needs a fresh copy (counter 0).  The plan region of
 * `workspace` is not used; size it with pa_decode_workspace_bytes as for
 * pa_decode.  context_lens must hold the lengths the plan was built from.
 */
int pa_decode_planned(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, int max_context_len,
                      float scale, void* out, int num_seqs, int num_heads,
                      int num_kv_heads, int head_dim, int block_size,
                      int num_blocks, int partition_size, const void* plan,
                      void* workspace, size_t workspace_bytes, int dtype,
                      void* stream);

/*
 * Prefill [Day6 paragraph 2; PAK section 3.1]: append the new tokens of
 * every sequence (a prompt, or several tokens at once), then causal
 * attention of each of them.  Sequence s owns rows query_start[s] ..
 * query_start[s+1]-1 of q, k, v (device int32 [num_seqs + 1], ascending,
 * query_start[num_seqs] <= num_tokens) and has context_lens[s] tokens after
 * the append (device int32, n_s <= context_lens[s] <= max_context_len);
 * its new token i sits at position p = context_lens[s] - n_s + i and gets
 *     out[row][h] = softmax(scale * K_s[0..p] q[row][h]) V_s[0..p]
 * (K_s, V_s gathered through block_tables[s] after the append, kv = h / g).
 *   q, out      device, [num_tokens][num_heads][head_dim] bf16
 *   k, v        device, [num_tokens][num_kv_heads][head_dim] bf16
 *   slot_mapping  device, [num_tokens] int64, as for pa_cache_append
 *   max_query_len  host bound of every n_s
 * bf16 only; heads per KV head 1, 2, 4 or 8; up to 65535 sequences and,
 * for head_dim 128, ceil(max_query_len * g / 128) <= 65535 (PA_ERR_UNSUPPORTED
 * beyond).  Lengths or offsets out of range set PA_STATUS_BAD_CONTEXT and
 * that sequence's rows are left unwritten.
 */
int pa_prefill(const void* q, const void* k, const void* v,
               const int64_t* slot_mapping, int num_tokens,
               const int32_t* query_start, const int32_t* context_lens,
               const int32_t* block_tables, int max_blocks_per_seq,
               int max_query_len, int max_context_len, float scale,
               void* k_cache, void* v_cache, void* out, int num_seqs,
               int num_heads, int num_kv_heads, int head_dim, int block_size,
               int num_blocks, int dtype, void* stream);

/*
 * Test hook for pa_prefill's split of a large batch; not for production
 * use.  A prefill kernel launch lists at most 440 work items per CTA, and a
 * batch with more is attended by several launches, each over a contiguous
 * range of the items.  This sets a smaller bound on the items of one launch
 * (items_per_launch >= 1), so that a small batch takes the several-launch
 * path; 0 restores the default.  It applies to the calls that follow, from
 * every thread.  Returns PA_OK, or PA_ERR_INVALID for a negative value.
 */
int pa_prefill_test_items_per_launch(int items_per_launch);

/*
 * Test hook for the prefill's failure detection (every pipeline wait of the
 * tcgen05 kernel gives up after 2 s, raises PA_STATUS_TIMEOUT, lets its
 * copies and products in flight finish and exits): from now on the key
 * producer of every CTA never issues its chunk number `chunk` (counted over
 * the CTA's chunks of keys, from 0), so that the waits for it run out; -1
 * restores normal operation.  Not for production.  Applies to the calls that
 * follow, from every thread.  Returns PA_OK, or PA_ERR_INVALID for a chunk
 * below -1.
 */
int pa_prefill_test_withhold(int chunk);

/*
 * Paged decode over FP8 caches written by pa_cache_append_fp8: the result of
 * pa_decode with K = e4m3(code) * k_scale and V = e4m3(code) * v_scale.  q
 * and out are bf16; head_dim 128; products in FP16 on tensor cores, sums in
 * FP32 [PAK section 6].  q must be finite with |q| < 65504 (it is taken to
 * FP16).  plan: NULL to build the work list on the device, else a list from
 * pa_decode_plan_host (as for pa_decode_planned).  Workspace as pa_decode.
 * Prefix groups are not supported with FP8 caches.
 */
int pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, int max_blocks_per_seq,
                  const int32_t* context_lens, int max_context_len,
                  float scale, float k_scale, float v_scale, void* out,
                  int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                  int block_size, int num_blocks, int partition_size,
                  const void* plan, void* workspace, size_t workspace_bytes,
                  void* stream);

/*
 * Shared-prefix decode [Day6 paragraph 5: sequences forked from one prompt
 * share its cache blocks].  The same result as pa_decode (and, with a plan,
 * pa_decode_planned), but each block a group of sequences shares is read
 * once per 128 / g members -- once per group for groups of up to 128 / g
 * sequences -- instead of once per member: a shared partition is attended,
 * per KV head, as one tile of 128 query rows (member x head) on the
 * 5th-generation tensor cores.
 *   groups      host, [num_groups][3] int32: first sequence, number of
 *               sequences, shared prefix length in tokens.  Group i is
 *               sequences first .. first + count - 1 of the batch; the
 *               ranges are ascending and disjoint; sequences in no group
 *               are decoded as by pa_decode.  0 <= num_groups <=
 *               PA_MAX_PREFIX_GROUPS; groups may be NULL when num_groups is 0.
 * The caller guarantees that the first `prefix` tokens of every member are
 * stored in the same physical blocks, listed in the table of the group's
 * first sequence, and that prefix <= max_context_len.  The whole partitions
 * of the prefix (floor(prefix / P) * P tokens, P the partition size, which
 * for partition_size 0 is pa_decode_partition_size_shared_prefix's) become
 * shared work items of the decode kernel, each attending one partition for
 * several members at once and storing their split-K partials; the members'
 * other partitions are decoded as usual and the log-sum-exp merge combines
 * them.  A member whose context ends inside the shared part is masked to
 * its own length.  Groups whose prefix is shorter than one partition, and
 * calls where no context spans two partitions, fall back to plain decode
 * for those sequences.  bf16 only; the workspace is sized as for pa_decode.
 */
#define PA_MAX_PREFIX_GROUPS 64
int pa_decode_shared_prefix(const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables,
                            int max_blocks_per_seq,
                            const int32_t* context_lens, int max_context_len,
                            float scale, void* out, int num_seqs,
                            int num_heads, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks,
                            int partition_size, const int32_t* groups,
                            int num_groups, void* workspace,
                            size_t workspace_bytes, int dtype, void* stream);

/*
 * Partition size that pa_decode_shared_prefix and
 * pa_decode_planned_shared_prefix use for these sizes and groups: the given
 * `partition_size` if > 0, else pa_decode_partition_size's choice doubled,
 * up to 1024 tokens, while every group's prefix still holds a whole
 * partition (fewer shared items and partials per group).  groups as for
 * pa_decode_shared_prefix (only the prefix lengths are read here).  Returns
 * the size, or a negative PA_ERR_* code.
 */
int pa_decode_partition_size_shared_prefix(int num_seqs, int num_kv_heads,
                                           int max_context_len,
                                           int partition_size,
                                           const int32_t* groups,
                                           int num_groups);

/* Host work list for pa_decode_planned_shared_prefix: the list of
 * pa_decode_plan_host with the groups' shared partitions as shared items
 * (same groups, head counts, partition size and lengths as the decode
 * call). */
int pa_decode_plan_host_shared_prefix(const int32_t* context_lens,
                                      int num_seqs, int max_context_len,
                                      int partition_size, int num_heads,
                                      int num_kv_heads, const int32_t* groups,
                                      int num_groups, void* plan);

/* pa_decode_planned for prefix groups; `plan` from
 * pa_decode_plan_host_shared_prefix with the same groups. */
int pa_decode_planned_shared_prefix(
    const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int max_context_len, float scale, void* out,
    int num_seqs, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int partition_size, const int32_t* groups,
    int num_groups, const void* plan, void* workspace, size_t workspace_bytes,
    int dtype, void* stream);

/*
 * Paged decode that allocates nothing: the same computation and arguments as
 * pa_decode, but the split-K scratch is a fixed device array inside this
 * library, so the caller passes no workspace.  The pages have no counterpart;
 * this entry point is for callers that cannot call cudaMalloc for a
 * workspace (device memory reserved up front by another allocator, or a loop
 * that must not make calls that may synchronize the device).
 *   - The array holds PA_STATIC_WORKSPACE_BYTES; sizes whose workspace
 *     (pa_decode_workspace_bytes) exceeds it return PA_ERR_INVALID.
 *   - Every GPU that loads the library holds the array until the process
 *     exits.  The first call on a device looks up the array's address there
 *     (cudaGetSymbolAddress), and so does the first call after the device's
 *     context was re-created (cudaDeviceReset); make that first call before
 *     any stream capture.
 *   - All calls share the array and it keeps the last call's contents;
 *     nothing in it needs to start at zero.  Calls whose kernels overlap on
 *     the GPU (different streams or threads) race on it: serialise them.
 *   - No cudaMalloc, cudaFree or other allocating call is made.
 */
#define PA_STATIC_WORKSPACE_BYTES (16u << 20)
int pa_decode_static_workspace(const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               int max_blocks_per_seq,
                               const int32_t* context_lens, int max_context_len,
                               float scale, void* out, int num_seqs,
                               int num_heads, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks,
                               int partition_size, int dtype, void* stream);

/* ------------------------------------------------------------------------
 * Host block allocator [Day6 paragraphs 2, 5, 6].  CPU only; no CUDA call.
 *
 * Free list: a stack.  A fresh allocator hands out free_order[0] first, then
 * free_order[1], ...; a freed block goes on top.  Sharing is ref-counted:
 * pa_seq_fork gives the child the parent's blocks and one more reference to
 * each.  Appending to a sequence whose last block is partly filled and
 * shared takes a new block and reports the copy (src -> dst) the caller must
 * apply with pa_copy_blocks before writing the token (copy-on-write).  A
 * call that fails (PA_ERR_OOM, PA_ERR_STATE, PA_ERR_INVALID) changes
 * nothing.  Not thread-safe: one allocator per thread at a time.
 * ------------------------------------------------------------------------ */
typedef struct pa_alloc pa_alloc;

/* New allocator over blocks 0..num_blocks-1.  free_order (host, nullable):
 * a permutation of 0..num_blocks-1 giving the hand-out order; NULL means
 * ascending.  *out receives the handle. */
int pa_alloc_create(int num_blocks, int block_size, const int32_t* free_order,
                    pa_alloc** out);
void pa_alloc_destroy(pa_alloc* a);
int pa_alloc_num_free(const pa_alloc* a);

/* Add sequence seq_id holding num_tokens tokens in ceil(num_tokens /
 * block_size) fresh blocks. */
int pa_seq_add(pa_alloc* a, int64_t seq_id, int num_tokens);
/* Child shares every block of parent (refcount + 1 each). */
int pa_seq_fork(pa_alloc* a, int64_t parent_id, int64_t child_id);
/* Reserve the slot of the sequence's next token.  *slot receives it;
 * *cow_src, *cow_dst receive the block copy to apply first, or -1, -1. */
int pa_seq_append_slot(pa_alloc* a, int64_t seq_id, int64_t* slot,
                       int32_t* cow_src, int32_t* cow_dst);
/* Drop the sequence: one reference less on each of its blocks, in table
 * order; blocks reaching zero go on top of the free list in that order. */
int pa_seq_free(pa_alloc* a, int64_t seq_id);
/* Token count of the sequence (>= 0), or a negative PA_ERR_* code. */
int pa_seq_num_tokens(const pa_alloc* a, int64_t seq_id);
/* Copy up to cap block ids of the sequence's table into out (host);
 * *n_out receives the table length (PA_ERR_INVALID if cap is too small). */
int pa_seq_block_table(const pa_alloc* a, int64_t seq_id, int32_t* out,
                       int cap, int* n_out);
/* Reference count of a block (>= 0), or a negative PA_ERR_* code. */
int pa_block_refcount(const pa_alloc* a, int block_id);

/*
 * Batched serving step on the host: reserve the next slot of each of the n
 * sequences seq_ids[0..n-1], in order.  Outputs (host):
 *   slot_mapping [n] int64; cow_pairs [n][2] int32 with *num_cow pairs used;
 *   block_tables [n][width] int32 (nullable): row i is updated in place
 *   where sequence i's table changed (rows are assumed to hold its table
 *   already; width must cover the grown table);
 *   context_lens [n] int32 (nullable): the new token counts.
 * If the pool cannot cover every new block of the batch, returns PA_ERR_OOM
 * and changes nothing.
 */
int pa_seqs_append_slots(pa_alloc* a, const int64_t* seq_ids, int n,
                         int64_t* slot_mapping, int32_t* cow_pairs,
                         int* num_cow, int32_t* block_tables, int width,
                         int32_t* context_lens);

/* Write the tables of seq_ids (host) into block_tables [n][width] (host),
 * padding with -1, and their token counts into context_lens [n] (nullable). */
int pa_seqs_block_tables(const pa_alloc* a, const int64_t* seq_ids, int n,
                         int32_t* block_tables, int width,
                         int32_t* context_lens);

/* ------------------------------------------------------------------------
 * Host side of a pipelined serving step [Day6 paragraph 2].
 *
 * The caller owns one pinned host buffer and two device buffers laid out by
 * pa_stepper_layout (offsets: work list, slot mapping int64[n], context
 * lengths int32[n], copy-on-write pairs int32[n][2], block tables
 * int32[n][width]).  Each step:
 *   pa_stepper_prepare  waits until the previous upload has read the host
 *                       buffer; reserves every sequence's next slot
 *                       (pa_seqs_append_slots, tables and lengths updated in
 *                       place); builds the decode work list
 *                       (pa_decode_plan_host, if partition_size > 0); on
 *                       upload_stream waits until the step that last read
 *                       device buffer k is over, copies the host buffer to
 *                       it and records an event; makes main_stream wait for
 *                       that event.  *buffer_index = k, *num_cow = copies the
 *                       caller must apply (pa_copy_blocks on main_stream)
 *                       before appending.
 *   ... the step's kernels on main_stream, reading device buffer k ...
 *   pa_stepper_finish   records on main_stream that buffer k is free again.
 * The stepper owns four CUDA events; everything else is the caller's.  The
 * allocator must not be changed by other calls between prepare and finish.
 * ------------------------------------------------------------------------ */
typedef struct pa_stepper pa_stepper;

int pa_stepper_layout(int num_seqs, int max_context_len, int block_size,
                      int partition_size, size_t* offsets /* [5] */,
                      size_t* total);
int pa_stepper_create(pa_alloc* alloc, const int64_t* seq_ids, int num_seqs,
                      int max_context_len, int block_size, int partition_size,
                      void* host_buf, void* dev_buf0, void* dev_buf1,
                      size_t buf_bytes, pa_stepper** out);
void pa_stepper_destroy(pa_stepper* st);
int pa_stepper_prepare(pa_stepper* st, void* upload_stream, void* main_stream,
                       int* buffer_index, int* num_cow);
int pa_stepper_finish(pa_stepper* st, void* main_stream);
/* Prefix groups of the stepper's batch (as for pa_decode_shared_prefix,
 * positions in seq_ids; copied) and the decode's head counts: work lists
 * built by later prepare calls are those of
 * pa_decode_plan_host_shared_prefix, for pa_decode_planned_shared_prefix.
 * num_groups = 0 removes them. */
int pa_stepper_set_prefix_groups(pa_stepper* st, const int32_t* groups,
                                 int num_groups, int num_heads,
                                 int num_kv_heads);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
