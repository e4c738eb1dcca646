// Host side of a pipelined serving step, in native code.
//
// Every decode step of a serving loop reserves each sequence's next slot in
// the block allocator ("Day 6/90 of Inference Engineering", PagedAttention
// notes, paragraph 2), and the slot mapping, context lengths, copy-on-write
// pairs, block tables and the decode work list must reach the device before
// the step's kernels run.  This object does all of that in one call:
//
//   prepare: wait until the previous upload has read the pinned buffer;
//            reserve the slots (tables and lengths updated in place);
//            build the work list; on the upload stream, wait until the step
//            that last read device buffer k is over, copy the pinned buffer
//            to it and record "uploaded"; make the main stream wait for it.
//   finish:  record "consumed" for buffer k on the main stream; k ^= 1.
//
// so a step costs the host one call on each side of its kernel launches.
// The buffers are the caller's (pinned host, two device copies); the object
// owns four CUDA events.

#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "kernels.h"
#include "pa.h"
#include "pa_internal.h"

struct pa_stepper {
  pa_alloc* alloc = nullptr;
  std::vector<int64_t> seq_ids;
  int max_context_len = 0;
  int partition_size = 0;
  int width = 0;
  char* host = nullptr;
  char* dev[2] = {nullptr, nullptr};
  size_t bytes = 0;
  size_t off[5] = {0, 0, 0, 0, 0};  // plan, slots, ctx, cow, tables
  cudaEvent_t uploaded[2] = {nullptr, nullptr};
  cudaEvent_t consumed[2] = {nullptr, nullptr};
  int k = 0;
  std::vector<int32_t> groups;  // prefix groups, [n][3]
  int num_heads = 1, num_kv_heads = 1;
};

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int cuda_error(cudaError_t e, const char* what) {
  static thread_local char buf[200];
  std::snprintf(buf, sizeof(buf), "%s: %s", what, cudaGetErrorString(e));
  return pa_fail(PA_ERR_CUDA, buf);
}

}  // namespace

extern "C" {

int pa_stepper_layout(int num_seqs, int max_context_len, int block_size, int partition_size, size_t* offsets,
                      size_t* total) {
  if (num_seqs <= 0 || max_context_len < 1 || block_size <= 0 || partition_size < 0 || !offsets || !total)
    return pa_fail(PA_ERR_INVALID, "pa_stepper_layout: bad arguments");
  const size_t plan = partition_size ? pa_decode_plan_bytes(num_seqs, max_context_len, partition_size) : 0;
  if (partition_size && plan == 0) return pa_fail(PA_ERR_INVALID, "pa_stepper_layout: partition size");
  const size_t width = (size_t)(max_context_len + block_size - 1) / block_size;
  const size_t s = (size_t)num_seqs;
  offsets[0] = 0;
  offsets[1] = align_up(plan, 256);
  offsets[2] = offsets[1] + 8 * s;
  offsets[3] = align_up(offsets[2] + 4 * s, 16);
  offsets[4] = align_up(offsets[3] + 8 * s, 16);
  *total = offsets[4] + 4 * s * width;
  return PA_OK;
}

int pa_stepper_create(pa_alloc* alloc, const int64_t* seq_ids, int num_seqs, int max_context_len, int block_size,
                      int partition_size, void* host_buf, void* dev_buf0, void* dev_buf1, size_t buf_bytes,
                      pa_stepper** out) {
  if (!alloc || !seq_ids || !host_buf || !dev_buf0 || !dev_buf1 || !out)
    return pa_fail(PA_ERR_INVALID, "pa_stepper_create: null argument");
  size_t off[5], total = 0;
  int rc = pa_stepper_layout(num_seqs, max_context_len, block_size, partition_size, off, &total);
  if (rc) return rc;
  if (buf_bytes < total) return pa_fail(PA_ERR_INVALID, "pa_stepper_create: buffers too small");
  if ((reinterpret_cast<uintptr_t>(host_buf) | reinterpret_cast<uintptr_t>(dev_buf0) |
       reinterpret_cast<uintptr_t>(dev_buf1)) & 255)
    return pa_fail(PA_ERR_INVALID, "pa_stepper_create: buffers must be 256-byte aligned");
  pa_stepper* st = new (std::nothrow) pa_stepper();
  if (!st) return pa_fail(PA_ERR_OOM, "pa_stepper_create: host allocation failed");
  st->alloc = alloc;
  st->seq_ids.assign(seq_ids, seq_ids + num_seqs);
  st->max_context_len = max_context_len;
  st->partition_size = partition_size;
  st->width = (max_context_len + block_size - 1) / block_size;
  st->host = static_cast<char*>(host_buf);
  st->dev[0] = static_cast<char*>(dev_buf0);
  st->dev[1] = static_cast<char*>(dev_buf1);
  st->bytes = total;
  std::memcpy(st->off, off, sizeof(off));
  for (int i = 0; i < 2; ++i) {
    cudaError_t e = cudaEventCreateWithFlags(&st->uploaded[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&st->consumed[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      pa_stepper_destroy(st);
      return cuda_error(e, "pa_stepper_create: cudaEventCreate");
    }
  }
  // the tables and lengths of the sequences as they stand
  rc = pa_seqs_block_tables(alloc, seq_ids, num_seqs, reinterpret_cast<int32_t*>(st->host + off[4]), st->width,
                            reinterpret_cast<int32_t*>(st->host + off[2]));
  if (rc) {
    pa_stepper_destroy(st);
    return rc;
  }
  *out = st;
  return PA_OK;
}

void pa_stepper_destroy(pa_stepper* st) {
  if (!st) return;
  for (int i = 0; i < 2; ++i) {
    if (st->uploaded[i]) cudaEventDestroy(st->uploaded[i]);
    if (st->consumed[i]) cudaEventDestroy(st->consumed[i]);
  }
  delete st;
}

int pa_stepper_set_prefix_groups(pa_stepper* st, const int32_t* groups, int num_groups, int num_heads,
                                 int num_kv_heads) {
  if (!st) return pa_fail(PA_ERR_INVALID, "pa_stepper_set_prefix_groups: null stepper");
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads)
    return pa_fail(PA_ERR_INVALID, "pa_stepper_set_prefix_groups: head counts");
  if (st->partition_size == 0 && num_groups != 0)
    return pa_fail(PA_ERR_INVALID, "pa_stepper_set_prefix_groups: the stepper builds no work list");
  if (num_groups != 0) {
    pa::PrefixGroups pg;
    int rc = pa_prefix_groups(groups, num_groups, (int)st->seq_ids.size(), st->max_context_len, st->partition_size,
                              &pg, "pa_stepper_set_prefix_groups");
    if (rc) return rc;
  }
  try {
    st->groups.assign(groups, groups + 3 * (size_t)num_groups);
    st->num_heads = num_heads;
    st->num_kv_heads = num_kv_heads;
  } catch (...) {
    return pa_fail(PA_ERR_OOM, "pa_stepper_set_prefix_groups: host allocation failed");
  }
  return PA_OK;
}

int pa_stepper_prepare(pa_stepper* st, void* upload_stream, void* main_stream, int* buffer_index, int* num_cow) {
  if (!st || !buffer_index || !num_cow) return pa_fail(PA_ERR_INVALID, "pa_stepper_prepare: null argument");
  const int k = st->k;
  // The previous upload read the pinned buffer; it must be done before the
  // allocator rewrites it.  (An event never recorded counts as done.)
  cudaError_t e = cudaEventSynchronize(st->uploaded[1 - k]);
  if (e != cudaSuccess) return cuda_error(e, "pa_stepper_prepare: cudaEventSynchronize");
  const int n = (int)st->seq_ids.size();
  int rc = pa_seqs_append_slots(st->alloc, st->seq_ids.data(), n, reinterpret_cast<int64_t*>(st->host + st->off[1]),
                                reinterpret_cast<int32_t*>(st->host + st->off[3]), num_cow,
                                reinterpret_cast<int32_t*>(st->host + st->off[4]), st->width,
                                reinterpret_cast<int32_t*>(st->host + st->off[2]));
  if (rc) return rc;
  if (st->partition_size) {
    rc = pa_decode_plan_host_shared_prefix(reinterpret_cast<const int32_t*>(st->host + st->off[2]), n,
                                           st->max_context_len, st->partition_size, st->num_heads,
                                           st->num_kv_heads, st->groups.empty() ? nullptr : st->groups.data(),
                                           (int)(st->groups.size() / 3), st->host + st->off[0]);
    if (rc) return rc;
  }
  cudaStream_t up = static_cast<cudaStream_t>(upload_stream);
  cudaStream_t mainst = static_cast<cudaStream_t>(main_stream);
  e = cudaStreamWaitEvent(up, st->consumed[k], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st->dev[k], st->host, st->bytes, cudaMemcpyHostToDevice, up);
  if (e == cudaSuccess) e = cudaEventRecord(st->uploaded[k], up);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(mainst, st->uploaded[k], 0);
  if (e != cudaSuccess) return cuda_error(e, "pa_stepper_prepare: upload");
  *buffer_index = k;
  return PA_OK;
}

int pa_stepper_finish(pa_stepper* st, void* main_stream) {
  if (!st) return pa_fail(PA_ERR_INVALID, "pa_stepper_finish: null argument");
  cudaError_t e = cudaEventRecord(st->consumed[st->k], static_cast<cudaStream_t>(main_stream));
  if (e != cudaSuccess) return cuda_error(e, "pa_stepper_finish: cudaEventRecord");
  st->k ^= 1;
  return PA_OK;
}

}  // extern "C"
