// Work list of the persistent decode kernel, built on the host.
//
// Same list as the device-side planner (decode_plan.cu): every full
// partition, then the partial ones from the longest remainder to the
// shortest, then one zero-length entry per empty context; a 256-byte header
// carries the work counter (0) and the list length.  A serving loop knows
// its context lengths on the host (the allocator holds them), so it can
// build the list there and upload it with the block tables instead of
// running the planner kernel on the critical path of every step.

#include <algorithm>
#include <cstring>
#include <vector>

#include "kernels.h"
#include "pa.h"
#include "pa_internal.h"

extern "C" {

size_t pa_decode_plan_bytes(int num_seqs, int max_context_len, int partition_size) {
  if (num_seqs <= 0 || max_context_len < 1 || partition_size < 32) return 0;
  const long long parts = (max_context_len + (long long)partition_size - 1) / partition_size;
  return sizeof(pa::PlanHeader) + (size_t)num_seqs * parts * sizeof(int32_t) * 2;
}

int pa_decode_plan_host(const int32_t* context_lens, int num_seqs, int max_context_len, int partition_size,
                        void* plan) {
  if (!context_lens || !plan || num_seqs <= 0 || max_context_len < 1 || partition_size < 32 ||
      partition_size % 32)
    return pa_fail(PA_ERR_INVALID, "pa_decode_plan_host: bad arguments");
  const long long parts = (max_context_len + (long long)partition_size - 1) / partition_size;
  if (num_seqs > 65535 || parts > 32767)
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode_plan_host: more than 65535 sequences or 32767 partitions");
  const int P = partition_size;
  auto* hdr = static_cast<pa::PlanHeader*>(plan);
  auto* list = reinterpret_cast<int32_t*>(static_cast<char*>(plan) + sizeof(pa::PlanHeader));
  size_t n = 0;
  for (int s = 0; s < num_seqs; ++s) {
    const int c = context_lens[s];
    if (c < 0 || c > max_context_len) return pa_fail(PA_ERR_INVALID, "pa_decode_plan_host: context length out of range");
    for (int p = 0; p < c / P; ++p) {
      list[2 * n] = s | (p << 16);
      list[2 * n + 1] = c;
      ++n;
    }
  }
  std::vector<int> partial;
  for (int s = 0; s < num_seqs; ++s)
    if (context_lens[s] % P) partial.push_back(s);
  std::stable_sort(partial.begin(), partial.end(),
                   [&](int a, int b) { return context_lens[a] % P > context_lens[b] % P; });
  for (int s : partial) {
    const int c = context_lens[s];
    list[2 * n] = s | ((c / P) << 16);
    list[2 * n + 1] = c;
    ++n;
  }
  for (int s = 0; s < num_seqs; ++s) {
    if (context_lens[s] != 0) continue;
    list[2 * n] = s;
    list[2 * n + 1] = 0;
    ++n;
  }
  std::memset(hdr, 0, sizeof(pa::PlanHeader));
  hdr->counter = 0;
  hdr->num_pairs = (int)n;
  return PA_OK;
}

}  // extern "C"
