// Work list of the persistent decode kernel, built on the host.
//
// Same list as the device-side planner (decode_plan.cu): every full
// partition, then the partial ones from the longest remainder to the
// shortest, then one zero-length entry per empty context; a 256-byte header
// carries the work counter (0) and the list length.  A serving loop knows
// its context lengths on the host (the allocator holds them), so it can
// build the list there and upload it with the block tables instead of
// running the planner kernel on the critical path of every step.
//
// Also validates prefix groups for the shared-prefix decode (shared with
// the device path in api.cu).

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <vector>

#include "kernels.h"
#include "pa.h"
#include "pa_internal.h"


int pa_prefix_groups(const int32_t* groups, int n, int num_seqs, int max_context_len, int partition_size,
                     pa::PrefixGroups* out, const char* who) {
  static thread_local char buf[200];
  std::memset(out, 0, sizeof(*out));
  if (n == 0) return PA_OK;
  if (n < 0 || !groups) {
    std::snprintf(buf, sizeof(buf), "%s: bad prefix group list", who);
    return pa_fail(PA_ERR_INVALID, buf);
  }
  if (n > pa::kMaxPrefixGroups) {
    std::snprintf(buf, sizeof(buf), "%s: more than %d prefix groups", who, pa::kMaxPrefixGroups);
    return pa_fail(PA_ERR_UNSUPPORTED, buf);
  }
  const long long max_parts = (max_context_len + (long long)partition_size - 1) / partition_size;
  int end = 0;  // one past the previous group's last sequence
  for (int i = 0; i < n; ++i) {
    const int first = groups[3 * i], count = groups[3 * i + 1], prefix = groups[3 * i + 2];
    if (first < end || count < 1 || (long long)first + count > num_seqs || prefix < 0 ||
        prefix > max_context_len) {
      std::snprintf(buf, sizeof(buf),
                    "%s: prefix group %d (first %d, count %d, prefix %d) is out of range, empty or overlaps the "
                    "previous one",
                    who, i, first, count, prefix);
      return pa_fail(PA_ERR_INVALID, buf);
    }
    end = first + count;
    // Whole partitions of the prefix; none when no context has a second
    // partition (there are no partial slots to write then).
    const int parts = max_parts > 1 ? prefix / partition_size : 0;
    if (parts == 0) continue;
    const int k = out->n++;
    out->first[k] = first;
    out->count[k] = count;
    out->parts[k] = parts;
  }
  return PA_OK;
}

extern "C" {

size_t pa_decode_plan_bytes(int num_seqs, int max_context_len, int partition_size) {
  if (num_seqs <= 0 || max_context_len < 1 || partition_size < 32) return 0;
  const long long parts = (max_context_len + (long long)partition_size - 1) / partition_size;
  return sizeof(pa::PlanHeader) + (size_t)num_seqs * parts * sizeof(int32_t) * 2;
}

int pa_decode_plan_host(const int32_t* context_lens, int num_seqs, int max_context_len, int partition_size,
                        void* plan) {
  return pa_decode_plan_host_shared_prefix(context_lens, num_seqs, max_context_len, partition_size, 1, 1, nullptr,
                                           0, plan);
}

int pa_decode_plan_host_shared_prefix(const int32_t* context_lens, int num_seqs, int max_context_len,
                                      int partition_size, int num_heads, int num_kv_heads, const int32_t* groups,
                                      int num_groups, void* plan) {
  if (!context_lens || !plan || num_seqs <= 0 || max_context_len < 1 || partition_size < 32 ||
      partition_size % 32)
    return pa_fail(PA_ERR_INVALID, "pa_decode_plan_host: bad arguments");
  const long long parts = (max_context_len + (long long)partition_size - 1) / partition_size;
  if (num_seqs > 65535 || parts > 32767)
    return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode_plan_host: more than 65535 sequences or 32767 partitions");
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads)
    return pa_fail(PA_ERR_INVALID, "pa_decode_plan_host: head counts");
  const int g = num_heads / num_kv_heads;
  pa::PrefixGroups pg;
  int rc = pa_prefix_groups(groups, num_groups, num_seqs, max_context_len, partition_size, &pg,
                            "pa_decode_plan_host");
  if (rc) return rc;
  for (int s = 0; s < num_seqs; ++s)
    if (context_lens[s] < 0 || context_lens[s] > max_context_len)
      return pa_fail(PA_ERR_INVALID, "pa_decode_plan_host: context length out of range");
  const int P = partition_size;
  auto* hdr = static_cast<pa::PlanHeader*>(plan);
  auto* list = reinterpret_cast<int32_t*>(static_cast<char*>(plan) + sizeof(pa::PlanHeader));
  size_t n = 0;
  // Shared partitions of prefix groups: shared-prefix items first; the
  // members' own items for them are left out.
  const int npre = pa::prefix_entries(pg, g);
  for (int e = 0; e < npre; ++e, ++n) {
    const int2 ent = pa::prefix_entry_at(pg, g, e);
    list[2 * n] = ent.x;
    list[2 * n + 1] = ent.y;
  }
  std::vector<int> skip(num_seqs);
  for (int s = 0; s < num_seqs; ++s) skip[s] = pa::prefix_parts_of(pg, s);
  for (int s = 0; s < num_seqs; ++s) {
    const int c = context_lens[s];
    for (int p = skip[s]; p < c / P; ++p) {
      list[2 * n] = s | (p << 16);
      list[2 * n + 1] = c;
      ++n;
    }
  }
  std::vector<int> partial;
  for (int s = 0; s < num_seqs; ++s)
    if (context_lens[s] % P && context_lens[s] / P >= skip[s]) partial.push_back(s);
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
