// Internal helpers shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>

// Record `msg` as the calling thread's last error and return `code`.
int pa_fail(int code, const char* msg);
// Clear the calling thread's last error.
void pa_clear_error();

#define PA_ABI_VERSION 1

namespace pa {
struct PrefixGroups;
}

// Validate prefix groups (host, [n][3]: first sequence, count, prefix tokens)
// against a decode call's sizes and fill `out` with the groups that share at
// least one whole partition.
int pa_prefix_groups(const int32_t* groups, int n, int num_seqs, int max_context_len, int partition_size,
                     pa::PrefixGroups* out, const char* who);
