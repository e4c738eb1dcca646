// Internal helpers shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>

// Record `msg` as the calling thread's last error and return `code`.
int pa_fail(int code, const char* msg);
// Clear the calling thread's last error.
void pa_clear_error();

#define PA_ABI_VERSION 1

// Identifier of the CUDA context current on the calling thread (unique
// within the process; a device's primary context gets a new one when it is
// re-created, e.g. after cudaDeviceReset), or 0 if none is current or it
// cannot be read.  Device addresses the library caches per device are keyed
// on it, so that they are looked up again in a new context.
unsigned long long pa_context_id();

namespace pa {
struct PrefixGroups;
}

// Validate prefix groups (host, [n][3]: first sequence, count, prefix tokens)
// against a decode call's sizes and fill `out` with the groups that share at
// least one whole partition.
int pa_prefix_groups(const int32_t* groups, int n, int num_seqs, int max_context_len, int partition_size,
                     pa::PrefixGroups* out, const char* who);
