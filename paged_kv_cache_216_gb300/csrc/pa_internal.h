// Internal helpers shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>

// Record `msg` as the calling thread's last error and return `code`.
int pa_fail(int code, const char* msg);
// Clear the calling thread's last error.
void pa_clear_error();

#define PA_ABI_VERSION 1
