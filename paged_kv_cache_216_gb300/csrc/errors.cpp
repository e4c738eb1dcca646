// Thread-local error reporting for the C ABI.
#include <string>

#include "pa.h"
#include "pa_internal.h"

namespace {
thread_local std::string g_last_error;
}

int pa_fail(int code, const char* msg) {
  g_last_error = msg ? msg : "";
  return code;
}

void pa_clear_error() { g_last_error.clear(); }

extern "C" const char* pa_last_error(void) { return g_last_error.c_str(); }

extern "C" int pa_version(void) { return PA_ABI_VERSION; }
