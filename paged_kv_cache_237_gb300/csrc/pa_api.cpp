// Library-wide C-ABI pieces: error reporting and version.
#include <cstring>
#include <string>

#include "pa.h"
#include "pa_internal.h"

namespace {
thread_local std::string g_last_error;
}

void pa_set_error(const char *msg) { g_last_error = msg ? msg : ""; }

int pa_fail(int code, const char *msg) {
    pa_set_error(msg);
    return code;
}

extern "C" const char *pa_last_error_string(void) { return g_last_error.c_str(); }

extern "C" int pa_version(void) { return (1 << 16) | 1; }
