// Library-wide entry points of the SPRINT C ABI (version, error strings).
#include <atomic>

#include "common.cuh"

static std::atomic<unsigned long long> g_launches{0};

void sprint::count_launches(int n) { g_launches.fetch_add((unsigned long long)n); }

extern "C" unsigned long long sprint_kernel_launches(void) { return g_launches.load(); }

extern "C" int sprint_version(void) { return SPRINT_VERSION; }

extern "C" int sprint_debug_checks(void) { return sprint::kDebugChecks ? 1 : 0; }

extern "C" const char *sprint_strerror(int code) {
  switch (code) {
    case SPRINT_OK: return "ok";
    case SPRINT_ERR_INVALID_ARG: return "invalid argument (null pointer, size or alignment)";
    case SPRINT_ERR_UNSUPPORTED: return "unsupported shape or layout";
    case SPRINT_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case SPRINT_ERR_WORKSPACE: return "workspace smaller than the *_workspace_bytes() size";
    case SPRINT_ERR_TOO_LARGE: return "request larger than the library's fixed scratch array";
    default: return "unknown sprint error code";
  }
}
