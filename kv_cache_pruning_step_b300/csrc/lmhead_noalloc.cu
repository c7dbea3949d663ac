// LM-head confidence for callers that cannot allocate device memory.
//
// Some hosts of this library may not call cudaMalloc at all: an inference
// server or plugin whose device memory belongs to a pool it must not go
// around, or a latency-critical serving loop where a cudaMalloc (and the
// synchronisation it can imply) is not acceptable.  This entry point gives
// them sprint_lmhead_confidence without a caller-provided workspace: the
// per-strip partials live in a fixed file-scope device array that every GPU
// which loads this library holds until the process exits.
//
// The array is shared by every call.  Nothing in it needs to start at zero:
// each call writes every partial it later reads.  Calls whose kernels
// overlap on the GPU (different streams, or different host threads) race on
// the array and must be serialised by the caller.
#include <mutex>

#include "common.cuh"

namespace {

__device__ __align__(256) unsigned char g_lmhead_scratch[SPRINT_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the symbol's host-side name is not a device address).
void *scratch_for_current_device(int *rc) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *rc = SPRINT_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_lmhead_scratch) != cudaSuccess || !p) {
      *rc = SPRINT_ERR_CUDA;
      return nullptr;
    }
    g_scratch_addr[dev] = p;
  }
  *rc = SPRINT_OK;
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int sprint_lmhead_confidence_noalloc(const void *h, const void *W, const float *temp,
                                                int M, int D, int V, int dtype,
                                                void *logits_out, float *conf_out,
                                                int32_t *argmax_out, int32_t *status,
                                                cudaStream_t stream) {
  if (M < 0 || D < 1 || V < 1) return SPRINT_ERR_INVALID_ARG;
  if (sprint_lmhead_workspace_bytes(M, D, V, dtype) > (size_t)SPRINT_NOALLOC_SCRATCH_BYTES)
    return SPRINT_ERR_TOO_LARGE;
  if (M == 0) return SPRINT_OK;
  int rc = SPRINT_OK;
  void *scratch = scratch_for_current_device(&rc);
  if (!scratch) return rc;
  return sprint_lmhead_confidence(h, W, temp, M, D, V, dtype, logits_out, conf_out, argmax_out,
                                  scratch, SPRINT_NOALLOC_SCRATCH_BYTES, status, stream);
}
