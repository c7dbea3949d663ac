// Non-uniform token unmasking.
//
// LLaDA2.0-Uni paper (arXiv 2604.20796), "Non-uniform Token Unmasking"
// paragraph: the fixed schedule unmasks ceil(m/T) tokens per step; SPRINT
// instead accepts, in one step, every masked position whose confidence
// exceeds tau, with at least ceil(m/(T-t)) acceptances per step so that
// every block finishes within T steps.
//
// One CTA per sequence, one thread per block position (LB <= 1024).  The
// rank of a masked position is the number of masked positions ahead of it
// in (confidence descending, position ascending) order, computed from a
// shared-memory copy of the block's confidences.
#include "common.cuh"
#include "unmask.cuh"

namespace sprint {

__global__ void unmask_kernel(const float *__restrict__ conf,
                              const int32_t *__restrict__ argmax,
                              uint8_t *__restrict__ mask, int32_t *__restrict__ tokens,
                              int32_t *__restrict__ m_out, int LB, int t, int T,
                              float tau, int mode, uint8_t *__restrict__ accepted_out,
                              int fresh, int32_t *status, Gate gate) {
  if (gate_closed(gate)) {  // the block finished earlier: nothing left to unmask
    unmask_gated(m_out, blockIdx.x, LB, accepted_out);
    return;
  }
  unmask_body(conf, argmax, mask, tokens, m_out, blockIdx.x, LB, t, T, tau, mode, accepted_out,
              fresh, status);
}

}  // namespace sprint

using namespace sprint;

int sprint::unmask_impl(const float *conf, const int32_t *argmax, uint8_t *mask, int32_t *tokens,
                        int32_t *m_out, int S, int LB, int t, int T, float tau, int mode,
                        uint8_t *accepted_out, int32_t *status, Gate gate,
                        cudaStream_t stream, int fresh) {
  if (S < 0 || LB < 1 || LB > 1024 || T < 1 || t < 0) return SPRINT_ERR_INVALID_ARG;
  if (mode != SPRINT_UNMASK_ADAPTIVE && mode != SPRINT_UNMASK_FIXED)
    return SPRINT_ERR_INVALID_ARG;
  if (S == 0) return SPRINT_OK;
  if (!conf || !argmax || !mask || !tokens || !m_out) return SPRINT_ERR_INVALID_ARG;
  const int threads = (LB + 31) / 32 * 32;
  unmask_kernel<<<S, threads, 0, stream>>>(conf, argmax, mask, tokens, m_out, LB, t, T, tau,
                                           mode, accepted_out, fresh, status, gate);
  return launch_status();
}

extern "C" int sprint_unmask(const float *conf, const int32_t *argmax, uint8_t *mask,
                             int32_t *tokens, int32_t *m_out, int S, int LB, int t, int T,
                             float tau, int mode, uint8_t *accepted_out, int32_t *status,
                             cudaStream_t stream) {
  return unmask_impl(conf, argmax, mask, tokens, m_out, S, LB, t, T, tau, mode, accepted_out,
                     status, Gate{nullptr, 0}, stream);
}
