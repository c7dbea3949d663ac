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

namespace sprint {

__global__ void unmask_kernel(const float *__restrict__ conf,
                              const int32_t *__restrict__ argmax,
                              uint8_t *__restrict__ mask, int32_t *__restrict__ tokens,
                              int32_t *__restrict__ m_out, int LB, int t, int T,
                              float tau, int mode, uint8_t *__restrict__ accepted_out,
                              int32_t *status, Gate gate) {
  if (gate_closed(gate)) {  // the block finished earlier: nothing left to unmask
    const size_t at = (size_t)blockIdx.x * LB + threadIdx.x;
    if (accepted_out && (int)threadIdx.x < LB) accepted_out[at] = 0;
    if (threadIdx.x == 0) m_out[blockIdx.x] = 0;
    return;
  }
  __shared__ float c_sh[1024];
  __shared__ uint8_t m_sh[1024];
  const int s = blockIdx.x, j = threadIdx.x;
  const size_t at = (size_t)s * LB + j;
  const bool active = j < LB;
  const float cj = active ? conf[at] : 0.f;
  const bool mj = active && mask[at] != 0;
  c_sh[j] = cj;
  m_sh[j] = mj;
  const int m = __syncthreads_count(mj);
  const int n_above = __syncthreads_count(mj && cj > tau);
  int rank = 0;
  if (mj)
    for (int i = 0; i < LB; ++i) {
      const float ci = c_sh[i];
      rank += m_sh[i] && (ci > cj || (ci == cj && i < j));
    }
  bool accept = false;
  if (mj) {
    if (mode == SPRINT_UNMASK_FIXED) {
      const int per_step = (LB + T - 1) / T;
      accept = rank < (per_step < m ? per_step : m);
    } else {
      const int left = T - t;
      const int k_min = left <= 1 ? m : (m + left - 1) / left;
      accept = n_above >= k_min ? cj > tau : rank < k_min;
    }
  }
  if (accept) {
    tokens[at] = argmax[at];
    mask[at] = 0;
  }
  if (active && accepted_out) accepted_out[at] = accept;
  const int n_acc = __syncthreads_count(accept);
  if (j == 0) m_out[s] = m - n_acc;
  if (kDebugChecks) {  // the count left equals the mask; unmasked positions hold tokens
    const bool still = active && mask[at] != 0;
    const int left = __syncthreads_count(still);
    if (j == 0) SPRINT_DCHECK(left == m - n_acc, status);
    if (active && !still) SPRINT_DCHECK(tokens[at] >= 0, status);
  }
}

}  // namespace sprint

using namespace sprint;

int sprint::unmask_impl(const float *conf, const int32_t *argmax, uint8_t *mask, int32_t *tokens,
                        int32_t *m_out, int S, int LB, int t, int T, float tau, int mode,
                        uint8_t *accepted_out, int32_t *status, Gate gate,
                        cudaStream_t stream) {
  if (S < 0 || LB < 1 || LB > 1024 || T < 1 || t < 0) return SPRINT_ERR_INVALID_ARG;
  if (mode != SPRINT_UNMASK_ADAPTIVE && mode != SPRINT_UNMASK_FIXED)
    return SPRINT_ERR_INVALID_ARG;
  if (S == 0) return SPRINT_OK;
  if (!conf || !argmax || !mask || !tokens || !m_out) return SPRINT_ERR_INVALID_ARG;
  const int threads = (LB + 31) / 32 * 32;
  unmask_kernel<<<S, threads, 0, stream>>>(conf, argmax, mask, tokens, m_out, LB, t, T, tau,
                                           mode, accepted_out, status, gate);
  return launch_status();
}

extern "C" int sprint_unmask(const float *conf, const int32_t *argmax, uint8_t *mask,
                             int32_t *tokens, int32_t *m_out, int S, int LB, int t, int T,
                             float tau, int mode, uint8_t *accepted_out, int32_t *status,
                             cudaStream_t stream) {
  return unmask_impl(conf, argmax, mask, tokens, m_out, S, LB, t, T, tau, mode, accepted_out,
                     status, Gate{nullptr, 0}, stream);
}
