// The unmask step of one sequence, shared by the unmask kernel and the
// native driver's fused combine-and-unmask kernel (lmhead.cu).
//
// LLaDA2.0-Uni paper (arXiv 2604.20796), "Non-uniform Token Unmasking"
// paragraph: accept every masked position whose confidence exceeds tau,
// at least ceil(m / (T - t)) of them per step (the most confident first);
// the fixed schedule accepts ceil(LB / T) per step.
#pragma once

#include "common.cuh"

namespace sprint {

// One unmask step of sequence s by the calling CTA (blockDim.x >= LB, every
// thread calls it): thread j < LB handles block position j.  fresh: the
// block's first step, every position masked whatever mask[] holds (the
// native driver then needs no separate initialisation of mask and tokens);
// positions not accepted get token -1.
__device__ __forceinline__ void unmask_body(const float *__restrict__ conf,
                                            const int32_t *__restrict__ argmax,
                                            uint8_t *__restrict__ mask,
                                            int32_t *__restrict__ tokens,
                                            int32_t *__restrict__ m_out, int s, int LB, int t,
                                            int T, float tau, int mode,
                                            uint8_t *__restrict__ accepted_out, int fresh,
                                            int32_t *status) {
  __shared__ float c_sh[1024];
  __shared__ uint8_t m_sh[1024];
  const int j = threadIdx.x;
  const size_t at = (size_t)s * LB + j;
  const bool active = j < LB;
  const float cj = active ? conf[at] : 0.f;
  const bool mj = active && (fresh || mask[at] != 0);
  if (active) {
    c_sh[j] = cj;
    m_sh[j] = mj;
  }
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
  } else if (fresh && active) {
    tokens[at] = -1;
    mask[at] = 1;
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

// Gated step of the native driver: the block finished at an earlier step.
__device__ __forceinline__ void unmask_gated(int32_t *__restrict__ m_out, int s, int LB,
                                             uint8_t *__restrict__ accepted_out) {
  const size_t at = (size_t)s * LB + threadIdx.x;
  if (accepted_out && (int)threadIdx.x < LB) accepted_out[at] = 0;
  if (threadIdx.x == 0) m_out[s] = 0;
}

}  // namespace sprint
