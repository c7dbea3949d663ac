// Native block driver: all denoising steps of one block enqueued at once.
//
// LLaDA2.0-Uni paper (arXiv 2604.20796), Sparse Prefix Retention and
// Non-uniform Token Unmasking paragraphs: a block of LB masked tokens is
// decoded in at most T steps; step 0 attends to the full prefix, later steps
// to the pruned one; each step unmasks at least ceil(m / (T - t)) positions.
//
// The host enqueues the T steps back to back; whether a step runs is decided
// on the GPU from the previous step's still-masked counts (the step gate in
// every kernel), so no step waits for a host round trip.
#include <mutex>

#include "common.cuh"

using namespace sprint;

namespace {

int record(void *const *events, int i, cudaStream_t stream) {
  if (!events || !events[i]) return SPRINT_OK;
  return cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) == cudaSuccess
             ? SPRINT_OK
             : SPRINT_ERR_CUDA;
}

// Without the residual chain nothing of a step reads the attention output,
// so each step's attention combine runs on a side stream while the LM head
// streams W.  One side stream and two events per device, made on first use;
// the mutex keeps calls from different host threads from interleaving their
// event records (the side stream then orders their combines one after the
// other, which is correct, if not concurrent).
struct SideSet {
  std::mutex mu;
  cudaStream_t side[PerDevice::kMax] = {};
  cudaEvent_t fork[PerDevice::kMax] = {}, join[PerDevice::kMax] = {};
};

SideSet &side_set() {
  static SideSet s;
  return s;
}

// Under ss.mu.
bool side_streams(SideSet &ss, int dev, SideStream *out) {
  if (!ss.fork[dev] && cudaEventCreateWithFlags(&ss.fork[dev], cudaEventDisableTiming) != cudaSuccess) {
    ss.fork[dev] = nullptr;
    return false;
  }
  if (!ss.join[dev] && cudaEventCreateWithFlags(&ss.join[dev], cudaEventDisableTiming) != cudaSuccess) {
    ss.join[dev] = nullptr;
    return false;
  }
  if (!ss.side[dev] && cudaStreamCreateWithFlags(&ss.side[dev], cudaStreamNonBlocking) != cudaSuccess) {
    ss.side[dev] = nullptr;
    return false;
  }
  *out = SideStream{ss.side[dev], ss.fork[dev], ss.join[dev]};
  return true;
}

}  // namespace

static int decode_steps_on(const sprint_steps_args *a, SideStream side, cudaStream_t stream);

extern "C" int sprint_decode_steps(const sprint_steps_args *a, cudaStream_t stream) {
  if (!a) return SPRINT_ERR_INVALID_ARG;
  if (a->S < 1 || a->LB < 1 || a->T < 1) return SPRINT_ERR_INVALID_ARG;
  if (!a->Q || !a->Kb || !a->Vb || !a->h || !a->mask || !a->tokens || !a->m_hist || !a->O ||
      !a->conf || !a->argmax || !a->status || !a->W)
    return SPRINT_ERR_INVALID_ARG;
  for (int t = 0; t < a->T; ++t)
    if (!a->Q[t] || !a->Kb[t] || !a->Vb[t] || !a->h[t]) return SPRINT_ERR_INVALID_ARG;
  if (a->residual && (!a->h_res || a->Hq * a->d != a->D)) return SPRINT_ERR_INVALID_ARG;
  if (a->residual && a->step0_given) return SPRINT_ERR_INVALID_ARG;
  SideStream side{nullptr, nullptr, nullptr};
  std::unique_lock<std::mutex> side_lock;
  if (!a->residual && a->dtype == SPRINT_BF16) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= PerDevice::kMax)
      return SPRINT_ERR_CUDA;
    SideSet &ss = side_set();
    side_lock = std::unique_lock<std::mutex>(ss.mu);
    if (!side_streams(ss, dev, &side)) return SPRINT_ERR_CUDA;
  }
  const int rc_all = decode_steps_on(a, side, stream);
  // The call's stream ends after the last combine, whatever happened.
  if (side.side && cudaStreamWaitEvent(stream, side.join, 0) != cudaSuccess && rc_all == SPRINT_OK)
    return SPRINT_ERR_CUDA;
  return rc_all;
}

static int decode_steps_on(const sprint_steps_args *a, SideStream side, cudaStream_t stream) {
  const int S = a->S, LB = a->LB, M = S * LB;
  // Fewer than 4096 block rows and blocks of at most kFusedMaxLB positions:
  // the LM head's strip partials are folded and the block unmasked by one
  // kernel per step.  Step 0's unmask starts from an all-masked block, so
  // mask and tokens need no separate initialisation.
  const bool fused = M < 4096 && LB <= kFusedMaxLB;
  for (int t = 0; t < a->T; ++t) {
    const Gate gate = t == 0 ? Gate{nullptr, 0} : Gate{a->m_hist + (size_t)(t - 1) * S, S};
    const bool full = t == 0, indexed = !full && a->kept_idx;
    const KvIndex kvi = indexed ? KvIndex{a->kept_idx, a->prefix_off, a->total_rows}
                                : KvIndex{nullptr, nullptr, 0};
    int rc = SPRINT_OK;
    // The previous step's combine has read the attention workspace.
    if (t > 0 && side.side && cudaStreamWaitEvent(stream, side.join, 0) != cudaSuccess)
      rc = SPRINT_ERR_CUDA;
    if (rc == SPRINT_OK) rc = record(a->events, 6 * t + 0, stream);
    if (rc == SPRINT_OK)
      rc = block_attn_impl(a->Q[t], full || indexed ? a->Kf : a->Kp,
                           full || indexed ? a->Vf : a->Vp, full ? a->prefix_off : a->kept_off,
                           full ? a->max_rows : a->max_kept,
                           full ? a->total_rows : a->total_kept, a->Kb[t], a->Vb[t], S, a->NL,
                           LB, a->Hq, a->Hkv, a->d, a->dtype, a->O, a->ws_attn,
                           a->ws_attn_bytes, a->status, kvi,
                           a->residual ? AttnResidual{a->h[t], a->h_res}
                                       : AttnResidual{nullptr, nullptr},
                           gate, stream, side);
    if (rc == SPRINT_OK) rc = record(a->events, 6 * t + 1, stream);
    if (rc == SPRINT_OK) rc = record(a->events, 6 * t + 2, stream);
    const void *h = a->residual ? a->h_res : a->h[t];
    const float *theta = a->theta ? a->theta[t] : nullptr;
    uint8_t *acc = a->accepted ? a->accepted + (size_t)t * M : nullptr;
    int32_t *m_t = a->m_hist + (size_t)t * S;
    const int fresh = t == 0;
    const bool head = !(t == 0 && a->step0_given);
    if (fused && head) {
      // the LM-head tiles, then one kernel folding the rows and unmasking
      // (its time is counted in the LM-head stage; the unmask events mark
      // an empty interval)
      if (rc == SPRINT_OK)
        rc = lmhead_tiles_impl(h, a->W, theta, M, a->D, a->vocab, a->dtype, a->logits, true,
                               a->ws_lm, a->ws_lm_bytes, a->status, gate, stream);
      if (rc == SPRINT_OK)
        rc = combine_unmask_impl(a->ws_lm, theta, S, LB, a->vocab, a->dtype, a->conf, a->argmax,
                                 a->mask, a->tokens, m_t, t, a->T, a->tau, a->mode, acc, fresh,
                                 a->status, gate, stream);
      if (rc == SPRINT_OK) rc = record(a->events, 6 * t + 3, stream);
      if (rc == SPRINT_OK) rc = record(a->events, 6 * t + 4, stream);
    } else {
      if (rc == SPRINT_OK && head)
        rc = lmhead_confidence_impl(h, a->W, theta, M, a->D, a->vocab, a->dtype, a->logits,
                                    a->conf, a->argmax, a->ws_lm, a->ws_lm_bytes, a->status,
                                    gate, stream);
      if (rc == SPRINT_OK) rc = record(a->events, 6 * t + 3, stream);
      if (rc == SPRINT_OK) rc = record(a->events, 6 * t + 4, stream);
      if (rc == SPRINT_OK)
        rc = unmask_impl(a->conf, a->argmax, a->mask, a->tokens, m_t, S, LB, t, a->T, a->tau,
                         a->mode, acc, a->status, gate, stream, fresh);
    }
    if (rc == SPRINT_OK) rc = record(a->events, 6 * t + 5, stream);
    if (rc != SPRINT_OK) return rc;
  }
  return SPRINT_OK;
}
