// Pruned prefix KV cache: gather of the kept rows of K and V.
//
// LLaDA2.0-Uni paper (arXiv 2604.20796), "Sparse Prefix Retention"
// paragraph: a pruned prefix KV cache is built once per block and every
// later step attends to it; evicted positions are dropped.
//
// HBM-bound copy.  One warp per kept position moves that position's row of
// every layer for K and for V (2 x NL rows of Hkv*d elements) with 16-byte
// loads and stores; all four 16-byte chunks of a lane for one layer (K and
// V) are loaded before any is stored, so each warp keeps 2 KB in flight.
#include "common.cuh"

namespace sprint {

__global__ void __launch_bounds__(256)
compact_kernel(const uint4 *__restrict__ K, const uint4 *__restrict__ V,
               const int32_t *__restrict__ prefix_off, int total_rows,
               const int32_t *__restrict__ kept_idx,
               const int32_t *__restrict__ kept_off, int S, int total_kept, int NL,
               int row_vecs, uint4 *__restrict__ Kp, uint4 *__restrict__ Vp,
               int32_t *status) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int g = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; g < total_kept; g += warps) {
    const int s = csr_owner(kept_off, S, g);
    const int k0 = __ldg(kept_off + s), k1 = __ldg(kept_off + s + 1);
    const int p0 = __ldg(prefix_off + s), p1 = __ldg(prefix_off + s + 1);
    if (k0 < 0 || k1 > total_kept || g < k0 || g >= k1 || p0 < 0 || p1 < p0 ||
        p1 > total_rows) {
      if (lane == 0) report(status, SPRINT_STATUS_BAD_OFFSETS);
      continue;
    }
    const int n = p1 - p0, ks = k1 - k0, j = g - k0;
    const int idx = __ldg(kept_idx + g);
    // Kept indices are stored in ascending position order.
    if (kDebugChecks && lane == 0 && j > 0) SPRINT_DCHECK(__ldg(kept_idx + g - 1) < idx, status);
    if (idx < 0 || idx >= n) {
      if (lane == 0) report(status, SPRINT_STATUS_BAD_INDEX);
      continue;
    }
    for (int l = 0; l < NL; ++l) {
      const size_t src = ((size_t)NL * p0 + (size_t)l * n + idx) * row_vecs;
      const size_t dst = ((size_t)NL * k0 + (size_t)l * ks + j) * row_vecs;
      for (int v = lane; v < row_vecs; v += 64) {
        const bool two = v + 32 < row_vecs;
        uint4 a = __ldg(K + src + v), b = __ldg(V + src + v), c, e;
        if (two) { c = __ldg(K + src + v + 32); e = __ldg(V + src + v + 32); }
        Kp[dst + v] = a;
        Vp[dst + v] = b;
        if (two) { Kp[dst + v + 32] = c; Vp[dst + v + 32] = e; }
      }
    }
  }
}

}  // namespace sprint

using namespace sprint;

extern "C" int sprint_compact_kv(const void *K, const void *V, int S,
                                 const int32_t *prefix_off, int total_rows, int NL,
                                 int Hkv, int d, int dtype, const int32_t *kept_idx,
                                 const int32_t *kept_off, int total_kept, void *Kp,
                                 void *Vp, int32_t *status, cudaStream_t stream) {
  if (S < 0 || total_rows < 0 || total_kept < 0 || NL < 1 || Hkv < 1 || d < 1)
    return SPRINT_ERR_INVALID_ARG;
  if (dtype != SPRINT_F32 && dtype != SPRINT_BF16) return SPRINT_ERR_INVALID_ARG;
  if (S == 0 || total_kept == 0) return SPRINT_OK;
  if (!K || !V || !prefix_off || !kept_idx || !kept_off || !Kp || !Vp || !status)
    return SPRINT_ERR_INVALID_ARG;
  const size_t row_bytes = (size_t)Hkv * d * (dtype == SPRINT_BF16 ? 2 : 4);
  if (row_bytes % 16 != 0 || !aligned16(K) || !aligned16(V) || !aligned16(Kp) ||
      !aligned16(Vp))
    return SPRINT_ERR_UNSUPPORTED;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int blocks = (total_kept + 7) / 8;
  blocks = blocks < sms * 8 ? blocks : sms * 8;
  compact_kernel<<<blocks, 256, 0, stream>>>(
      static_cast<const uint4 *>(K), static_cast<const uint4 *>(V), prefix_off, total_rows,
      kept_idx, kept_off, S, total_kept, NL, (int)(row_bytes / 16), static_cast<uint4 *>(Kp),
      static_cast<uint4 *>(Vp), status);
  return launch_status();
}
