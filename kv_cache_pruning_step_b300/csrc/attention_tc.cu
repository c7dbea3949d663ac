// bf16 attention chunks.  Placeholder that routes to the CUDA-core chunk
// kernel until the tcgen05 kernel is in place.
#include "attention.cuh"
#include "common.cuh"

int sprint::attn_tc_chunk_keys(int S, int NL, int Hkv, int LB, int max_kv_rows) {
  return attn_chunk_keys(S, NL, Hkv, LB, max_kv_rows, 4 * 148);
}

int sprint::attn_tc_chunks(const __nv_bfloat16 *Q, const __nv_bfloat16 *Kp,
                           const __nv_bfloat16 *Vp, const int32_t *kv_off, int total_kv_rows,
                           const __nv_bfloat16 *Kb, const __nv_bfloat16 *Vb, int S, int NL,
                           int LB, int Hq, int Hkv, int d, const AttnWs &w, int32_t *status,
                           cudaStream_t stream) {
  return attn_simt_chunks_bf16(Q, Kp, Vp, kv_off, total_kv_rows, Kb, Vb, S, NL, LB, Hq, Hkv, d,
                               w, status, stream);
}
