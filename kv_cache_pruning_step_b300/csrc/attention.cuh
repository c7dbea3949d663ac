// Internal interface between the attention entry point and its chunk kernels.
#pragma once

#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace sprint {

// Split-KV partials: unit u = ((s * NL + l) * Hkv + g) * chunks + chunk holds
// R = LB * Hq / Hkv rows of (unnormalised O row [d], row max in log2 units,
// row sum of exp2(score - max)).
struct AttnWs {
  float *o;        // [units][R][d]
  float *ml;       // [units][R][2]
  int chunks;      // key chunks per (sequence, layer, KV head)
  int chunk_keys;  // keys per chunk
  size_t bytes;    // workspace bytes of this layout
};

AttnWs attn_ws_layout(void *ws, int S, int NL, int LB, int Hq, int Hkv, int d, int max_kv_rows,
                      int chunk_keys);
int attn_chunk_keys(int S, int NL, int Hkv, int LB, int max_kv_rows, int target_units);

// bf16 path on the tcgen05 tensor cores (attention_tc.cu): workspace size
// and the whole call (chunk kernel and combine).
size_t attn_tc_workspace_bytes(int S, int NL, int Hkv, int d);
int attn_tc_forward(const __nv_bfloat16 *Q, const __nv_bfloat16 *Kp, const __nv_bfloat16 *Vp,
                    const int32_t *kv_off, int total_kv_rows, const __nv_bfloat16 *Kb,
                    const __nv_bfloat16 *Vb, int S, int NL, int LB, int Hq, int Hkv, int d,
                    void *O, void *ws, int32_t *status, KvIndex kvi, AttnResidual res,
                    Gate gate, cudaStream_t stream, SideStream side);
// The prefix's own attention (bf16, tcgen05; attention_tc.cu).
int attn_tc_prefix(const __nv_bfloat16 *Qp, const __nv_bfloat16 *K, const __nv_bfloat16 *V,
                   const int32_t *prefix_off, int total_rows, int S, int NL, int Hq, int Hkv,
                   int d, __nv_bfloat16 *Op, int32_t *status, cudaStream_t stream);

}  // namespace sprint
