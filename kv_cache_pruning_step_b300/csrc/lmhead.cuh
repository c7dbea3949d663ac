// Internal interface between the LM-head entry point and its tile kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace sprint {

// Vocabulary columns folded into one (max, sum-exp, argmax) partial per row
// (the tensor-core tile width in bf16): 256 by default; 224 for bf16 calls
// with few rows (block steps), where the column tiles are the whole grid's
// work, 702 tiles of 224 spread over 148 SMs more evenly than 614 of 256,
// and a 44 KB stage leaves room for a 5-deep TMA ring.  (For many rows the
// 256-wide MMA is the faster one.)
constexpr int kPartCols = 256;
constexpr int kPartColsNarrow = 224;
constexpr int kNarrowMaxRows = 4096;

inline int lmhead_strip_cols(int M, int dtype) {
  return dtype == SPRINT_BF16 && M < kNarrowMaxRows ? kPartColsNarrow : kPartCols;
}

struct LmheadWs {
  float *pmax;    // [strips][M] max of the raw fp32 dot products in the strip
  float *psum;    // [strips][M] sum of exp(z - z_stripmax) over the strip
  int32_t *parg;  // [strips][M] first column attaining the strip max
                  // (nullptr: the caller wants no greedy token)
  int strips;     // ceil(V / cols)
  int cols;       // vocabulary columns per strip
};

LmheadWs lmhead_ws_layout(void *ws, int M, int V, int cols);

// bf16 tiles on the tcgen05 tensor cores; writes the strip partials (and
// the temperature-scaled logits when `logits` is not null).
int lmhead_tc_tiles(const __nv_bfloat16 *h, const __nv_bfloat16 *W, const float *temp, int M,
                    int D, int V, __nv_bfloat16 *logits, const LmheadWs &p, int32_t *status,
                    Gate gate, cudaStream_t stream);

}  // namespace sprint
