// LM head reduced to top-1 softmax confidence and greedy token.
//
// LLaDA2.0-Uni paper (arXiv 2604.20796): c_i = max_v p(v | x_t) scores every
// prefix position ("Sparse Prefix Retention" paragraph) and c_n = p(x0_hat^n
// | x_t) drives unmasking ("Non-uniform Token Unmasking" paragraph).  With
// logits z_v = (h . W_v) / theta, c = 1 / sum_v exp(z_v - max z): the
// probability vector is never formed.
//
// Column tiles of kPartCols vocabulary entries each produce, per row, a
// partial (max of the raw fp32 dot products, sum of exp(z - z_tilemax),
// first column attaining the max); lmhead_combine_kernel folds the tiles in
// ascending order.  The bf16 path computes the tiles on the tcgen05 tensor
// cores (lmhead_tc.cu); this file holds the fp32 SIMT tile kernel, the
// combine kernel and the entry point.
#include <math.h>

#include "common.cuh"
#include "lmhead.cuh"

namespace sprint {

constexpr float kLog2e = 1.4426950408889634f;

// 64 x 64 output tile per pass, 4 passes cover one kPartCols strip.
template <typename T>
__global__ void __launch_bounds__(256)
lmhead_simt_kernel(const T *__restrict__ h, const T *__restrict__ W,
                   const float *__restrict__ temp, int M, int D, int V,
                   T *__restrict__ logits, float *__restrict__ pmax,
                   float *__restrict__ psum, int32_t *__restrict__ parg,
                   int32_t *status, Gate gate) {
  if (gate_closed(gate)) return;
  constexpr int BM = 64, BN = 64, BK = 16;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ float Zs[BM][BN + 1];
  __shared__ float r_max[BM], r_sum[BM], r_scale[BM], r_inv[BM];
  __shared__ int r_arg[BM];

  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * BM;
  const int strip = blockIdx.x;
  if (tid < BM) {
    const int row = m0 + tid;
    float th = 1.0f;
    if (temp && row < M) {
      th = temp[row];
      if (!(th > 0.0f) || !isfinite(th)) {
        report(status, SPRINT_STATUS_BAD_TEMPERATURE);
        th = 1.0f;
      }
    }
    r_inv[tid] = 1.0f / th;
    r_scale[tid] = kLog2e / th;
    r_max[tid] = -INFINITY;
    r_sum[tid] = 0.f;
    r_arg[tid] = 0;
  }
  for (int sub = 0; sub < kPartCols / BN; ++sub) {
    const int n0 = strip * kPartCols + sub * BN;
    if (n0 >= V) break;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < D; k0 += BK) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = tid + 256 * q, r = e >> 4, k = e & 15;
        const int gm = m0 + r, gn = n0 + r, gk = k0 + k;
        As[k][r] = (gm < M && gk < D) ? to_f32(h[(size_t)gm * D + gk]) : 0.f;
        Bs[k][r] = (gn < V && gk < D) ? to_f32(W[(size_t)gn * D + gk]) : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < BK; ++k) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) { a[i] = As[k][ty * 4 + i]; b[i] = Bs[k][tx * 4 + i]; }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = ty * 4 + i, c = tx * 4 + j;
        Zs[r][c] = acc[i][j];
        if (logits && m0 + r < M && n0 + c < V)
          logits[(size_t)(m0 + r) * V + n0 + c] = from_f32<T>(acc[i][j] * r_inv[r]);
      }
    __syncthreads();
    if (tid < BM) {
      const int ncols = V - n0 < BN ? V - n0 : BN;
      float mx = Zs[tid][0];
      int am = 0;
      for (int c = 1; c < ncols; ++c)
        if (Zs[tid][c] > mx) { mx = Zs[tid][c]; am = c; }
      const float sc = r_scale[tid];
      const float new_max = fmaxf(r_max[tid], mx);
      float sum = r_sum[tid] * exp2f((r_max[tid] - new_max) * sc);
      for (int c = 0; c < ncols; ++c) sum += exp2f((Zs[tid][c] - new_max) * sc);
      if (mx > r_max[tid]) r_arg[tid] = n0 + am;
      r_max[tid] = new_max;
      r_sum[tid] = sum;
    }
    __syncthreads();
  }
  if (tid < BM && m0 + tid < M) {
    const size_t at = (size_t)strip * M + m0 + tid;
    pmax[at] = r_max[tid];
    psum[at] = r_sum[tid];
    if (parg) parg[at] = r_arg[tid];
  }
}

struct Part {
  float m, s;
  int a;
};

// Fold of two partials of one row: max, rescaled sum, lowest column on ties.
__device__ __forceinline__ Part fold(Part x, Part y, float sc) {
  if (x.m == -INFINITY) return y;
  if (y.m == -INFINITY) return x;
  const float m = fmaxf(x.m, y.m);
  Part r;
  r.m = m;
  r.s = x.s * exp2f((x.m - m) * sc) + y.s * exp2f((y.m - m) * sc);
  r.a = x.m > y.m ? x.a : (y.m > x.m ? y.a : min(x.a, y.a));
  return r;
}

// Debug build: a row's greedy token lies in [0, V) and its confidence, a
// maximum probability, in [1/V, 1] (with room for rounding).
__device__ __forceinline__ void debug_check_row(float c, int a, int V, int32_t *status) {
  (void)c; (void)a; (void)V; (void)status;
  SPRINT_DCHECK(a >= 0 && a < V, status);
  SPRINT_DCHECK(c >= (1.0f / (float)V) * (1.0f - 1e-3f) && c <= 1.0f + 1e-5f, status);
}

// Many rows: a CTA of 32 rows x 8 strip groups.  Thread (x, y) folds strips
// y, y + 8, ... of row x (loads coalesced over x), then the 8 group partials
// of each row are folded in ascending y.  Deterministic for given M, V.
constexpr int kCombRows = 32, kCombGroups = 8;

__global__ void __launch_bounds__(kCombRows * kCombGroups)
lmhead_combine_kernel(const float *__restrict__ pmax, const float *__restrict__ psum,
                      const int32_t *__restrict__ parg, const float *__restrict__ temp, int M,
                      int strips, int V, float *__restrict__ conf, int32_t *__restrict__ argmax,
                      int32_t *status, Gate gate) {
  if (gate_closed(gate)) return;
  __shared__ Part sh[kCombGroups][kCombRows];
  const int x = threadIdx.x, y = threadIdx.y;
  const int row = blockIdx.x * kCombRows + x;
  float th = 1.0f;
  if (row < M && temp) th = temp[row];
  if (!(th > 0.0f) || !isfinite(th)) th = 1.0f;
  const float sc = kLog2e / th;
  Part acc{-INFINITY, 0.f, 0};
  if (row < M) {
#pragma unroll 4
    for (int t = y; t < strips; t += kCombGroups) {
      const size_t at = (size_t)t * M + row;
      acc = fold(acc, Part{pmax[at], psum[at], parg ? parg[at] : 0}, sc);
    }
  }
  sh[y][x] = acc;
  __syncthreads();
  if (y == 0 && row < M) {
    Part r = sh[0][x];
#pragma unroll
    for (int g = 1; g < kCombGroups; ++g) r = fold(r, sh[g][x], sc);
    conf[row] = 1.0f / r.s;
    if (argmax) argmax[row] = r.a;
    debug_check_row(1.0f / r.s, argmax ? r.a : 0, V, status);
  }
}

// Few rows: one CTA per row, threads stride over the strips, then a fixed
// shuffle/shared-memory tree (deterministic).
__global__ void __launch_bounds__(128)
lmhead_combine_rows_kernel(const float *__restrict__ pmax, const float *__restrict__ psum,
                           const int32_t *__restrict__ parg, const float *__restrict__ temp,
                           int M, int strips, int V, float *__restrict__ conf,
                           int32_t *__restrict__ argmax, int32_t *status, Gate gate) {
  if (gate_closed(gate)) return;
  __shared__ Part sh[4];
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float th = temp ? temp[row] : 1.0f;
  if (!(th > 0.0f) || !isfinite(th)) th = 1.0f;
  const float sc = kLog2e / th;
  Part acc{-INFINITY, 0.f, 0};
  for (int t = tid; t < strips; t += 128) {
    const size_t at = (size_t)t * M + row;
    acc = fold(acc, Part{pmax[at], psum[at], parg ? parg[at] : 0}, sc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Part y{__shfl_xor_sync(0xffffffffu, acc.m, o), __shfl_xor_sync(0xffffffffu, acc.s, o),
           __shfl_xor_sync(0xffffffffu, acc.a, o)};
    acc = (lane & o) ? fold(y, acc, sc) : fold(acc, y, sc);
  }
  if (lane == 0) sh[warp] = acc;
  __syncthreads();
  if (tid == 0) {
    Part r = fold(fold(sh[0], sh[1], sc), fold(sh[2], sh[3], sc), sc);
    conf[row] = 1.0f / r.s;
    if (argmax) argmax[row] = r.a;
    debug_check_row(1.0f / r.s, argmax ? r.a : 0, V, status);
  }
}

LmheadWs lmhead_ws_layout(void *ws, int M, int V, int cols) {
  const int strips = (V + cols - 1) / cols;
  const size_t one = align_up((size_t)strips * M * 4, 256);
  char *p = static_cast<char *>(ws);
  return {reinterpret_cast<float *>(p), reinterpret_cast<float *>(p + one),
          reinterpret_cast<int32_t *>(p + 2 * one), strips, cols};
}

}  // namespace sprint

using namespace sprint;

extern "C" size_t sprint_lmhead_workspace_bytes(int M, int D, int V, int dtype) {
  (void)D;
  if (M < 0 || V < 1) return 0;
  const int cols = lmhead_strip_cols(M, dtype);
  const int strips = (V + cols - 1) / cols;
  return 3 * align_up((size_t)strips * M * 4, 256);
}

int sprint::lmhead_confidence_impl(const void *h, const void *W, const float *temp, int M,
                                   int D, int V, int dtype, void *logits_out, float *conf_out,
                                   int32_t *argmax_out, void *ws, size_t ws_bytes,
                                   int32_t *status, Gate gate, cudaStream_t stream) {
  if (M < 0 || D < 1 || V < 1) return SPRINT_ERR_INVALID_ARG;
  if (dtype != SPRINT_F32 && dtype != SPRINT_BF16) return SPRINT_ERR_INVALID_ARG;
  if (M == 0) return SPRINT_OK;
  if (!h || !W || !conf_out || !ws || !status) return SPRINT_ERR_INVALID_ARG;
  if (ws_bytes < sprint_lmhead_workspace_bytes(M, D, V, dtype)) return SPRINT_ERR_WORKSPACE;
  LmheadWs p = lmhead_ws_layout(ws, M, V, lmhead_strip_cols(M, dtype));
  if (!argmax_out) p.parg = nullptr;  // no greedy token wanted: skip its tracking
  if (dtype == SPRINT_BF16) {
    if (D % 8 != 0 || !aligned16(h) || !aligned16(W)) return SPRINT_ERR_UNSUPPORTED;
    const int rc = lmhead_tc_tiles(static_cast<const __nv_bfloat16 *>(h),
                                   static_cast<const __nv_bfloat16 *>(W), temp, M, D, V,
                                   static_cast<__nv_bfloat16 *>(logits_out), p, status, gate,
                                   stream);
    if (rc != SPRINT_OK) return rc;
  } else {
    dim3 grid(p.strips, (M + 63) / 64);
    lmhead_simt_kernel<float><<<grid, 256, 0, stream>>>(
        static_cast<const float *>(h), static_cast<const float *>(W), temp, M, D, V,
        static_cast<float *>(logits_out), p.pmax, p.psum, p.parg, status, gate);
    if (launch_status() != SPRINT_OK) return SPRINT_ERR_CUDA;
  }
  if (M < 4096)
    lmhead_combine_rows_kernel<<<M, 128, 0, stream>>>(p.pmax, p.psum, p.parg, temp, M, p.strips,
                                                      V, conf_out, argmax_out, status, gate);
  else
    lmhead_combine_kernel<<<(M + kCombRows - 1) / kCombRows, dim3(kCombRows, kCombGroups), 0,
                            stream>>>(p.pmax, p.psum, p.parg, temp, M, p.strips, V, conf_out,
                                      argmax_out, status, gate);
  return launch_status();
}

extern "C" int sprint_lmhead_confidence(const void *h, const void *W, const float *temp,
                                        int M, int D, int V, int dtype, void *logits_out,
                                        float *conf_out, int32_t *argmax_out, void *ws,
                                        size_t ws_bytes, int32_t *status,
                                        cudaStream_t stream) {
  return lmhead_confidence_impl(h, W, temp, M, D, V, dtype, logits_out, conf_out, argmax_out, ws,
                                ws_bytes, status, Gate{nullptr, 0}, stream);
}
