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

#include <cooperative_groups.h>

#include "common.cuh"
#include "unmask.cuh"
#include "lmhead.cuh"

namespace sprint {

namespace cg = cooperative_groups;

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

__device__ __forceinline__ float row_scale(const float *__restrict__ temp, int row) {
  float th = temp ? temp[row] : 1.0f;
  if (!(th > 0.0f) || !isfinite(th)) th = 1.0f;
  return kLog2e / th;
}

// Few rows (M < 4096): the strip partials of a tile of up to 32 rows are
// folded by a cluster of kFoldCtas CTAs.  Strip group g < kFoldGroups folds
// strips g, g + kFoldGroups, ... of each row in order; the groups' partials
// are then folded by a complete binary tree over the groups in order, the
// lower group always the first operand (a fixed tree: deterministic, ties to
// the lowest column).  CTA r holds groups [r G, r G + G) (G =
// kGroupsPerCta, one warp per group, lane = row of the tile) and folds their
// subtree in shared memory; rank 0 folds the CTAs' subtrees, which the other
// CTAs write into its shared memory.
constexpr int kFoldCtas = 8, kGroupsPerCta = 16, kFoldGroups = kFoldCtas * kGroupsPerCta;
constexpr int kFoldThreads = 32 * kGroupsPerCta;
static_assert(kFoldThreads == kFusedMaxLB, "one unmask thread per block position");

struct FoldSmem {
  float m[kGroupsPerCta][33], s[kGroupsPerCta][33];
  int a[kGroupsPerCta][33];
  float cm[kFoldCtas][32], cs[kFoldCtas][32];  // the CTAs' subtrees (read in rank 0)
  int ca[kFoldCtas][32];
};

// Every thread of every CTA of the cluster calls it; warp 0 of rank 0 gets
// the row's partial (lane = row of the tile).
__device__ __forceinline__ Part fold_rows_cluster(cg::cluster_group &cluster,
                                                  const float *__restrict__ pmax,
                                                  const float *__restrict__ psum,
                                                  const int32_t *__restrict__ parg, int M,
                                                  int strips, int row0, int nrows, float sc,
                                                  FoldSmem &sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned rank = cluster.block_rank();
  const int g = (int)rank * kGroupsPerCta + w;
  Part acc{-INFINITY, 0.f, 0};
  if (lane < nrows) {
    const int row = row0 + lane;
#pragma unroll 8
    for (int t = g; t < strips; t += kFoldGroups) {
      const size_t at = (size_t)t * M + row;
      acc = fold(acc, Part{pmax[at], psum[at], parg ? parg[at] : 0}, sc);
    }
  }
  sh.m[w][lane] = acc.m;
  sh.s[w][lane] = acc.s;
  sh.a[w][lane] = acc.a;
  __syncthreads();
#pragma unroll
  for (int o = 1; o < kGroupsPerCta; o <<= 1) {
    if ((w & (2 * o - 1)) == 0) {
      acc = fold(acc, Part{sh.m[w + o][lane], sh.s[w + o][lane], sh.a[w + o][lane]}, sc);
      sh.m[w][lane] = acc.m;
      sh.s[w][lane] = acc.s;
      sh.a[w][lane] = acc.a;
    }
    __syncthreads();
  }
  if (w == 0) {
    FoldSmem *dst = cluster.map_shared_rank(&sh, 0);
    dst->cm[rank][lane] = acc.m;
    dst->cs[rank][lane] = acc.s;
    dst->ca[rank][lane] = acc.a;
  }
  cluster.sync();  // rank 0 holds every CTA's subtree
  if (rank == 0 && w == 0) {
    Part p[kFoldCtas];
#pragma unroll
    for (int c = 0; c < kFoldCtas; ++c) p[c] = Part{sh.cm[c][lane], sh.cs[c][lane], sh.ca[c][lane]};
#pragma unroll
    for (int o = 1; o < kFoldCtas; o <<= 1)
#pragma unroll
      for (int c = 0; c < kFoldCtas; c += 2 * o) p[c] = fold(p[c], p[c + o], sc);
    acc = p[0];
  }
  return acc;
}

// One cluster per tile of 32 rows.
__global__ void __launch_bounds__(kFoldThreads)
lmhead_combine_rows_kernel(const float *__restrict__ pmax, const float *__restrict__ psum,
                           const int32_t *__restrict__ parg, const float *__restrict__ temp,
                           int M, int strips, int V, float *__restrict__ conf,
                           int32_t *__restrict__ argmax, int32_t *status, Gate gate) {
  if (gate_closed(gate)) return;  // the same decision in every CTA of the cluster
  __shared__ FoldSmem sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int row0 = (int)(blockIdx.x / kFoldCtas) * 32, nrows = min(32, M - row0);
  const int row = row0 + min((int)(threadIdx.x & 31), nrows - 1);
  const Part r = fold_rows_cluster(cluster, pmax, psum, parg, M, strips, row0, nrows,
                                   row_scale(temp, row), sh);
  if (cluster.block_rank() == 0 && (int)threadIdx.x < nrows) {
    conf[row] = 1.0f / r.s;
    if (argmax) argmax[row] = r.a;
    debug_check_row(1.0f / r.s, argmax ? r.a : 0, V, status);
  }
}

// Native block driver: one cluster per sequence folds the strip partials of
// the sequence's LB rows (32 rows at a time, exactly as
// lmhead_combine_rows_kernel); rank 0 (blockDim.x = 512 >= LB) then takes
// the step's unmask decision for the block (exactly as unmask_kernel): one
// launch instead of two.
__global__ void __launch_bounds__(kFoldThreads)
lmhead_combine_unmask_kernel(const float *__restrict__ pmax, const float *__restrict__ psum,
                             const int32_t *__restrict__ parg, const float *__restrict__ temp,
                             int LB, int M, int strips, int V, float *__restrict__ conf,
                             int32_t *__restrict__ argmax, uint8_t *__restrict__ mask,
                             int32_t *__restrict__ tokens, int32_t *__restrict__ m_out, int t,
                             int T, float tau, int mode, uint8_t *__restrict__ accepted_out,
                             int fresh, int32_t *status, Gate gate) {
  cg::cluster_group cluster = cg::this_cluster();
  const bool lead = cluster.block_rank() == 0;
  const int s = (int)(blockIdx.x / kFoldCtas);
  if (gate_closed(gate)) {
    if (lead) unmask_gated(m_out, s, LB, accepted_out);
    return;
  }
  __shared__ FoldSmem sh;
  const int lane = threadIdx.x & 31;
  for (int j0 = 0; j0 < LB; j0 += 32) {
    if (j0) cluster.sync();  // rank 0 has read the previous tile's subtrees
    const int row0 = s * LB + j0, nrows = min(32, LB - j0);
    const int row = row0 + min(lane, nrows - 1);
    const Part r = fold_rows_cluster(cluster, pmax, psum, parg, M, strips, row0, nrows,
                                     row_scale(temp, row), sh);
    if (lead && (int)threadIdx.x < nrows) {
      conf[row] = 1.0f / r.s;
      argmax[row] = r.a;
      debug_check_row(1.0f / r.s, r.a, V, status);
    }
  }
  if (!lead) return;
  __syncthreads();  // the block's confidences are written (read back from global below)
  unmask_body(conf, argmax, mask, tokens, m_out, s, LB, t, T, tau, mode, accepted_out, fresh,
              status);
}

template <typename... KArgs, typename... Args>
int launch_fold(void (*kern)(KArgs...), int clusters, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kFoldCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(clusters * kFoldCtas);
  cfg.blockDim = dim3(kFoldThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, args...) != cudaSuccess) return SPRINT_ERR_CUDA;
  return launch_status();
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
    return launch_fold(lmhead_combine_rows_kernel, (M + 31) / 32, stream, (const float *)p.pmax,
                       (const float *)p.psum, (const int32_t *)p.parg, temp, M, p.strips, V,
                       conf_out, argmax_out, status, gate);
  lmhead_combine_kernel<<<(M + kCombRows - 1) / kCombRows, dim3(kCombRows, kCombGroups), 0,
                            stream>>>(p.pmax, p.psum, p.parg, temp, M, p.strips, V, conf_out,
                                      argmax_out, status, gate);
  return launch_status();
}

int sprint::lmhead_tiles_impl(const void *h, const void *W, const float *temp, int M, int D,
                              int V, int dtype, void *logits_out, bool want_argmax, void *ws,
                              size_t ws_bytes, int32_t *status, Gate gate, cudaStream_t stream) {
  if (M < 1 || M >= 4096 || D < 1 || V < 1 || !h || !W || !ws || !status)
    return SPRINT_ERR_INVALID_ARG;
  if (ws_bytes < sprint_lmhead_workspace_bytes(M, D, V, dtype)) return SPRINT_ERR_WORKSPACE;
  LmheadWs p = lmhead_ws_layout(ws, M, V, lmhead_strip_cols(M, dtype));
  if (!want_argmax) p.parg = nullptr;
  if (dtype == SPRINT_BF16) {
    if (D % 8 != 0 || !aligned16(h) || !aligned16(W)) return SPRINT_ERR_UNSUPPORTED;
    return lmhead_tc_tiles(static_cast<const __nv_bfloat16 *>(h),
                           static_cast<const __nv_bfloat16 *>(W), temp, M, D, V,
                           static_cast<__nv_bfloat16 *>(logits_out), p, status, gate, stream);
  }
  dim3 grid(p.strips, (M + 63) / 64);
  lmhead_simt_kernel<float><<<grid, 256, 0, stream>>>(
      static_cast<const float *>(h), static_cast<const float *>(W), temp, M, D, V,
      static_cast<float *>(logits_out), p.pmax, p.psum, p.parg, status, gate);
  return launch_status();
}

int sprint::combine_unmask_impl(void *ws, const float *temp, int S, int LB, int V, int dtype,
                                float *conf_out, int32_t *argmax_out, uint8_t *mask,
                                int32_t *tokens, int32_t *m_out, int t, int T, float tau,
                                int mode, uint8_t *accepted_out, int fresh, int32_t *status,
                                Gate gate, cudaStream_t stream) {
  const int M = S * LB;
  if (S < 1 || LB < 1 || LB > kFusedMaxLB || M >= 4096 || !ws || !conf_out || !argmax_out || !mask ||
      !tokens || !m_out)
    return SPRINT_ERR_INVALID_ARG;
  const LmheadWs p = lmhead_ws_layout(ws, M, V, lmhead_strip_cols(M, dtype));
  return launch_fold(lmhead_combine_unmask_kernel, S, stream, (const float *)p.pmax,
                     (const float *)p.psum, (const int32_t *)p.parg, temp, LB, M, p.strips, V,
                     conf_out, argmax_out, mask, tokens, m_out, t, T, tau, mode, accepted_out,
                     fresh, status, gate);
}

extern "C" int sprint_lmhead_confidence(const void *h, const void *W, const float *temp,
                                        int M, int D, int V, int dtype, void *logits_out,
                                        float *conf_out, int32_t *argmax_out, void *ws,
                                        size_t ws_bytes, int32_t *status,
                                        cudaStream_t stream) {
  return lmhead_confidence_impl(h, W, temp, M, D, V, dtype, logits_out, conf_out, argmax_out, ws,
                                ws_bytes, status, Gate{nullptr, 0}, stream);
}
