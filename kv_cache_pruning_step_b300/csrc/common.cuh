// Shared device helpers of the SPRINT kernels: status reporting, vector
// loads of bf16/fp32 rows, warp/block reductions, CSR lookups.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/sprint.h"

namespace sprint {

// Host: one int per device ordinal, computed once per device under a lock.
// Function attributes and occupancy belong to one device's context, so a
// process that calls the library on several devices (or from several host
// threads) needs them per device.
struct PerDevice {
  static constexpr int kMax = 64;
  std::mutex mu;
  int value[kMax] = {};
  bool ready[kMax] = {};
  // *out = the current device's value; init(dev, &v) computes it the first
  // time.  False when the device cannot be read or init fails (init is then
  // tried again on the next call).
  template <typename F> bool get(int *out, F init) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMax) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
      int v = 0;
      if (!init(dev, &v)) return false;
      value[dev] = v;
      ready[dev] = true;
    }
    *out = value[dev];
    return true;
  }
};

// Host: kernel launches made by this library in this process.
void count_launches(int n);

// Host: map a launch error to the ABI code; counts one successful launch.
static inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return SPRINT_ERR_CUDA;
  count_launches(1);
  return SPRINT_OK;
}

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

__device__ __forceinline__ void report(int32_t *status, uint32_t bit) {
  if (status) atomicOr(reinterpret_cast<unsigned int *>(status), bit);
}

// Invariant checks compiled into the debug build only (SPRINT_DEBUG_CHECKS
// defined non-zero): a failed check ORs SPRINT_STATUS_DEBUG_CHECK into the
// status word and the kernel carries on; nothing traps.
#if defined(SPRINT_DEBUG_CHECKS) && SPRINT_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#define SPRINT_DCHECK(cond, status)                                      \
  do {                                                                   \
    if (!(cond)) ::sprint::report((status), SPRINT_STATUS_DEBUG_CHECK);  \
  } while (0)
#else
constexpr bool kDebugChecks = false;
#define SPRINT_DCHECK(cond, status) \
  do {                              \
  } while (0)
#endif

// Eight consecutive elements of a row, widened to fp32.
template <typename T> struct Vec8;

template <> struct Vec8<float> {
  static __device__ __forceinline__ void load(const float *p, float (&x)[8]) {
    float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
};

template <> struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&x)[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Inclusive warp scan of ints.
__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Exclusive block scan of one int per thread (blockDim.x multiple of 32,
// at most 1024).  `sh` holds >= 33 ints.  Returns the exclusive prefix;
// *total receives the block total.
__device__ __forceinline__ int block_excl_scan(int v, int *sh, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int incl = warp_incl_scan(v);
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? sh[lane] : 0;
    int wi = warp_incl_scan(w);
    if (lane < nw) sh[lane] = wi - w;
    if (lane == nw - 1) sh[32] = wi;
  }
  __syncthreads();
  int out = sh[warp] + incl - v;
  *total = sh[32];
  __syncthreads();
  return out;
}

// Canonical sum of the key-norm means u over the n positions of one
// sequence, the numerator of the mean in I_i.  Its bits do not depend on
// how a launch divides the work, so kernels that split the positions
// differently (the two-modality selection in clusters of CTAs, the keep
// pools in one CTA) reach the same mean:
//   * a leaf is kLeaf = 1024 consecutive positions; lane j of a warp adds
//     positions j, j + 32, ..., j + 992 of the leaf in fp32 in that order,
//     and the 32 lane sums are added in fp64 by an xor butterfly;
//   * the leaves are added by a complete binary tree over the leaf index,
//     padded with zero leaves to a power of two.
// Any division of that tree into aligned power-of-two blocks of leaves
// (adding +0 changes nothing) gives the same result.
constexpr int kLeaf = 1024;

__device__ __forceinline__ int next_pow2(int x) { return x <= 1 ? 1 : 1 << (32 - __clz(x - 1)); }

// Sum of leaf g; the same value in every lane.
__device__ __forceinline__ double u_leaf_sum(const float *__restrict__ u, int n, int g,
                                             int lane) {
  const int base = g * kLeaf;
  float v[32];  // all 32 loads in flight before the in-order sum
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int p = base + i * 32 + lane;
    v[i] = p < n ? __ldg(u + p) : 0.f;
  }
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) acc += v[i];
  return warp_sum((double)acc);
}

// Tree sum of the aligned block of `count` leaves (a power of two) that
// starts at leaf `first`; leaves at or past G are zero.  Whole warp.
__device__ __forceinline__ double u_subtree_sum(const float *__restrict__ u, int n, int G,
                                                int first, int count, int lane) {
  if (first >= G) return 0.0;
  double stack[32];
  int level_top = 0;
  for (int j = 0; j < count; ++j) {
    const int g = first + j;
    double v = g < G ? u_leaf_sum(u, n, g, lane) : 0.0;
    int level = 0;
    while ((j >> level) & 1) {  // merge complete left subtrees (binary carry)
      v = stack[level] + v;
      ++level;
    }
    stack[level] = v;
    level_top = level;
  }
  return stack[level_top];
}

// In-place complete binary tree over v[0..cnt) (cnt a power of two); the
// sum lands in v[0].
__device__ __forceinline__ void tree_fold(double *v, int cnt) {
  for (int step = 1; step < cnt; step <<= 1)
    for (int q = 0; q + step < cnt; q += 2 * step) v[q] = v[q] + v[q + step];
}

// Sequence that owns global row `row` under CSR offsets off[0..S].
__device__ __forceinline__ int csr_owner(const int32_t *off, int S, int row) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(off + mid) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Step gate of the native block driver (sprint_decode_steps): the kernels
// of a step after the first do nothing once every sequence finished at an
// earlier step, i.e. when the previous step's still-masked counts
// m_prev[0..S) are all zero.  m_prev == nullptr: always open.
struct Gate {
  const int32_t *m_prev;
  int S;
};

// Block-uniform test; every thread of the block must call it, before any
// other barrier of the kernel.
__device__ __forceinline__ bool gate_closed(const Gate &g) {
  if (!g.m_prev) return false;
  __shared__ int closed_sh;
  if (threadIdx.x == 0 && threadIdx.y == 0) {
    int any = 0;
    for (int s = 0; s < g.S; ++s) any |= __ldg(g.m_prev + s);
    closed_sh = any == 0;
  }
  __syncthreads();
  return closed_sh != 0;
}

// Prefix keys read through an index instead of a compacted copy: key i of
// sequence s is row idx[kv_off[s] + i] of that sequence's full prefix, which
// starts at row prefix_off[s] of the full K / V and has prefix_off[s+1] -
// prefix_off[s] rows.  idx == nullptr: the prefix keys are stored
// contiguously (a compacted or full cache located by kv_off).
struct KvIndex {
  const int32_t *idx;
  const int32_t *prefix_off;
  int total_prefix_rows;
};

// Residual epilogue of the attention (optional): for the last layer, also
// write h_out = h_in + O with the heads concatenated ([S * LB][Hq * d], the
// storage type of O), O rounded to its storage type first.  h_out ==
// nullptr: off.
struct AttnResidual {
  const void *h_in;
  void *h_out;
};

// Entry points with a step gate, shared by the C ABI (gate open) and the
// native block driver.
int lmhead_confidence_impl(const void *h, const void *W, const float *temp, int M, int D, int V,
                           int dtype, void *logits_out, float *conf_out, int32_t *argmax_out,
                           void *ws, size_t ws_bytes, int32_t *status, Gate gate,
                           cudaStream_t stream);
// Native driver: the bf16 attention's combine kernel may run on a side
// stream (forked after the chunk kernel with `fork`, joined through `join`,
// which the caller waits on before the workspace or O is touched again).
struct SideStream {
  cudaStream_t side;  // nullptr: the combine runs on the call's stream
  cudaEvent_t fork, join;
};
int block_attn_impl(const void *Q, const void *Kp, const void *Vp, const int32_t *kv_off,
                    int max_kv_rows, int total_kv_rows, const void *Kb, const void *Vb, int S,
                    int NL, int LB, int Hq, int Hkv, int d, int dtype, void *O, void *ws,
                    size_t ws_bytes, int32_t *status, KvIndex kvi, AttnResidual res,
                    Gate gate, cudaStream_t stream, SideStream side = {nullptr, nullptr, nullptr});
int unmask_impl(const float *conf, const int32_t *argmax, uint8_t *mask, int32_t *tokens,
                int32_t *m_out, int S, int LB, int t, int T, float tau, int mode,
                uint8_t *accepted_out, int32_t *status, Gate gate, cudaStream_t stream,
                int fresh = 0);
// Native driver, block steps of fewer than 4096 rows and blocks of at most
// kFusedMaxLB positions: the LM-head tiles only (strip partials in ws), then
// one kernel that folds each sequence's rows and unmasks its block
// (lmhead.cu).
constexpr int kFusedMaxLB = 512;
int lmhead_tiles_impl(const void *h, const void *W, const float *temp, int M, int D, int V,
                      int dtype, void *logits_out, bool want_argmax, void *ws, size_t ws_bytes,
                      int32_t *status, Gate gate, cudaStream_t stream);
int combine_unmask_impl(void *ws, const float *temp, int S, int LB, int V, int dtype,
                        float *conf_out, int32_t *argmax_out, uint8_t *mask, int32_t *tokens,
                        int32_t *m_out, int t, int T, float tau, int mode,
                        uint8_t *accepted_out, int fresh, int32_t *status, Gate gate,
                        cudaStream_t stream);

// Key-norm pass of the scoring (score_prune.cu): u[row] = mean over layers
// of the L2 norm of the row's keys concatenated over KV heads.
int keynorm_launch(const void *K, const int32_t *prefix_off, int S, int total_rows, int NL,
                   int row_elems, int dtype, float *u, int32_t *status, cudaStream_t stream);

// Orderable unsigned key of a float: a > b  <=>  key(a) > key(b); -0 == +0.
__device__ __forceinline__ uint32_t float_key(float f) {
  if (f == 0.0f) f = 0.0f;
  uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

}  // namespace sprint
