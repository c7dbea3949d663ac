// Sparse Prefix Retention scoring and modality-aware selection.
//
// LLaDA2.0-Uni paper (arXiv 2604.20796), Inference section, "Sparse Prefix
// Retention" paragraph: every prefix position i gets the mean-normalised key
// norm I_i and the top-1 confidence c_i, blended into s_i (alpha = 0.5);
// within each modality the top floor(r n) positions by s_i are kept.
//
// Two kernels:
//   keynorm_kernel  HBM-bound: one warp per prefix position reads that
//                   position's key rows of every layer (NL x Hkv*d elements,
//                   1 KB per layer at Hkv*d = 512 bf16) with 16-byte loads,
//                   eight layers' loads in flight at once, and writes
//                   u_i = mean over layers of the L2 norm of the
//                   concatenated KV heads.
//   select_kernel   latency-bound: one 1024-thread CTA per sequence.  Mean of
//                   u (fp32 per thread, fp64 across threads), composite score
//                   s_i in fp32, then a 4-pass
//                   8-bit radix select on the orderable 32-bit key of s_i for
//                   both modalities at once, ties at the threshold resolved
//                   by ascending position with a block scan, and a stable
//                   block-scan compaction writing kept indices in ascending
//                   position order.  The sequence's keys and modality tags
//                   are staged in shared memory (5 bytes per position) when
//                   they fit, so global memory is read once and the six
//                   passes run at shared-memory latency; longer sequences
//                   keep them in the workspace.
#include <math.h>

#include "common.cuh"

namespace sprint {

// Eight consecutive elements as raw loaded bits, squared and summed in
// element order after the load has landed.
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
  typedef uint4 type;
  static __device__ __forceinline__ uint4 load(const __nv_bfloat16 *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
  }
  static __device__ __forceinline__ float sum_sq(uint4 u, float acc) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = __uint_as_float(w[i] << 16), b = __uint_as_float(w[i] & 0xffff0000u);
      acc = fmaf(a, a, acc);
      acc = fmaf(b, b, acc);
    }
    return acc;
  }
};
template <> struct Raw8<float> {
  struct type { float4 a, b; };
  static __device__ __forceinline__ type load(const float *p) {
    return {__ldg(reinterpret_cast<const float4 *>(p)),
            __ldg(reinterpret_cast<const float4 *>(p) + 1)};
  }
  static __device__ __forceinline__ float sum_sq(type v, float acc) {
    const float x[8] = {v.a.x, v.a.y, v.a.z, v.a.w, v.b.x, v.b.y, v.b.z, v.b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(x[i], x[i], acc);
    return acc;
  }
};

template <typename T>
__global__ void __launch_bounds__(256, 2)
keynorm_kernel(const T *__restrict__ K, const int32_t *__restrict__ prefix_off,
               int S, int total_rows, int NL, int row_elems,
               float *__restrict__ u, int32_t *status) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < total_rows;
       row += warps) {
    const int s = csr_owner(prefix_off, S, row);
    const int p0 = __ldg(prefix_off + s), p1 = __ldg(prefix_off + s + 1);
    const int i = row - p0;
    if (p0 < 0 || p1 > total_rows || i < 0 || i >= p1 - p0) {
      if (lane == 0) report(status, SPRINT_STATUS_BAD_OFFSETS);
      continue;
    }
    const size_t layer_stride = (size_t)(p1 - p0) * row_elems;
    const T *base = K + ((size_t)NL * p0 + i) * row_elems;
    float acc = 0.f;
    // Up to LG layers x two 16-byte chunks per lane are loaded before any is
    // used: 256 bytes per lane (8 KB per warp) in flight for bf16.
    constexpr int LG = sizeof(T) == 2 ? 8 : 4;
    for (int l0 = 0; l0 < NL; l0 += LG) {
      const int nl = min(LG, NL - l0);
      float ss[LG];
#pragma unroll
      for (int q = 0; q < LG; ++q) ss[q] = 0.f;
      for (int e = lane * 8; e < row_elems; e += 512) {
        const bool second = e + 256 < row_elems;
        typename Raw8<T>::type x[LG], y[LG];
#pragma unroll
        for (int q = 0; q < LG; ++q) {
          if (q < nl) {
            const T *p = base + (size_t)(l0 + q) * layer_stride + e;
            x[q] = Raw8<T>::load(p);
            if (second) y[q] = Raw8<T>::load(p + 256);
          }
        }
#pragma unroll
        for (int q = 0; q < LG; ++q) {
          if (q < nl) {
            ss[q] = Raw8<T>::sum_sq(x[q], ss[q]);
            if (second) ss[q] = Raw8<T>::sum_sq(y[q], ss[q]);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < LG; ++q)
        if (q < nl) acc += sqrtf(warp_sum(ss[q]));
    }
    if (lane == 0) u[row] = acc / (float)NL;
  }
}

constexpr int kSelThreads = 1024;
constexpr int kSelPer = 8;  // consecutive positions per thread per chunk
// Longest sequence whose keys and tags are staged in shared memory:
// 40,960 x 5 bytes = 200 KB of the 227 KB a CTA may hold.
constexpr int kStageMax = 40960;

__device__ __forceinline__ int keep_count_dev(int n, double r) {
  return (int)floor(r * (double)n + 1e-9);
}

__global__ void __launch_bounds__(kSelThreads)
select_kernel(const float *__restrict__ u, const float *__restrict__ conf,
              const uint8_t *__restrict__ modality,
              const int32_t *__restrict__ prefix_off,
              const int32_t *__restrict__ kept_off, int S, int total_rows,
              float alpha, double r_text, double r_img,
              uint32_t *__restrict__ keys_ws, int32_t *__restrict__ kept_idx,
              float *__restrict__ score_out, int32_t *status, int stage_cap) {
  extern __shared__ uint32_t stage_sh[];  // [stage_cap] keys, then [stage_cap] tags
  __shared__ uint32_t hist[2][256];
  __shared__ int scan_sh[33];
  __shared__ double dsum_sh[32];
  __shared__ int cnt_sh[32];
  __shared__ uint32_t thresh_sh[2];
  __shared__ int need_sh[2];
  __shared__ int mode_sh[2];  // 0 keep none, 1 keep all, 2 threshold

  const int s = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int p0 = prefix_off[s], p1 = prefix_off[s + 1];
  const int k0 = kept_off[s], k1 = kept_off[s + 1];
  if (p0 < 0 || p1 < p0 || p1 > total_rows || k0 < 0 || k1 < k0) {
    if (tid == 0) report(status, SPRINT_STATUS_BAD_OFFSETS);
    return;
  }
  const int n = p1 - p0;
  // Keys and modality tags of this sequence: staged in shared memory when
  // they fit, else read from the workspace / the caller's array.
  const bool staged = n <= stage_cap;
  uint32_t *keys = staged ? stage_sh : keys_ws + p0;
  uint8_t *mod_sh = reinterpret_cast<uint8_t *>(stage_sh + stage_cap);
  const uint8_t *mods = staged ? mod_sh : modality + p0;

  // Pass 1: sum of u and the image count; u is kept (as raw bits) where the
  // keys will go.  Each thread sums its positions in fp32; the 1024 thread
  // sums are added in fp64 (FP64 throughput is low on this GPU, so fp64 is
  // kept off the per-position path).
  float su_f = 0.f;
  int nimg = 0;
#pragma unroll 8
  for (int i = tid; i < n; i += kSelThreads) {
    const float ui = u[p0 + i];
    const uint8_t mi = modality[p0 + i] != 0;
    su_f += ui;
    nimg += mi;
    if (staged) {
      keys[i] = __float_as_uint(ui);
      mod_sh[i] = mi;
    }
  }
  double su = warp_sum((double)su_f);
  nimg = warp_sum(nimg);
  if (lane == 0) { dsum_sh[warp] = su; cnt_sh[warp] = nimg; }
  __syncthreads();
  if (warp == 0) {
    double v = dsum_sh[lane];
    int c = cnt_sh[lane];
    v = warp_sum(v);
    c = warp_sum(c);
    if (lane == 0) { dsum_sh[0] = v; cnt_sh[0] = c; }
  }
  __syncthreads();
  const double mean = n > 0 ? dsum_sh[0] / (double)n : 0.0;
  const int n_img = cnt_sh[0], n_txt = n - n_img;
  const int k_txt = keep_count_dev(n_txt, r_text), k_img = keep_count_dev(n_img, r_img);
  if (k1 - k0 != k_txt + k_img) {
    if (tid == 0) report(status, SPRINT_STATUS_KEPT_MISMATCH);
    return;
  }

  // Pass 2: composite score s_i = alpha I_i + (1 - alpha) c_i in fp32
  // (I_i = u_i / mean, an fp32 division by the fp32-rounded mean).
  const float one_m_alpha = 1.0f - alpha;
  const float mean_f = (float)mean;
#pragma unroll 8
  for (int i = tid; i < n; i += kSelThreads) {
    const float ui = staged ? __uint_as_float(keys[i]) : u[p0 + i];
    const float imp = mean_f > 0.0f ? ui / mean_f : 0.0f;
    const float sc = fmaf(alpha, imp, one_m_alpha * conf[p0 + i]);
    keys[i] = float_key(sc);
    if (score_out) score_out[p0 + i] = sc;
  }
  if (tid < 2) {
    const int k = tid == 0 ? k_txt : k_img, nm = tid == 0 ? n_txt : n_img;
    mode_sh[tid] = k <= 0 ? 0 : (k >= nm ? 1 : 2);
    need_sh[tid] = k;
    thresh_sh[tid] = 0u;
  }
  __syncthreads();

  // Radix select, most significant byte first, both modalities together:
  // find the k-th largest key T and how many keys equal to T are kept.
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 512; b += kSelThreads) (&hist[0][0])[b] = 0u;
    __syncthreads();
    const uint32_t hi_mask = shift == 24 ? 0u : (0xffffffffu << (shift + 8));
    const uint32_t pre0 = thresh_sh[0], pre1 = thresh_sh[1];
    const bool act0 = mode_sh[0] == 2, act1 = mode_sh[1] == 2;
    for (int base = 0; base < n; base += kSelThreads) {
      const int i = base + tid;
      int bin = -1;
      if (i < n) {
        const uint32_t key = keys[i];
        const int mu = mods[i] != 0;
        const uint32_t pre = mu ? pre1 : pre0;
        const bool act = mu ? act1 : act0;
        if (act && ((key ^ pre) & hi_mask) == 0u) bin = mu * 256 + ((key >> shift) & 255u);
      }
      // Warp-aggregated histogram update: one atomic per distinct bin.
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (bin >= 0 && lane == __ffs(peers) - 1)
        atomicAdd(&hist[0][0] + bin, (uint32_t)__popc(peers));
    }
    __syncthreads();
    if (warp < 2 && mode_sh[warp] == 2) {
      // Lane L owns bins 255-8L .. 248-8L (descending); find the bin where
      // the running count from the top reaches `need`.
      const int mu = warp;
      uint32_t c[8];
      uint32_t mine = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) { c[q] = hist[mu][255 - 8 * lane - q]; mine += c[q]; }
      uint32_t incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - mine;
      const uint32_t need = (uint32_t)need_sh[mu];
      const bool hit = excl < need && incl >= need;
      const unsigned who = __ballot_sync(0xffffffffu, hit);
      if (hit) {
        uint32_t run = excl;
        int q = 0;
        for (; q < 8; ++q) {
          if (run + c[q] >= need) break;
          run += c[q];
        }
        const uint32_t digit = 255u - 8u * lane - q;
        thresh_sh[mu] |= digit << shift;
        need_sh[mu] = (int)(need - run);
      }
      (void)who;
    }
    __syncthreads();
  }

  // Pass 3: stable compaction in ascending position order.  A position is
  // kept if its key exceeds its modality's threshold, or equals it and it
  // is among the first need_sh ties by position.
  const uint32_t T0 = thresh_sh[0], T1 = thresh_sh[1];
  const int m0 = mode_sh[0], m1 = mode_sh[1];
  const int need0 = need_sh[0], need1 = need_sh[1];
  int tie_base0 = 0, tie_base1 = 0, out_base = 0;
  for (int c0 = 0; c0 < n; c0 += kSelThreads * kSelPer) {
    const int first = c0 + tid * kSelPer;
    uint32_t kk[kSelPer];
    uint8_t mm[kSelPer];
    int ties = 0;  // text ties in the low 16 bits, image ties in the high 16
#pragma unroll
    for (int q = 0; q < kSelPer; ++q) {
      const int i = first + q;
      kk[q] = 0u;
      mm[q] = 0;
      if (i < n) {
        kk[q] = keys[i];
        mm[q] = mods[i] != 0;
        if (mm[q] == 0 && m0 == 2 && kk[q] == T0) ties += 1;
        if (mm[q] != 0 && m1 == 2 && kk[q] == T1) ties += 1 << 16;
      }
    }
    int ties_total;
    const int ties_excl = block_excl_scan(ties, scan_sh, &ties_total);
    int run0 = tie_base0 + (ties_excl & 0xffff), run1 = tie_base1 + (ties_excl >> 16);
    uint32_t keep_bits = 0u;
#pragma unroll
    for (int q = 0; q < kSelPer; ++q) {
      const int i = first + q;
      if (i >= n) continue;
      bool keep;
      if (mm[q] == 0) {
        keep = m0 == 1 || (m0 == 2 && (kk[q] > T0 || (kk[q] == T0 && run0 < need0)));
        if (m0 == 2 && kk[q] == T0) ++run0;
      } else {
        keep = m1 == 1 || (m1 == 2 && (kk[q] > T1 || (kk[q] == T1 && run1 < need1)));
        if (m1 == 2 && kk[q] == T1) ++run1;
      }
      keep_bits |= (uint32_t)keep << q;
    }
    int kept_total;
    int out = out_base + block_excl_scan(__popc(keep_bits), scan_sh, &kept_total);
#pragma unroll
    for (int q = 0; q < kSelPer; ++q)
      if (keep_bits >> q & 1u) {
        if (out < k1 - k0) kept_idx[k0 + out] = first + q;
        else report(status, SPRINT_STATUS_KEPT_MISMATCH);
        ++out;
      }
    tie_base0 += ties_total & 0xffff;
    tie_base1 += ties_total >> 16;
    out_base += kept_total;
  }
}

}  // namespace sprint

using namespace sprint;

extern "C" size_t sprint_score_prune_workspace_bytes(int S, int total_rows) {
  if (S < 0 || total_rows < 0) return 0;
  return align_up((size_t)total_rows * sizeof(float), 256) +
         align_up((size_t)total_rows * sizeof(uint32_t), 256);
}

extern "C" int sprint_score_prune(const void *K, int S, const int32_t *prefix_off,
                                  int total_rows, int NL, int Hkv, int d, int dtype,
                                  const float *conf, const uint8_t *modality,
                                  float alpha, double r_text, double r_img,
                                  int32_t *kept_idx, const int32_t *kept_off,
                                  float *score_out, void *ws, size_t ws_bytes,
                                  int32_t *status, cudaStream_t stream) {
  if (S < 0 || total_rows < 0 || NL < 1 || Hkv < 1 || d < 1) return SPRINT_ERR_INVALID_ARG;
  if (dtype != SPRINT_F32 && dtype != SPRINT_BF16) return SPRINT_ERR_INVALID_ARG;
  if (!(r_text >= 0.0 && r_text <= 1.0 && r_img >= 0.0 && r_img <= 1.0))
    return SPRINT_ERR_INVALID_ARG;
  if (!(alpha == alpha)) return SPRINT_ERR_INVALID_ARG;
  if (S == 0) return SPRINT_OK;
  if (!prefix_off || !kept_off || !status) return SPRINT_ERR_INVALID_ARG;
  if (total_rows > 0 && (!K || !conf || !modality || !ws)) return SPRINT_ERR_INVALID_ARG;
  const int row_elems = Hkv * d;
  if (row_elems % 8 != 0 || (K && !aligned16(K))) return SPRINT_ERR_UNSUPPORTED;
  if (ws_bytes < sprint_score_prune_workspace_bytes(S, total_rows)) return SPRINT_ERR_WORKSPACE;

  float *u = static_cast<float *>(ws);
  uint32_t *keys = reinterpret_cast<uint32_t *>(static_cast<char *>(ws) +
                                                align_up((size_t)total_rows * 4, 256));
  if (total_rows > 0) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // One wave: two 256-thread CTAs per SM (register-limited), each warp
    // striding over rows.
    int blocks = (total_rows + 7) / 8;
    blocks = blocks < sms * 2 ? blocks : sms * 2;
    if (dtype == SPRINT_BF16)
      keynorm_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
          static_cast<const __nv_bfloat16 *>(K), prefix_off, S, total_rows, NL, row_elems, u,
          status);
    else
      keynorm_kernel<float><<<blocks, 256, 0, stream>>>(
          static_cast<const float *>(K), prefix_off, S, total_rows, NL, row_elems, u, status);
    if (launch_status() != SPRINT_OK) return SPRINT_ERR_CUDA;
  }
  // Stage up to kStageMax positions per sequence in shared memory (5 bytes
  // each); the capacity follows the longest sequence the call can hold.
  const int stage_cap = total_rows < kStageMax ? total_rows : kStageMax;
  const size_t stage_bytes = (size_t)stage_cap * 5 + 16;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)((size_t)kStageMax * 5 + 16)) != cudaSuccess)
      return SPRINT_ERR_CUDA;
    attr_set = true;
  }
  select_kernel<<<S, kSelThreads, stage_bytes, stream>>>(u, conf, modality, prefix_off,
                                                         kept_off, S, total_rows, alpha, r_text,
                                                         r_img, keys, kept_idx, score_out,
                                                         status, stage_cap);
  return launch_status();
}

extern "C" int sprint_keep_count(int n, double r) {
  if (n < 0 || !(r >= 0.0 && r <= 1.0)) return -1;
  return (int)floor(r * (double)n + 1e-9);
}
