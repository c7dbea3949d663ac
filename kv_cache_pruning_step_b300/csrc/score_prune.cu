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
//                   s_i in fp32 and its orderable 32-bit key; then a radix
//                   select on the key minus its modality's smallest key,
//                   12 bits at a time from the top (4096-bin histograms,
//                   both modalities at once), giving each modality's
//                   threshold key and how many keys equal to it are kept;
//                   then a stable compaction: each warp counts its range's
//                   definite keeps and threshold ties with ballots, the warp
//                   totals are scanned, and each warp writes its kept
//                   positions (ties by ascending position) to consecutive
//                   output slots.  The sequence's keys and modality tags are
//                   staged in shared memory (5 bytes per position) when they
//                   fit, so global memory is read once; longer sequences
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
constexpr int kDigit = 12, kBins = 1 << kDigit;  // radix digit of the selection
// Longest sequence whose keys and tags are staged in shared memory:
// 36,864 x 5 bytes = 180 KB, next to 34 KB of histograms and scan space.
constexpr int kStageMax = 36864;

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
  extern __shared__ uint4 stage_raw[];  // [stage_cap rounded up to 4] keys, then tags
  uint32_t *stage_sh = reinterpret_cast<uint32_t *>(stage_raw);
  __shared__ uint32_t hist[2][kBins];
  __shared__ uint32_t kmin_sh[2], kmax_sh[2], prefix_sh[2];
  __shared__ int shift_sh[2];
  __shared__ int scan_sh[33];
  __shared__ double dsum_sh[32];
  __shared__ int cnt_sh[32];
  __shared__ float mean_sh;
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
  // The tags start 16-byte aligned (the key area is rounded up to 4 keys):
  // the compaction reads 8 tags at a time with one 8-byte load.
  uint8_t *mod_sh = reinterpret_cast<uint8_t *>(stage_sh + ((stage_cap + 3) & ~3));
  const uint8_t *mods = staged ? mod_sh : modality + p0;

  // Pass 1: sum of u and the image count; u is kept (as raw bits) where the
  // keys will go.  Each thread sums its positions in fp32; the 1024 thread
  // sums are added in fp64 (FP64 throughput is low on this GPU, so fp64 is
  // kept off the per-position path).  Loads come in batches of kB per
  // thread, all issued before any store (stores through `keys` might alias
  // the byte-typed tag loads, so the compiler would not reorder them).
  constexpr int kB = 8;
  float su_f = 0.f;
  int nimg = 0;
  for (int i0 = tid; i0 < n; i0 += kB * kSelThreads) {
    float ub[kB];
    uint8_t mb[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int i = i0 + j * kSelThreads;
      ub[j] = i < n ? __ldg(u + p0 + i) : 0.f;
      mb[j] = i < n ? (__ldg(modality + p0 + i) != 0) : 0;
    }
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int i = i0 + j * kSelThreads;
      su_f += ub[j];
      nimg += mb[j];
      if (staged && i < n) {
        keys[i] = __float_as_uint(ub[j]);
        mod_sh[i] = mb[j];
      }
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
    if (lane == 0) {
      // One thread does the fp64 division and the keep counts.
      const int ni = c, nt = n - c;
      mean_sh = n > 0 ? (float)(v / (double)n) : 0.f;
      cnt_sh[0] = ni;
      cnt_sh[1] = keep_count_dev(nt, r_text);
      cnt_sh[2] = keep_count_dev(ni, r_img);
    }
  }
  __syncthreads();
  const float mean_f = mean_sh;
  const int n_img = cnt_sh[0], n_txt = n - n_img;
  const int k_txt = cnt_sh[1], k_img = cnt_sh[2];
  if (k1 - k0 != k_txt + k_img) {
    if (tid == 0) report(status, SPRINT_STATUS_KEPT_MISMATCH);
    return;
  }

  // Pass 2: composite score s_i = alpha I_i + (1 - alpha) c_i in fp32
  // (I_i = u_i / mean, an fp32 division by the fp32-rounded mean), its
  // orderable key, and the smallest and largest key of each modality.
  if (tid < 2) {
    kmin_sh[tid] = 0xffffffffu;
    kmax_sh[tid] = 0u;
  }
  __syncthreads();
  const float one_m_alpha = 1.0f - alpha;
  uint32_t lo0 = 0xffffffffu, lo1 = 0xffffffffu, hi0 = 0u, hi1 = 0u;
  for (int i0 = tid; i0 < n; i0 += kB * kSelThreads) {
    float ub[kB], cb[kB];
    bool ib[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int i = i0 + j * kSelThreads;
      ub[j] = i < n ? (staged ? __uint_as_float(keys[i]) : __ldg(u + p0 + i)) : 0.f;
      cb[j] = i < n ? __ldg(conf + p0 + i) : 0.f;
      ib[j] = i < n && mods[i] != 0;
    }
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int i = i0 + j * kSelThreads;
      if (i >= n) continue;
      const float imp = mean_f > 0.0f ? ub[j] / mean_f : 0.0f;
      const float sc = fmaf(alpha, imp, one_m_alpha * cb[j]);
      const uint32_t key = float_key(sc);
      keys[i] = key;
      if (ib[j]) {
        lo1 = min(lo1, key);
        hi1 = max(hi1, key);
      } else {
        lo0 = min(lo0, key);
        hi0 = max(hi0, key);
      }
      if (score_out) score_out[p0 + i] = sc;
    }
  }
  lo0 = __reduce_min_sync(0xffffffffu, lo0);
  lo1 = __reduce_min_sync(0xffffffffu, lo1);
  hi0 = __reduce_max_sync(0xffffffffu, hi0);
  hi1 = __reduce_max_sync(0xffffffffu, hi1);
  if (lane == 0) {
    atomicMin(&kmin_sh[0], lo0);
    atomicMin(&kmin_sh[1], lo1);
    atomicMax(&kmax_sh[0], hi0);
    atomicMax(&kmax_sh[1], hi1);
  }
  __syncthreads();
  if (tid < 2) {
    const int k = tid == 0 ? k_txt : k_img, nm = tid == 0 ? n_txt : n_img;
    mode_sh[tid] = k <= 0 ? 0 : (k >= nm ? 1 : 2);
    need_sh[tid] = k;
    // Keys of the modality relative to its smallest key span `shift` bits;
    // the selection resolves them kDigit bits at a time from the top.
    const uint32_t range = kmax_sh[tid] - kmin_sh[tid];
    shift_sh[tid] = mode_sh[tid] == 2 && range ? 32 - __clz(range) : 0;
    prefix_sh[tid] = 0u;
  }
  __syncthreads();

  // Radix select on d = key - (smallest key of the modality), kDigit bits at
  // a time from the top, both modalities together: find the k-th largest
  // key T and how many keys equal to T are kept (ties then go by position).
  // Range reduction and 4096 bins keep atomic collisions rare.
  while (__syncthreads_or(tid < 2 && shift_sh[tid] > 0)) {
    for (int b = tid; b < 2 * kBins; b += kSelThreads) (&hist[0][0])[b] = 0u;
    __syncthreads();
    const int sh0 = shift_sh[0], sh1 = shift_sh[1];
    const int w0 = sh0 < kDigit ? sh0 : kDigit, w1 = sh1 < kDigit ? sh1 : kDigit;
    const uint32_t pre0 = prefix_sh[0], pre1 = prefix_sh[1];
    const uint32_t base0 = kmin_sh[0], base1 = kmin_sh[1];
    // Read before the scans below: one thread rewrites need_sh after them.
    const uint32_t needv0 = (uint32_t)need_sh[0], needv1 = (uint32_t)need_sh[1];
#pragma unroll 4
    for (int i = tid; i < n; i += kSelThreads) {
      const bool img = mods[i] != 0;
      const int sh = img ? sh1 : sh0, w = img ? w1 : w0;
      if (sh == 0) continue;
      const uint64_t d = (uint64_t)(keys[i] - (img ? base1 : base0));
      if ((uint32_t)(d >> sh) == (img ? pre1 : pre0))
        atomicAdd(&hist[img][(uint32_t)(d >> (sh - w)) & ((1u << w) - 1u)], 1u);
    }
    __syncthreads();
    // Counts above each thread's 4 bins (bins in descending order), one
    // block scan per modality.
    uint32_t c0[4], c1[4];
    int mine0 = 0, mine1 = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int bin = kBins - 1 - 4 * tid - q;
      c0[q] = hist[0][bin];
      c1[q] = hist[1][bin];
      mine0 += (int)c0[q];
      mine1 += (int)c1[q];
    }
    int total;
    const int above0 = block_excl_scan(mine0, scan_sh, &total);
    const int above1 = block_excl_scan(mine1, scan_sh, &total);
#pragma unroll
    for (int mu = 0; mu < 2; ++mu) {
      const int sh = mu ? sh1 : sh0, w = mu ? w1 : w0;
      if (sh == 0) continue;
      const uint32_t need = mu ? needv1 : needv0;
      uint32_t run = (uint32_t)(mu ? above1 : above0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t cq = mu ? c1[q] : c0[q];
        if (run < need && run + cq >= need) {  // the k-th largest lies in this bin
          const uint32_t digit = (uint32_t)(kBins - 1 - 4 * tid - q);
          prefix_sh[mu] = ((mu ? pre1 : pre0) << w) | digit;
          need_sh[mu] = (int)(need - run);
          shift_sh[mu] = sh - w;
        }
        run += cq;
      }
    }
    __syncthreads();
  }
  if (tid < 2) thresh_sh[tid] = kmin_sh[tid] + prefix_sh[tid];
  __syncthreads();

  // Pass 3: stable compaction in ascending position order.  A position is
  // kept if its key exceeds its modality's threshold (or the modality keeps
  // everything), or equals the threshold and is among the first need_sh
  // such ties by position.  Warp w owns positions [w R, (w+1) R): it counts
  // its definite keeps and ties with ballots, the 32 warp totals are
  // scanned, then every warp walks its range again and writes its kept
  // positions at consecutive output slots (coalesced stores).
  const uint32_t T0 = thresh_sh[0], T1 = thresh_sh[1];
  const int m0 = mode_sh[0], m1 = mode_sh[1];
  const int need0 = need_sh[0], need1 = need_sh[1];
  const int k_all = k1 - k0;
  const int per_warp = ((n + 32 * 32 - 1) / (32 * 32)) * 32;  // multiple of 32
  const int w_lo = warp * per_warp, w_hi = min(n, w_lo + per_warp);
  auto classify = [&](int i, bool &def, bool &tie0, bool &tie1) {
    def = tie0 = tie1 = false;
    if (i >= w_hi) return;
    const uint32_t key = keys[i];
    if (mods[i] != 0) {
      def = m1 == 1 || (m1 == 2 && key > T1);
      tie1 = m1 == 2 && key == T1;
    } else {
      def = m0 == 1 || (m0 == 2 && key > T0);
      tie0 = m0 == 2 && key == T0;
    }
  };
  int c_def = 0, c_t0 = 0, c_t1 = 0;
  for (int i0 = w_lo; i0 < w_hi; i0 += 32) {
    bool d, t0, t1;
    classify(i0 + lane, d, t0, t1);
    c_def += __popc(__ballot_sync(0xffffffffu, d));
    c_t0 += __popc(__ballot_sync(0xffffffffu, t0));
    c_t1 += __popc(__ballot_sync(0xffffffffu, t1));
  }
  // Exclusive scan of the warp totals (thread w of warp 0 handles warp w).
  __shared__ int wdef[32], wt0[32], wt1[32];
  if (lane == 0) { wdef[warp] = c_def; wt0[warp] = c_t0; wt1[warp] = c_t1; }
  __syncthreads();
  if (warp == 0) {
    const int a = wdef[lane], b = wt0[lane], c = wt1[lane];
    const int ia = warp_incl_scan(a), ib = warp_incl_scan(b), ic = warp_incl_scan(c);
    wdef[lane] = ia - a;
    wt0[lane] = ib - b;
    wt1[lane] = ic - c;
  }
  __syncthreads();
  int r_def = wdef[warp], r_t0 = wt0[warp], r_t1 = wt1[warp];
  const unsigned lt = (1u << lane) - 1u;
  for (int i0 = w_lo; i0 < w_hi; i0 += 32) {
    bool d, t0, t1;
    classify(i0 + lane, d, t0, t1);
    const unsigned bd = __ballot_sync(0xffffffffu, d);
    const unsigned b0 = __ballot_sync(0xffffffffu, t0);
    const unsigned b1 = __ballot_sync(0xffffffffu, t1);
    const bool keep = d || (t0 && r_t0 + __popc(b0 & lt) < need0) ||
                      (t1 && r_t1 + __popc(b1 & lt) < need1);
    const unsigned bk = __ballot_sync(0xffffffffu, keep);
    // kept before this group = definite keeps + the first `need` ties
    const int base = r_def + min(r_t0, need0) + min(r_t1, need1);
    if (keep) {
      const int out = base + __popc(bk & lt);
      if (out < k_all) kept_idx[k0 + out] = i0 + lane;
      else report(status, SPRINT_STATUS_KEPT_MISMATCH);
    }
    r_def += __popc(bd);
    r_t0 += __popc(b0);
    r_t1 += __popc(b1);
  }
}

int keynorm_launch(const void *K, const int32_t *prefix_off, int S, int total_rows, int NL,
                   int row_elems, int dtype, float *u, int32_t *status, cudaStream_t stream) {
  if (total_rows <= 0) return SPRINT_OK;
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
    keynorm_kernel<float><<<blocks, 256, 0, stream>>>(static_cast<const float *>(K), prefix_off,
                                                      S, total_rows, NL, row_elems, u, status);
  return launch_status();
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
  if (keynorm_launch(K, prefix_off, S, total_rows, NL, row_elems, dtype, u, status, stream) !=
      SPRINT_OK)
    return SPRINT_ERR_CUDA;
  // Stage up to kStageMax positions per sequence in shared memory (5 bytes
  // each); the capacity follows the longest sequence the call can hold.
  const int stage_cap = total_rows < kStageMax ? total_rows : kStageMax;
  const size_t stage_bytes = (size_t)((stage_cap + 3) & ~3) * 4 + (size_t)stage_cap + 16;
  static PerDevice attr_set;
  int set = 0;
  if (!attr_set.get(&set, [](int, int *v) {
        *v = 1;
        return cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)((size_t)kStageMax * 5 + 16)) == cudaSuccess;
      }))
    return SPRINT_ERR_CUDA;
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
