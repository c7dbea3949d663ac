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
#include <cooperative_groups.h>
#include <math.h>

#include "common.cuh"

namespace cg = cooperative_groups;

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

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxBpt = (1 << 12) / kSelThreads;  // digits per thread in a scan, at most
constexpr int kDigit = 12, kBins = 1 << kDigit;  // radix digit of the selection
constexpr int kMaxCluster = 8;                     // CTAs per sequence, at most
// Positions a CTA's slice aims at when the cluster size is chosen, and the
// longest slice whose keys and tags are staged in shared memory (5 bytes
// per position); longer slices keep their keys in the workspace.
constexpr int kSliceTarget = 2048;
constexpr int kStageCta = 16384;

__device__ __forceinline__ int keep_count_dev(int n, double r) {
  return (int)floor(r * (double)n + 1e-9);
}

// What each CTA of a sequence's cluster publishes to the others (read
// through distributed shared memory after a cluster barrier).
struct SelXchg {
  double tree;        // this CTA's block of the canonical sum of u
  int nimg;           // image positions in the slice
  uint32_t lo[2];     // smallest / largest key per modality in the slice
  uint32_t hi[2];
  uint32_t tot[2];    // keys of the current radix pass in the digits this CTA owns
  int cnt[3];         // definite keeps, text ties, image ties in the slice
};

// Dynamic shared memory: histograms [2][kBins], the cluster sums of the
// digits this CTA owns [2][kBins / cl] (cl > 1), then the staged keys and
// tags of the slice.
__host__ __device__ inline size_t select_smem_bytes(int cl, int cap) {
  return (size_t)2 * kBins * 4 + (cl > 1 ? (size_t)2 * (kBins / cl) * 4 : 0) + (size_t)cap * 5;
}

// One cluster of cl CTAs per sequence (cl = 1, 2, 4 or 8, the same for the
// whole launch); CTA `rank` owns the slice [rank L, rank L + L) of the
// sequence's positions and the radix digits [rank kBins/cl, ...).
//   1. the canonical sum of u (common.cuh), the image count, the mean and
//      the keep counts; every CTA folds the cluster's partials in rank order;
//   2. s_i = alpha I_i + (1 - alpha) c_i in fp32 with I_i = u_i / mean (an
//      fp32 division by the fp32-rounded mean), its orderable key, and each
//      modality's smallest and largest key;
//   3. radix select of each modality's k-th largest key on keys reduced to
//      the modality's range, 12 bits per pass from the top: every CTA
//      histograms its slice, each CTA sums its own digits over the cluster,
//      and the CTA whose digits hold the k-th key finds the digit;
//   4. stable compaction in ascending position order: warps count their
//      definite keeps and threshold ties with ballots, counts are scanned
//      over the warps and over the cluster's CTAs, and every warp writes its
//      kept positions to consecutive output slots (ties by ascending
//      position).
__global__ void __launch_bounds__(kSelThreads, 1)
select_kernel(const float *__restrict__ u, const float *__restrict__ conf,
              const uint8_t *__restrict__ modality, const int32_t *__restrict__ prefix_off,
              const int32_t *__restrict__ kept_off, int total_rows, float alpha,
              double r_text, double r_img, uint32_t *__restrict__ keys_ws,
              int32_t *__restrict__ kept_idx, float *__restrict__ score_out, int32_t *status,
              int stage_cap) {
  cg::cluster_group cluster = cg::this_cluster();
  const int cl = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  const int s = blockIdx.x / cl;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  extern __shared__ __align__(16) uint8_t sel_smem[];
  const int W = kBins / cl;  // digits this CTA owns
  uint32_t *hist = reinterpret_cast<uint32_t *>(sel_smem);
  uint32_t *hsum = cl > 1 ? hist + 2 * kBins : hist;  // [2][W]
  uint32_t *stage_keys = hist + 2 * kBins + (cl > 1 ? 2 * W : 0);
  uint8_t *stage_tags = reinterpret_cast<uint8_t *>(stage_keys + stage_cap);
  __shared__ SelXchg xc;
  __shared__ double wtree[kSelWarps];
  __shared__ int scan_sh[33];
  __shared__ int wcnt[3][32];
  __shared__ float mean_sh;
  __shared__ int info_sh[4];  // image count, text keep, image keep, counts consistent
  __shared__ uint32_t lmin_sh[2], lmax_sh[2], kmin_sh[2], prefix_sh[2];
  __shared__ int shift_sh[2], need_sh[2], mode_sh[2], qstar_sh[2], above_sh[2], dneed_sh[2];
  __shared__ uint32_t digit_sh[2];

  const int p0 = prefix_off[s], p1 = prefix_off[s + 1];
  const int k0 = kept_off[s], k1 = kept_off[s + 1];
  // Every CTA of the cluster reads the same offsets, so all of them return
  // here or none does (before any cluster barrier).
  if (p0 < 0 || p1 < p0 || p1 > total_rows || k0 < 0 || k1 < k0) {
    if (rank == 0 && tid == 0) report(status, SPRINT_STATUS_BAD_OFFSETS);
    return;
  }
  const int n = p1 - p0;
  const int L = ((n + cl - 1) / cl + 31) & ~31;
  const int lo_i = min(n, rank * L), m = min(n, lo_i + L) - lo_i;
  const int g0 = p0 + lo_i;  // first global row of the slice
  const bool staged = L <= stage_cap;
  uint32_t *keys = staged ? stage_keys : keys_ws + g0;
  const uint8_t *tags = staged ? stage_tags : modality + g0;
  if (tid < 2) {
    lmin_sh[tid] = 0xffffffffu;
    lmax_sh[tid] = 0u;
  }

  // ---- 1. canonical sum of u; image count; staging of u bits and tags
  {
    const int G = (n + kLeaf - 1) / kLeaf, P = next_pow2(G);
    const int workers = cl * kSelWarps, B = P > workers ? P / workers : 1;
    const int wk = rank * kSelWarps + warp;
    const double v = wk * B < P ? u_subtree_sum(u + p0, n, G, wk * B, B, lane) : 0.0;
    if (lane == 0) wtree[warp] = v;
  }
  constexpr int kB = 4;
  int nimg = 0;
  for (int j0 = tid; j0 < m; j0 += kB * kSelThreads) {
    float ub[kB];
    uint8_t mb[kB];
#pragma unroll
    for (int q = 0; q < kB; ++q) {
      const int j = j0 + q * kSelThreads;
      ub[q] = j < m ? __ldg(u + g0 + j) : 0.f;
      mb[q] = j < m ? (__ldg(modality + g0 + j) != 0) : 0;
    }
#pragma unroll
    for (int q = 0; q < kB; ++q) {
      const int j = j0 + q * kSelThreads;
      nimg += mb[q];
      if (staged && j < m) {
        stage_keys[j] = __float_as_uint(ub[q]);
        stage_tags[j] = mb[q];
      }
    }
  }
  nimg = warp_sum(nimg);
  if (lane == 0) wcnt[0][warp] = nimg;
  __syncthreads();
  if (tid == 0) {
    double v[kSelWarps];
    int t = 0;
    for (int i = 0; i < kSelWarps; ++i) {
      v[i] = wtree[i];
      t += wcnt[0][i];
    }
    tree_fold(v, kSelWarps);
    xc.tree = v[0];
    xc.nimg = t;
  }
  cluster.sync();
  if (tid == 0) {
    double v[kMaxCluster];
    int nq[kMaxCluster];
#pragma unroll
    for (int q = 0; q < kMaxCluster; ++q) {  // all remote loads in flight
      const SelXchg *r = cluster.map_shared_rank(&xc, q < cl ? q : 0);
      v[q] = q < cl ? r->tree : 0.0;
      nq[q] = q < cl ? r->nimg : 0;
    }
    int ni = 0;
#pragma unroll
    for (int q = 0; q < kMaxCluster; ++q) ni += nq[q];
    tree_fold(v, cl);
    mean_sh = n > 0 ? (float)(v[0] / (double)n) : 0.f;
    info_sh[0] = ni;
    info_sh[1] = keep_count_dev(n - ni, r_text);
    info_sh[2] = keep_count_dev(ni, r_img);
    info_sh[3] = k1 - k0 == info_sh[1] + info_sh[2];
  }
  __syncthreads();
  const float mean_f = mean_sh;
  const int n_img = info_sh[0], n_txt = n - n_img;
  const int k_txt = info_sh[1], k_img = info_sh[2];

  // ---- 2. scores, keys, key range per modality
  const float one_m_alpha = 1.0f - alpha;
  uint32_t lo0 = 0xffffffffu, lo1 = 0xffffffffu, hi0 = 0u, hi1 = 0u;
  for (int j0 = tid; j0 < m; j0 += kB * kSelThreads) {
    float ub[kB], cb[kB];
    bool ib[kB];
#pragma unroll
    for (int q = 0; q < kB; ++q) {
      const int j = j0 + q * kSelThreads;
      ub[q] = j < m ? (staged ? __uint_as_float(stage_keys[j]) : __ldg(u + g0 + j)) : 0.f;
      cb[q] = j < m ? __ldg(conf + g0 + j) : 0.f;
      ib[q] = j < m && tags[j] != 0;
    }
#pragma unroll
    for (int q = 0; q < kB; ++q) {
      const int j = j0 + q * kSelThreads;
      if (j >= m) continue;
      const float imp = mean_f > 0.0f ? ub[q] / mean_f : 0.0f;
      const float sc = fmaf(alpha, imp, one_m_alpha * cb[q]);
      const uint32_t key = float_key(sc);
      keys[j] = key;
      if (ib[q]) {
        lo1 = min(lo1, key);
        hi1 = max(hi1, key);
      } else {
        lo0 = min(lo0, key);
        hi0 = max(hi0, key);
      }
      if (score_out) score_out[g0 + j] = sc;
    }
  }
  lo0 = __reduce_min_sync(0xffffffffu, lo0);
  lo1 = __reduce_min_sync(0xffffffffu, lo1);
  hi0 = __reduce_max_sync(0xffffffffu, hi0);
  hi1 = __reduce_max_sync(0xffffffffu, hi1);
  if (lane == 0) {
    atomicMin(&lmin_sh[0], lo0);
    atomicMin(&lmin_sh[1], lo1);
    atomicMax(&lmax_sh[0], hi0);
    atomicMax(&lmax_sh[1], hi1);
  }
  __syncthreads();
  if (tid < 2) {
    xc.lo[tid] = lmin_sh[tid];
    xc.hi[tid] = lmax_sh[tid];
  }
  cluster.sync();
  if (!info_sh[3]) {  // the same decision in every CTA of the cluster
    if (rank == 0 && tid == 0) report(status, SPRINT_STATUS_KEPT_MISMATCH);
    cluster.sync();  // nobody leaves while another CTA may still read its xc
    return;
  }
  if (tid < 2) {
    const int mu = tid;
    uint32_t lo[kMaxCluster], hi[kMaxCluster];
#pragma unroll
    for (int q = 0; q < kMaxCluster; ++q) {
      const SelXchg *r = cluster.map_shared_rank(&xc, q < cl ? q : 0);
      lo[q] = r->lo[mu];
      hi[q] = r->hi[mu];
    }
    uint32_t kmn = 0xffffffffu, kmx = 0u;
#pragma unroll
    for (int q = 0; q < kMaxCluster; ++q) {
      kmn = min(kmn, lo[q]);
      kmx = max(kmx, hi[q]);
    }
    const int k = mu ? k_img : k_txt, nm = mu ? n_img : n_txt;
    mode_sh[mu] = k <= 0 ? 0 : (k >= nm ? 1 : 2);
    need_sh[mu] = k;
    kmin_sh[mu] = kmn;
    prefix_sh[mu] = 0u;
    // Keys of the modality relative to its smallest key span `shift` bits;
    // the selection resolves them kDigit bits at a time from the top.
    const uint32_t range = kmx - kmn;
    shift_sh[mu] = mode_sh[mu] == 2 && range ? 32 - __clz(range) : 0;
  }
  __syncthreads();

  // ---- 3. radix select, both modalities together.  The loop condition and
  // every decision below come from values that are identical in all CTAs
  // of the cluster, so they pass the same cluster barriers.
  while (shift_sh[0] > 0 || shift_sh[1] > 0) {
    for (int b = tid; b < 2 * kBins; b += kSelThreads) hist[b] = 0u;
    __syncthreads();
    const int sh0 = shift_sh[0], sh1 = shift_sh[1];
    const int w0 = sh0 < kDigit ? sh0 : kDigit, w1 = sh1 < kDigit ? sh1 : kDigit;
    const uint32_t pre0 = prefix_sh[0], pre1 = prefix_sh[1];
    const uint32_t base0 = kmin_sh[0], base1 = kmin_sh[1];
#pragma unroll 4
    for (int j = tid; j < m; j += kSelThreads) {
      const bool img = tags[j] != 0;
      const int sh = img ? sh1 : sh0, w = img ? w1 : w0;
      if (sh == 0) continue;
      const uint64_t d = (uint64_t)(keys[j] - (img ? base1 : base0));
      if ((uint32_t)(d >> sh) == (img ? pre1 : pre0))
        atomicAdd(&hist[(img ? kBins : 0) + ((uint32_t)(d >> (sh - w)) & ((1u << w) - 1u))], 1u);
    }
    cluster.sync();  // every CTA's histogram is complete
    if (cl > 1) {
      // all cl remote loads of a digit in flight at once
      for (int idx = tid; idx < 2 * W; idx += kSelThreads) {
        const int mu = idx >= W, b = rank * W + (idx - mu * W);
        uint32_t c[kMaxCluster];
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q)
          c[q] = q < cl ? cluster.map_shared_rank(hist, q)[mu * kBins + b] : 0u;
        uint32_t t = 0u;
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q) t += c[q];
        hsum[idx] = t;
      }
      __syncthreads();
    }
    uint32_t t0 = 0u, t1 = 0u;
    for (int b = tid; b < W; b += kSelThreads) {
      t0 += hsum[b];
      t1 += hsum[W + b];
    }
    t0 = __reduce_add_sync(0xffffffffu, t0);
    t1 = __reduce_add_sync(0xffffffffu, t1);
    if (lane == 0) {
      wcnt[0][warp] = (int)t0;
      wcnt[1][warp] = (int)t1;
    }
    __syncthreads();
    if (tid < 2) {
      uint32_t t = 0u;
      for (int i = 0; i < kSelWarps; ++i) t += (uint32_t)wcnt[tid][i];
      xc.tot[tid] = t;
    }
    cluster.sync();  // every CTA's digit totals are published
    if (tid < 2) {
      const int mu = tid;
      int qs = -1;
      uint32_t above = 0u, run = 0u;
      const uint32_t need = (uint32_t)need_sh[mu];
      if (shift_sh[mu] > 0) {
        uint32_t tot[kMaxCluster];
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q)
          tot[q] = q < cl ? cluster.map_shared_rank(&xc, q)->tot[mu] : 0u;
        for (int q = cl - 1; q >= 0; --q) {  // higher ranks own larger digits
          const uint32_t tq = tot[q];
          if (qs < 0 && run < need && run + tq >= need) {
            qs = q;
            above = run;
          }
          run += tq;
        }
      }
      qstar_sh[mu] = qs;
      above_sh[mu] = (int)above;
    }
    __syncthreads();
    // Every CTA finds the threshold digit itself from the digit totals of
    // the CTA that owns it (read through distributed shared memory), so no
    // barrier publishes it.  That CTA rewrites its totals only after the
    // next pass's first cluster barrier, which every reader reaches after
    // these reads.
    for (int mu = 0; mu < 2; ++mu) {
      const int qs = qstar_sh[mu];
      if (shift_sh[mu] <= 0 || qs < 0) continue;  // uniform in the CTA
      const uint32_t *src = cl > 1 ? cluster.map_shared_rank(hsum, qs) : hsum;
      // Digits of CTA qs in descending order, bpt per thread; counts above
      // each thread's digits by one block scan.
      const int bpt = (W + kSelThreads - 1) / kSelThreads;
      uint32_t c[kMaxBpt];
      int mine = 0;
#pragma unroll
      for (int q = 0; q < kMaxBpt; ++q) {
        const int jd = tid * bpt + q;
        c[q] = (q < bpt && jd < W) ? src[mu * W + (W - 1 - jd)] : 0u;
        mine += (int)c[q];
      }
      int total;
      const int above_in = block_excl_scan(mine, scan_sh, &total);
      const uint32_t need = (uint32_t)need_sh[mu];
      uint32_t run = (uint32_t)above_sh[mu] + (uint32_t)above_in;
#pragma unroll
      for (int q = 0; q < kMaxBpt; ++q) {
        const int jd = tid * bpt + q;
        if (q < bpt && jd < W) {
          if (run < need && run + c[q] >= need) {  // the k-th largest lies in this digit
            digit_sh[mu] = (uint32_t)(qs * W + (W - 1 - jd));
            dneed_sh[mu] = (int)(need - run);
          }
          run += c[q];
        }
      }
    }
    __syncthreads();
    if (tid < 2 && shift_sh[tid] > 0) {
      const int mu = tid, sh = shift_sh[mu], w = sh < kDigit ? sh : kDigit;
      if (qstar_sh[mu] >= 0) {
        prefix_sh[mu] = (prefix_sh[mu] << w) | digit_sh[mu];
        need_sh[mu] = dneed_sh[mu];
        shift_sh[mu] = sh - w;
      } else {  // counts inconsistent with the keep count: cannot happen
        report(status, SPRINT_STATUS_KEPT_MISMATCH);
        shift_sh[mu] = 0;
      }
    }
    __syncthreads();
  }

  // ---- 4. stable compaction in ascending position order.  A position is
  // kept if its key exceeds its modality's threshold (or the modality keeps
  // everything), or equals the threshold and is among the first need_sh
  // such ties by position.  Warp w owns positions [w R, (w+1) R) of the
  // slice.
  const uint32_t T0 = kmin_sh[0] + prefix_sh[0], T1 = kmin_sh[1] + prefix_sh[1];
  const int m0 = mode_sh[0], m1 = mode_sh[1];
  const int need0 = need_sh[0], need1 = need_sh[1];
  const int k_all = k1 - k0;
  const int per_warp = ((m + kSelWarps * 32 - 1) / (kSelWarps * 32)) * 32;  // multiple of 32
  const int w_lo = warp * per_warp, w_hi = min(m, w_lo + per_warp);
  auto classify = [&](int j, bool &def, bool &tie0, bool &tie1) {
    def = tie0 = tie1 = false;
    if (j >= w_hi) return;
    const uint32_t key = keys[j];
    if (tags[j] != 0) {
      def = m1 == 1 || (m1 == 2 && key > T1);
      tie1 = m1 == 2 && key == T1;
    } else {
      def = m0 == 1 || (m0 == 2 && key > T0);
      tie0 = m0 == 2 && key == T0;
    }
  };
  int c_def = 0, c_t0 = 0, c_t1 = 0;
  for (int j0 = w_lo; j0 < w_hi; j0 += 32) {
    bool d, t0, t1;
    classify(j0 + lane, d, t0, t1);
    c_def += __popc(__ballot_sync(0xffffffffu, d));
    c_t0 += __popc(__ballot_sync(0xffffffffu, t0));
    c_t1 += __popc(__ballot_sync(0xffffffffu, t1));
  }
  if (lane == 0) {
    wcnt[0][warp] = c_def;
    wcnt[1][warp] = c_t0;
    wcnt[2][warp] = c_t1;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scans of the warp totals; the CTA's totals
    const bool w_ok = lane < kSelWarps;
    const int a = w_ok ? wcnt[0][lane] : 0, b = w_ok ? wcnt[1][lane] : 0,
              c = w_ok ? wcnt[2][lane] : 0;
    const int ia = warp_incl_scan(a), ib = warp_incl_scan(b), ic = warp_incl_scan(c);
    wcnt[0][lane] = ia - a;
    wcnt[1][lane] = ib - b;
    wcnt[2][lane] = ic - c;
    if (lane == 31) {
      xc.cnt[0] = ia;
      xc.cnt[1] = ib;
      xc.cnt[2] = ic;
    }
  }
  cluster.sync();  // every CTA's totals are published
  __shared__ int cbase_sh[3];
  if (tid < 3) {
    int c[kMaxCluster];
#pragma unroll
    for (int q = 0; q < kMaxCluster; ++q)
      c[q] = q < rank ? cluster.map_shared_rank(&xc, q)->cnt[tid] : 0;
    int t = 0;
#pragma unroll
    for (int q = 0; q < kMaxCluster; ++q) t += c[q];
    cbase_sh[tid] = t;
  }
  __syncthreads();
  int r_def = cbase_sh[0] + wcnt[0][warp], r_t0 = cbase_sh[1] + wcnt[1][warp],
      r_t1 = cbase_sh[2] + wcnt[2][warp];
  const unsigned lt = (1u << lane) - 1u;
  for (int j0 = w_lo; j0 < w_hi; j0 += 32) {
    bool d, t0, t1;
    classify(j0 + lane, d, t0, t1);
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
      if (out < k_all) kept_idx[k0 + out] = lo_i + j0 + lane;
      else report(status, SPRINT_STATUS_KEPT_MISMATCH);
    }
    r_def += __popc(bd);
    r_t0 += __popc(b0);
    r_t1 += __popc(b1);
  }
  if (kDebugChecks && rank == cl - 1 && tid == 0) {
    // positions written by the whole cluster = the sequence's kept count
    const int written = cbase_sh[0] + xc.cnt[0] + min(cbase_sh[1] + xc.cnt[1], need0) +
                        min(cbase_sh[2] + xc.cnt[2], need1);
    SPRINT_DCHECK(written == k_all, status);
  }
  cluster.sync();  // nobody leaves while another CTA may still read its counts
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

namespace {

// select_kernel over every sequence, on key norms u already in memory; keys
// is the [total_rows] key scratch.
int select_launch(const float *u, int S, const int32_t *prefix_off, int total_rows,
                  const float *conf, const uint8_t *modality, float alpha, double r_text,
                  double r_img, int32_t *kept_idx, const int32_t *kept_off, float *score_out,
                  uint32_t *keys, int32_t *status, cudaStream_t stream) {
  // One cluster per sequence, sized so that a CTA's slice is about
  // kSliceTarget positions of an average sequence; slices up to kStageCta
  // positions are staged in shared memory.
  const int avg = total_rows / S;
  int cl = 1;
  while (cl < kMaxCluster && cl * kSliceTarget < avg) cl <<= 1;
  int cap = ((total_rows + cl - 1) / cl + 31) & ~31;
  if (cap > kStageCta) cap = kStageCta;
  static PerDevice attr_set;
  int set = 0;
  if (!attr_set.get(&set, [](int, int *v) {
        *v = 1;
        size_t most = 0;
        for (int c = 1; c <= kMaxCluster; c <<= 1) {
          const size_t b = select_smem_bytes(c, kStageCta);
          most = b > most ? b : most;
        }
        return cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)most) == cudaSuccess;
      }))
    return SPRINT_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(S * cl);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = select_smem_bytes(cl, cap);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, select_kernel, u, conf, modality, prefix_off, kept_off,
                         total_rows, alpha, r_text, r_img, keys, kept_idx, score_out, status,
                         cap) != cudaSuccess)
    return SPRINT_ERR_CUDA;
  return launch_status();
}


bool select_args_ok(int S, int total_rows, float alpha, double r_text, double r_img) {
  return S >= 0 && total_rows >= 0 && r_text >= 0.0 && r_text <= 1.0 && r_img >= 0.0 &&
         r_img <= 1.0 && alpha == alpha;
}

}  // namespace

extern "C" int sprint_key_norms(const void *K, int S, const int32_t *prefix_off, int total_rows,
                                int NL, int Hkv, int d, int dtype, float *u_out,
                                int32_t *status, cudaStream_t stream) {
  if (S < 0 || total_rows < 0 || NL < 1 || Hkv < 1 || d < 1) return SPRINT_ERR_INVALID_ARG;
  if (dtype != SPRINT_F32 && dtype != SPRINT_BF16) return SPRINT_ERR_INVALID_ARG;
  if (S == 0 || total_rows == 0) return SPRINT_OK;
  if (!prefix_off || !status || !K || !u_out) return SPRINT_ERR_INVALID_ARG;
  const int row_elems = Hkv * d;
  if (row_elems % 8 != 0 || !aligned16(K)) return SPRINT_ERR_UNSUPPORTED;
  return keynorm_launch(K, prefix_off, S, total_rows, NL, row_elems, dtype, u_out, status,
                        stream) == SPRINT_OK
             ? SPRINT_OK
             : SPRINT_ERR_CUDA;
}

extern "C" size_t sprint_select_kept_workspace_bytes(int S, int total_rows) {
  if (S < 0 || total_rows < 0) return 0;
  return align_up((size_t)total_rows * sizeof(uint32_t), 256);
}

extern "C" int sprint_select_kept(const float *u, int S, const int32_t *prefix_off,
                                  int total_rows, const float *conf, const uint8_t *modality,
                                  float alpha, double r_text, double r_img, int32_t *kept_idx,
                                  const int32_t *kept_off, float *score_out, void *ws,
                                  size_t ws_bytes, int32_t *status, cudaStream_t stream) {
  if (!select_args_ok(S, total_rows, alpha, r_text, r_img)) return SPRINT_ERR_INVALID_ARG;
  if (S == 0) return SPRINT_OK;
  if (!prefix_off || !kept_off || !status) return SPRINT_ERR_INVALID_ARG;
  if (total_rows > 0 && (!u || !conf || !modality || !ws)) return SPRINT_ERR_INVALID_ARG;
  if (ws_bytes < sprint_select_kept_workspace_bytes(S, total_rows)) return SPRINT_ERR_WORKSPACE;
  return select_launch(u, S, prefix_off, total_rows, conf, modality, alpha, r_text, r_img,
                       kept_idx, kept_off, score_out, static_cast<uint32_t *>(ws), status,
                       stream);
}

extern "C" int sprint_score_prune(const void *K, int S, const int32_t *prefix_off,
                                  int total_rows, int NL, int Hkv, int d, int dtype,
                                  const float *conf, const uint8_t *modality,
                                  float alpha, double r_text, double r_img,
                                  int32_t *kept_idx, const int32_t *kept_off,
                                  float *score_out, void *ws, size_t ws_bytes,
                                  int32_t *status, cudaStream_t stream) {
  if (NL < 1 || Hkv < 1 || d < 1) return SPRINT_ERR_INVALID_ARG;
  if (dtype != SPRINT_F32 && dtype != SPRINT_BF16) return SPRINT_ERR_INVALID_ARG;
  if (!select_args_ok(S, total_rows, alpha, r_text, r_img)) return SPRINT_ERR_INVALID_ARG;
  if (S == 0) return SPRINT_OK;
  if (!prefix_off || !kept_off || !status) return SPRINT_ERR_INVALID_ARG;
  if (total_rows > 0 && (!K || !conf || !modality || !ws)) return SPRINT_ERR_INVALID_ARG;
  const int row_elems = Hkv * d;
  if (row_elems % 8 != 0 || (K && !aligned16(K))) return SPRINT_ERR_UNSUPPORTED;
  if (ws_bytes < sprint_score_prune_workspace_bytes(S, total_rows)) return SPRINT_ERR_WORKSPACE;
  // The key norms, then the selection on them: sprint_key_norms followed by
  // sprint_select_kept.
  float *u = static_cast<float *>(ws);
  uint32_t *keys = reinterpret_cast<uint32_t *>(static_cast<char *>(ws) +
                                                align_up((size_t)total_rows * 4, 256));
  if (keynorm_launch(K, prefix_off, S, total_rows, NL, row_elems, dtype, u, status, stream) !=
      SPRINT_OK)
    return SPRINT_ERR_CUDA;
  return select_launch(u, S, prefix_off, total_rows, conf, modality, alpha, r_text, r_img,
                       kept_idx, kept_off, score_out, keys, status, stream);
}

extern "C" int sprint_keep_count(int n, double r) {
  if (n < 0 || !(r >= 0.0 && r <= 1.0)) return -1;
  return (int)floor(r * (double)n + 1e-9);
}
