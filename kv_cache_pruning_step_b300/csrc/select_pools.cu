// Selection with keep pools: the top positions of every pool, each pool with
// its own keep count.
//
// LLaDA2.0-Uni paper (arXiv 2604.20796), Inference section, "Sparse Prefix
// Retention" paragraph: positions are scored by s_i = alpha I_i + (1 -
// alpha) c_i and, within each group, the top positions by s_i are retained.
// The paper's groups are the two modalities (sprint_score_prune); here every
// position carries a pool id (text, one pool per image, or one pool for the
// whole prefix) and the caller gives each pool's keep count.
//
// Kernels (all latency-bound; the key norms come from keynorm_kernel):
//   pool_score_kernel    one thread-block cluster of cl CTAs (1024 threads
//                        each) per sequence, CTA r taking slice r of its
//                        positions: the mean of u and s_i with exactly the
//                        arithmetic of select_kernel (so the two modality
//                        pools reproduce its kept set bit for bit), the
//                        orderable key of every s_i, and each pool's size
//                        and smallest / largest key (warp-aggregated
//                        shared-memory atomics, merged by rank 0 through
//                        distributed shared memory).  Rank 0 checks the keep
//                        counts against the pool sizes and the kept offsets.
//   pool_select_kernel   one 1024-thread CTA per (sequence, pool): radix
//                        select of the pool's keep-th largest key T on keys
//                        reduced to the pool's range, 12 bits per pass, then
//                        the position of the last tie at T that is kept
//                        (ties go by ascending position).
//   pool_compact_kernel  one cluster of cl CTAs per sequence: stable
//                        compaction of the kept positions in ascending order
//                        (warp ballots, a scan of the 32 warp totals, the
//                        totals of the lower-ranked CTAs read through
//                        distributed shared memory, coalesced stores).
#include <limits.h>
#include <math.h>

#include <cooperative_groups.h>

#include "common.cuh"

namespace sprint {
namespace {

namespace cg = cooperative_groups;

constexpr int kThreads = 1024;
constexpr int kMaxCl = 8;           // CTAs per sequence, at most
constexpr int kPoolSlice = 4096;    // positions a CTA's slice aims at
constexpr int kDigit = 12, kBins = 1 << kDigit;
constexpr int kMaxPools = 256;

// Per (sequence, pool) record in the workspace.
struct PoolRec {
  int size;        // members
  int keep;        // keep count
  uint32_t kmin;   // smallest and largest key of the pool
  uint32_t kmax;
  int mode;        // 0 keep none, 1 keep all, 2 threshold
  uint32_t thresh; // threshold key T (mode 2)
  int tie_cut;     // keys equal to T are kept at positions <= tie_cut
  int ok;          // the sequence passed its checks
};

// What each CTA of a sequence's cluster publishes (read through distributed
// shared memory after a cluster barrier).
struct PoolXchg {
  double tree;  // this CTA's block of the canonical sum of u
  int bad;      // a position of the slice names no pool
  int kept;     // kept positions in the slice (compaction)
};

__global__ void __launch_bounds__(kThreads)
pool_score_kernel(const float *__restrict__ u, const float *__restrict__ conf,
                  const uint8_t *__restrict__ pool, int n_pools,
                  const int32_t *__restrict__ keep, const int32_t *__restrict__ prefix_off,
                  const int32_t *__restrict__ kept_off, int total_rows, int total_kept,
                  float alpha, uint32_t *__restrict__ keys, float *__restrict__ score_out,
                  PoolRec *__restrict__ rec, int32_t *status) {
  cg::cluster_group cluster = cg::this_cluster();
  const int cl = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  __shared__ double dsum_sh[32];
  __shared__ PoolXchg xc;
  __shared__ float mean_sh;
  __shared__ int cnt_sh[kMaxPools];
  __shared__ uint32_t kmin_sh[kMaxPools], kmax_sh[kMaxPools];
  __shared__ int bad_sh, ok_sh;
  const int s = blockIdx.x / cl, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  PoolRec *r = rec + (size_t)s * n_pools;
  const int p0 = prefix_off[s], p1 = prefix_off[s + 1];
  const int k0 = kept_off[s], k1 = kept_off[s + 1];
  // Every CTA of the cluster reads the same offsets, so all of them return
  // here or none does (before any cluster barrier).
  if (p0 < 0 || p1 < p0 || p1 > total_rows || k0 < 0 || k1 < k0 || k1 > total_kept) {
    if (rank == 0) {
      if (tid == 0) report(status, SPRINT_STATUS_BAD_OFFSETS);
      for (int p = tid; p < n_pools; p += kThreads) r[p].ok = 0;
    }
    return;
  }
  const int n = p1 - p0;
  const int L = ((n + cl - 1) / cl + 31) & ~31;
  const int lo = min(n, rank * L), hi = min(n, lo + L);
  for (int p = tid; p < kMaxPools; p += kThreads) {
    cnt_sh[p] = 0;
    kmin_sh[p] = 0xffffffffu;
    kmax_sh[p] = 0u;
  }
  if (tid == 0) bad_sh = 0;

  // Mean of u: the canonical sum (common.cuh) with the cluster's cl x 32
  // warps as the workers, the same bits as the two-modality selection's.
  {
    const int G = (n + kLeaf - 1) / kLeaf, P = next_pow2(G);
    const int workers = cl * 32, B = P > workers ? P / workers : 1;
    const int wk = rank * 32 + warp;
    const double v = wk * B < P ? u_subtree_sum(u + p0, n, G, wk * B, B, lane) : 0.0;
    if (lane == 0) dsum_sh[warp] = v;
  }
  __syncthreads();
  if (tid == 0) {
    double v[32];
    for (int i = 0; i < 32; ++i) v[i] = dsum_sh[i];
    tree_fold(v, 32);
    xc.tree = v[0];
  }
  cluster.sync();
  if (tid == 0) {
    double v[kMaxCl];
#pragma unroll
    for (int q = 0; q < kMaxCl; ++q)  // all remote loads in flight
      v[q] = q < cl ? cluster.map_shared_rank(&xc, q)->tree : 0.0;
    tree_fold(v, cl);
    mean_sh = n > 0 ? (float)(v[0] / (double)n) : 0.f;
  }
  __syncthreads();
  const float mean_f = mean_sh;

  // s_i, its key, and per-pool size and key range over the slice.
  const float one_m_alpha = 1.0f - alpha;
  for (int i0 = lo; i0 < hi; i0 += kThreads) {
    const int i = i0 + tid;
    const bool in = i < hi;
    const int pid = in ? (int)__ldg(pool + p0 + i) : -1;
    uint32_t key = 0u;
    if (in) {
      const float ui = __ldg(u + p0 + i), ci = __ldg(conf + p0 + i);
      const float imp = mean_f > 0.0f ? ui / mean_f : 0.0f;
      const float sc = fmaf(alpha, imp, one_m_alpha * ci);
      key = float_key(sc);
      keys[p0 + i] = key;
      if (score_out) score_out[p0 + i] = sc;
    }
    const bool member = in && pid < n_pools;
    if (in && !member) bad_sh = 1;
    // Lanes of one pool combine their count and key range; their lowest
    // lane updates the pool's shared entries.
    const unsigned grp = __match_any_sync(0xffffffffu, member ? pid : -1);
    const uint32_t klo = __reduce_min_sync(grp, key), khi = __reduce_max_sync(grp, key);
    if (member && lane == __ffs(grp) - 1) {
      atomicAdd(&cnt_sh[pid], __popc(grp));
      atomicMin(&kmin_sh[pid], klo);
      atomicMax(&kmax_sh[pid], khi);
    }
  }
  __syncthreads();
  if (tid == 0) xc.bad = bad_sh;
  cluster.sync();  // every CTA's pool counts and ranges are complete
  if (rank == 0) {
    // Pool sizes and key ranges over the cluster (rank 0's own entries are
    // read before they are overwritten, by the same thread).
    for (int p = tid; p < n_pools; p += kThreads) {
      int c[kMaxCl];
      uint32_t a[kMaxCl], z[kMaxCl];
#pragma unroll
      for (int q = 0; q < kMaxCl; ++q) {
        c[q] = q < cl ? cluster.map_shared_rank(cnt_sh, q)[p] : 0;
        a[q] = q < cl ? cluster.map_shared_rank(kmin_sh, q)[p] : 0xffffffffu;
        z[q] = q < cl ? cluster.map_shared_rank(kmax_sh, q)[p] : 0u;
      }
      int ct = 0;
      uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
      for (int q = 0; q < kMaxCl; ++q) {
        ct += c[q];
        mn = min(mn, a[q]);
        mx = max(mx, z[q]);
      }
      cnt_sh[p] = ct;
      kmin_sh[p] = mn;
      kmax_sh[p] = mx;
    }
    if (tid == 0) {
      int b = 0;
      for (int q = 0; q < cl; ++q) b |= cluster.map_shared_rank(&xc, q)->bad;
      bad_sh = b;
    }
    __syncthreads();
    // Keep counts: each within its pool, and together the sequence's kept rows.
    int sum = 0, bad = 0;
    for (int p = tid; p < n_pools; p += kThreads) {
      const int k = keep[(size_t)s * n_pools + p];
      bad |= k < 0 || k > cnt_sh[p];
      sum += k;
    }
    sum = warp_sum(sum);
    bad = __any_sync(0xffffffffu, bad);
    __shared__ int wsum_sh[32], wbad_sh[32];
    if (lane == 0) { wsum_sh[warp] = sum; wbad_sh[warp] = bad; }
    __syncthreads();
    if (warp == 0) {
      const int t = warp_sum(wsum_sh[lane]);
      const int b = __any_sync(0xffffffffu, wbad_sh[lane]);
      if (lane == 0) {
        ok_sh = !b && t == k1 - k0 && !bad_sh;
        if (b || t != k1 - k0) report(status, SPRINT_STATUS_KEPT_MISMATCH);
        if (bad_sh) report(status, SPRINT_STATUS_BAD_INDEX);
      }
    }
    __syncthreads();
    for (int p = tid; p < n_pools; p += kThreads) {
      const int k = keep[(size_t)s * n_pools + p];
      r[p].size = cnt_sh[p];
      r[p].keep = k;
      r[p].kmin = kmin_sh[p];
      r[p].kmax = kmax_sh[p];
      r[p].mode = k <= 0 ? 0 : (k >= cnt_sh[p] ? 1 : 2);
      r[p].thresh = 0u;
      r[p].tie_cut = INT_MAX;
      r[p].ok = ok_sh;
    }
  }
  cluster.sync();  // no CTA leaves while rank 0 may still read its shared memory
}

__global__ void __launch_bounds__(kThreads)
pool_select_kernel(const uint8_t *__restrict__ pool, int n_pools,
                   const int32_t *__restrict__ prefix_off, const uint32_t *__restrict__ keys,
                   PoolRec *__restrict__ rec) {
  __shared__ uint32_t hist[kBins];
  __shared__ int scan_sh[33];
  __shared__ uint32_t prefix_sh;
  __shared__ int shift_sh, need_sh, last_cnt_sh, cut_sh;
  const int s = blockIdx.x, p = blockIdx.y, tid = threadIdx.x;
  PoolRec &r = rec[(size_t)s * n_pools + p];
  if (!r.ok || r.mode != 2) return;
  const int p0 = prefix_off[s], n = prefix_off[s + 1] - p0;
  const uint8_t *pl = pool + p0;
  const uint32_t *ky = keys + p0;
  const uint32_t base = r.kmin, range = r.kmax - r.kmin;
  if (tid == 0) {
    prefix_sh = 0u;
    shift_sh = range ? 32 - __clz(range) : 0;
    need_sh = r.keep;
    last_cnt_sh = r.size;  // all keys equal: every member ties at T
  }
  __syncthreads();
  // Radix select on d = key - base, kDigit bits at a time from the top:
  // the keep-th largest key T, and need = how many keys equal to T are kept.
  while (shift_sh > 0) {
    const int sh = shift_sh, w = sh < kDigit ? sh : kDigit;
    const uint32_t pre = prefix_sh;
    const uint32_t need = (uint32_t)need_sh;
    for (int b = tid; b < kBins; b += kThreads) hist[b] = 0u;
    __syncthreads();
#pragma unroll 4
    for (int i = tid; i < n; i += kThreads) {
      if (__ldg(pl + i) != p) continue;
      const uint64_t d = (uint64_t)(__ldg(ky + i) - base);
      if ((uint32_t)(d >> sh) == pre)
        atomicAdd(&hist[(uint32_t)(d >> (sh - w)) & ((1u << w) - 1u)], 1u);
    }
    __syncthreads();
    uint32_t c[4];
    int mine = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      c[q] = hist[kBins - 1 - 4 * tid - q];
      mine += (int)c[q];
    }
    int total;
    uint32_t run = (uint32_t)block_excl_scan(mine, scan_sh, &total);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (run < need && run + c[q] >= need) {  // the keep-th largest is in this bin
        prefix_sh = (pre << w) | (uint32_t)(kBins - 1 - 4 * tid - q);
        need_sh = (int)(need - run);
        shift_sh = sh - w;
        last_cnt_sh = (int)c[q];
      }
      run += c[q];
    }
    __syncthreads();
  }
  const uint32_t T = base + prefix_sh;
  const int need = need_sh;
  // Ties: when fewer than all keys equal to T are kept, find the position of
  // the need-th of them in ascending order.
  if (need < last_cnt_sh) {
    int before = 0;
    if (tid == 0) cut_sh = INT_MAX;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kThreads) {
      const int i = i0 + tid;
      const int t = i < n && __ldg(pl + i) == p && __ldg(ky + i) == T;
      int total;
      const int excl = block_excl_scan(t, scan_sh, &total);
      if (before + total >= need) {
        if (t && before + excl + 1 == need) cut_sh = i;
        break;  // uniform: every thread sees the same totals
      }
      before += total;
    }
    __syncthreads();
  } else if (tid == 0) {
    cut_sh = INT_MAX;
  }
  __syncthreads();
  if (tid == 0) {
    r.thresh = T;
    r.tie_cut = cut_sh;
  }
}

__global__ void __launch_bounds__(kThreads)
pool_compact_kernel(const uint8_t *__restrict__ pool, int n_pools,
                    const int32_t *__restrict__ prefix_off, const int32_t *__restrict__ kept_off,
                    const uint32_t *__restrict__ keys, const PoolRec *__restrict__ rec,
                    int32_t *__restrict__ kept_idx, int32_t *status) {
  cg::cluster_group cluster = cg::this_cluster();
  const int cl = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  __shared__ int mode_sh[kMaxPools], cut_sh[kMaxPools];
  __shared__ uint32_t thr_sh[kMaxPools];
  __shared__ int wcnt[32];
  __shared__ PoolXchg xc;
  const int s = blockIdx.x / cl, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const PoolRec *r = rec + (size_t)s * n_pools;
  if (!r[0].ok) return;  // the same decision in every CTA of the cluster
  for (int p = tid; p < n_pools; p += kThreads) {
    mode_sh[p] = r[p].mode;
    thr_sh[p] = r[p].thresh;
    cut_sh[p] = r[p].tie_cut;
  }
  __syncthreads();
  const int p0 = prefix_off[s], n = prefix_off[s + 1] - p0;
  const int k0 = kept_off[s], k_all = kept_off[s + 1] - k0;
  // CTA rank takes positions [lo, hi); warp w of it a range of a multiple
  // of 32 positions.
  const int L = ((n + cl - 1) / cl + 31) & ~31;
  const int lo = min(n, rank * L), hi = min(n, lo + L);
  const int per_warp = ((hi - lo + 32 * 32 - 1) / (32 * 32)) * 32;
  const int w_lo = lo + warp * per_warp, w_hi = min(hi, w_lo + per_warp);
  auto kept = [&](int i) {
    if (i >= w_hi) return false;
    const int pid = __ldg(pool + p0 + i);
    if (pid >= n_pools) return false;
    const int m = mode_sh[pid];
    if (m != 2) return m == 1;
    const uint32_t key = __ldg(keys + p0 + i), T = thr_sh[pid];
    return key > T || (key == T && i <= cut_sh[pid]);
  };
  int c = 0;
  for (int i0 = w_lo; i0 < w_hi; i0 += 32) c += __popc(__ballot_sync(0xffffffffu, kept(i0 + lane)));
  if (lane == 0) wcnt[warp] = c;
  __syncthreads();
  if (warp == 0) {
    const int a = wcnt[lane];
    const int incl = warp_incl_scan(a);
    wcnt[lane] = incl - a;
    if (lane == 31) xc.kept = incl;
  }
  __shared__ int base_sh;
  cluster.sync();  // every CTA's kept count is published
  if (tid == 0) {  // kept positions in the lower-ranked CTAs' slices
    int v[kMaxCl], base = 0;
#pragma unroll
    for (int q = 0; q < kMaxCl; ++q) v[q] = q < rank ? cluster.map_shared_rank(&xc, q)->kept : 0;
#pragma unroll
    for (int q = 0; q < kMaxCl; ++q) base += v[q];
    base_sh = base;
  }
  __syncthreads();
  int out = base_sh + wcnt[warp];
  const unsigned lt = (1u << lane) - 1u;
  for (int i0 = w_lo; i0 < w_hi; i0 += 32) {
    const bool k = kept(i0 + lane);
    const unsigned b = __ballot_sync(0xffffffffu, k);
    if (k) {
      const int o = out + __popc(b & lt);
      if (o < k_all) kept_idx[k0 + o] = i0 + lane;
      else report(status, SPRINT_STATUS_KEPT_MISMATCH);
    }
    out += __popc(b);
  }
  cluster.sync();  // no CTA leaves while another may still read its count
}

}  // namespace
}  // namespace sprint

using namespace sprint;

extern "C" size_t sprint_select_kept_pools_workspace_bytes(int S, int total_rows, int n_pools) {
  if (S < 0 || total_rows < 0 || n_pools < 1 || n_pools > kMaxPools) return 0;
  return align_up((size_t)total_rows * sizeof(uint32_t), 256) +
         align_up((size_t)S * n_pools * sizeof(PoolRec), 256);
}

extern "C" size_t sprint_score_prune_pools_workspace_bytes(int S, int total_rows, int n_pools) {
  if (S < 0 || total_rows < 0 || n_pools < 1 || n_pools > kMaxPools) return 0;
  return align_up((size_t)total_rows * sizeof(float), 256) +
         sprint_select_kept_pools_workspace_bytes(S, total_rows, n_pools);
}

namespace {

int pools_args_ok(int S, int total_rows, int total_kept, int n_pools, float alpha) {
  return S >= 0 && total_rows >= 0 && total_kept >= 0 && n_pools >= 1 && n_pools <= kMaxPools &&
         alpha == alpha;
}

// The three pool kernels on key norms u already in memory; ws holds the
// keys and the pool records.
int pools_launch(const float *u, int S, const int32_t *prefix_off, int total_rows,
                 const float *conf, const uint8_t *pool, int n_pools, const int32_t *keep,
                 float alpha, int32_t *kept_idx, const int32_t *kept_off, int total_kept,
                 float *score_out, void *ws, int32_t *status, cudaStream_t stream) {
  char *w = static_cast<char *>(ws);
  uint32_t *keys = reinterpret_cast<uint32_t *>(w);
  w += align_up((size_t)total_rows * 4, 256);
  PoolRec *rec = reinterpret_cast<PoolRec *>(w);
  // One cluster per sequence for scoring and compaction, sized so that a
  // CTA's slice is about kPoolSlice positions of an average sequence.
  const int avg = total_rows / S;
  int cl = 1;
  while (cl < kMaxCl && cl * kPoolSlice < avg) cl <<= 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(S * cl);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, pool_score_kernel, u, conf, pool, n_pools, keep, prefix_off,
                         kept_off, total_rows, total_kept, alpha, keys, score_out, rec,
                         status) != cudaSuccess ||
      launch_status() != SPRINT_OK)
    return SPRINT_ERR_CUDA;
  pool_select_kernel<<<dim3(S, n_pools), kThreads, 0, stream>>>(pool, n_pools, prefix_off, keys,
                                                                rec);
  if (launch_status() != SPRINT_OK) return SPRINT_ERR_CUDA;
  if (cudaLaunchKernelEx(&cfg, pool_compact_kernel, pool, n_pools, prefix_off, kept_off,
                         (const uint32_t *)keys, (const PoolRec *)rec, kept_idx,
                         status) != cudaSuccess)
    return SPRINT_ERR_CUDA;
  return launch_status();
}

}  // namespace

extern "C" int sprint_select_kept_pools(const float *u, int S, const int32_t *prefix_off,
                                        int total_rows, const float *conf, const uint8_t *pool,
                                        int n_pools, const int32_t *keep, float alpha,
                                        int32_t *kept_idx, const int32_t *kept_off,
                                        int total_kept, float *score_out, void *ws,
                                        size_t ws_bytes, int32_t *status, cudaStream_t stream) {
  if (!pools_args_ok(S, total_rows, total_kept, n_pools, alpha)) return SPRINT_ERR_INVALID_ARG;
  if (S == 0) return SPRINT_OK;
  if (!prefix_off || !kept_off || !keep || !status || !ws) return SPRINT_ERR_INVALID_ARG;
  if (total_rows > 0 && (!u || !conf || !pool)) return SPRINT_ERR_INVALID_ARG;
  if (total_kept > 0 && !kept_idx) return SPRINT_ERR_INVALID_ARG;
  if (ws_bytes < sprint_select_kept_pools_workspace_bytes(S, total_rows, n_pools))
    return SPRINT_ERR_WORKSPACE;
  return pools_launch(u, S, prefix_off, total_rows, conf, pool, n_pools, keep, alpha, kept_idx,
                      kept_off, total_kept, score_out, ws, status, stream);
}

extern "C" int sprint_score_prune_pools(const void *K, int S, const int32_t *prefix_off,
                                        int total_rows, int NL, int Hkv, int d, int dtype,
                                        const float *conf, const uint8_t *pool, int n_pools,
                                        const int32_t *keep, float alpha, int32_t *kept_idx,
                                        const int32_t *kept_off, int total_kept,
                                        float *score_out, void *ws, size_t ws_bytes,
                                        int32_t *status, cudaStream_t stream) {
  if (!pools_args_ok(S, total_rows, total_kept, n_pools, alpha) || NL < 1 || Hkv < 1 || d < 1)
    return SPRINT_ERR_INVALID_ARG;
  if (dtype != SPRINT_F32 && dtype != SPRINT_BF16) return SPRINT_ERR_INVALID_ARG;
  if (S == 0) return SPRINT_OK;
  if (!prefix_off || !kept_off || !keep || !status || !ws) return SPRINT_ERR_INVALID_ARG;
  if (total_rows > 0 && (!K || !conf || !pool)) return SPRINT_ERR_INVALID_ARG;
  if (total_kept > 0 && !kept_idx) return SPRINT_ERR_INVALID_ARG;
  const int row_elems = Hkv * d;
  if (row_elems % 8 != 0 || (K && !aligned16(K))) return SPRINT_ERR_UNSUPPORTED;
  if (ws_bytes < sprint_score_prune_pools_workspace_bytes(S, total_rows, n_pools))
    return SPRINT_ERR_WORKSPACE;
  // The key norms, then the pool selection on them: sprint_key_norms
  // followed by sprint_select_kept_pools.
  float *u = static_cast<float *>(ws);
  void *rest = static_cast<char *>(ws) + align_up((size_t)total_rows * 4, 256);
  if (keynorm_launch(K, prefix_off, S, total_rows, NL, row_elems, dtype, u, status, stream) !=
      SPRINT_OK)
    return SPRINT_ERR_CUDA;
  return pools_launch(u, S, prefix_off, total_rows, conf, pool, n_pools, keep, alpha, kept_idx,
                      kept_off, total_kept, score_out, rest, status, stream);
}
