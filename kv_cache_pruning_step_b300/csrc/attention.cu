// Bidirectional in-block attention over [prefix ; block], split over keys.
//
// LLaDA2.0-Uni paper (arXiv 2604.20796), "Sparse Prefix Retention"
// paragraph: the first step of a block attends to the full prefix, every
// later step to the pruned prefix; block diffusion (BDLM paragraph) gives
// bidirectional attention inside the block.
//
// Work unit: (sequence, layer, KV head g, key chunk).  The R = LB * Hq/Hkv
// query rows that share KV head g (GQA group) are processed together, row
// r = j * G + hh for block position j and head g * G + hh.  Each unit writes
// an unnormalised partial (row max m in log2 units, row sum l, O row) to the
// workspace; attn_combine_kernel merges the chunks in ascending order.
// This file holds the CUDA-core (SIMT) chunk kernel used for fp32 and the
// combine kernel and entry point; bf16 runs on tcgen05 (attention_tc.cu).
#include <math.h>

#include "attention.cuh"
#include "common.cuh"

namespace sprint {

constexpr float kLog2e = 1.4426950408889634f;

template <typename T, int D>
__global__ void __launch_bounds__(256)
attn_simt_kernel(const T *__restrict__ Q, const T *__restrict__ Kp, const T *__restrict__ Vp,
                 const int32_t *__restrict__ kv_off, int total_kv_rows,
                 const T *__restrict__ Kb, const T *__restrict__ Vb, int NL, int LB, int Hq,
                 int Hkv, AttnWs ws, int32_t *status, KvIndex kvi, Gate gate) {
  constexpr int TK = 32;
  if (gate_closed(gate)) return;
  extern __shared__ float smem[];
  const int G = Hq / Hkv, R = LB * G;
  float *Qs = smem;                  // [R][D]
  float *Ks = Qs + R * D;            // [TK][D + 1]
  float *Vs = Ks + TK * (D + 1);     // [TK][D]

  const int chunk = blockIdx.x, s = blockIdx.z;
  const int l = blockIdx.y / Hkv, g = blockIdx.y % Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int o0 = kv_off[s], o1 = kv_off[s + 1];
  const size_t unit = (((size_t)s * NL + l) * Hkv + g) * ws.chunks + chunk;
  float *out_o = ws.o + unit * R * D;
  float *out_ml = ws.ml + unit * R * 2;
  if (o0 < 0 || o1 < o0 || o1 > total_kv_rows) {
    if (tid == 0) report(status, SPRINT_STATUS_BAD_OFFSETS);
    for (int r = tid; r < R; r += 256) { out_ml[2 * r] = -INFINITY; out_ml[2 * r + 1] = 0.f; }
    for (int e = tid; e < R * D; e += 256) out_o[e] = 0.f;
    return;
  }
  // Rows of the prefix keys: contiguous from NL * o0 + l * kn, or (indexed)
  // row idx[o0 + key] of layer l of the sequence's full prefix.
  int pf0 = 0, n_full = 0;
  if (kvi.idx) {
    pf0 = kvi.prefix_off[s];
    const int pf1 = kvi.prefix_off[s + 1];
    if (pf0 < 0 || pf1 < pf0 || pf1 > kvi.total_prefix_rows) {
      if (tid == 0 && chunk == 0) report(status, SPRINT_STATUS_BAD_OFFSETS);
      pf0 = 0;
    } else {
      n_full = pf1 - pf0;
    }
  }
  const int kn = o1 - o0, N = kn + LB;
  const int lo = chunk * ws.chunk_keys;
  const int hi = min(N, lo + ws.chunk_keys);
  if (lo >= hi) {
    for (int r = tid; r < R; r += 256) { out_ml[2 * r] = -INFINITY; out_ml[2 * r + 1] = 0.f; }
    for (int e = tid; e < R * D; e += 256) out_o[e] = 0.f;
    return;
  }
  // Queries, pre-scaled so that scores come out in log2 units.
  const float qscale = kLog2e / sqrtf((float)D);
  for (int e = tid; e < R * D; e += 256) {
    const int r = e / D, x = e % D, j = r / G, hh = r % G;
    Qs[e] = to_f32(Q[((((size_t)s * NL + l) * LB + j) * Hq + g * G + hh) * D + x]) * qscale;
  }
  constexpr int ROWS_MAX = 16;  // R <= 128 rows over 8 warps
  float m_run[ROWS_MAX], l_run[ROWS_MAX], o_run[ROWS_MAX][D / 32];
#pragma unroll
  for (int i = 0; i < ROWS_MAX; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int q = 0; q < D / 32; ++q) o_run[i][q] = 0.f;
  }
  for (int k0 = lo; k0 < hi; k0 += TK) {
    __syncthreads();
    for (int e = tid; e < TK * D; e += 256) {
      const int kk = e / D, x = e % D, key = k0 + kk;
      float kv = 0.f, vv = 0.f;
      if (key < hi) {
        size_t at;
        if (key < kn) {
          size_t row = (size_t)NL * o0 + (size_t)l * kn + key;
          bool ok = true;
          if (kvi.idx) {
            const int src = kvi.idx[o0 + key];
            ok = src >= 0 && src < n_full;
            if (!ok && x == 0) report(status, SPRINT_STATUS_BAD_INDEX);
            row = (size_t)NL * pf0 + (size_t)l * n_full + (ok ? src : 0);
          }
          at = (row * Hkv + g) * D + x;
          kv = ok ? to_f32(Kp[at]) : 0.f;
          vv = ok ? to_f32(Vp[at]) : 0.f;
        } else {
          at = ((((size_t)s * NL + l) * LB + (key - kn)) * Hkv + g) * D + x;
          kv = to_f32(Kb[at]);
          vv = to_f32(Vb[at]);
        }
      }
      Ks[kk * (D + 1) + x] = kv;
      Vs[kk * D + x] = vv;
    }
    __syncthreads();
    const bool valid = k0 + lane < hi;
#pragma unroll
    for (int i = 0; i < ROWS_MAX; ++i) {
      const int r = warp + 8 * i;
      if (r >= R) break;
      const float *qr = Qs + r * D;
      const float *kr = Ks + lane * (D + 1);
      float sc = 0.f;
#pragma unroll 8
      for (int x = 0; x < D; ++x) sc = fmaf(qr[x], kr[x], sc);
      sc = valid ? sc : -INFINITY;
      const float m_new = fmaxf(m_run[i], warp_max(sc));
      const float p = exp2f(sc - m_new);
      const float corr = exp2f(m_run[i] - m_new);
      l_run[i] = l_run[i] * corr + warp_sum(p);
      m_run[i] = m_new;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) o_run[i][q] *= corr;
      for (int kk = 0; kk < TK; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, p, kk);
#pragma unroll
        for (int q = 0; q < D / 32; ++q) o_run[i][q] = fmaf(pk, Vs[kk * D + lane + 32 * q], o_run[i][q]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < ROWS_MAX; ++i) {
    const int r = warp + 8 * i;
    if (r >= R) break;
    if (lane == 0) { out_ml[2 * r] = m_run[i]; out_ml[2 * r + 1] = l_run[i]; }
#pragma unroll
    for (int q = 0; q < D / 32; ++q) out_o[(size_t)r * D + lane + 32 * q] = o_run[i][q];
  }
}

// One warp per output row (sequence, layer, KV head, group row): merge the
// chunk partials in ascending chunk order and normalise.
template <typename T>
__global__ void attn_combine_kernel(AttnWs ws, int S, int NL, int LB, int Hq, int Hkv, int D,
                                    T *__restrict__ O, AttnResidual res, Gate gate) {
  if (gate_closed(gate)) return;
  const int G = Hq / Hkv, R = LB * G;
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)S * NL * Hkv * R) return;
  const int r = (int)(row % R);
  const long long sg = row / R;  // ((s * NL + l) * Hkv + g)
  const int g = (int)(sg % Hkv);
  const long long sl = sg / Hkv;  // s * NL + l
  const size_t base_unit = (size_t)sg * ws.chunks;
  float mx = -INFINITY;
  for (int c = 0; c < ws.chunks; ++c) mx = fmaxf(mx, ws.ml[((base_unit + c) * R + r) * 2]);
  float den = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c = 0; c < ws.chunks; ++c) {
    const size_t u = base_unit + c;
    const float mc = ws.ml[(u * R + r) * 2];
    if (mc == -INFINITY) continue;
    const float w = exp2f(mc - mx);
    den = fmaf(w, ws.ml[(u * R + r) * 2 + 1], den);
    const float *oc = ws.o + (u * R + r) * D;
    for (int q = 0; q * 32 < D; ++q) acc[q] = fmaf(w, oc[lane + 32 * q], acc[q]);
  }
  const int j = r / G, hh = r % G;
  const size_t at = ((size_t)sl * LB + j) * Hq * D + (size_t)(g * G + hh) * D;
  T *dst = O + at;
  const float inv = 1.0f / den;
  // Residual epilogue on the last layer: h_out[s][j] = h_in[s][j] + O (heads
  // concatenated), from O as stored.
  const bool last = res.h_out && (int)(sl % NL) == NL - 1;
  const size_t hat = ((size_t)(sl / NL) * LB + j) * Hq * D + (size_t)(g * G + hh) * D;
  for (int q = 0; q * 32 < D; ++q) {
    const T o = from_f32<T>(acc[q] * inv);
    dst[lane + 32 * q] = o;
    if (last)
      static_cast<T *>(res.h_out)[hat + lane + 32 * q] =
          from_f32<T>(to_f32(static_cast<const T *>(res.h_in)[hat + lane + 32 * q]) + to_f32(o));
  }
}

// h_out = h_in + O of the last layer, heads concatenated: one thread per
// element of h ([S * LB][Hq * d]).
template <typename T>
__global__ void residual_kernel(const T *__restrict__ h_in, const T *__restrict__ O, int NL,
                                int LB, int width, long long total, T *__restrict__ h_out) {
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const long long row = e / width, c = e % width;  // row = s * LB + j
    const long long s = row / LB, j = row % LB;
    const T o = O[((s * NL + (NL - 1)) * LB + j) * width + c];
    h_out[e] = from_f32<T>(to_f32(h_in[e]) + to_f32(o));
  }
}

int attn_chunk_keys(int S, int NL, int Hkv, int LB, int max_kv_rows, int target_units) {
  const long long pairs = (long long)S * NL * Hkv;
  const int n_max = max_kv_rows + LB;
  long long want = (target_units + pairs - 1) / pairs;
  if (want < 1) want = 1;
  int ck = (int)((n_max + want - 1) / want);
  ck = (ck + 127) / 128 * 128;
  if (ck < 128) ck = 128;
  return ck;
}

AttnWs attn_ws_layout(void *ws, int S, int NL, int LB, int Hq, int Hkv, int d, int max_kv_rows,
                      int chunk_keys) {
  const int R = LB * (Hq / Hkv);
  const int chunks = (max_kv_rows + LB + chunk_keys - 1) / chunk_keys;
  const size_t units = (size_t)S * NL * Hkv * chunks;
  char *p = static_cast<char *>(ws);
  AttnWs w;
  w.o = reinterpret_cast<float *>(p);
  w.ml = reinterpret_cast<float *>(p + align_up(units * R * d * 4, 256));
  w.chunks = chunks;
  w.chunk_keys = chunk_keys;
  w.bytes = align_up(units * R * d * 4, 256) + align_up(units * R * 2 * 4, 256);
  return w;
}

}  // namespace sprint

using namespace sprint;

// The fp32 SIMT kernel is arithmetic-bound: spread it over ~4 units per SM.
static int attn_chunk_policy(int S, int NL, int Hkv, int LB, int max_kv_rows) {
  return attn_chunk_keys(S, NL, Hkv, LB, max_kv_rows, 4 * 148);
}

extern "C" size_t sprint_block_attn_workspace_bytes(int S, int NL, int LB, int Hq, int Hkv,
                                                    int d, int max_kv_rows, int dtype) {
  if (S < 1 || NL < 1 || LB < 1 || Hq < 1 || Hkv < 1 || d < 1 || max_kv_rows < 0 ||
      Hq % Hkv != 0)
    return 0;
  if (dtype == SPRINT_BF16) return attn_tc_workspace_bytes(S, NL, Hkv, d);
  const int ck = attn_chunk_policy(S, NL, Hkv, LB, max_kv_rows);
  return attn_ws_layout(nullptr, S, NL, LB, Hq, Hkv, d, max_kv_rows, ck).bytes;
}

int sprint::block_attn_impl(const void *Q, const void *Kp, const void *Vp,
                            const int32_t *kv_off, int max_kv_rows, int total_kv_rows,
                            const void *Kb, const void *Vb, int S, int NL, int LB, int Hq,
                            int Hkv, int d, int dtype, void *O, void *ws, size_t ws_bytes,
                            int32_t *status, KvIndex kvi, AttnResidual res, Gate gate,
                            cudaStream_t stream, SideStream side) {
  if (S < 0 || NL < 1 || LB < 1 || Hq < 1 || Hkv < 1 || max_kv_rows < 0 || total_kv_rows < 0)
    return SPRINT_ERR_INVALID_ARG;
  if (dtype != SPRINT_F32 && dtype != SPRINT_BF16) return SPRINT_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return SPRINT_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return SPRINT_ERR_UNSUPPORTED;
  if (LB * (Hq / Hkv) > 128) return SPRINT_ERR_UNSUPPORTED;
  if (S == 0) return SPRINT_OK;
  if (!Q || !kv_off || !Kb || !Vb || !O || !ws || !status) return SPRINT_ERR_INVALID_ARG;
  if (total_kv_rows > 0 && (!Kp || !Vp)) return SPRINT_ERR_INVALID_ARG;
  if (kvi.idx && (!kvi.prefix_off || kvi.total_prefix_rows < total_kv_rows))
    return SPRINT_ERR_INVALID_ARG;
  if (res.h_out && !res.h_in) return SPRINT_ERR_INVALID_ARG;
  if (ws_bytes < sprint_block_attn_workspace_bytes(S, NL, LB, Hq, Hkv, d, max_kv_rows, dtype))
    return SPRINT_ERR_WORKSPACE;
  if (dtype == SPRINT_BF16) {
    if (!aligned16(Q) || !aligned16(Kb) || !aligned16(Vb) || (Kp && !aligned16(Kp)) ||
        (Vp && !aligned16(Vp)))
      return SPRINT_ERR_UNSUPPORTED;
    return attn_tc_forward(static_cast<const __nv_bfloat16 *>(Q),
                           static_cast<const __nv_bfloat16 *>(Kp),
                           static_cast<const __nv_bfloat16 *>(Vp), kv_off, total_kv_rows,
                           static_cast<const __nv_bfloat16 *>(Kb),
                           static_cast<const __nv_bfloat16 *>(Vb), S, NL, LB, Hq, Hkv, d, O, ws,
                           status, kvi, res, gate, stream, side);
  }
  const int ck = attn_chunk_policy(S, NL, Hkv, LB, max_kv_rows);
  const AttnWs w = attn_ws_layout(ws, S, NL, LB, Hq, Hkv, d, max_kv_rows, ck);
  const int R = LB * (Hq / Hkv);
  {
    dim3 grid(w.chunks, NL * Hkv, S);
    const size_t sm = ((size_t)R * d + 32 * (d + 1) + 32 * d) * 4;
    if (d == 64) {
      cudaFuncSetAttribute(attn_simt_kernel<float, 64>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      attn_simt_kernel<float, 64><<<grid, 256, sm, stream>>>(
          static_cast<const float *>(Q), static_cast<const float *>(Kp),
          static_cast<const float *>(Vp), kv_off, total_kv_rows, static_cast<const float *>(Kb),
          static_cast<const float *>(Vb), NL, LB, Hq, Hkv, w, status, kvi, gate);
    } else {
      cudaFuncSetAttribute(attn_simt_kernel<float, 128>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      attn_simt_kernel<float, 128><<<grid, 256, sm, stream>>>(
          static_cast<const float *>(Q), static_cast<const float *>(Kp),
          static_cast<const float *>(Vp), kv_off, total_kv_rows, static_cast<const float *>(Kb),
          static_cast<const float *>(Vb), NL, LB, Hq, Hkv, w, status, kvi, gate);
    }
    if (launch_status() != SPRINT_OK) return SPRINT_ERR_CUDA;
  }
  const long long rows = (long long)S * NL * Hkv * R;
  const int blocks = (int)((rows * 32 + 255) / 256);
  attn_combine_kernel<float><<<blocks, 256, 0, stream>>>(w, S, NL, LB, Hq, Hkv, d,
                                                         static_cast<float *>(O), res, gate);
  return launch_status();
}

extern "C" int sprint_block_attn(const void *Q, const void *Kp, const void *Vp,
                                 const int32_t *kv_off, int max_kv_rows, int total_kv_rows,
                                 const void *Kb, const void *Vb, int S, int NL, int LB, int Hq,
                                 int Hkv, int d, int dtype, void *O, void *ws, size_t ws_bytes,
                                 int32_t *status, cudaStream_t stream) {
  return block_attn_impl(Q, Kp, Vp, kv_off, max_kv_rows, total_kv_rows, Kb, Vb, S, NL, LB, Hq,
                         Hkv, d, dtype, O, ws, ws_bytes, status, KvIndex{nullptr, nullptr, 0},
                         AttnResidual{nullptr, nullptr}, Gate{nullptr, 0}, stream);
}

extern "C" int sprint_block_attn_indexed(const void *Q, const void *K, const void *V,
                                         const int32_t *prefix_off, int total_rows,
                                         const int32_t *kept_idx, const int32_t *kept_off,
                                         int max_kept, int total_kept, const void *Kb,
                                         const void *Vb, int S, int NL, int LB, int Hq, int Hkv,
                                         int d, int dtype, void *O, void *ws, size_t ws_bytes,
                                         int32_t *status, cudaStream_t stream) {
  if ((!kept_idx && total_kept > 0) || !prefix_off || total_rows < 0)
    return SPRINT_ERR_INVALID_ARG;
  // Nothing kept: only the block's own keys, as in the contiguous layout.
  const KvIndex kvi = total_kept > 0 ? KvIndex{kept_idx, prefix_off, total_rows}
                                     : KvIndex{nullptr, nullptr, 0};
  return block_attn_impl(Q, K, V, kept_off, max_kept, total_kept, Kb, Vb, S, NL, LB, Hq, Hkv, d,
                         dtype, O, ws, ws_bytes, status, kvi, AttnResidual{nullptr, nullptr},
                         Gate{nullptr, 0}, stream);
}

extern "C" int sprint_prefix_attn(const void *Qp, const void *K, const void *V,
                                  const int32_t *prefix_off, int total_rows, int S, int NL,
                                  int Hq, int Hkv, int d, int dtype, void *Op, int32_t *status,
                                  cudaStream_t stream) {
  if (S < 0 || total_rows < 0 || NL < 1 || Hq < 1 || Hkv < 1) return SPRINT_ERR_INVALID_ARG;
  if (dtype != SPRINT_F32 && dtype != SPRINT_BF16) return SPRINT_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return SPRINT_ERR_INVALID_ARG;
  if (dtype != SPRINT_BF16 || (d != 64 && d != 128)) return SPRINT_ERR_UNSUPPORTED;
  if (S == 0 || total_rows == 0) return SPRINT_OK;
  if (!Qp || !K || !V || !prefix_off || !Op || !status) return SPRINT_ERR_INVALID_ARG;
  if ((long long)NL * total_rows > 0x7fffffffLL) return SPRINT_ERR_UNSUPPORTED;
  if (!aligned16(Qp) || !aligned16(K) || !aligned16(V) || !aligned16(Op))
    return SPRINT_ERR_UNSUPPORTED;
  return attn_tc_prefix(static_cast<const __nv_bfloat16 *>(Qp),
                        static_cast<const __nv_bfloat16 *>(K),
                        static_cast<const __nv_bfloat16 *>(V), prefix_off, total_rows, S, NL, Hq,
                        Hkv, d, static_cast<__nv_bfloat16 *>(Op), status, stream);
}

extern "C" int sprint_residual_hidden(const void *h_in, const void *O, int S, int NL, int LB,
                                      int Hq, int d, int dtype, void *h_out,
                                      cudaStream_t stream) {
  if (S < 0 || NL < 1 || LB < 1 || Hq < 1 || d < 1) return SPRINT_ERR_INVALID_ARG;
  if (dtype != SPRINT_F32 && dtype != SPRINT_BF16) return SPRINT_ERR_INVALID_ARG;
  if (S == 0) return SPRINT_OK;
  if (!h_in || !O || !h_out) return SPRINT_ERR_INVALID_ARG;
  const long long total = (long long)S * LB * Hq * d;
  const int blocks = (int)((total + 255) / 256 < 148 * 16 ? (total + 255) / 256 : 148 * 16);
  if (dtype == SPRINT_BF16)
    residual_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(h_in), static_cast<const __nv_bfloat16 *>(O), NL, LB,
        Hq * d, total, static_cast<__nv_bfloat16 *>(h_out));
  else
    residual_kernel<float><<<blocks, 256, 0, stream>>>(static_cast<const float *>(h_in),
                                                       static_cast<const float *>(O), NL, LB,
                                                       Hq * d, total,
                                                       static_cast<float *>(h_out));
  return launch_status();
}
