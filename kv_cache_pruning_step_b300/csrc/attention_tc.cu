// bf16 block attention on the tcgen05 tensor cores, split over keys.
//
// LLaDA2.0-Uni paper (arXiv 2604.20796), "Sparse Prefix Retention"
// paragraph: the block's first step attends to the full prefix, later steps
// to the pruned prefix; attention inside the block is bidirectional.
//
// Work decomposition (stream-K).  For sequence s the keys of one (layer l,
// KV head g) pair are ceil(k_s / 128) prefix tiles of 128 keys plus one tile
// holding the block's LB keys.  All tiles of all pairs form one ordered list
// of T tiles; CTA c (of G = #SMs, one per SM) takes tiles
// [c T / G, (c+1) T / G).  A CTA's range splits into segments at pair
// boundaries; each segment writes one unnormalised partial (O rows, row max,
// row sum) into slot  pair(x) + min(G, ceil((x+1) G / T)) - 1  (x = the
// segment's first tile), which is unique over all segments and below
// #pairs + G.  attn_tc_combine_kernel enumerates the segments of every pair
// the same way and merges them in tile order.
//
// Per segment (192 threads):
//   warp 0      TMA: the pair's 128 query rows (LB block positions x G heads of
//               the group, one 3-D box per 64 head-dim columns), then K and V
//               tiles (128 keys x d) into a 2-stage ring (128-byte swizzle);
//   warp 1      owns 512 TMEM columns: S double buffer (2 x 128) and O (d);
//               one lane issues S = Q K^T (M=128, N=128) and O += P V
//               (M=128, N=d, V read MN-major), QK of tile t+1 ahead of PV of t;
//   warps 2-5   softmax, one query row per thread: tile max from S, lazy
//               rescale of O and l only when the max grows by more than 2^8,
//               P = exp2(S * log2e/sqrt(d) - m) written as bf16 into the
//               swizzled shared-memory A operand of the PV MMA; at the end of
//               the segment O, m, l go to the workspace.
#include <cuda.h>
#include <math.h>

#include "attention.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace sprint {

bool make_tmap_bf16_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                       uint64_t row_stride_elems, uint32_t box_inner, uint32_t box_rows);
unsigned long long wait_cap_ns();
int sm_count();

namespace {

constexpr int TILE = 128;       // keys per tile
constexpr int ROWS = 128;       // query rows per MMA tile (LB x G <= 128)
constexpr int THREADS = 192;
constexpr int MAX_SEQ = 1024;   // sequences per call on this path
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <int D> struct Layout {
  static constexpr int BOX = ROWS * 128;           // one 128-row x 64-col box
  static constexpr int Q_BYTES = (D / 64) * BOX;
  static constexpr int K_BYTES = (D / 64) * BOX;   // 128 keys x d
  static constexpr int STAGE = 2 * K_BYTES;        // K then V
  static constexpr int P_BYTES = 2 * BOX;          // 128 rows x 128 keys
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = Q_BYTES;
  static constexpr int OFF_P = OFF_KV + 2 * STAGE;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int OFF_SEQ = OFF_BAR + 256;
  static constexpr size_t SMEM = 1024 + OFF_SEQ + 4 * (MAX_SEQ + 1) * 4;
  static constexpr uint32_t TMEM_O = 2 * TILE;     // S buffers at 0 and 128
};

struct Problem {
  const int32_t *kv_off;
  int total_kv_rows, S, NL, LB, Hq, Hkv;
  float *ws_o, *ws_ml;
  int32_t *status;
  unsigned long long cap_ns;
};

// Per-sequence tables: ts[s] = first global tile of sequence s; nt[s] =
// tiles per (layer, KV head) pair = ceil(k_s/128) + 1; ks[s] = prefix keys
// (0 when the offsets are invalid); k0[s] = kv_off[s].
__device__ void build_seq_tables(const Problem &pb, int *ts, int *nt, int *ks, int *k0,
                                 int32_t *status) {
  if (threadIdx.x == 0) {
    int acc = 0;
    bool bad = false;
    for (int s = 0; s < pb.S; ++s) {
      int a = pb.kv_off[s], b = pb.kv_off[s + 1];
      int k = b - a;
      if (a < 0 || k < 0 || b > pb.total_kv_rows) { bad = true; k = 0; a = 0; }
      ts[s] = acc;
      nt[s] = (k + TILE - 1) / TILE + 1;
      ks[s] = k;
      k0[s] = a;
      acc += pb.NL * pb.Hkv * nt[s];
    }
    ts[pb.S] = acc;
    if (bad && blockIdx.x == 0) report(status, SPRINT_STATUS_BAD_OFFSETS);
  }
}

struct Seg {
  int s, l, g, pair;       // sequence, layer, KV head, global pair index
  int first_tile, ntile;   // tile index within the pair, tiles in the segment
  int n_pair, k_s, kv0;    // tiles of the pair, prefix keys, kv_off[s]
  int slot;
};

__device__ __forceinline__ int seq_of(const int *ts, int S, int x) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (ts[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ long long starts_le(long long x, int G, long long T) {
  long long c = ((x + 1) * G + T - 1) / T;
  return c < G ? c : G;
}

__device__ __forceinline__ Seg locate(const Problem &pb, const int *ts, const int *nt,
                                      const int *ks, const int *k0, int x, int end, int G,
                                      int T) {
  Seg sg;
  sg.s = seq_of(ts, pb.S, x);
  const int y = x - ts[sg.s];
  sg.n_pair = nt[sg.s];
  const int pis = y / sg.n_pair;
  sg.first_tile = y - pis * sg.n_pair;
  sg.l = pis / pb.Hkv;
  sg.g = pis - sg.l * pb.Hkv;
  sg.pair = sg.s * pb.NL * pb.Hkv + pis;
  const int pair_end = ts[sg.s] + (pis + 1) * sg.n_pair;
  sg.ntile = min(end, pair_end) - x;
  sg.kv0 = k0[sg.s];
  sg.k_s = ks[sg.s];
  sg.slot = sg.pair + (int)starts_le(x, G, T) - 1;
  return sg;
}

// Swizzled (128-byte) address of 16-byte chunk `ch` (0..15 over 128 keys) of
// row r in the P operand: two 64-key column blocks of 128 rows x 128 bytes.
__device__ __forceinline__ uint32_t p_chunk_addr(uint32_t p_base, int r, int ch) {
  const int blk = ch >> 3, c = ch & 7;
  return p_base + blk * (ROWS * 128) + r * 128 + ((c ^ (r & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
               const __grid_constant__ CUtensorMap tm_vp,
               const __grid_constant__ CUtensorMap tm_kb,
               const __grid_constant__ CUtensorMap tm_vb, Problem pb) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint64_t *q_full = bar + 0, *k_full = bar + 1, *v_full = bar + 3, *kv_empty = bar + 5;
  uint64_t *s_full = bar + 7, *s_free = bar + 9, *p_ready = bar + 11, *pv_done = bar + 12;
  uint64_t *o_full = bar + 13, *drain = bar + 14;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 15);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *ts = reinterpret_cast<int *>(smem + L::OFF_SEQ);
  int *nt = ts + (MAX_SEQ + 1), *ks = nt + (MAX_SEQ + 1), *k0 = ks + (MAX_SEQ + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int GQ = pb.Hq / pb.Hkv, R = pb.LB * GQ;

  // Zero every operand buffer once: rows TMA never writes (query rows >= R,
  // key rows past a short tile) then hold finite values.
  for (int i = threadIdx.x * 16; i < L::OFF_BAR; i += THREADS * 16)
    *reinterpret_cast<uint4 *>(smem + i) = make_uint4(0, 0, 0, 0);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  build_seq_tables(pb, ts, nt, ks, k0, pb.status);
  if (threadIdx.x == 0) {
    tc::mbar_init(tc::smem_u32(q_full), 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(tc::smem_u32(k_full + i), 1);
      tc::mbar_init(tc::smem_u32(v_full + i), 1);
      tc::mbar_init(tc::smem_u32(kv_empty + i), 1);
      tc::mbar_init(tc::smem_u32(s_full + i), 1);
      tc::mbar_init(tc::smem_u32(s_free + i), 4);
    }
    tc::mbar_init(tc::smem_u32(p_ready), 4);
    tc::mbar_init(tc::smem_u32(pv_done), 1);
    tc::mbar_init(tc::smem_u32(o_full), 1);
    tc::mbar_init(tc::smem_u32(drain), 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int T = ts[pb.S];
  const int x_begin = (int)((long long)blockIdx.x * T / G);
  const int x_end = (int)((long long)(blockIdx.x + 1) * T / G);
  const uint32_t sQ = tc::smem_u32(smem + L::OFF_Q);
  const uint32_t sKV = tc::smem_u32(smem + L::OFF_KV);
  const uint32_t sP = tc::smem_u32(smem + L::OFF_P);
  const float qk_scale = kLog2e * rsqrtf((float)D);

  // Counters shared in meaning by all roles (each role keeps its own copy).
  uint32_t seg_no = 0, tile_no = 0, qk_no = 0, pv_no = 0;
  // Producer bookkeeping for the final drain.
  uint32_t issued = 0, last_par = 0;

  for (int x = x_begin; x < x_end; ++seg_no) {
    const Seg sg = locate(pb, ts, nt, ks, k0, x, x_end, G, T);
    x += sg.ntile;
    const bool run = !*abort_flag;
    if (warp == 0 && lane == 0 && run) {
      // ------------------------------------------------ producer
      const uint32_t qb = tc::smem_u32(q_full);
      tc::mbar_arrive_expect_tx(qb, (uint32_t)((D / 64) * R * 128));
      const int qrow = (sg.s * pb.NL + sg.l) * pb.LB;
      for (int b = 0; b < D / 64; ++b)
        tc::tma_load_3d(sQ + b * L::BOX, &tm_q, qb, b * 64, sg.g * GQ, qrow);
      for (int t = 0; t < sg.ntile; ++t) {
        const int stage = (tile_no + t) & 1;
        const uint32_t ph = ((tile_no + t) >> 1) & 1;
        if (!tc::mbar_wait(tc::smem_u32(kv_empty + stage), ph ^ 1, pb.cap_ns, abort_flag)) break;
        const int i = sg.first_tile + t;
        const uint32_t kdst = sKV + stage * L::STAGE, vdst = kdst + L::K_BYTES;
        const uint32_t kb = tc::smem_u32(k_full + stage), vb = tc::smem_u32(v_full + stage);
        if (i < sg.n_pair - 1) {
          const int z = pb.NL * sg.kv0 + sg.l * sg.k_s + i * TILE;
          tc::mbar_arrive_expect_tx(kb, L::K_BYTES);
          for (int b = 0; b < D / 64; ++b) tc::tma_load_3d(kdst + b * L::BOX, &tm_kp, kb, b * 64, sg.g, z);
          tc::mbar_arrive_expect_tx(vb, L::K_BYTES);
          for (int b = 0; b < D / 64; ++b) tc::tma_load_3d(vdst + b * L::BOX, &tm_vp, vb, b * 64, sg.g, z);
        } else {
          const int z = (sg.s * pb.NL + sg.l) * pb.LB;
          const uint32_t bytes = (uint32_t)((D / 64) * pb.LB * 128);
          tc::mbar_arrive_expect_tx(kb, bytes);
          for (int b = 0; b < D / 64; ++b) tc::tma_load_3d(kdst + b * L::BOX, &tm_kb, kb, b * 64, sg.g, z);
          tc::mbar_arrive_expect_tx(vb, bytes);
          for (int b = 0; b < D / 64; ++b) tc::tma_load_3d(vdst + b * L::BOX, &tm_vb, vb, b * 64, sg.g, z);
        }
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (ph << stage);
      }
    } else if (warp == 1 && lane == 0 && run) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(ROWS, TILE, false, false);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(ROWS, D, false, true);
      bool ok = tc::mbar_wait(tc::smem_u32(q_full), seg_no & 1, pb.cap_ns, abort_flag);
      auto issue_pv = [&](int u) -> bool {
        const int stage = (tile_no + u) & 1;
        const uint32_t ph = ((tile_no + u) >> 1) & 1;
        if (!tc::mbar_wait(tc::smem_u32(p_ready), (pv_no + u) & 1, pb.cap_ns, abort_flag)) return false;
        if (!tc::mbar_wait(tc::smem_u32(v_full + stage), ph, pb.cap_ns, abort_flag)) return false;
        tc::fence_after_sync();
        const uint32_t vbase = sKV + stage * L::STAGE + L::K_BYTES;
#pragma unroll
        for (int k = 0; k < TILE / 16; ++k) {
          const uint64_t a = tc::desc_kmajor_sw128(sP + (k >> 2) * L::BOX + (k & 3) * 32);
          const uint64_t b = tc::desc_mnmajor_sw128(vbase + k * 16 * 128, L::BOX);
          tc::mma_bf16(tmem + L::TMEM_O, a, b, idesc_pv, (u > 0 || k > 0) ? 1u : 0u);
        }
        tc::mma_commit(tc::smem_u32(pv_done));
        tc::mma_commit(tc::smem_u32(kv_empty + stage));
        return true;
      };
      for (int t = 0; ok && t < sg.ntile; ++t) {
        const int stage = (tile_no + t) & 1;
        const uint32_t ph = ((tile_no + t) >> 1) & 1;
        const uint32_t q = qk_no + t, sb = q & 1;
        if (!tc::mbar_wait(tc::smem_u32(k_full + stage), ph, pb.cap_ns, abort_flag) ||
            !tc::mbar_wait(tc::smem_u32(s_free + sb), ((q >> 1) & 1) ^ 1, pb.cap_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t kbase = sKV + stage * L::STAGE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * L::BOX + (k & 3) * 32;
          tc::mma_bf16(tmem + sb * TILE, tc::desc_kmajor_sw128(sQ + off),
                       tc::desc_kmajor_sw128(kbase + off), idesc_qk, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(tc::smem_u32(s_full + sb));
        if (t > 0 && !issue_pv(t - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_pv(sg.ntile - 1);
      if (ok) tc::mma_commit(tc::smem_u32(o_full));
    } else if (warp >= 2 && run) {
      // ------------------------------------------------ softmax
      const int q4 = warp & 3, r = q4 * 32 + lane;
      const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
      float m_used = -INFINITY, l_sum = 0.f;
      bool ok = true;
      for (int t = 0; t < sg.ntile; ++t) {
        const uint32_t q = qk_no + t, sb = q & 1;
        const int i = sg.first_tile + t;
        const int nvalid = i < sg.n_pair - 1 ? min(TILE, sg.k_s - i * TILE) : pb.LB;
        if (!__all_sync(0xffffffffu,
                        tc::mbar_wait(tc::smem_u32(s_full + sb), (q >> 1) & 1, pb.cap_ns, abort_flag))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t s_addr = tmem + lane_off + sb * TILE;
        float mx = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < TILE / 32; ++c) {
          float v[32];
          tc::tmem_ld32(s_addr + c * 32, v);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c * 32 + j < nvalid) mx = fmaxf(mx, v[j] * qk_scale);
        }
        // P buffer and O are free once the previous PV has completed.
        if (t > 0 && !__all_sync(0xffffffffu, tc::mbar_wait(tc::smem_u32(pv_done),
                                                            (pv_no + t - 1) & 1, pb.cap_ns,
                                                            abort_flag))) {
          ok = false;
          break;
        }
        // Lazy rescale: a row moves its reference max only when the tile max
        // exceeds it by more than 2^8; O rows are rescaled in TMEM (the
        // tcgen05.ld/st are warp-collective, the factor is per row).
        const bool need = mx > m_used + kRescaleLog2;
        const float alpha = need ? exp2f(m_used - mx) : 1.0f;
        if (need) {
          l_sum *= alpha;
          m_used = mx;
        }
        if (t > 0 && __any_sync(0xffffffffu, need)) {
          tc::fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tc::tmem_ld32(tmem + lane_off + L::TMEM_O + c * 32, o);
            tc::tmem_wait_ld();
            uint32_t u[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(o[j] * alpha);
            asm volatile(
                "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
                "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
                ::"r"(tmem + lane_off + L::TMEM_O + c * 32),
                "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]),
                "r"(u[7]), "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]),
                "r"(u[13]), "r"(u[14]), "r"(u[15]), "r"(u[16]), "r"(u[17]), "r"(u[18]),
                "r"(u[19]), "r"(u[20]), "r"(u[21]), "r"(u[22]), "r"(u[23]), "r"(u[24]),
                "r"(u[25]), "r"(u[26]), "r"(u[27]), "r"(u[28]), "r"(u[29]), "r"(u[30]),
                "r"(u[31])
                : "memory");
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        // P = exp2(S * scale - m) in bf16, written to the swizzled A operand.
#pragma unroll 1
        for (int c = 0; c < TILE / 32; ++c) {
          float v[32];
          tc::tmem_ld32(s_addr + c * 32, v);
          tc::tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float p0 = c * 32 + j < nvalid ? exp2f(fmaf(v[j], qk_scale, -m_used)) : 0.f;
            const float p1 = c * 32 + j + 1 < nvalid ? exp2f(fmaf(v[j + 1], qk_scale, -m_used)) : 0.f;
            l_sum += p0 + p1;
            __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
            pk[j >> 1] = *reinterpret_cast<uint32_t *>(&h2);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t addr = p_chunk_addr(sP, r, c * 4 + u);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * u]),
                         "r"(pk[4 * u + 1]), "r"(pk[4 * u + 2]), "r"(pk[4 * u + 3])
                         : "memory");
          }
        }
        tc::fence_before_sync();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(tc::smem_u32(s_free + sb));
          tc::mbar_arrive(tc::smem_u32(p_ready));
        }
      }
      if (ok && __all_sync(0xffffffffu, tc::mbar_wait(tc::smem_u32(o_full), seg_no & 1,
                                                      pb.cap_ns, abort_flag))) {
        tc::fence_after_sync();
        float *dst = pb.ws_o + ((size_t)sg.slot * ROWS + r) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tc::tmem_ld32(tmem + lane_off + L::TMEM_O + c * 32, o);
          tc::tmem_wait_ld();
          if (r < R) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4 *>(dst + c * 32 + j) =
                  make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
          }
        }
        if (r < R) {
          pb.ws_ml[((size_t)sg.slot * ROWS + r) * 2] = m_used;
          pb.ws_ml[((size_t)sg.slot * ROWS + r) * 2 + 1] = l_sum;
        }
        tc::fence_before_sync();
      }
    }
    tile_no += sg.ntile;
    qk_no += sg.ntile;
    pv_no += sg.ntile;
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  }

  // Drain: no copy or MMA of this CTA may be in flight when it exits.
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < 2; ++s)
      if (issued >> s & 1u) {
        volatile int no_abort = 0;
        tc::mbar_wait(tc::smem_u32(k_full + s), last_par >> s & 1u, pb.cap_ns, &no_abort);
        tc::mbar_wait(tc::smem_u32(v_full + s), last_par >> s & 1u, pb.cap_ns, &no_abort);
      }
  }
  if (warp == 1 && lane == 0) {
    tc::mma_commit(tc::smem_u32(drain));
    volatile int no_abort = 0;
    tc::mbar_wait(tc::smem_u32(drain), 0, pb.cap_ns, &no_abort);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (threadIdx.x == 0 && *abort_flag) report(pb.status, SPRINT_STATUS_TIMEOUT);
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// One warp per (pair, query row): merge the pair's segments in tile order.
template <int D>
__global__ void attn_tc_combine_kernel(Problem pb, int G, __nv_bfloat16 *__restrict__ O) {
  __shared__ int ts[MAX_SEQ + 1], nt[MAX_SEQ + 1], ks[MAX_SEQ + 1], k0[MAX_SEQ + 1];
  build_seq_tables(pb, ts, nt, ks, k0, nullptr);
  __syncthreads();
  const int GQ = pb.Hq / pb.Hkv, R = pb.LB * GQ;
  const int lane = threadIdx.x & 31;
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long pairs = (long long)pb.S * pb.NL * pb.Hkv;
  if (w >= pairs * R) return;
  const int pair = (int)(w / R), r = (int)(w % R);
  const int per_seq = pb.NL * pb.Hkv;
  const int s = pair / per_seq, pis = pair % per_seq;
  const int l = pis / pb.Hkv, g = pis % pb.Hkv;
  const long long T = ts[pb.S];
  const int p0 = ts[s] + pis * nt[s], p1 = p0 + nt[s];
  float mx = -INFINITY;
  for (long long x = p0; x < p1;) {
    const long long c = starts_le(x, G, T);
    const long long nxt = c < G ? c * T / G : T;
    const int slot = pair + (int)c - 1;
    mx = fmaxf(mx, pb.ws_ml[((size_t)slot * ROWS + r) * 2]);
    x = nxt < p1 ? nxt : p1;
  }
  float den = 0.f, acc[D / 32];
#pragma unroll
  for (int q = 0; q < D / 32; ++q) acc[q] = 0.f;
  for (long long x = p0; x < p1;) {
    const long long c = starts_le(x, G, T);
    const long long nxt = c < G ? c * T / G : T;
    const int slot = pair + (int)c - 1;
    const float mc = pb.ws_ml[((size_t)slot * ROWS + r) * 2];
    if (mc != -INFINITY) {
      const float wgt = exp2f(mc - mx);
      den = fmaf(wgt, pb.ws_ml[((size_t)slot * ROWS + r) * 2 + 1], den);
      const float *oc = pb.ws_o + ((size_t)slot * ROWS + r) * D;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) acc[q] = fmaf(wgt, oc[lane + 32 * q], acc[q]);
    }
    x = nxt < p1 ? nxt : p1;
  }
  const int j = r / GQ, hh = r % GQ;
  __nv_bfloat16 *dst =
      O + (((size_t)(s * pb.NL + l) * pb.LB + j) * pb.Hq + (size_t)(g * GQ + hh)) * D;
  const float inv = 1.0f / den;
#pragma unroll
  for (int q = 0; q < D / 32; ++q) dst[lane + 32 * q] = __float2bfloat16_rn(acc[q] * inv);
}

EncodeTiledFn encode3() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 [rows][heads][D] tensor; box {64, box_heads, box_rows}, 128-byte swizzle.
bool make_tmap_3d(CUtensorMap *m, const void *base, int D, int heads, uint64_t rows,
                  int box_heads, int box_rows) {
  EncodeTiledFn fn = encode3();
  if (!fn || rows == 0) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, rows};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
  const cuuint32_t box[3] = {64u, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
int launch(const __nv_bfloat16 *Q, const __nv_bfloat16 *Kp, const __nv_bfloat16 *Vp,
           const int32_t *kv_off, int total_kv_rows, const __nv_bfloat16 *Kb,
           const __nv_bfloat16 *Vb, int S, int NL, int LB, int Hq, int Hkv, void *O, void *ws,
           int32_t *status, cudaStream_t stream) {
  using Lt = Layout<D>;
  const int GQ = Hq / Hkv;
  CUtensorMap tq, tkp, tvp, tkb, tvb;
  const uint64_t brows = (uint64_t)S * NL * LB;
  if (!make_tmap_3d(&tq, Q, D, Hq, brows, GQ, LB) || !make_tmap_3d(&tkb, Kb, D, Hkv, brows, 1, LB) ||
      !make_tmap_3d(&tvb, Vb, D, Hkv, brows, 1, LB))
    return SPRINT_ERR_CUDA;
  if (total_kv_rows > 0) {
    if (!make_tmap_3d(&tkp, Kp, D, Hkv, (uint64_t)NL * total_kv_rows, 1, TILE) ||
        !make_tmap_3d(&tvp, Vp, D, Hkv, (uint64_t)NL * total_kv_rows, 1, TILE))
      return SPRINT_ERR_CUDA;
  } else {  // no prefix rows at all: never dereferenced
    tkp = tkb;
    tvp = tvb;
  }
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Lt::SMEM) != cudaSuccess)
      return SPRINT_ERR_CUDA;
    attr = true;
  }
  const int G = sm_count();
  const size_t pairs = (size_t)S * NL * Hkv;
  Problem pb;
  pb.kv_off = kv_off;
  pb.total_kv_rows = total_kv_rows;
  pb.S = S; pb.NL = NL; pb.LB = LB; pb.Hq = Hq; pb.Hkv = Hkv;
  pb.ws_o = static_cast<float *>(ws);
  pb.ws_ml = reinterpret_cast<float *>(static_cast<char *>(ws) +
                                       align_up((pairs + G) * ROWS * D * 4, 256));
  pb.status = status;
  pb.cap_ns = wait_cap_ns();
  attn_tc_kernel<D><<<G, THREADS, Lt::SMEM, stream>>>(tq, tkp, tvp, tkb, tvb, pb);
  if (launch_status() != SPRINT_OK) return SPRINT_ERR_CUDA;
  const long long warps = (long long)pairs * LB * GQ;
  attn_tc_combine_kernel<D><<<(int)((warps * 32 + 255) / 256), 256, 0, stream>>>(
      pb, G, static_cast<__nv_bfloat16 *>(O));
  return launch_status();
}

}  // namespace

size_t attn_tc_workspace_bytes(int S, int NL, int Hkv, int d) {
  const size_t slots = (size_t)S * NL * Hkv + (size_t)sm_count();
  return align_up(slots * ROWS * d * 4, 256) + align_up(slots * ROWS * 2 * 4, 256);
}

int attn_tc_forward(const __nv_bfloat16 *Q, const __nv_bfloat16 *Kp, const __nv_bfloat16 *Vp,
                    const int32_t *kv_off, int total_kv_rows, const __nv_bfloat16 *Kb,
                    const __nv_bfloat16 *Vb, int S, int NL, int LB, int Hq, int Hkv, int d,
                    void *O, void *ws, int32_t *status, cudaStream_t stream) {
  if (S > MAX_SEQ) return SPRINT_ERR_UNSUPPORTED;
  return d == 64 ? launch<64>(Q, Kp, Vp, kv_off, total_kv_rows, Kb, Vb, S, NL, LB, Hq, Hkv, O,
                              ws, status, stream)
                 : launch<128>(Q, Kp, Vp, kv_off, total_kv_rows, Kb, Vb, S, NL, LB, Hq, Hkv, O,
                               ws, status, stream);
}

}  // namespace sprint
