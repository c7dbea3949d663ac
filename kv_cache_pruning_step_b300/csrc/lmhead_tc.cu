// bf16 LM-head tiles on the tcgen05 tensor cores with the vocabulary
// softmax reduction fused into the epilogue.
//
// LLaDA2.0-Uni paper (arXiv 2604.20796): the block's first step scores every
// prefix position by its top-1 softmax confidence c_i ("Sparse Prefix
// Retention" paragraph) and every step ranks the block's predictions by
// c_n ("Non-uniform Token Unmasking" paragraph).  Both are max_v softmax
// of z = (h . W_v) / theta; the probability vector is never formed.
//
// Design (one persistent CTA per SM, 192 threads, 1 CTA/SM):
//   warp 0      TMA producer: 128x64 tiles of h and BNx64 tiles of W (bf16,
//               128-byte swizzle) into a shared-memory ring of as many
//               stages as fit in 227 KB; BN = 256, or 224 when the call has
//               few rows: the column tiles are then all the work, and 702
//               of them spread over 148 SMs more evenly than 614;
//   warp 1      allocates 512 TMEM columns; one lane issues
//               tcgen05.mma.kind::f16 (K=16) into one of two fp32
//               accumulators (TMEM columns 0 and 256);
//   warps 2-5   epilogue: each thread owns one accumulator row (TMEM lane),
//               reads its BN columns 32 at a time with tcgen05.ld, and folds
//               them into (max of raw dot products, first column reaching it
//               when the caller wants the greedy token, sum of exp2((acc -
//               max) * log2(e) / theta), one FMA and one ex2.approx per
//               element); optional logits (acc / theta in bf16).  Warps
//               whose rows all lie past M skip the reduction.  The second
//               accumulator lets the MMA of the next tile overlap this
//               epilogue.
// Calls with one row tile (block steps) run one CTA per tile with
// cta_group::1 MMAs of M=128, N=BN.  Calls with two or more row tiles (the
// prefix) run clusters of two CTAs whose MMAs are one cta_group::2 product
// of M=256, N=BN: each CTA loads its own h tile and half of the W tile, so
// W crosses from L2 into the SMs once per pair and each SM's tensor core
// reads half as much W from shared memory per MMA.
// Output tiles are visited in bands along one operand (at most 32 MB of h
// rows, or of W columns) that stays in L2 while the other operand's tiles
// stream past it once per band.
#include <cuda.h>
#include <math.h>
#include <stdlib.h>

#include <algorithm>

#include "common.cuh"
#include "lmhead.cuh"
#include "tc_ptx.cuh"

namespace sprint {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_STRIDE = 256;  // TMEM columns between the two accumulators
constexpr int THREADS = 192;
constexpr float kLog2e = 1.4426950408889634f;

// Tile shape per column width BN (256, or 224 for calls with few rows).  A
// CTA of a pair (kPair) loads half of each W tile: BN/2 rows.
template <int BN, bool kPair> struct Tiles {
  static constexpr int B_ROWS = kPair ? BN / 2 : BN;
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // As many stages as fit in 227 KB: 5 of 44 KB at BN = 224, 4 of 48 KB at
  // 256; 7 of 30 or 32 KB per CTA of a pair.
  static constexpr int STAGES = (227 * 1024 - 1024 - 256) / STAGE_BYTES;
  static constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 256;
  static_assert(STAGE_BYTES % 1024 == 0, "stages must stay 1024-byte aligned");
  static_assert(BN % 32 == 0 && BN <= 256, "epilogue reads 32 columns at a time");
  static_assert(8 * (2 * STAGES + 7) <= 256, "barriers, TMEM slot and abort flag fit in 256 bytes");
};

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x with the hardware approximation (relative error about 2^-22);
// results below 2^-126 flush to zero (terms that small do not change a sum
// that contains 2^0).
__device__ __forceinline__ float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Tile order for L2 reuse: tiles are visited in bands of `band` consecutive
// tiles along the kept operand's axis (row units of h, or column tiles of
// W); inside a band the other operand's tiles are the outer loop, so each
// of them streams from DRAM once per band while the band's tiles of the
// kept operand stay in L2 (every one is touched again after about one band
// of reads).  Consecutive tile numbers run on concurrent CTAs, which
// therefore share the streamed tile.
struct TileOrder {
  int keep_h;  // 1: bands of h row units, 0: bands of W column tiles
  int band;    // tiles of the kept operand per band
};

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, TileOrder o, int &m,
                                            int &n) {
  const int kept = o.keep_h ? num_m : num_n, streamed = o.keep_h ? num_n : num_m;
  const int per_band = o.band * streamed;
  const int b = t / per_band;
  const int idx = t - b * per_band;
  const int bw = min(o.band, kept - b * o.band);
  const int k = b * o.band + idx % bw, q = idx / bw;
  m = o.keep_h ? k : q;
  n = o.keep_h ? q : k;
}

// kArg: also track the first column reaching each row's maximum (the
// greedy token).  Without it the chunk maximum is a three-input max tree.
// kPair: the grid is made of clusters of two CTAs that run their MMAs as
// one cta_group::2 product of M = 256 rows: rank 0 and rank 1 take row
// tiles 2i and 2i+1 of the same column tile, and each loads its own h tile
// and its own half (BN/2 rows) of the W tile, so W is read once per pair.
// Rank 0 issues the MMAs; both CTAs' copies complete on rank 0's full
// barrier, its commits arrive on both CTAs' empty and accumulator-full
// barriers, and rank 1's epilogue hands the accumulator back on rank 0's
// accumulator-empty barrier.  Each CTA's tensor memory holds its own 128
// rows of the 128 x BN product: columns [0, BN/2) from rank 0's W half,
// [BN/2, BN) from rank 1's.
template <int BN, bool kArg, bool kPair>
__global__ void __launch_bounds__(THREADS, 1)
lmhead_tc_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                 const float *__restrict__ temp, int M, int D, int V,
                 __nv_bfloat16 *__restrict__ logits, float *__restrict__ pmax,
                 float *__restrict__ psum, int32_t *__restrict__ parg, int32_t *status,
                 unsigned long long cap_ns, int stall_test, TileOrder order, Gate gate) {
  if (gate_closed(gate)) return;
  // The final waits for in-flight copies and MMAs ignore the abort flag and
  // get at least one second.
  const unsigned long long drain_ns = cap_ns > 1000000000ull ? cap_ns : 1000000000ull;
  constexpr int STAGE_BYTES = Tiles<BN, kPair>::STAGE_BYTES;
  constexpr int STAGES = Tiles<BN, kPair>::STAGES;
  constexpr int B_ROWS = Tiles<BN, kPair>::B_ROWS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  uint64_t *full = bars, *empty = bars + STAGES;
  uint64_t *tfull = bars + 2 * STAGES, *tempty = tfull + 2, *drain = tempty + 2;
  uint64_t *never = drain + 1;  // no one arrives: the stall test waits on it
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(never + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = (M + BM - 1) / BM, num_n = (V + BN - 1) / BN;
  // Scheduling units: one CTA, or one pair of CTAs (rank 0 / 1 take row
  // tiles 2 mu and 2 mu + 1).
  const uint32_t rank = kPair ? tc::cluster_ctarank() : 0u;
  const int unit = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int units = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int num_mu = kPair ? (num_m + 1) / 2 : num_m;
  const int tiles = num_mu * num_n, nk = (D + BK - 1) / BK;
  auto coords = [&](int t, int &m, int &n) {
    int mu;
    tile_coords(t, num_mu, num_n, order, mu, n);
    m = kPair ? 2 * mu + (int)rank : mu;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(tc::smem_u32(full + s), 1);   // the expect-tx arrive (rank 0 of a pair)
      tc::mbar_init(tc::smem_u32(empty + s), 1);  // one MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(tc::smem_u32(tfull + b), 1);
      tc::mbar_init(tc::smem_u32(tempty + b), kPair ? 8 : 4);  // epilogue warps (of both CTAs)
    }
    tc::mbar_init(tc::smem_u32(drain), 1);
    tc::mbar_init(tc::smem_u32(never), 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    if (kPair) {
      tc::tmem_alloc_pair(tc::smem_u32(tmem_slot), TMEM_COLS);
      tc::tmem_relinquish_pair();
    } else {
      tc::tmem_alloc(tc::smem_u32(tmem_slot), TMEM_COLS);
      tc::tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tm_h);
    tc::prefetch_tmap(&tm_w);
  }
  tc::fence_before_sync();
  __syncthreads();
  // The peer CTA signals this CTA's barriers: both must be initialised.
  if (kPair) tc::cluster_sync();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs of a pair)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_parity = 0;  // bit s: stage s has a load issued
      for (int t = unit; t < tiles; t += units) {
        int m, n;
        coords(t, m, n);
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(tc::smem_u32(empty + stage), phase ^ 1, cap_ns, abort_flag))
            goto producer_done;
          const uint32_t fb = tc::smem_u32(full + stage);
          const uint32_t sa = tc::smem_u32(smem + stage * STAGE_BYTES);
          if (kPair) {
            // Both CTAs' tiles complete on rank 0's full barrier, armed by
            // rank 0 for the two CTAs' bytes.
            const uint32_t fb0 = tc::map_to_rank(fb, 0);
            if (rank == 0) tc::mbar_arrive_expect_tx(fb, 2 * STAGE_BYTES);
            tc::tma_load_2d_pair(sa, &tm_h, fb0, kb * BK, m * BM);
            tc::tma_load_2d_pair(sa + A_BYTES, &tm_w, fb0, kb * BK, n * BN + (int)rank * B_ROWS);
          } else {
            tc::mbar_arrive_expect_tx(fb, STAGE_BYTES);  // h tile + W tile
            tc::tma_load_2d(sa, &tm_h, fb, kb * BK, m * BM);
            tc::tma_load_2d(sa + A_BYTES, &tm_w, fb, kb * BK, n * BN);
          }
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
    producer_done:
      // Never leave with a copy in flight: wait (bounded) for the last load
      // issued into every stage.  Rank 0's full barriers also count rank
      // 1's copies; rank 1 stays resident until rank 0 has drained (the
      // cluster barrier before exit).
      if (!kPair || rank == 0)
        for (int s = 0; s < STAGES; ++s)
          if (issued >> s & 1u) {
            volatile int no_abort = 0;
            tc::mbar_wait(tc::smem_u32(full + s), last_parity >> s & 1u, drain_ns, &no_abort);
          }
    }
  } else if (warp == 1) {
    if (lane == 0 && (!kPair || rank == 0)) {
      // ---------------- MMA issuer (rank 0 of a pair)
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kPair ? 2 * BM : BM, BN, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      // Failure-path test: wait on a barrier no one arrives on, so the
      // bounded wait expires and the CTA takes its abort path.
      if (stall_test) tc::mbar_wait(tc::smem_u32(never), 0, cap_ns, abort_flag);
      for (int t = unit; t < tiles && !*abort_flag; t += units, ++it) {
        const int buf = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!tc::mbar_wait(tc::smem_u32(tempty + buf), (use & 1u) ^ 1u, cap_ns, abort_flag))
          break;
        tc::fence_after_sync();
        const uint32_t d = tmem + (uint32_t)buf * ACC_STRIDE;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(tc::smem_u32(full + stage), phase, cap_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sa = tc::smem_u32(smem + stage * STAGE_BYTES);
          const uint64_t adesc = tc::desc_kmajor_sw128(sa);
          const uint64_t bdesc = tc::desc_kmajor_sw128(sa + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {  // +32 bytes along K per step
            if (kPair)
              tc::mma_bf16_pair(d, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
            else
              tc::mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
          }
          if (kPair)
            tc::mma_commit_pair_multicast(tc::smem_u32(empty + stage), 0x3);
          else
            tc::mma_commit(tc::smem_u32(empty + stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if (kPair)
          tc::mma_commit_pair_multicast(tc::smem_u32(tfull + buf), 0x3);
        else
          tc::mma_commit(tc::smem_u32(tfull + buf));
      }
      // Every MMA this thread issued has finished once `drain` completes.
      if (kPair)
        tc::mma_commit_pair(tc::smem_u32(drain));
      else
        tc::mma_commit(tc::smem_u32(drain));
      volatile int no_abort = 0;
      tc::mbar_wait(tc::smem_u32(drain), 0, drain_ns, &no_abort);
    }
  } else {
    // ---------------- epilogue: one accumulator row per thread
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r_tile = q * 32 + lane;
    int it = 0;
    for (int t = unit; t < tiles; t += units, ++it) {
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      int m, n;
      coords(t, m, n);
      if (!tc::mbar_wait(tc::smem_u32(tfull + buf), use & 1u, cap_ns, abort_flag)) break;
      tc::fence_after_sync();
      const int row = m * BM + r_tile;
      const bool vrow = row < M;
      float th = 1.0f;
      if (temp && vrow) {
        th = temp[row];
        if (!(th > 0.0f) || !isfinite(th)) {
          report(status, SPRINT_STATUS_BAD_TEMPERATURE);
          th = 1.0f;
        }
      }
      const float sc = kLog2e / th, inv = 1.0f / th;
      float run_max = -INFINITY, run_sum = 0.f;
      int arg = 0;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)buf * ACC_STRIDE;
      const int col0 = n * BN;
      // A warp whose 32 rows all lie past M (a call with few rows) has
      // nothing to reduce: it only hands the accumulator back.
      const bool live = m * BM + q * 32 < M;
#pragma unroll 1
      for (int c = 0; live && c < BN / 32; ++c) {
        const int cb = col0 + c * 32;
        const int ncol = min(32, V - cb);
        if (ncol <= 0) break;  // uniform across the warp
        float v[32];
        tc::tmem_ld32(taddr + (uint32_t)(c * 32), v);
        if (ncol < 32) {  // past the vocabulary: no maximum, no probability
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i >= ncol) v[i] = -INFINITY;
        }
        float cm;
        int ca = 0;
        if (kArg) {
          cm = v[0];
#pragma unroll
          for (int i = 1; i < 32; ++i)
            if (v[i] > cm) { cm = v[i]; ca = i; }
        } else {
          float t[11];
#pragma unroll
          for (int i = 0; i < 10; ++i) t[i] = max3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
          t[10] = fmaxf(v[30], v[31]);
          cm = max3(max3(t[0], t[1], t[2]), max3(t[3], t[4], t[5]),
                    max3(max3(t[6], t[7], t[8]), t[9], t[10]));
        }
        if (cm > run_max) {
          run_sum *= fast_exp2((run_max - cm) * sc);
          run_max = cm;
          arg = cb + ca;
        }
        // exp2((v - max) * log2(e) / theta) as one FMA each, four partial sums
        const float nb = -run_max * sc;
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 32; ++i) s4[i & 3] += fast_exp2(fmaf(v[i], sc, nb));
        run_sum += (s4[0] + s4[1]) + (s4[2] + s4[3]);
        if (logits && vrow) {
          __nv_bfloat16 *dst = logits + (size_t)row * V + cb;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < ncol) dst[i] = __float2bfloat16_rn(v[i] * inv);
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        // Rank 0's MMA issuer reuses the buffer once every epilogue warp of
        // the pair has read it.
        if (kPair)
          tc::mbar_arrive_cluster(tc::map_to_rank(tc::smem_u32(tempty + buf), 0));
        else
          tc::mbar_arrive(tc::smem_u32(tempty + buf));
      }
      if (vrow) {
        const size_t at = (size_t)n * M + row;
        pmax[at] = run_max;
        psum[at] = run_sum;
        if (kArg) parg[at] = arg;
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  // Neither CTA of a pair leaves, or frees its tensor memory, while the
  // other may still signal it or write into it (rank 0's MMAs are done once
  // its drain wait above has completed).
  if (kPair) tc::cluster_sync();
  tc::fence_after_sync();
  if (threadIdx.x == 0 && *abort_flag) report(status, SPRINT_STATUS_TIMEOUT);
  if (warp == 1) {
    if (kPair)
      tc::tmem_dealloc_pair(tmem, TMEM_COLS);
    else
      tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

EncodeTiledFn encode_fn() {
  // Looked up once per process (a thread-safe static initialisation).
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
  }();
  return fn;
}

// bf16 row-major [rows][inner] tensor map with a (box_inner x box_rows) box
// in the 128-byte swizzle; out-of-range elements read as zero.
bool make_tmap_bf16_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                       uint64_t row_stride_elems, uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_stride_elems * 2};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int stall_test_enabled() {
  static const int v = [] {
    const char *e = getenv("SPRINT_TEST_STALL");
    return (e && e[0] == '1') ? 1 : 0;
  }();
  return v;
}

unsigned long long wait_cap_ns() {
  static const unsigned long long cap = [] {
    const char *e = getenv("SPRINT_WAIT_CAP_NS");
    const unsigned long long c = e ? strtoull(e, nullptr, 10) : 2000000000ull;
    return c ? c : 1ull;
  }();
  return cap;
}

int sm_count() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

template <int BN, bool kArg, bool kPair>
int launch_kernel(const CUtensorMap &tm_h, const CUtensorMap &tm_w, const float *temp, int M,
                  int D, int V, __nv_bfloat16 *logits, const LmheadWs &p, int32_t *status,
                  Gate gate, int units, TileOrder order, cudaStream_t stream) {
  constexpr size_t SMEM_BYTES = Tiles<BN, kPair>::SMEM_BYTES;
  auto kern = lmhead_tc_kernel<BN, kArg, kPair>;
  static PerDevice attr_set;
  int set = 0;
  if (!attr_set.get(&set, [&](int, int *v) {
        *v = 1;
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)SMEM_BYTES) == cudaSuccess;
      }))
    return SPRINT_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  int grid = units;
  if (kPair) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Clusters resident at once (pairs of SMs in a GPC); every pair keeps
    // its tiles, so more pairs than fit would only run later.
    static PerDevice pairs_cache;
    int max_pairs = 1;
    if (!pairs_cache.get(&max_pairs, [&](int, int *v) {
          cfg.gridDim = dim3(2 * units);
          int mp = 0;
          if (cudaOccupancyMaxActiveClusters(&mp, kern, &cfg) != cudaSuccess || mp < 1) {
            (void)cudaGetLastError();  // not a launch error: fall back to one pair
            mp = 1;
          }
          *v = mp;
          return true;
        }))
      return SPRINT_ERR_CUDA;
    grid = 2 * (units < max_pairs ? units : max_pairs);
  }
  cfg.gridDim = dim3(grid);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tm_h, tm_w, temp, M, D, V, logits,
                                           p.pmax, p.psum, p.parg, status, wait_cap_ns(),
                                           stall_test_enabled(), order, gate);
  if (e != cudaSuccess) return SPRINT_ERR_CUDA;
  return launch_status();
}

// The kept operand's band is at most kKeepBytes; the order with the smaller
// estimate of DRAM reads wins: keeping h reads h once and W once per band of
// rows, keeping W the other way round.  32 MB is what measured best at the
// 32K-row prefix (both orders, bands of 16 to 64 MB, with and without L2
// eviction hints): far less than the 126 MB L2 stays useful to tiles that
// all 148 SMs read.
constexpr size_t kKeepBytes = size_t(32) << 20;

TileOrder tile_order(int num_m, int num_n, size_t m_tile_bytes, size_t n_tile_bytes) {
  auto banding = [](int tiles, size_t tile_bytes, int &band) {
    const int most = (int)std::max<size_t>(1, kKeepBytes / tile_bytes);
    const int bands = (tiles + most - 1) / most;
    band = (tiles + bands - 1) / bands;
    return bands;
  };
  int band_m, band_n;
  const double h = (double)num_m * m_tile_bytes, w = (double)num_n * n_tile_bytes;
  const double keep_h = h + w * banding(num_m, m_tile_bytes, band_m);
  const double keep_w = w + h * banding(num_n, n_tile_bytes, band_n);
  return keep_h <= keep_w ? TileOrder{1, band_m} : TileOrder{0, band_n};
}

template <int BN>
int launch_tiles(const __nv_bfloat16 *h, const __nv_bfloat16 *W, const float *temp, int M, int D,
                 int V, __nv_bfloat16 *logits, const LmheadWs &p, int32_t *status, Gate gate,
                 cudaStream_t stream) {
  CUtensorMap tm_h, tm_w;
  const int num_m = (M + BM - 1) / BM, num_n = (V + BN - 1) / BN;
  // Calls with two or more row tiles run as CTA pairs; a CTA of a pair
  // loads BN/2 rows of each W tile.
  const bool pair = num_m >= 2;
  if (!make_tmap_bf16_2d(&tm_h, h, D, M, D, BK, BM) ||
      !make_tmap_bf16_2d(&tm_w, W, D, V, D, BK, pair ? BN / 2 : BN))
    return SPRINT_ERR_CUDA;
  const int sms = sm_count();
  const int num_mu = pair ? (num_m + 1) / 2 : num_m;
  const TileOrder order = tile_order(num_mu, num_n, (size_t)(pair ? 2 * BM : BM) * D * 2,
                                     (size_t)BN * D * 2);
  if (pair) {
    const int pair_tiles = num_mu * num_n;
    const int pairs = pair_tiles < sms / 2 ? pair_tiles : sms / 2;
    return p.parg ? launch_kernel<BN, true, true>(tm_h, tm_w, temp, M, D, V, logits, p, status,
                                                   gate, pairs, order, stream)
                  : launch_kernel<BN, false, true>(tm_h, tm_w, temp, M, D, V, logits, p, status,
                                                    gate, pairs, order, stream);
  }
  const int tiles = num_m * num_n;
  const int grid = tiles < sms ? tiles : sms;
  return p.parg ? launch_kernel<BN, true, false>(tm_h, tm_w, temp, M, D, V, logits, p, status,
                                                  gate, grid, order, stream)
                : launch_kernel<BN, false, false>(tm_h, tm_w, temp, M, D, V, logits, p, status,
                                                   gate, grid, order, stream);
}

int lmhead_tc_tiles(const __nv_bfloat16 *h, const __nv_bfloat16 *W, const float *temp, int M,
                    int D, int V, __nv_bfloat16 *logits, const LmheadWs &p, int32_t *status,
                    Gate gate, cudaStream_t stream) {
  if (p.cols == kPartColsNarrow)
    return launch_tiles<kPartColsNarrow>(h, W, temp, M, D, V, logits, p, status, gate, stream);
  if (p.cols == kPartCols)
    return launch_tiles<kPartCols>(h, W, temp, M, D, V, logits, p, status, gate, stream);
  return SPRINT_ERR_UNSUPPORTED;
}

}  // namespace sprint
