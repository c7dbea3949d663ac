// bf16 block attention on the tcgen05 tensor cores, split over keys.
//
// LLaDA2.0-Uni paper (arXiv 2604.20796), "Sparse Prefix Retention"
// paragraph: the block's first step attends to the full prefix, later steps
// to the pruned prefix; attention inside the block is bidirectional.
//
// Work decomposition (stream-K).  For sequence s the keys of one (layer l,
// KV head g) pair are ceil(k_s / 128) prefix tiles of 128 keys plus
// ceil(LB / 128) tiles of the block's own keys.  All tiles of all pairs form
// one ordered list of T tiles, split over G CTAs (one per SM) in contiguous
// ranges.  The split charges every pair start kPairCost tiles: tile x of
// pair p sits at virtual position v(x) = x + kPairCost (p + 1) of VT = T +
// kPairCost #pairs, and CTA c takes the tiles with v(x) in [c VT / G,
// (c+1) VT / G), so a CTA whose range takes in a pair start gets fewer tiles.
// A CTA's range splits into segments at pair boundaries; each segment writes
// two unnormalised partials (O rows, row max, row sum; one per softmax
// warpgroup) into slots 2 * slot + {0, 1} with slot = pair(x) + min(G,
// ceil((v(x)+1) G / VT)) - 1 (x = the segment's first tile, the second term
// its CTA), which is unique over all segments and below #pairs + G.
// attn_tc_combine_kernel enumerates the segments of every pair the same way
// and merges them in tile order.
//
// Per segment (352 threads):
//   warp 0      TMA: the pair's 128 query rows (LB block positions x G heads of
//               the group, one 3-D box per 64 head-dim columns), then K and V
//               tiles (128 keys x d) into a ring of as many 64 KB stages as
//               fit (3 for a few sequences; 128-byte swizzle);
//   warp 1      owns 512 TMEM columns: two S buffers (128 columns each) and
//               two O accumulators (d each); one lane issues S = Q K^T
//               (M=128, N=128) for tile q into S[q & 1] once the PV of tile
//               q-2 (whose P lives there) is done;
//   warp 10     one lane issues O[q & 1] += P V (M=128, N=d, K=128, P read
//               from tensor memory as the A operand, V MN-major from shared
//               memory); with one thread issuing both products the issue
//               rate, not HBM, bounded the kernel;
//   warps 2-9   softmax in two warpgroups that take alternate tiles:
//               warpgroup h owns the tiles q with q & 1 == h, with its own S
//               buffer and O accumulator, and runs its own online softmax
//               (row max m_h, row sum l_h), one query row per thread.  A
//               first pass over S in TMEM finds the tile max; the reference
//               max moves only when the tile max exceeds it by more than 2^8
//               (O_h is then rescaled in TMEM); a second pass writes P =
//               exp2(S * log2e/sqrt(d) - m_h) as bf16 pairs over the first 64
//               columns of S_h, where the PV product reads it.  P is handed
//               to the PV issuer in quarters of 32 keys, each with its own
//               barrier, so the products of a quarter run while the next is
//               computed and little of the PV is left once the softmax ends.
//               At the end of the segment each warpgroup writes its (O_h,
//               m_h, l_h) partial, O in column quads of 32-row runs so that
//               every store of a warp is 512 contiguous bytes.
//
// Segments of a CTA follow each other without a CTA-wide barrier: the
// producer loads the next segment's first K/V tile while the last tiles of
// the current one are still being computed, and its query once the
// segment's last QK has read Q (q_empty); each warpgroup writes its partial
// as soon as its own last PV is done (o_full[h]) and goes on to the next
// segment, whose first PV into its accumulator follows from the P hand-over.
//
// Indexed prefix (no compacted copy): the kept rows are gathered from the
// full cache through the kept indices.  Then warps 0 and 11 each load half
// of a prefix tile with 16-byte cp.async copies (a 256-byte head row per 16
// lanes) into the same 128-byte-swizzled layout the TMA writes; each lane
// waits for its own copies, fences them for the tensor cores (generic to
// async proxy) and arrives on the stage's full barrier itself (64 arrivals:
// every lane's release follows its own fence); the MMA issuers fence again
// after their wait, before the tensor cores read the stage.
// With three or more stages a warp does not wait for tile q's copies right
// after issuing them: it arrives for tile q once it has issued the first
// quarter of tile q+1 (the stage of q+1 frees when the PV of tile q-2 ends,
// which is also when the QK of tile q may start).
#include <cuda.h>
#include <math.h>

#include <type_traits>

#include "attention.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace sprint {

bool make_tmap_bf16_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                       uint64_t row_stride_elems, uint32_t box_inner, uint32_t box_rows);
unsigned long long wait_cap_ns();
int stall_test_enabled();
int sm_count();

namespace {

constexpr int TILE = 128;       // keys per tile
constexpr int MAX_STAGES = 4;   // K/V ring depth at most (as many as fit)
// mbarriers (21 + 2 MAX_STAGES), the TMEM address and the abort flag share
// a 256-byte block.
static_assert((21 + 2 * MAX_STAGES) * 8 + 8 <= 256, "barrier block overflows");
constexpr int ROWS = 128;       // query rows per MMA tile (LB x G <= 128)
constexpr int THREADS = 352;
// The indexed-prefix kernel adds a second gathering warp; 384 threads still
// leave 168 registers per thread.
constexpr int GATHER_WARP = 11;
constexpr int THREADS_INDEXED = 384;
constexpr int MAX_SEQ = 1024;   // sequences per call on this path
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <int D> struct Layout {
  static constexpr int QBOX = ROWS * 128;          // 128 query rows x 64 cols
  static constexpr int KBOX = TILE * 128;          // 128 keys x 64 cols
  static constexpr int Q_BYTES = (D / 64) * QBOX;
  static constexpr int K_BYTES = (D / 64) * KBOX;  // 128 keys x d
  static constexpr int STAGE = 2 * K_BYTES;        // K then V
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = Q_BYTES;
  // Dynamic shared memory of a launch with `stages` ring stages and S
  // sequences: [Q][stages x (K, V)][barriers 256 B][4 x (S+1) int tables].
  static size_t smem_bytes(int stages, int S) {
    return 1024 + (size_t)OFF_KV + (size_t)stages * STAGE + 256 + 16 * (size_t)(S + 1);
  }
  // TMEM columns: S[0], S[1] at 0 and 128 (P[h] overwrites the first 64
  // columns of S[h] as bf16 pairs), O[0], O[1] after them.
  static constexpr uint32_t TMEM_O = 2 * TILE;
};

struct Problem {
  const int32_t *kv_off;
  int total_kv_rows, S, NL, LB, Hq, Hkv;
  float *ws_o, *ws_ml;
  int32_t *status;
  unsigned long long cap_ns;    // limit of every pipeline wait
  unsigned long long drain_ns;  // limit of the final waits for in-flight work
  int stall_test;               // failure-path test: the MMA role stalls first
  Gate gate;                    // step gate of the native block driver
  int stages;                   // K/V ring stages of this launch (2..MAX_STAGES)
  KvIndex kvi;                  // indexed prefix (kvi.idx != nullptr): gathered
  const __nv_bfloat16 *Kf, *Vf; // from these full caches
  __nv_bfloat16 *Op;            // prefix self-attention: output [NL][n][Hq][d] per sequence
  bool prefix;                  // prefix self-attention (no block keys, one unit per
                                // (layer, query head, 128-row query tile), whole key range)
};

// Per-sequence tables: ts[s] = first global unit of sequence s (decode: its
// first tile); nt[s] = tiles per (layer, KV head) pair = ceil(k_s / TILE) +
// ceil(LB / TILE) (prefix mode: ceil(k_s / TILE)); ks[s] = prefix keys (0
// when the offsets are invalid); k0[s] = kv_off[s].
//
// kParallel (decode and the combine): one thread per sequence reads its
// offsets, and warp 0 turns the per-sequence unit counts into ts by an
// exclusive scan (each lane over a contiguous run of sequences); every
// thread of the CTA calls it.  Otherwise thread 0 walks the sequences (the
// prefix self-attention's units are long, and its registers are tight).
template <bool kParallel>
__device__ void build_seq_tables(const Problem &pb, int *ts, int *nt, int *ks, int *k0,
                                 int32_t *status) {
  const int per_pair = pb.prefix ? pb.NL * pb.Hkv * (pb.Hq / pb.Hkv) : pb.NL * pb.Hkv;
  // Prefix mode: units (layer, KV head, query tile, head of the group) of
  // ceil(k / TILE) key tiles each; decode: the prefix tiles and the block's
  // own key tiles of every (layer, KV head) pair.
  auto seq = [&](int s, bool &bad) {
    int a = pb.kv_off[s], b = pb.kv_off[s + 1];
    int k = b - a;
    if (a < 0 || k < 0 || b > pb.total_kv_rows) { bad = true; k = 0; a = 0; }
    ks[s] = k;
    k0[s] = a;
    nt[s] = pb.prefix ? (k + TILE - 1) / TILE : (k + TILE - 1) / TILE + (pb.LB + TILE - 1) / TILE;
  };
  if (!kParallel) {
    if (threadIdx.x == 0) {
      int acc = 0;
      bool bad = false;
      for (int s = 0; s < pb.S; ++s) {
        seq(s, bad);
        ts[s] = acc;
        acc += per_pair * nt[s];
      }
      ts[pb.S] = acc;
      if (bad && blockIdx.x == 0) report(status, SPRINT_STATUS_BAD_OFFSETS);
    }
    return;
  }
  bool bad = false;
  for (int s = threadIdx.x; s < pb.S; s += blockDim.x) seq(s, bad);
  if (bad && blockIdx.x == 0) report(status, SPRINT_STATUS_BAD_OFFSETS);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int run = (pb.S + 31) / 32, lo = min(pb.S, lane * run), hi = min(pb.S, lo + run);
    int sum = 0;
    for (int s = lo; s < hi; ++s) sum += per_pair * nt[s];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int acc = incl - sum;
    for (int s = lo; s < hi; ++s) {
      ts[s] = acc;
      acc += per_pair * nt[s];
    }
    if (lane == 31) ts[pb.S] = incl;
  }
}

struct Seg {
  int s, l, g, pair;       // sequence, layer, KV head, global pair index
  int first_tile, ntile;   // tile index within the pair, tiles in the segment
  int n_pair, k_s, kv0;    // tiles of the pair, prefix keys, kv_off[s]
  int slot;
  int qt, hh;              // prefix self-attention: query tile, head within the group
};


__device__ __forceinline__ int seq_of(const int *ts, int S, int x) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (ts[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Number of CTAs c in [0, G) whose virtual range starts at or below
// virtual position v: floor(c VT / G) <= v.
__device__ __forceinline__ long long starts_le(long long v, int G, long long VT) {
  long long c = ((v + 1) * G + VT - 1) / VT;
  return c < G ? c : G;
}

// Cost-aware split.  Every pair start costs a CTA about kPairCost tiles'
// time (its query load behind the last QK of the previous pair, the first
// tiles of a fresh softmax and the partials' write), so the
// list is split over a virtual axis on which pair p takes kPairCost + n_p
// positions: kPairCost for its start, then one per tile.  Tile x of pair p
// sits at v(x) = x + kPairCost (p + 1); CTA c takes the virtual range
// [c VT / G, (c+1) VT / G) and with it the tiles whose v(x) fall there.
constexpr int kPairCost = 3;

__device__ __forceinline__ long long virt_total(const Problem &pb, long long T) {
  return T + (long long)kPairCost * pb.S * pb.NL * pb.Hkv;
}

// Number of tiles x with v(x) < v, for 0 <= v <= VT: the first real tile of
// the CTA whose virtual range starts at v.
__device__ __forceinline__ int real_of(const Problem &pb, const int *ts, const int *nt,
                                       long long v) {
  const long long per_seq = (long long)pb.NL * pb.Hkv;
  int lo = 0, hi = pb.S - 1;  // the last sequence whose virtual start is <= v
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (ts[mid] + kPairCost * per_seq * mid <= v) lo = mid; else hi = mid - 1;
  }
  const long long y = v - (ts[lo] + kPairCost * per_seq * lo);
  const long long span = nt[lo] + kPairCost;
  const long long pis = y / span, rem = y - pis * span;
  return (int)(ts[lo] + pis * nt[lo] + (rem > kPairCost ? rem - kPairCost : 0));
}

__device__ __forceinline__ Seg locate(const Problem &pb, const int *ts, const int *nt,
                                      const int *ks, const int *k0, int x, int end, int G,
                                      long long VT) {
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
  sg.slot = sg.pair + (int)starts_le(x + (long long)kPairCost * (sg.pair + 1), G, VT) - 1;
  return sg;
}

// Unit u of the prefix self-attention: sequence s, then (layer, KV head),
// then query tile, then the head within the group (fastest, so the heads
// that share a KV head run at the same time and share its tiles in L2).
__device__ __forceinline__ Seg locate_prefix(const Problem &pb, const int *ts, const int *nt,
                                             const int *ks, const int *k0, int u) {
  Seg sg;
  sg.s = seq_of(ts, pb.S, u);
  const int GQ = pb.Hq / pb.Hkv;
  const int per_pair = nt[sg.s] * GQ;
  const int y = u - ts[sg.s];
  const int pis = y / per_pair, rem = y - pis * per_pair;
  sg.l = pis / pb.Hkv;
  sg.g = pis - sg.l * pb.Hkv;
  sg.pair = sg.s * pb.NL * pb.Hkv + pis;
  sg.qt = rem / GQ;
  sg.hh = rem - sg.qt * GQ;
  sg.first_tile = 0;
  sg.ntile = nt[sg.s];
  sg.n_pair = nt[sg.s];
  sg.k_s = ks[sg.s];
  sg.kv0 = k0[sg.s];
  sg.slot = 0;
  return sg;
}

// 16-byte global -> shared copy (L2 only); src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x with the hardware approximation (relative error about 2^-22);
// results below 2^-126 flush to zero, as do probabilities that small.
__device__ __forceinline__ float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Two f32 lanes in one 64-bit register pair (Blackwell's packed FP32 path:
// one fma / add instruction for both lanes, each lane rounded as the scalar
// instruction would round it).
__device__ __forceinline__ uint64_t pack2(float x, float y) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &x, float &y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Tensor-memory stores, each waited for in the same statement: tcgen05.st
// reads its source registers asynchronously until tcgen05.wait::st, and the
// compiler, seeing the registers as read by the store itself, may reuse
// them for the next values before then.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16: A (bf16 pairs packed in
// 32-bit columns, one row per lane) read from tensor memory.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int D, bool kIndexed, bool kPrefix>
__global__ void __launch_bounds__(kIndexed ? THREADS_INDEXED : THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
               const __grid_constant__ CUtensorMap tm_vp,
               const __grid_constant__ CUtensorMap tm_kb,
               const __grid_constant__ CUtensorMap tm_vb, Problem pb) {
  using L = Layout<D>;
  if (gate_closed(pb.gate)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stages = pb.stages;
  const int off_bar = L::OFF_KV + stages * L::STAGE;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + off_bar);
  uint64_t *q_full = bar;                        // 1
  uint64_t *kv_full = bar + 1;                   // MAX_STAGES
  uint64_t *kv_empty = kv_full + MAX_STAGES;     // MAX_STAGES
  uint64_t *s_full = kv_empty + MAX_STAGES;      // 2
  uint64_t *p_ready = s_full + 2;                // 8: [warpgroup][key quarter]
  uint64_t *pv_done = p_ready + 8;               // 2
  // o_full[h]: the segment's last PV of warpgroup h is done (prefix mode:
  // o_full[0], every PV of the unit).  drain[2]: one per issuer.
  uint64_t *o_full = pv_done + 2, *drain = o_full + 2;
  uint64_t *never = drain + 2;  // no one arrives: the stall test waits on it
  uint64_t *ml_ready = never + 1;  // 2: prefix mode, a warpgroup's (m, l) are published
  uint64_t *q_empty = ml_ready + 2;  // decode: the segment's last QK has read Q
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(q_empty + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *ts = reinterpret_cast<int *>(smem + off_bar + 256);
  int *nt = ts + (pb.S + 1), *ks = nt + (pb.S + 1), *k0 = ks + (pb.S + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  // Query rows of a tile: the block's LB rows of every head of the group,
  // or (prefix mode) 128 prefix positions of one head.
  const int GQ = pb.Hq / pb.Hkv, R = kPrefix ? ROWS : pb.LB * GQ;
  const int BR = pb.LB < TILE ? pb.LB : TILE;  // rows of a block-key box

  // Zero the query and K/V buffers once: rows TMA never writes (query rows
  // >= R, key rows past a short tile) then hold finite values.
  for (int i = threadIdx.x * 16; i < off_bar; i += (int)blockDim.x * 16)
    *reinterpret_cast<uint4 *>(smem + i) = make_uint4(0, 0, 0, 0);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  build_seq_tables<!kPrefix>(pb, ts, nt, ks, k0, pb.status);
  if (threadIdx.x == 0) {
    tc::mbar_init(tc::smem_u32(q_full), 1);
    for (int i = 0; i < MAX_STAGES; ++i) {
      tc::mbar_init(tc::smem_u32(kv_full + i), kIndexed ? 64 : 1);  // every producer lane
      tc::mbar_init(tc::smem_u32(kv_empty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(tc::smem_u32(s_full + i), 1);
      for (int k4 = 0; k4 < 4; ++k4)  // the 4 warps of warpgroup i, one per key quarter
        tc::mbar_init(tc::smem_u32(p_ready + 4 * i + k4), 4);
      tc::mbar_init(tc::smem_u32(pv_done + i), 1);
    }
    tc::mbar_init(tc::smem_u32(o_full), 1);
    tc::mbar_init(tc::smem_u32(o_full + 1), 1);
    tc::mbar_init(tc::smem_u32(q_empty), 1);
    tc::mbar_init(tc::smem_u32(drain), 1);
    tc::mbar_init(tc::smem_u32(drain + 1), 1);
    tc::mbar_init(tc::smem_u32(never), 1);
    tc::mbar_init(tc::smem_u32(ml_ready), 4);      // the 4 warps of warpgroup 0
    tc::mbar_init(tc::smem_u32(ml_ready + 1), 4);  // and of warpgroup 1
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
  // Decode: a contiguous range of the tile list (stream-K).  Prefix mode:
  // units blockIdx.x, blockIdx.x + G, ... (whole key ranges).
  const int T = ts[pb.S];
  const long long VT = kPrefix ? T : virt_total(pb, T);
  const int x_begin =
      kPrefix ? (int)blockIdx.x : real_of(pb, ts, nt, (long long)blockIdx.x * VT / G);
  const int x_end = kPrefix ? T : real_of(pb, ts, nt, (long long)(blockIdx.x + 1) * VT / G);
  const uint32_t sQ = tc::smem_u32(smem + L::OFF_Q);
  const uint32_t sKV = tc::smem_u32(smem + L::OFF_KV);
  const float qk_scale = kLog2e * rsqrtf((float)D);

  // Global tile counter (same in every role) and segment counter.
  uint32_t seg_no = 0, tile_no = 0;
  uint32_t o_phase = 0;  // softmax, decode: segments in which this warpgroup had a tile
  // Producer bookkeeping for the final drain.
  uint32_t issued = 0, last_par = 0, q_issued = 0, q_par = 0;

  for (int x = x_begin; x < x_end; ++seg_no) {
    const Seg sg = kPrefix ? locate_prefix(pb, ts, nt, ks, k0, x)
                           : locate(pb, ts, nt, ks, k0, x, x_end, G, VT);
    x += kPrefix ? G : sg.ntile;
    const int np = (sg.k_s + TILE - 1) / TILE;  // prefix tiles of the pair
    const bool run = !*abort_flag;
    if (kIndexed && (warp == 0 || warp == GATHER_WARP) && run) {
      // ------------------------------------------------ producers, indexed prefix
      // Warps 0 and GATHER_WARP each gather half of a prefix tile's rows
      // (gw = 0: rows 0-63, gw = 1: rows 64-127); every lane of both arrives
      // on the stage's full barrier (count 64); lane 0 of warp 0 also loads
      // Q and the block's own key tiles by TMA (its arrival carries the
      // expected bytes).
      const int gw = warp == 0 ? 0 : 1;
      // The query follows the segment's first tile (lane 0 of warp 0 only),
      // once the previous segment's last QK has read Q.
      auto load_q = [&]() {
        if (gw != 0 || lane != 0) return true;
        if (seg_no > 0 &&
            !tc::mbar_wait(tc::smem_u32(q_empty), (seg_no - 1) & 1, pb.cap_ns, abort_flag))
          return false;
        const uint32_t qb = tc::smem_u32(q_full);
        tc::mbar_arrive_expect_tx(qb, (uint32_t)((D / 64) * R * 128));
        const int qrow = (sg.s * pb.NL + sg.l) * pb.LB;
        for (int b = 0; b < D / 64; ++b)
          tc::tma_load_3d(sQ + b * L::QBOX, &tm_q, qb, b * 64, sg.g * GQ, qrow);
        q_issued = 1;
        q_par = seg_no & 1;
        return true;
      };
      // The sequence's full prefix: rows [pf0, pf1) of every layer.
      int pf0 = __ldg(pb.kvi.prefix_off + sg.s), pf1 = __ldg(pb.kvi.prefix_off + sg.s + 1);
      if (pf0 < 0 || pf1 < pf0 || pf1 > pb.kvi.total_prefix_rows) {
        if (lane == 0 && gw == 0) report(pb.status, SPRINT_STATUS_BAD_OFFSETS);
        pf0 = pf1 = 0;
      }
      const int n_full = pf1 - pf0;
      constexpr int CH = D / 8, RPI = 32 / CH;  // 16-byte chunks per row, rows per pass
      const int sub = lane / CH, c16 = lane % CH;
      const int chunk = c16 & 7;
      // This lane's chunk of row 0 of (layer l, KV head g) of the sequence
      // (row 0 is a valid address whenever the sequence has prefix rows).
      const size_t lane_off =
          n_full ? ((size_t)pb.NL * pf0 + (size_t)sg.l * n_full) * ((size_t)pb.Hkv * D) +
                       (size_t)sg.g * D + (size_t)c16 * 8
                 : 0;
      const __nv_bfloat16 *kl = pb.Kf + lane_off, *vl = pb.Vf + lane_off;
      const uint32_t row_bytes = (uint32_t)pb.Hkv * D * 2;
      // Shared-memory offset of this lane's chunk in row 64 gw + j RPI + sub:
      // box (c16 / 8), row, and the 128-byte swizzle (chunk ^ (row % 8)),
      // where row % 8 = (j RPI % 8 + sub) % 8 takes 8 / RPI values.
      uint32_t xo[8 / RPI];
#pragma unroll
      for (int m = 0; m < 8 / RPI; ++m)
        xo[m] = (c16 >> 3) * L::KBOX + (64 * gw + sub) * 128 +
                ((chunk ^ ((m * RPI + sub) & 7)) << 4);
      const int lag = stages >= 3 ? 1 : 0;  // gathered tiles whose arrival is deferred
      int pend_stage = -1;                  // the deferred tile's stage
      auto arrive_pending = [&](bool all) {
        if (pend_stage < 0) return;
        if (all) cp_async_wait<0>(); else cp_async_wait<1>();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc::mbar_arrive(tc::smem_u32(kv_full + pend_stage));
        pend_stage = -1;
      };
      for (int t = 0; t < sg.ntile; ++t) {
        const uint32_t q = tile_no + t;
        const int stage = q % stages;
        const uint32_t ph = (q / stages) & 1;
        if (t == 1 && !__all_sync(0xffffffffu, load_q())) break;
        if (!__all_sync(0xffffffffu, tc::mbar_wait(tc::smem_u32(kv_empty + stage), ph ^ 1,
                                                   pb.cap_ns, abort_flag)))
          break;
        const int i = sg.first_tile + t;
        const uint32_t kdst = sKV + stage * L::STAGE, vdst = kdst + L::K_BYTES;
        if (i < np) {
          // Kept indices of this warp's 64 rows: row 64 gw + lane in ixa,
          // row 64 gw + 32 + lane in ixb; -1 past the tile's keys or for an
          // index outside the sequence's prefix (reported).
          const int nvalid = min(TILE, sg.k_s - i * TILE) - 64 * gw;
          const int32_t *ip = pb.kvi.idx + sg.kv0 + i * TILE + 64 * gw;
          int ixa = lane < nvalid ? __ldg(ip + lane) : -1;
          int ixb = lane + 32 < nvalid ? __ldg(ip + lane + 32) : -1;
          const bool bad = (lane < nvalid && (ixa < 0 || ixa >= n_full)) ||
                           (lane + 32 < nvalid && (ixb < 0 || ixb >= n_full));
          if (ixa >= n_full) ixa = -1;
          if (ixb >= n_full) ixb = -1;
          if (__any_sync(0xffffffffu, bad) && lane == 0)
            report(pb.status, SPRINT_STATUS_BAD_INDEX);
          // Rows [32 p, 32 p + 32) of this warp's half, as one copy group.
          auto issue_rows = [&](int p) {
#pragma unroll
            for (int jj = 0; jj < 32 / RPI; ++jj) {
              const int j = p * (32 / RPI) + jj;
              const int src = __shfl_sync(0xffffffffu, p ? ixb : ixa, (jj * RPI + sub) & 31);
              const uint32_t n = src >= 0 ? 16u : 0u;
              const size_t go = (size_t)(uint32_t)max(src, 0) * row_bytes;
              const uint32_t so = xo[((j * RPI) & 7) / RPI] + j * RPI * 128;
              cp_async16(kdst + so, reinterpret_cast<const char *>(kl) + go, n);
              cp_async16(vdst + so, reinterpret_cast<const char *>(vl) + go, n);
            }
            cp_async_commit();
          };
          // The deferred arrival of the previous gathered tile comes after
          // the first group of this one (only that group may still be in
          // flight), so the QK of that tile waits for a quarter tile's
          // issue, not a whole one.
          issue_rows(0);
          if (lag) arrive_pending(false);
          issue_rows(1);
          pend_stage = stage;
          if (!lag) arrive_pending(true);
          issued &= ~(1u << stage);  // nothing of the TMA in flight on this stage
        } else {
          arrive_pending(true);
          const uint32_t fb = tc::smem_u32(kv_full + stage);
          if (gw == 0 && lane == 0) {
            const int z = (sg.s * pb.NL + sg.l) * pb.LB + (i - np) * TILE;
            tc::mbar_arrive_expect_tx(fb, (uint32_t)(2 * (D / 64) * BR * 128));
            for (int b = 0; b < D / 64; ++b) {
              tc::tma_load_3d(kdst + b * L::KBOX, &tm_kb, fb, b * 64, sg.g, z);
              tc::tma_load_3d(vdst + b * L::KBOX, &tm_vb, fb, b * 64, sg.g, z);
            }
          } else {
            tc::mbar_arrive(fb);  // the other 63 of the barrier's 64 arrivals
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (ph << stage);
        }
        if (t == 0 && sg.ntile == 1 && !__all_sync(0xffffffffu, load_q())) break;
      }
      arrive_pending(true);
    } else if (warp == 0 && lane == 0 && run) {
      // ------------------------------------------------ producer
      // Decode: the segment's first K/V tile goes out before its query, so
      // that it loads while the previous segment's last QK still reads Q.
      auto load_q = [&]() {
        if (!kPrefix && seg_no > 0 &&
            !tc::mbar_wait(tc::smem_u32(q_empty), (seg_no - 1) & 1, pb.cap_ns, abort_flag))
          return false;
        const uint32_t qb = tc::smem_u32(q_full);
        tc::mbar_arrive_expect_tx(qb, (uint32_t)((D / 64) * R * 128));
        if (kPrefix) {  // 128 prefix positions of head g GQ + hh
          const int qrow = pb.NL * sg.kv0 + sg.l * sg.k_s + sg.qt * TILE;
          for (int b = 0; b < D / 64; ++b)
            tc::tma_load_3d(sQ + b * L::QBOX, &tm_q, qb, b * 64, sg.g * GQ + sg.hh, qrow);
        } else {
          const int qrow = (sg.s * pb.NL + sg.l) * pb.LB;
          for (int b = 0; b < D / 64; ++b)
            tc::tma_load_3d(sQ + b * L::QBOX, &tm_q, qb, b * 64, sg.g * GQ, qrow);
        }
        q_issued = 1;
        q_par = seg_no & 1;
        return true;
      };
      if (kPrefix) load_q();  // never waits in prefix mode
      for (int t = 0; t < sg.ntile; ++t) {
        if (!kPrefix && t == 1 && !load_q()) break;
        const uint32_t q = tile_no + t;
        const int stage = q % stages;
        const uint32_t ph = (q / stages) & 1;
        if (!tc::mbar_wait(tc::smem_u32(kv_empty + stage), ph ^ 1, pb.cap_ns, abort_flag)) break;
        const int i = sg.first_tile + t;
        const uint32_t kdst = sKV + stage * L::STAGE, vdst = kdst + L::K_BYTES;
        const uint32_t fb = tc::smem_u32(kv_full + stage);
        if (i < np) {
          const int z = pb.NL * sg.kv0 + sg.l * sg.k_s + i * TILE;
          tc::mbar_arrive_expect_tx(fb, 2 * L::K_BYTES);
          for (int b = 0; b < D / 64; ++b) {
            tc::tma_load_3d(kdst + b * L::KBOX, &tm_kp, fb, b * 64, sg.g, z);
            tc::tma_load_3d(vdst + b * L::KBOX, &tm_vp, fb, b * 64, sg.g, z);
          }
        } else {
          const int z = (sg.s * pb.NL + sg.l) * pb.LB + (i - np) * TILE;
          tc::mbar_arrive_expect_tx(fb, (uint32_t)(2 * (D / 64) * BR * 128));
          for (int b = 0; b < D / 64; ++b) {
            tc::tma_load_3d(kdst + b * L::KBOX, &tm_kb, fb, b * 64, sg.g, z);
            tc::tma_load_3d(vdst + b * L::KBOX, &tm_vb, fb, b * 64, sg.g, z);
          }
        }
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (ph << stage);
        if (!kPrefix && t == 0 && sg.ntile == 1) load_q();
      }
    } else if (warp == 1 && lane == 0 && run) {
      // ------------------------------------------------ QK issuer
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(ROWS, TILE, false, false);
      // Failure-path test: wait on a barrier no one arrives on, so the
      // bounded wait expires and the CTA takes its abort path.
      if (pb.stall_test) tc::mbar_wait(tc::smem_u32(never), 0, pb.cap_ns, abort_flag);
      bool ok = !*abort_flag &&
                tc::mbar_wait(tc::smem_u32(q_full), seg_no & 1, pb.cap_ns, abort_flag);
      // Shared-memory descriptors, built once and advanced by constant
      // offsets (16-byte units; no carry: every address is below 256 KB).
      const uint64_t qd = tc::desc_kmajor_sw128(sQ);
      const uint64_t kd0 = tc::desc_kmajor_sw128(sKV);
      constexpr uint64_t kStageD = L::STAGE >> 4;
      for (int t = 0; ok && t < sg.ntile; ++t) {
        const uint32_t q = tile_no + t;
        const int stage = q % stages, h = q & 1;
        const uint32_t ph = (q / stages) & 1;
        // S[h] also holds P of tile q - 2, which may belong to the previous
        // segment: its PV must be done first.
        if (!tc::mbar_wait(tc::smem_u32(kv_full + stage), ph, pb.cap_ns, abort_flag) ||
            (q >= 2 && !tc::mbar_wait(tc::smem_u32(pv_done + h), ((q >> 1) & 1) ^ 1, pb.cap_ns,
                                      abort_flag))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (kIndexed) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const uint64_t kd = kd0 + (uint64_t)stage * kStageD;
        const uint32_t sd = tmem + h * TILE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          constexpr int kQBoxD = L::QBOX >> 4, kKBoxD = L::KBOX >> 4;
          tc::mma_bf16(sd, qd + (k >> 2) * kQBoxD + (k & 3) * 2, kd + (k >> 2) * kKBoxD + (k & 3) * 2,
                       idesc_qk, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(tc::smem_u32(s_full + h));
      }
      // Decode: Q is free for the next segment's query once these QKs are done.
      if (!kPrefix && ok) tc::mma_commit(tc::smem_u32(q_empty));
    } else if (warp == 10 && lane == 0 && run) {
      // ------------------------------------------------ PV issuer
      // O[h] += P[h] V for every tile (h = q & 1); P is the A operand, read
      // from tensor memory where the softmax left it.  A second issuing
      // thread: one thread issuing both products could not keep up with HBM.
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(ROWS, D, false, true);
      const uint64_t vd0 = tc::desc_mnmajor_sw128(sKV + L::K_BYTES, L::KBOX);
      constexpr uint64_t kStageD = L::STAGE >> 4;
      bool ok = true;
      for (int u = 0; u < sg.ntile; ++u) {
        const uint32_t q = tile_no + u;
        const int stage = q % stages, h = q & 1;
        const uint32_t ph = (q / stages) & 1;
        const uint64_t vd = vd0 + (uint64_t)stage * kStageD;
        const uint32_t pa = tmem + h * TILE;          // P[h]: 64 columns of bf16 pairs
        const uint32_t od = tmem + L::TMEM_O + h * D;
        // P arrives in quarters of 32 keys: a quarter's products run while
        // the softmax still computes the next.
#pragma unroll
        for (int half = 0; half < 4; ++half) {  // quarters of 32 keys
          if (!tc::mbar_wait(tc::smem_u32(p_ready + 4 * h + half), (q >> 1) & 1, pb.cap_ns,
                             abort_flag) ||
              (half == 0 &&
               !tc::mbar_wait(tc::smem_u32(kv_full + stage), ph, pb.cap_ns, abort_flag))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          if (kIndexed && half == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {  // 16 keys: 8 columns of P, 16 rows of V
            const int k = half * 2 + kk;
            // A warpgroup's first tile of the segment (u < 2) starts its O.
            mma_bf16_ts(od, pa + 8 * k, vd + (16 * 128 >> 4) * k, idesc_pv,
                        (u >= 2 || k > 0) ? 1u : 0u);
          }
        }
        if (!ok) break;
        tc::mma_commit(tc::smem_u32(pv_done + h));
        tc::mma_commit(tc::smem_u32(kv_empty + stage));
        // Decode: warpgroup h's accumulator is final after its last tile of
        // the segment (u = ntile - 1 or ntile - 2; one of each parity).
        if (!kPrefix && u >= sg.ntile - 2) tc::mma_commit(tc::smem_u32(o_full + h));
      }
      if (kPrefix && ok) tc::mma_commit(tc::smem_u32(o_full));
    } else if (warp >= 2 && warp < 10 && run) {
      // ------------------------------------------------ softmax, warpgroup h
      const int h = (warp - 2) >> 2;
      const int q4 = warp & 3, r = q4 * 32 + lane;
      const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
      const uint32_t o_addr = tmem + lane_off + L::TMEM_O + h * D;
      const uint32_t s_addr = tmem + lane_off + h * TILE;
      float m_used = -INFINITY, l_sum = 0.f;
      bool ok = true, mine = false;
      for (int t = 0; t < sg.ntile; ++t) {
        const uint32_t q = tile_no + t;
        if ((int)(q & 1) != h) continue;
        mine = true;
        const int i = sg.first_tile + t;
        const int nvalid = i < np ? min(TILE, sg.k_s - i * TILE)
                                  : min(TILE, pb.LB - (i - np) * TILE);
        // S of tile q is complete, and (by the issue order) so is the PV of
        // tile q - 2: O[h] is stable and S[h] may take P.
        if (!__all_sync(0xffffffffu, tc::mbar_wait(tc::smem_u32(s_full + h), (q >> 1) & 1,
                                                   pb.cap_ns, abort_flag))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        float mraw = -INFINITY;
#pragma unroll
        for (int c = 0; c < TILE / 32; ++c) {
          float v[32];
          tc::tmem_ld32(s_addr + c * 32, v);
          if (nvalid < TILE) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c * 32 + j >= nvalid) v[j] = -INFINITY;
          }
          float a0 = v[0], a1 = v[1], a2 = v[2], a3 = v[3];
#pragma unroll
          for (int j = 4; j < 32; j += 8) {
            a0 = max3(a0, v[j], v[j + 1]);
            a1 = max3(a1, v[j + 2], v[j + 3]);
            a2 = max3(a2, v[j + 4], v[j + 5]);
            a3 = max3(a3, v[j + 6], v[j + 7]);
          }
          mraw = max3(mraw, max3(a0, a1, a2), a3);
        }
        const float mx = mraw * qk_scale;
        // Lazy rescale: a row moves its reference max only when the tile max
        // exceeds it by more than 2^8; O rows are then rescaled in TMEM.
        const bool need = mx > m_used + kRescaleLog2;
        const float alpha = need ? exp2f(m_used - mx) : 1.0f;
        if (need) {
          l_sum *= alpha;
          m_used = mx;
        }
        if (t >= 2 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tc::tmem_ld32(o_addr + c * 32, o);
            uint32_t u[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(o[j] * alpha);
            tmem_st32(o_addr + c * 32, u);
          }
        }
        const float nm = -m_used;
        // Exponent arguments s * log2e/sqrt(d) - m two keys per instruction
        // (each lane one fma, as fmaf), and the row sum in two lanes (even
        // and odd keys), added at the end of the tile.
        const uint64_t scale2 = pack2(qk_scale, qk_scale), nm2 = pack2(nm, nm);
        uint64_t lsum2 = pack2(0.f, 0.f);
        // Decode: unrolled by two, not four: at the 168-register cap of three
        // warps per sub-partition the full unroll spilled registers and was
        // slower.  Prefix mode keeps the full unroll, which measured faster
        // there in spite of a small spill.
        // The same pass for a full tile (no key to mask, the common case;
        // the branch is uniform over the CTA) and for a partial one.
        auto exp_pass = [&](auto masked) {
#pragma unroll(kPrefix ? 4 : 2)
          for (int c = 0; c < TILE / 32; ++c) {
            float v[32];
            tc::tmem_ld32(s_addr + c * 32, v);
            uint32_t pk[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              const int j = 2 * u;
              float x0, x1;
              unpack2(fma2(pack2(v[j], v[j + 1]), scale2, nm2), x0, x1);
              float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              if (decltype(masked)::value) {
                if (c * 32 + j >= nvalid) p0 = 0.f;
                if (c * 32 + j + 1 >= nvalid) p1 = 0.f;
              }
              lsum2 = add2(lsum2, pack2(p0, p1));
              __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
              pk[u] = *reinterpret_cast<uint32_t *>(&h2);
            }
            tmem_st16(s_addr + c * 16, pk);
            {  // every 32-key quarter of P is handed over on its own
              tc::fence_before_sync();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(tc::smem_u32(p_ready + 4 * h + c));
            }
          }
        };
        if (nvalid >= TILE)
          exp_pass(std::false_type{});
        else
          exp_pass(std::true_type{});
        float ls0, ls1;
        unpack2(lsum2, ls0, ls1);
        l_sum += ls0 + ls1;
      }
      if (kPrefix && ok &&
          __all_sync(0xffffffffu, tc::mbar_wait(tc::smem_u32(o_full), seg_no & 1, pb.cap_ns,
                                                abort_flag))) {
        // Prefix mode: merge the two warpgroups' accumulators of each row
        // and write the normalised output.  The warpgroups publish (m, l)
        // in the Q buffer (no QK of this unit is left to read it) and each
        // writes half of the row's columns.
        tc::fence_after_sync();
        float2 *ml_sh = reinterpret_cast<float2 *>(smem + L::OFF_Q);
        ml_sh[h * ROWS + r] = mine ? make_float2(m_used, l_sum) : make_float2(-INFINITY, 0.f);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(ml_ready + h));
        if (__all_sync(0xffffffffu, tc::mbar_wait(tc::smem_u32(ml_ready + (h ^ 1)), seg_no & 1,
                                                  pb.cap_ns, abort_flag))) {
          const float2 a = ml_sh[r], b = ml_sh[ROWS + r];
          const float M = fmaxf(a.x, b.x);
          const float w0 = a.x == -INFINITY ? 0.f : exp2f(a.x - M);
          const float w1 = b.x == -INFINITY ? 0.f : exp2f(b.x - M);
          const float den = (w0 > 0.f ? w0 * a.y : 0.f) + (w1 > 0.f ? w1 * b.y : 0.f);
          const float inv = 1.0f / den;
          const int i = sg.qt * TILE + r;
          __nv_bfloat16 *dst =
              pb.Op + (((size_t)pb.NL * sg.kv0 + (size_t)sg.l * sg.k_s + i) * pb.Hq +
                       (size_t)(sg.g * GQ + sg.hh)) * D;
          const uint32_t o0 = tmem + lane_off + L::TMEM_O, o1 = o0 + D;
#pragma unroll 1
          for (int c = h * (D / 64); c < (h + 1) * (D / 64); ++c) {
            float x0[32], x1[32];
            tc::tmem_ld32(o0 + c * 32, x0);
            tc::tmem_ld32(o1 + c * 32, x1);
            if (i < sg.k_s) {
              uint32_t pk[16];
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                // a warpgroup without keys in this unit left its
                // accumulator unwritten: its weight 0 selects nothing of it
                const float e0 = (w0 > 0.f ? x0[2 * u] * w0 : 0.f) +
                                 (w1 > 0.f ? x1[2 * u] * w1 : 0.f);
                const float e1 = (w0 > 0.f ? x0[2 * u + 1] * w0 : 0.f) +
                                 (w1 > 0.f ? x1[2 * u + 1] * w1 : 0.f);
                __nv_bfloat162 h2 = __floats2bfloat162_rn(e0 * inv, e1 * inv);
                pk[u] = *reinterpret_cast<uint32_t *>(&h2);
              }
              uint4 *out = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v)
                out[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
          }
        }
        // The next unit's Q lands here by TMA (async proxy) after the
        // generic accesses above.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc::fence_before_sync();
      } else if (!kPrefix && ok &&
                 (!mine || __all_sync(0xffffffffu,
                                      tc::mbar_wait(tc::smem_u32(o_full + h), o_phase++ & 1,
                                                    pb.cap_ns, abort_flag)))) {
        // o_full[h] completes once per segment in which warpgroup h has a
        // tile, so its phase counts those segments.
        tc::fence_after_sync();
        const size_t part = (size_t)(2 * sg.slot + h) * ROWS + r;
        if (mine) {
          // Partial O in [part][D/4 column quads][ROWS rows]: the warp's 32
          // rows of one quad are 512 contiguous bytes, so every store below
          // is coalesced (one row per thread, as tensor memory hands it out).
          float4 *dst = reinterpret_cast<float4 *>(pb.ws_o) +
                        (size_t)(2 * sg.slot + h) * (D / 4) * ROWS + r;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tc::tmem_ld32(o_addr + c * 32, o);
            if (r < R) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                dst[(size_t)(c * 8 + j) * ROWS] =
                    make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            }
          }
        }
        // A warpgroup with no tile in this segment leaves an empty partial.
        if (r < R) *reinterpret_cast<float2 *>(pb.ws_ml + part * 2) = make_float2(m_used, l_sum);
        tc::fence_before_sync();
      }
    }
    tile_no += sg.ntile;
    // Prefix mode: the next unit's query lands where the (m, l) of this one
    // were exchanged, so every role finishes the unit first.  Decode roles
    // run on into the next segment; their hand-overs are the barriers above
    // (the K/V ring, q_empty, pv_done and o_full).
    if (kPrefix) {
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
    }
  }

  // Drain: no copy or MMA of this CTA may be in flight when it exits.  These
  // waits ignore the abort flag and use the longer drain limit.
  if (kIndexed && (warp == 0 || warp == GATHER_WARP))
    asm volatile("cp.async.wait_all;" ::: "memory");
  if (warp == 0 && lane == 0) {
    volatile int no_abort = 0;
    if (q_issued) tc::mbar_wait(tc::smem_u32(q_full), q_par, pb.drain_ns, &no_abort);
    for (int s = 0; s < stages; ++s)
      if (issued >> s & 1u)
        tc::mbar_wait(tc::smem_u32(kv_full + s), last_par >> s & 1u, pb.drain_ns, &no_abort);
  }
  if ((warp == 1 || warp == 10) && lane == 0) {  // each issuer drains its own MMAs
    const uint32_t db = tc::smem_u32(drain + (warp == 10));
    tc::mma_commit(db);
    volatile int no_abort = 0;
    tc::mbar_wait(db, 0, pb.drain_ns, &no_abort);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (threadIdx.x == 0 && *abort_flag) report(pb.status, SPRINT_STATUS_TIMEOUT);
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// One CTA per (pair, group of 32 query rows): merge both warpgroup partials
// of every segment of the pair in tile order (max of the row maxima, then
// the weighted sums).  Lane i of every warp takes row 32 group + i, and warp
// w the column quads [w PER, (w+1) PER), so each load of a partial reads the
// 512 contiguous bytes that one warp of the chunk kernel stored.  PER = 1
// (D/4 warps) spreads few pairs over many warps; with many pairs, eight
// warps of D/32 quads each keep more loads in flight per thread and read
// the row maxima fewer times.  The bf16 rows go out through shared memory,
// 16 bytes per thread and store.
template <int D, int PER> constexpr int combine_threads() { return 32 * (D / 4) / PER; }

template <int D, int PER>
__global__ void __launch_bounds__(combine_threads<D, PER>())
attn_tc_combine_kernel(Problem pb, int G, __nv_bfloat16 *__restrict__ O, AttnResidual res) {
  if (gate_closed(pb.gate)) return;
  constexpr int C4 = D / 4;       // float4 column quads of a row
  constexpr int PITCH = D + 8;    // bf16 row pitch of the staging tile (16-byte multiple)
  __shared__ int ts[MAX_SEQ + 1], nt[MAX_SEQ + 1], ks[MAX_SEQ + 1], k0[MAX_SEQ + 1];
  __shared__ __align__(16) __nv_bfloat16 tile[32 * PITCH];
  build_seq_tables<true>(pb, ts, nt, ks, k0, nullptr);
  __syncthreads();
  const int GQ = pb.Hq / pb.Hkv, R = pb.LB * GQ;
  const int groups = (R + 31) / 32;
  const int pair = (int)(blockIdx.x / groups), rg = (int)(blockIdx.x % groups);
  if (pair >= pb.S * pb.NL * pb.Hkv) return;  // whole CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = rg * 32 + lane;
  const bool live = r < R;
  const int per_seq = pb.NL * pb.Hkv;
  const int s = pair / per_seq, pis = pair % per_seq;
  const int l = pis / pb.Hkv, g = pis % pb.Hkv;
  const long long VT = virt_total(pb, ts[pb.S]);
  const int p0 = ts[s] + pis * nt[s], p1 = p0 + nt[s];
  // The CTAs whose tile ranges meet [p0, p1) are c_first..c_last (found from
  // the tiles' virtual positions), and CTA c wrote this pair's partials into
  // slot pair + c.  A CTA between them whose virtual range is empty (VT < G)
  // holds no segment and is skipped; one with a non-empty range there holds
  // tiles of this pair, since the virtual positions between v(p0) and
  // v(p1 - 1) are all tiles of it.
  const long long vp = (long long)kPairCost * (pair + 1);
  const int c_first = (int)starts_le(p0 + vp, G, VT) - 1;
  const int c_last = (int)starts_le(p1 - 1 + vp, G, VT) - 1;
  const bool dense = VT >= G;
  auto holds = [&](int c) {
    return dense || (long long)c * VT / G < (long long)(c + 1) * VT / G;
  };
  const float2 *ml_all = reinterpret_cast<const float2 *>(pb.ws_ml);
  const float4 *o_all = reinterpret_cast<const float4 *>(pb.ws_o);
  float acc[4 * PER];
#pragma unroll
  for (int q = 0; q < 4 * PER; ++q) acc[q] = 0.f;
  float den = 0.f;
  if (live) {
    // Pass 1: the largest row max over all partials (independent loads).
    float mx = -INFINITY;
#pragma unroll 4
    for (int c = c_first; c <= c_last; ++c) {
      if (!holds(c)) continue;
      const size_t part = (size_t)(2 * (pair + c)) * ROWS + r;
      mx = fmaxf(mx, fmaxf(ml_all[part].x, ml_all[part + ROWS].x));
    }
    // Pass 2: weighted sum of the partials in tile order.
#pragma unroll 2
    for (int c = c_first; c <= c_last; ++c) {
      if (!holds(c)) continue;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const size_t pidx = (size_t)(2 * (pair + c) + h);
        const float2 ml = ml_all[pidx * ROWS + r];
        // A warpgroup that saw no key of the segment left m = -inf: weight 0.
        const bool none = ml.x == -INFINITY;
        const float wgt = none ? 0.f : exp2f(ml.x - mx);
        den = fmaf(wgt, none ? 0.f : ml.y, den);
        const float4 *oc = o_all + (pidx * C4 + (size_t)warp * PER) * ROWS + r;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
          const float4 o = oc[(size_t)k * ROWS];
          acc[4 * k + 0] = fmaf(wgt, none ? 0.f : o.x, acc[4 * k + 0]);
          acc[4 * k + 1] = fmaf(wgt, none ? 0.f : o.y, acc[4 * k + 1]);
          acc[4 * k + 2] = fmaf(wgt, none ? 0.f : o.z, acc[4 * k + 2]);
          acc[4 * k + 3] = fmaf(wgt, none ? 0.f : o.w, acc[4 * k + 3]);
        }
      }
    }
    const float inv = 1.0f / den;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      __nv_bfloat162 a = __floats2bfloat162_rn(acc[4 * k] * inv, acc[4 * k + 1] * inv);
      __nv_bfloat162 b = __floats2bfloat162_rn(acc[4 * k + 2] * inv, acc[4 * k + 3] * inv);
      uint2 v;
      v.x = *reinterpret_cast<uint32_t *>(&a);
      v.y = *reinterpret_cast<uint32_t *>(&b);
      *reinterpret_cast<uint2 *>(tile + lane * PITCH + (warp * PER + k) * 4) = v;
    }
  }
  __syncthreads();
  // Rows out: O[s][l][j][g GQ + hh][:] for row r = j GQ + hh, 16 bytes per
  // thread.  Residual epilogue on the last layer: h_out[s][j] = h_in[s][j] +
  // O (heads concatenated), from O as stored (bf16).
  constexpr int V16 = D / 8;  // 16-byte pieces of a row
  const bool last = res.h_out && l == pb.NL - 1;
  const __nv_bfloat16 *h_in = static_cast<const __nv_bfloat16 *>(res.h_in);
  __nv_bfloat16 *h_out = static_cast<__nv_bfloat16 *>(res.h_out);
  // The caller's buffers need only bf16 alignment: 16-byte stores only when
  // every one of them allows it (the same for the whole grid).
  const bool vec = ((reinterpret_cast<uintptr_t>(O) |
                     (last ? reinterpret_cast<uintptr_t>(h_in) | reinterpret_cast<uintptr_t>(h_out)
                           : 0)) & 15) == 0;
  for (int idx = threadIdx.x; idx < 32 * V16; idx += blockDim.x) {
    const int rr = idx / V16, v = idx % V16, row = rg * 32 + rr;
    if (row >= R) continue;
    const int j = row / GQ, hh = row % GQ;
    const uint4 val = *reinterpret_cast<const uint4 *>(tile + rr * PITCH + v * 8);
    const __nv_bfloat16 *oi = reinterpret_cast<const __nv_bfloat16 *>(&val);
    __nv_bfloat16 *dst =
        O + (((size_t)(s * pb.NL + l) * pb.LB + j) * pb.Hq + (size_t)(g * GQ + hh)) * D + v * 8;
    if (vec) {
      *reinterpret_cast<uint4 *>(dst) = val;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) dst[e] = oi[e];
    }
    if (last) {
      const size_t hat = (((size_t)s * pb.LB + j) * pb.Hq + (size_t)(g * GQ + hh)) * D + v * 8;
      uint4 hin, out;
      __nv_bfloat16 *hi = reinterpret_cast<__nv_bfloat16 *>(&hin);
      __nv_bfloat16 *ho = reinterpret_cast<__nv_bfloat16 *>(&out);
      if (vec) {
        hin = *reinterpret_cast<const uint4 *>(h_in + hat);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) hi[e] = h_in[hat + e];
      }
#pragma unroll
      for (int e = 0; e < 8; ++e)
        ho[e] = __float2bfloat16_rn(__bfloat162float(hi[e]) + __bfloat162float(oi[e]));
      if (vec) {
        *reinterpret_cast<uint4 *>(h_out + hat) = out;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) h_out[hat + e] = ho[e];
      }
    }
  }
}

EncodeTiledFn encode3() {
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

// Largest dynamic shared memory a CTA may use, with every variant of the
// kernel opted in to it (once per device).
template <int D> bool smem_optin(int *optin) {
  static PerDevice optin_cache;
  return optin_cache.get(optin, [](int dev, int *v) {
    return cudaDeviceGetAttribute(v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) ==
               cudaSuccess &&
           cudaFuncSetAttribute(attn_tc_kernel<D, false, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, *v - 256) ==
               cudaSuccess &&
           cudaFuncSetAttribute(attn_tc_kernel<D, true, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, *v - 256) ==
               cudaSuccess &&
           cudaFuncSetAttribute(attn_tc_kernel<D, false, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, *v - 256) ==
               cudaSuccess;
  });
}

template <int D>
int launch(const __nv_bfloat16 *Q, const __nv_bfloat16 *Kp, const __nv_bfloat16 *Vp,
           const int32_t *kv_off, int total_kv_rows, const __nv_bfloat16 *Kb,
           const __nv_bfloat16 *Vb, int S, int NL, int LB, int Hq, int Hkv, void *O, void *ws,
           int32_t *status, KvIndex kvi, AttnResidual res, Gate gate, cudaStream_t stream,
           SideStream side) {
  using Lt = Layout<D>;
  const int GQ = Hq / Hkv;
  CUtensorMap tq, tkp, tvp, tkb, tvb;
  const uint64_t brows = (uint64_t)S * NL * LB;
  const int BR = LB < TILE ? LB : TILE;
  if (!make_tmap_3d(&tq, Q, D, Hq, brows, GQ, LB) || !make_tmap_3d(&tkb, Kb, D, Hkv, brows, 1, BR) ||
      !make_tmap_3d(&tvb, Vb, D, Hkv, brows, 1, BR))
    return SPRINT_ERR_CUDA;
  if (total_kv_rows > 0 && !kvi.idx) {
    if (!make_tmap_3d(&tkp, Kp, D, Hkv, (uint64_t)NL * total_kv_rows, 1, TILE) ||
        !make_tmap_3d(&tvp, Vp, D, Hkv, (uint64_t)NL * total_kv_rows, 1, TILE))
      return SPRINT_ERR_CUDA;
  } else {  // no contiguous prefix rows: never dereferenced
    tkp = tkb;
    tvp = tvb;
  }
  // As many ring stages as fit next to Q, the barriers and the tables.
  int optin = 0;
  if (!smem_optin<D>(&optin)) return SPRINT_ERR_CUDA;
  int stages = MAX_STAGES;
  while (stages > 2 && Lt::smem_bytes(stages, S) > (size_t)(optin - 256)) --stages;
  const size_t smem = Lt::smem_bytes(stages, S);
  if (smem > (size_t)(optin - 256)) return SPRINT_ERR_UNSUPPORTED;
  const int G = sm_count();
  const size_t pairs = (size_t)S * NL * Hkv;
  Problem pb;
  pb.kv_off = kv_off;
  pb.total_kv_rows = total_kv_rows;
  pb.S = S; pb.NL = NL; pb.LB = LB; pb.Hq = Hq; pb.Hkv = Hkv;
  pb.ws_o = static_cast<float *>(ws);
  pb.ws_ml = reinterpret_cast<float *>(static_cast<char *>(ws) +
                                       align_up(2 * (pairs + G) * ROWS * D * 4, 256));
  pb.status = status;
  pb.cap_ns = wait_cap_ns();
  pb.drain_ns = pb.cap_ns > 1000000000ull ? pb.cap_ns : 1000000000ull;
  pb.stall_test = stall_test_enabled();
  pb.gate = gate;
  pb.stages = stages;
  pb.kvi = kvi;
  pb.Kf = kvi.idx ? Kp : nullptr;
  pb.Vf = kvi.idx ? Vp : nullptr;
  pb.Op = nullptr;
  pb.prefix = false;
  if (kvi.idx)
    attn_tc_kernel<D, true, false><<<G, THREADS_INDEXED, smem, stream>>>(tq, tkp, tvp, tkb, tvb,
                                                                         pb);
  else
    attn_tc_kernel<D, false, false><<<G, THREADS, smem, stream>>>(tq, tkp, tvp, tkb, tvb, pb);
  if (launch_status() != SPRINT_OK) return SPRINT_ERR_CUDA;
  cudaStream_t cs = stream;
  if (side.side) {  // the combine on the side stream, after the chunk kernel
    if (cudaEventRecord(side.fork, stream) != cudaSuccess ||
        cudaStreamWaitEvent(side.side, side.fork, 0) != cudaSuccess)
      return SPRINT_ERR_CUDA;
    cs = side.side;
  }
  // Few CTAs (a few sequences): one warp per column quad; many: eight warps.
  const long long ctas = (long long)pairs * ((LB * GQ + 31) / 32);
  constexpr int kWide = D / 32;
  if (ctas >= 2 * (long long)G)
    attn_tc_combine_kernel<D, kWide><<<(int)ctas, combine_threads<D, kWide>(), 0, cs>>>(
        pb, G, static_cast<__nv_bfloat16 *>(O), res);
  else
    attn_tc_combine_kernel<D, 1><<<(int)ctas, combine_threads<D, 1>(), 0, cs>>>(
        pb, G, static_cast<__nv_bfloat16 *>(O), res);
  const int rc = launch_status();
  if (rc == SPRINT_OK && side.side && cudaEventRecord(side.join, side.side) != cudaSuccess)
    return SPRINT_ERR_CUDA;
  return rc;
}

// Prefix self-attention: one unit per (sequence, layer, query head, 128-row
// query tile) over all of the sequence's prefix keys; no workspace, no
// combine (each unit merges its two warpgroups' accumulators and writes
// its normalised rows).
template <int D>
int launch_prefix(const __nv_bfloat16 *Qp, const __nv_bfloat16 *K, const __nv_bfloat16 *V,
                  const int32_t *prefix_off, int total_rows, int S, int NL, int Hq, int Hkv,
                  __nv_bfloat16 *Op, int32_t *status, cudaStream_t stream) {
  using Lt = Layout<D>;
  CUtensorMap tq, tk, tv;
  const uint64_t rows = (uint64_t)NL * total_rows;
  if (!make_tmap_3d(&tq, Qp, D, Hq, rows, 1, TILE) || !make_tmap_3d(&tk, K, D, Hkv, rows, 1, TILE) ||
      !make_tmap_3d(&tv, V, D, Hkv, rows, 1, TILE))
    return SPRINT_ERR_CUDA;
  int optin = 0;
  if (!smem_optin<D>(&optin)) return SPRINT_ERR_CUDA;
  int stages = MAX_STAGES;
  while (stages > 2 && Lt::smem_bytes(stages, S) > (size_t)(optin - 256)) --stages;
  const size_t smem = Lt::smem_bytes(stages, S);
  if (smem > (size_t)(optin - 256)) return SPRINT_ERR_UNSUPPORTED;
  Problem pb;
  pb.kv_off = prefix_off;
  pb.total_kv_rows = total_rows;
  pb.S = S; pb.NL = NL; pb.LB = 0; pb.Hq = Hq; pb.Hkv = Hkv;
  pb.ws_o = nullptr;
  pb.ws_ml = nullptr;
  pb.status = status;
  pb.cap_ns = wait_cap_ns();
  pb.drain_ns = pb.cap_ns > 1000000000ull ? pb.cap_ns : 1000000000ull;
  pb.stall_test = stall_test_enabled();
  pb.gate = Gate{nullptr, 0};
  pb.stages = stages;
  pb.kvi = KvIndex{nullptr, nullptr, 0};
  pb.Kf = nullptr;
  pb.Vf = nullptr;
  pb.Op = Op;
  pb.prefix = true;
  attn_tc_kernel<D, false, true><<<sm_count(), THREADS, smem, stream>>>(tq, tk, tv, tk, tv, pb);
  return launch_status();
}

}  // namespace

int attn_tc_prefix(const __nv_bfloat16 *Qp, const __nv_bfloat16 *K, const __nv_bfloat16 *V,
                   const int32_t *prefix_off, int total_rows, int S, int NL, int Hq, int Hkv,
                   int d, __nv_bfloat16 *Op, int32_t *status, cudaStream_t stream) {
  if (S > MAX_SEQ) return SPRINT_ERR_UNSUPPORTED;
  return d == 64 ? launch_prefix<64>(Qp, K, V, prefix_off, total_rows, S, NL, Hq, Hkv, Op, status,
                                     stream)
                 : launch_prefix<128>(Qp, K, V, prefix_off, total_rows, S, NL, Hq, Hkv, Op,
                                      status, stream);
}

size_t attn_tc_workspace_bytes(int S, int NL, int Hkv, int d) {
  const size_t parts = 2 * ((size_t)S * NL * Hkv + (size_t)sm_count());
  return align_up(parts * ROWS * d * 4, 256) + align_up(parts * ROWS * 2 * 4, 256);
}

int attn_tc_forward(const __nv_bfloat16 *Q, const __nv_bfloat16 *Kp, const __nv_bfloat16 *Vp,
                    const int32_t *kv_off, int total_kv_rows, const __nv_bfloat16 *Kb,
                    const __nv_bfloat16 *Vb, int S, int NL, int LB, int Hq, int Hkv, int d,
                    void *O, void *ws, int32_t *status, KvIndex kvi, AttnResidual res,
                    Gate gate, cudaStream_t stream, SideStream side) {
  if (S > MAX_SEQ) return SPRINT_ERR_UNSUPPORTED;
  return d == 64 ? launch<64>(Q, Kp, Vp, kv_off, total_kv_rows, Kb, Vb, S, NL, LB, Hq, Hkv, O,
                              ws, status, kvi, res, gate, stream, side)
                 : launch<128>(Q, Kp, Vp, kv_off, total_kv_rows, Kb, Vb, S, NL, LB, Hq, Hkv, O,
                               ws, status, kvi, res, gate, stream, side);
}

}  // namespace sprint
