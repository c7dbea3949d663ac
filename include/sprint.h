/*
 * sprint.h -- C ABI of the SPRINT block-decode step on NVIDIA B300 (sm_103a).
 *
 * SPRINT ("Sparse Prefix Retention with Inference-time Non-uniform Token
 * Unmasking") is the training-free decode accelerator of LLaDA2.0-Uni
 * (arXiv 2604.20796, Inference section).  A block of LB masked tokens is
 * decoded in at most T steps.  On the block's first step every prefix
 * position is scored, the prefix KV cache is pruned per modality, and every
 * step attends, predicts and unmasks:
 *
 *   sprint_lmhead_confidence  top-1 softmax confidence c and greedy token of
 *                             LM-head rows (prefix rows on step 0, the block's
 *                             rows on every step); optional logits
 *   sprint_score_prune        key-norm importance, composite score, and the
 *                             per-modality top-floor(r n) kept set
 *   sprint_score_prune_pools  the same scores, kept set with one keep count
 *                             per pool (per-image or whole-prefix pools)
 *   sprint_key_norms,         the two halves of the above as separate calls
 *   sprint_select_kept(_pools) (key norms; scores and kept set)
 *   sprint_compact_kv         gather of the kept rows of K and V
 *   sprint_block_attn         bidirectional block attention over
 *                             [pruned prefix ; block]
 *   sprint_block_attn_indexed the same, reading the kept rows of the full
 *                             cache through the kept indices (no compaction)
 *   sprint_unmask             confidence-adaptive (or fixed) unmasking
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.    Every tensor pointer is a DEVICE pointer owned by the caller.
 *            The library allocates nothing and frees nothing.  Scratch
 *            memory is a caller-provided workspace of at least the size the
 *            matching *_workspace_bytes() function returns (16-byte aligned).
 * Streams.   Every call enqueues work on the caller's stream and returns
 *            without synchronising.  Calls on one stream run in order.
 * Layouts.   Dense, row-major, no padding.  Tensors of several sequences are
 *            concatenated; sequence s starts at the row offset given by a
 *            CSR offset array (int32 [S+1], device, off[0] = 0).
 *              K, V        per sequence [NL][n_s][Hkv][d]
 *              Kb, Vb      [S][NL][LB][Hkv][d]
 *              Q, O        [S][NL][LB][Hq][d]
 *              W           [V][D]  (nn.Linear weight layout)
 *              h           [M][D]
 * dtype.     SPRINT_F32: fp32 storage and arithmetic.
 *            SPRINT_BF16: bf16 storage, fp32 accumulation; the LM head and
 *            attention run on the tcgen05 tensor cores.
 * Errors.    Return value: SPRINT_OK, or a negative SPRINT_ERR_* code when
 *            the host-side checks reject the call (nothing is launched) or a
 *            launch fails.  Data-dependent errors found on the device (bad
 *            offsets or indices, a wait that timed out) are OR-ed into the
 *            caller's int32 device word `status` as SPRINT_STATUS_* bits;
 *            the caller zeroes it and reads it when convenient.
 */
#ifndef SPRINT_H
#define SPRINT_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPRINT_VERSION 100 /* 1.0.0 */

/* Return codes. */
#define SPRINT_OK 0
#define SPRINT_ERR_INVALID_ARG (-1) /* null pointer, bad size, misaligned  */
#define SPRINT_ERR_UNSUPPORTED (-2) /* valid but not implemented (e.g. d)   */
#define SPRINT_ERR_CUDA (-3)        /* a CUDA call or launch failed         */
#define SPRINT_ERR_WORKSPACE (-5)   /* workspace smaller than required      */
#define SPRINT_ERR_TOO_LARGE (-6)   /* beyond a fixed-size internal buffer  */

/* Bits of the device status word. */
#define SPRINT_STATUS_BAD_OFFSETS 1u   /* CSR offsets not monotone / too big */
#define SPRINT_STATUS_KEPT_MISMATCH 2u /* kept_off disagrees with floor(r n) */
#define SPRINT_STATUS_TIMEOUT 4u       /* a bounded device wait expired      */
#define SPRINT_STATUS_BAD_INDEX 8u     /* kept index outside its prefix      */
#define SPRINT_STATUS_BAD_TEMPERATURE 16u /* temperature <= 0 or not finite  */
#define SPRINT_STATUS_DEBUG_CHECK 32u  /* an invariant checked only by the
                                          debug build failed (see below)     */

/* Storage types. */
#define SPRINT_F32 0
#define SPRINT_BF16 1

/* Unmask schedules. */
#define SPRINT_UNMASK_ADAPTIVE 0
#define SPRINT_UNMASK_FIXED 1

int sprint_version(void);
const char *sprint_strerror(int code);

/* Kernels this library has launched in this process (a diagnostic counter;
 * every successful launch adds one). */
unsigned long long sprint_kernel_launches(void);

/* 1 when this library is the debug build (compiled with SPRINT_DEBUG_CHECKS,
 * `python -m kv_cache_pruning_step_b300.build --debug`, libsprint_debug.so),
 * else 0.  The debug build also checks invariants that the release build
 * trusts, and reports a failed one as SPRINT_STATUS_DEBUG_CHECK in the
 * call's status word; no check traps or stops a kernel.  Checked: the kept
 * indices of every sequence are strictly ascending (sprint_compact_kv, as
 * sprint_score_prune writes them); the selection wrote exactly the kept
 * count of every sequence (sprint_score_prune); the still-masked count m
 * equals the number of set mask bytes after every unmask, and every
 * unmasked position holds a token (sprint_unmask); every greedy token lies
 * in [0, V) and every confidence in [1/V, 1] within rounding
 * (sprint_lmhead_confidence).  Not a counterpart of anything in the paper. */
int sprint_debug_checks(void);

/*
 * floor(r * n) keep count of one modality.  LLaDA2.0-Uni paper, Sparse
 * Prefix Retention paragraph: within each modality the top floor(r n)
 * positions are retained.  Computed in double as floor(r n + 1e-9), which
 * is the exact floor for decimal ratios with up to 6 digits and n < 2^31.
 * Returns -1 when n < 0 or r is outside [0, 1].  Host function.
 */
int sprint_keep_count(int n, double r);

/*
 * sprint_lmhead_confidence -- LM-head logits reduced to the top-1 softmax
 * confidence and the greedy token, without materialising probabilities.
 *
 * LLaDA2.0-Uni paper, Sparse Prefix Retention paragraph: c_i = max_v
 * p(v | x_t), the top-1 softmax confidence of prefix position i; and
 * Non-uniform Token Unmasking paragraph: c_n = p(x0_hat^n | x_t) of the
 * predicted token x0_hat^n.  Logits are z[i][v] = (h[i] . W[v]) / temp[i].
 *
 *   h          [M][D]  hidden states (dtype)
 *   W          [V][D]  LM-head weight (dtype)
 *   temp       [M] fp32 per-row logit temperature, > 0; NULL means 1
 *   logits_out [M][V]  (dtype) temperature-scaled logits, or NULL
 *   conf_out   [M] fp32  c = 1 / sum_v exp(z_v - max_v z)
 *   argmax_out [M] int32 smallest v attaining max_v z, or NULL when only
 *              the confidence is wanted (the scoring of prefix rows): the
 *              kernels then skip tracking the greedy token
 *   ws         workspace of sprint_lmhead_workspace_bytes(M, D, V, dtype)
 *
 * M >= 0, D >= 1, V >= 1; bf16 needs D % 8 == 0 and 16-byte aligned h, W.
 * Device status: SPRINT_STATUS_BAD_TEMPERATURE, SPRINT_STATUS_TIMEOUT.
 */
size_t sprint_lmhead_workspace_bytes(int M, int D, int V, int dtype);
int sprint_lmhead_confidence(const void *h, const void *W, const float *temp,
                             int M, int D, int V, int dtype, void *logits_out,
                             float *conf_out, int32_t *argmax_out, void *ws,
                             size_t ws_bytes, int32_t *status,
                             cudaStream_t stream);

/*
 * sprint_lmhead_confidence_noalloc -- sprint_lmhead_confidence for callers
 * that cannot allocate device memory (for example a serving host or plugin
 * whose device memory all comes from a pool it may not bypass, or a
 * latency-critical loop that must not call cudaMalloc).  It takes no
 * workspace; the partials live in a fixed file-scope device array of
 * SPRINT_NOALLOC_SCRATCH_BYTES that every GPU which loads this library holds
 * until the process exits.  The LLaDA2.0-Uni paper has no counterpart to
 * this entry point: it is a memory-management variant of the one above.
 *
 * Arguments, layouts and results are those of sprint_lmhead_confidence.
 * Limit: sprint_lmhead_workspace_bytes(M, D, V, dtype) must not exceed
 * SPRINT_NOALLOC_SCRATCH_BYTES (4 MiB: 3 x 4 bytes x M x ceil(V / 224) for
 * bf16 below 4096 rows, e.g. up to 497 rows at a 157,184-entry vocabulary;
 * ceil(V / 256) strips otherwise); larger calls return
 * SPRINT_ERR_TOO_LARGE and launch nothing.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture.  All
 * calls share the array: calls whose kernels overlap on the GPU race and
 * must be serialised by the caller.  Nothing in the array needs clearing.
 */
#define SPRINT_NOALLOC_SCRATCH_BYTES (4u << 20)
int sprint_lmhead_confidence_noalloc(const void *h, const void *W, const float *temp,
                                     int M, int D, int V, int dtype, void *logits_out,
                                     float *conf_out, int32_t *argmax_out,
                                     int32_t *status, cudaStream_t stream);

/*
 * sprint_score_prune -- per-modality kept set of every sequence's prefix.
 *
 * LLaDA2.0-Uni paper, Sparse Prefix Retention paragraph:
 *   key-norm importance  I_i = ||k_i|| / ((1/L) sum_j ||k_j||), where ||k_i||
 *                        is the L2 norm of position i's keys concatenated
 *                        over the KV heads, averaged over the NL layers, and
 *                        the mean runs over all L = n_s prefix positions;
 *   composite score      s_i = alpha I_i + (1 - alpha) c_i  (the paper's
 *                        equation is not reproduced; this blend is the
 *                        convention, alpha = 0.5 in the paper);
 *   modality-aware keep  within each modality mu the top floor(r_mu n_mu)
 *                        positions by (s descending, index ascending).
 *
 *   K            keys, per sequence [NL][n_s][Hkv][d] (dtype)
 *   prefix_off   int32 [S+1] device CSR offsets of the prefixes
 *   total_rows   prefix_off[S] (host copy; sizes the launch)
 *   conf         fp32 [total_rows] top-1 confidence of every prefix row
 *   modality     uint8 [total_rows], 0 = text, any other value = image
 *   kept_off     int32 [S+1] device CSR offsets of the kept sets; sequence
 *                s must have kept_off[s+1]-kept_off[s] = k_text + k_img
 *                with k = sprint_keep_count(n_mu, r_mu)
 *   kept_idx     int32 [kept_off[S]] OUT: kept positions of each sequence,
 *                ascending, as indices local to the sequence's prefix
 *   score_out    fp32 [total_rows] OUT composite scores, or NULL
 *   ws           workspace of sprint_score_prune_workspace_bytes(...)
 *
 * Device status: SPRINT_STATUS_BAD_OFFSETS, SPRINT_STATUS_KEPT_MISMATCH
 * (that sequence's kept_idx range is left unwritten).
 */
size_t sprint_score_prune_workspace_bytes(int S, int total_rows);
int sprint_score_prune(const void *K, int S, const int32_t *prefix_off,
                       int total_rows, int NL, int Hkv, int d, int dtype,
                       const float *conf, const uint8_t *modality, float alpha,
                       double r_text, double r_img, int32_t *kept_idx,
                       const int32_t *kept_off, float *score_out, void *ws,
                       size_t ws_bytes, int32_t *status, cudaStream_t stream);

/*
 * sprint_score_prune_pools -- kept set with a keep count per pool.
 *
 * LLaDA2.0-Uni paper, Sparse Prefix Retention paragraph: scores as for
 * sprint_score_prune; within each group the top positions by s_i are
 * retained.  The paper's groups are the two modalities; here position i of
 * sequence s belongs to pool pool[i] and that pool keeps its keep[s][pool]
 * highest-scoring members (s descending, index ascending).  With pool =
 * modality and keep = sprint_keep_count(n_mu, r_mu) the result equals
 * sprint_score_prune's bit for bit.  Other groupings: text plus one pool
 * per image (each image at r_img), or a single pool for the whole prefix
 * (one budget floor(r n) for both modalities).
 *
 *   K, prefix_off, total_rows, NL, Hkv, d, dtype, conf, alpha, score_out
 *                as for sprint_score_prune
 *   pool         uint8 [total_rows] pool id of every prefix position,
 *                below n_pools
 *   n_pools      pools per sequence, 1..256
 *   keep         int32 [S][n_pools] device: keep count of every pool
 *                (0 <= keep <= pool size)
 *   kept_off     int32 [S+1] device CSR offsets of the kept sets; sequence
 *                s must have kept_off[s+1]-kept_off[s] = sum_p keep[s][p]
 *   total_kept   kept_off[S] (host copy; bounds the offsets)
 *   kept_idx     int32 [total_kept] OUT: kept positions of each sequence,
 *                ascending, local to the sequence's prefix
 *   ws           workspace of sprint_score_prune_pools_workspace_bytes(S,
 *                total_rows, n_pools)
 *
 * Device status: SPRINT_STATUS_BAD_OFFSETS, SPRINT_STATUS_KEPT_MISMATCH (a
 * keep count outside its pool or not summing to the kept offsets),
 * SPRINT_STATUS_BAD_INDEX (a pool id >= n_pools); a sequence with any of
 * these keeps nothing (its kept_idx range is left unwritten).
 */
size_t sprint_score_prune_pools_workspace_bytes(int S, int total_rows, int n_pools);
int sprint_score_prune_pools(const void *K, int S, const int32_t *prefix_off,
                             int total_rows, int NL, int Hkv, int d, int dtype,
                             const float *conf, const uint8_t *pool, int n_pools,
                             const int32_t *keep, float alpha, int32_t *kept_idx,
                             const int32_t *kept_off, int total_kept,
                             float *score_out, void *ws, size_t ws_bytes,
                             int32_t *status, cudaStream_t stream);

/*
 * The two halves of sprint_score_prune / sprint_score_prune_pools as
 * separate calls, so that the key norms (HBM-bound, they read every prefix
 * key once) can run on another stream while the prefix LM head (tensor-
 * bound) computes the confidences the selection needs.  The pair gives the
 * combined call's kept set and scores bit for bit.
 *
 * sprint_key_norms -- u_out[i] = (1/NL) sum_l ||k_i^(l)||, the numerator of
 * the key-norm importance I_i (Sparse Prefix Retention paragraph): the L2
 * norm of position i's keys concatenated over the KV heads, averaged over
 * the layers.
 *   K, S, prefix_off, total_rows, NL, Hkv, d, dtype   as for sprint_score_prune
 *   u_out        fp32 [total_rows] OUT
 * Device status: SPRINT_STATUS_BAD_OFFSETS.
 *
 * sprint_select_kept -- the composite scores and the per-modality kept set
 * of sprint_score_prune, from key norms u (fp32 [total_rows], as written by
 * sprint_key_norms); the other arguments as for sprint_score_prune, ws of
 * sprint_select_kept_workspace_bytes(S, total_rows) bytes.
 *
 * sprint_select_kept_pools -- the same for sprint_score_prune_pools, ws of
 * sprint_select_kept_pools_workspace_bytes(S, total_rows, n_pools) bytes.
 */
int sprint_key_norms(const void *K, int S, const int32_t *prefix_off, int total_rows, int NL,
                     int Hkv, int d, int dtype, float *u_out, int32_t *status,
                     cudaStream_t stream);
size_t sprint_select_kept_workspace_bytes(int S, int total_rows);
int sprint_select_kept(const float *u, int S, const int32_t *prefix_off, int total_rows,
                       const float *conf, const uint8_t *modality, float alpha,
                       double r_text, double r_img, int32_t *kept_idx,
                       const int32_t *kept_off, float *score_out, void *ws,
                       size_t ws_bytes, int32_t *status, cudaStream_t stream);
size_t sprint_select_kept_pools_workspace_bytes(int S, int total_rows, int n_pools);
int sprint_select_kept_pools(const float *u, int S, const int32_t *prefix_off,
                             int total_rows, const float *conf, const uint8_t *pool,
                             int n_pools, const int32_t *keep, float alpha,
                             int32_t *kept_idx, const int32_t *kept_off, int total_kept,
                             float *score_out, void *ws, size_t ws_bytes, int32_t *status,
                             cudaStream_t stream);

/*
 * sprint_compact_kv -- pruned prefix cache: Kp[l][j] = K[l][kept_idx[j]],
 * the same for V, every layer, per sequence.  LLaDA2.0-Uni paper, Sparse
 * Prefix Retention paragraph: a pruned prefix KV cache is constructed once
 * per block; evicted positions are dropped.
 *
 *   K, V         per sequence [NL][n_s][Hkv][d] (dtype), offsets prefix_off
 *   total_rows   prefix_off[S] (host copy; bounds the reads)
 *   kept_idx     int32, per sequence local ascending indices, offsets kept_off
 *   Kp, Vp       OUT per sequence [NL][k_s][Hkv][d] (dtype), offsets kept_off
 *   total_kept   kept_off[S] (host copy; sizes the launch)
 *
 * Rows are copied bit for bit.  Device status: SPRINT_STATUS_BAD_OFFSETS,
 * SPRINT_STATUS_BAD_INDEX (that row is skipped).
 */
int sprint_compact_kv(const void *K, const void *V, int S,
                      const int32_t *prefix_off, int total_rows, int NL,
                      int Hkv, int d,
                      int dtype, const int32_t *kept_idx,
                      const int32_t *kept_off, int total_kept, void *Kp,
                      void *Vp, int32_t *status, cudaStream_t stream);

/*
 * sprint_block_attn -- bidirectional in-block attention of the block's
 * queries over [prefix keys ; block keys], every layer and query head.
 * LLaDA2.0-Uni paper, Sparse Prefix Retention paragraph: the block's first
 * step attends to the full prefix, every later step to the much shorter
 * pruned prefix.  Block diffusion gives no causal mask inside the block.
 *
 *   O[l][j][h] = sum_i softmax_i(Q[l][j][h] . key_i / sqrt(d)) value_i over
 *   key_i in [Kp[l][0..k_s) ; Kb[l][0..LB)] of KV head g = floor(h Hkv / Hq).
 *
 *   Q            [S][NL][LB][Hq][d] (dtype)
 *   Kp, Vp       prefix keys/values, per sequence [NL][k_s][Hkv][d], located
 *                by kv_off (int32 [S+1], device); the full prefix on step 0
 *   max_kv_rows  max_s k_s (host; sizes the launch)
 *   total_kv_rows kv_off[S] (host; bounds the reads)
 *   Kb, Vb       [S][NL][LB][Hkv][d] the block's own keys/values
 *   O            OUT [S][NL][LB][Hq][d] (dtype); element alignment suffices
 *                (16-byte aligned O is written with 16-byte stores)
 *   ws           workspace of sprint_block_attn_workspace_bytes(...)
 *
 * d in {64, 128}; Hq % Hkv == 0; LB * Hq / Hkv <= 128 for bf16.
 * Device status: SPRINT_STATUS_BAD_OFFSETS, SPRINT_STATUS_TIMEOUT.
 */
size_t sprint_block_attn_workspace_bytes(int S, int NL, int LB, int Hq, int Hkv,
                                         int d, int max_kv_rows, int dtype);
int sprint_block_attn(const void *Q, const void *Kp, const void *Vp,
                      const int32_t *kv_off, int max_kv_rows,
                      int total_kv_rows, const void *Kb,
                      const void *Vb, int S, int NL, int LB, int Hq, int Hkv,
                      int d, int dtype, void *O, void *ws, size_t ws_bytes,
                      int32_t *status, cudaStream_t stream);

/*
 * sprint_block_attn_indexed -- sprint_block_attn over the pruned prefix
 * without the compacted copy: the kept rows are read from the full cache
 * through the kept indices.  LLaDA2.0-Uni paper, Sparse Prefix Retention
 * paragraph: later steps attend only to the retained prefix positions; this
 * call computes exactly what sprint_compact_kv followed by sprint_block_attn
 * computes (bit for bit on the same device), without writing Kp / Vp.
 *
 *   key i of sequence s (i < k_s = kept_off[s+1] - kept_off[s]) is prefix
 *   row kept_idx[kept_off[s] + i] of that sequence, i.e. K[l] row
 *   NL * prefix_off[s] + l * n_s + kept_idx[...] with n_s =
 *   prefix_off[s+1] - prefix_off[s].
 *
 *   Q, Kb, Vb, O  as for sprint_block_attn
 *   K, V          the full prefix cache, per sequence [NL][n_s][Hkv][d]
 *   prefix_off    int32 [S+1] (device); total_rows = prefix_off[S] (host)
 *   kept_idx      int32 [total_kept] (device), local to each sequence, as
 *                 sprint_score_prune writes them (any order is accepted;
 *                 the keys are summed in the order given); may be NULL
 *                 when total_kept = 0
 *   kept_off      int32 [S+1] (device); max_kept, total_kept (host)
 *   ws            workspace of sprint_block_attn_workspace_bytes(S, NL, LB,
 *                 Hq, Hkv, d, max_kept, dtype)
 *
 * Constraints as for sprint_block_attn; total_kept <= total_rows.
 * Device status: SPRINT_STATUS_BAD_OFFSETS, SPRINT_STATUS_BAD_INDEX (an
 * index outside [0, n_s): that key is read as zeros), SPRINT_STATUS_TIMEOUT.
 */
int sprint_block_attn_indexed(const void *Q, const void *K, const void *V,
                              const int32_t *prefix_off, int total_rows,
                              const int32_t *kept_idx, const int32_t *kept_off,
                              int max_kept, int total_kept, const void *Kb,
                              const void *Vb, int S, int NL, int LB, int Hq,
                              int Hkv, int d, int dtype, void *O, void *ws,
                              size_t ws_bytes, int32_t *status,
                              cudaStream_t stream);

/*
 * sprint_prefix_attn -- the prefix's own attention in the full forward pass
 * of a block's first step.  LLaDA2.0-Uni paper, Sparse Prefix Retention
 * paragraph: the first step of each block runs a full forward pass that
 * yields the logits and the complete KV cache of the prefix.  Every prefix
 * position attends to every prefix position of its sequence (no causal
 * mask: the prefix is one clean context), softmax scale 1/sqrt(d), query
 * head h reads KV head floor(h Hkv / Hq):
 *   Op[l][i][h] = sum_j softmax_j(Qp[l][i][h] . K[l][j][g] / sqrt(d)) V[l][j][g]
 * over j < n_s.  An optional part of the step (the bench's --prefix-attn):
 * the pruning itself needs only the cache, not this output.
 *
 *   Qp, Op      per sequence [NL][n_s][Hq][d], sequences concatenated
 *               (dtype; Op written, caller-owned)
 *   K, V        per sequence [NL][n_s][Hkv][d] (dtype)
 *   prefix_off  int32 [S+1] (device); total_rows = prefix_off[S] (host)
 *
 * bf16 only, on the tcgen05 tensor cores: d in {64, 128}, Hq % Hkv == 0,
 * S <= 1024, all pointers 16-byte aligned, NL * total_rows < 2^31
 * (SPRINT_ERR_UNSUPPORTED otherwise, e.g. for fp32).  No workspace.
 * Device status: SPRINT_STATUS_BAD_OFFSETS, SPRINT_STATUS_TIMEOUT.
 */
int sprint_prefix_attn(const void *Qp, const void *K, const void *V,
                       const int32_t *prefix_off, int total_rows, int S, int NL,
                       int Hq, int Hkv, int d, int dtype, void *Op, int32_t *status,
                       cudaStream_t stream);

/*
 * sprint_residual_hidden -- h_out = h_in + O of the last layer, the heads
 * concatenated: h_out[s*LB + j][h*d + c] = h_in[...] + O[s][NL-1][j][h][c]
 * (added in fp32 and stored in dtype).  An optional link of the decode
 * step, not part of the LLaDA2.0-Uni paper's method (whose backbone is not
 * reproduced here): it makes the block LM head read the step's attention
 * output.
 *
 *   h_in, h_out  [S*LB][Hq*d] (dtype); h_out may alias h_in
 *   O            [S][NL][LB][Hq][d] (dtype), as sprint_block_attn writes it
 */
int sprint_residual_hidden(const void *h_in, const void *O, int S, int NL,
                           int LB, int Hq, int d, int dtype, void *h_out,
                           cudaStream_t stream);

/*
 * sprint_unmask -- one unmask decision per sequence.  LLaDA2.0-Uni paper,
 * Non-uniform Token Unmasking paragraph:
 *   ADAPTIVE  accept every masked position whose confidence exceeds tau
 *             (strictly); if fewer than ceil(m / (T - t)) qualify, accept
 *             the ceil(m / (T - t)) most confident instead (m = positions
 *             still masked, t = 0-based step; t >= T - 1 accepts all);
 *   FIXED     accept the min(m, ceil(LB / T)) most confident (a block
 *             starts fully masked, so LB is its initial masked count).
 * Ranking is by (confidence descending, position ascending), in fp32.
 * Accepted positions take their argmax token and are never re-masked.
 *
 *   conf, argmax   [S][LB] fp32 / int32 (from sprint_lmhead_confidence)
 *   mask           [S][LB] uint8 IN/OUT, nonzero = still masked
 *   tokens         [S][LB] int32 IN/OUT
 *   m_out          [S] int32 OUT positions still masked after this step
 *   accepted_out   [S][LB] uint8 OUT 1 where accepted this step, or NULL
 *
 * 1 <= LB <= 1024, T >= 1, 0 <= t.
 */
int sprint_unmask(const float *conf, const int32_t *argmax, uint8_t *mask,
                  int32_t *tokens, int32_t *m_out, int S, int LB, int t, int T,
                  float tau, int mode, uint8_t *accepted_out, int32_t *status,
                  cudaStream_t stream);

/*
 * sprint_decode_steps -- every denoising step of one block, enqueued in one
 * call (the library's native block driver).  LLaDA2.0-Uni paper, Sparse
 * Prefix Retention and Non-uniform Token Unmasking paragraphs: step 0
 * attends to the full prefix, steps t >= 1 to the pruned prefix; every step
 * predicts the block's tokens and unmasks a confidence-adaptive number of
 * them, at least ceil(m / (T - t)), so the block ends within T steps.
 *
 * For step t = 0 .. T-1 the call enqueues sprint_block_attn, then
 * sprint_lmhead_confidence on the block rows, then sprint_unmask, on
 * `stream`, without any device-to-host synchronisation.  With fewer than
 * 4096 block rows (S * LB < 4096) the LM head's strip partials are folded
 * and the block unmasked by one kernel (the same arithmetic as the two
 * separate calls, bit for bit).  Whether a step runs is decided on the
 * device: the kernels of step t >= 1 read the still-masked counts
 * m_hist[t-1][0..S) written by step t-1 and return at once when all are
 * zero (the block finished earlier).  Step 0's unmask treats every
 * position as masked whatever mask holds, and leaves mask and tokens fully
 * written (1 / -1 where not accepted).  The prefix pass
 * (prefix confidences, sprint_score_prune, sprint_compact_kv) is not part
 * of this call.  With kept_idx set, steps t >= 1 attend as
 * sprint_block_attn_indexed does (kept rows of Kf / Vf read through
 * kept_idx; Kp / Vp are ignored and may be NULL).
 *
 * Steps executed = 1 + the number of t in [1, T) with some m_hist[t-1][s]
 * > 0; the caller reads m_hist after synchronising.
 *
 * bf16 without the residual chain: each step's attention combine (which
 * only writes O) runs on an internal stream of the library, one per
 * device, forked from `stream` by an event after the step's attention and
 * joined back before the next step's attention and before the call
 * returns, so all work of the call is ordered before later work on
 * `stream` (and the call can be captured into a CUDA graph from `stream`).
 * Calls from several host threads on one device are serialised while they
 * enqueue.
 *
 * Every step's inputs (Q, Kb, Vb, h, theta) are given up front: this
 * driver suits step inputs that are already resident (for example produced
 * by device work enqueued earlier on the same stream).
 *
 * Fields (all device pointers unless noted; layouts as for the five calls):
 *   S, NL, LB, Hq, Hkv, d, D, vocab, dtype   shapes and storage type
 *   T, tau, mode                             step budget and unmask rule
 *   Kf, Vf, prefix_off, max_rows, total_rows the full prefix (step 0)
 *   Kp, Vp, kept_off, max_kept, total_kept   the pruned prefix (t >= 1)
 *   W                                        LM-head weight [vocab][D]
 *   Q, Kb, Vb, h, theta                      HOST arrays of T device pointers
 *                                            (theta entries may be NULL)
 *   O                                        [S][NL][LB][Hq][d] attention out
 *   logits                                   [S*LB][vocab] or NULL
 *   conf, argmax                             [S*LB] last executed step's c
 *   mask, tokens                             [S][LB] state, set at step 0
 *   m_hist                                   int32 [T][S] masked after step t
 *   accepted                                 uint8 [T][S][LB] or NULL
 *   ws_attn / ws_lm (+ bytes)                workspaces of the two calls
 *   status                                   device status word
 *   events                                   NULL or a HOST array of 6*T
 *                                            cudaEvent_t: per step, start and
 *                                            end of attention, LM head, unmask
 *                                            (NULL entries are not recorded;
 *                                            an event between two kernels
 *                                            keeps them from overlapping)
 *   kept_idx                                 NULL, or int32 [total_kept]: the
 *                                            indexed pruned prefix (t >= 1)
 *   step0_given                              != 0: conf and argmax already
 *                                            hold step 0's block confidences
 *                                            (computed by the caller, e.g.
 *                                            with the prefix rows in one LM-
 *                                            head call); step 0 skips its LM
 *                                            head (not with residual)
 *   residual, h_res                          residual != 0: every step's LM
 *                                            head reads h_res = h[t] + O of
 *                                            the last layer (heads
 *                                            concatenated; needs Hq d = D),
 *                                            written by the attention;
 *                                            h_res is [S*LB][D] (dtype)
 * Returns the first non-zero code of the enqueued calls (nothing after it
 * is enqueued), SPRINT_ERR_INVALID_ARG for a missing field.
 */
typedef struct sprint_steps_args {
  int S, NL, LB, Hq, Hkv, d, D, vocab, dtype;
  int T;
  float tau;
  int mode;
  const void *Kf, *Vf;
  const int32_t *prefix_off;
  int max_rows, total_rows;
  const void *Kp, *Vp;
  const int32_t *kept_off;
  int max_kept, total_kept;
  const void *W;
  const void *const *Q, *const *Kb, *const *Vb, *const *h;
  const float *const *theta;
  void *O, *logits;
  float *conf;
  int32_t *argmax;
  uint8_t *mask;
  int32_t *tokens, *m_hist;
  uint8_t *accepted;
  void *ws_attn;
  size_t ws_attn_bytes;
  void *ws_lm;
  size_t ws_lm_bytes;
  int32_t *status;
  void *const *events;
  const int32_t *kept_idx;
  int residual;
  void *h_res;
  int step0_given;
} sprint_steps_args;

int sprint_decode_steps(const sprint_steps_args *args, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPRINT_H */
