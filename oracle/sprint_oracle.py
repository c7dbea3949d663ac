"""Plain CPU oracle of the SPRINT block-decode step (fp64, numpy).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import or run this module.
The CUDA library never calls it and shares no code with it.

Every function restates one step of SPRINT ("Sparse Prefix Retention with
Inference-time Non-uniform Token Unmasking") as the LLaDA2.0-Uni paper
describes it (arXiv 2604.20796, Inference section: "Sparse Prefix Retention"
and "Non-uniform Token Unmasking" paragraphs).  Arithmetic is fp64 on values
expanded exactly from the inputs' storage type.  Each function is the plain
definition: no blocking, fusion or reordering.  Rows of independent outputs
may be processed a slice at a time to bound memory.

Readings taken where the paper is silent or its equation was lost in
extraction:
  R1  composite score s_i = alpha * I_i + (1 - alpha) * c_i, alpha = 0.5
      (the paper's equation for s_i is missing; parity unpinned against it);
  R2  ||k_i|| is the L2 norm of position i's keys concatenated over KV heads,
      taken per layer and averaged over layers; one kept set serves all layers;
  R3  the mean in the denominator of I_i runs over all L prefix positions of
      the sequence, both modalities; if that mean is 0 every I_i is 0;
  R4  top-floor(r n) within a modality ranks by (s descending, index
      ascending); floor(r n) is exact for the decimal ratio r;
  R5  kept positions are stored in ascending position order;
  R6  fixed schedule: ceil(LB / T) per step, LB = masked count at block start;
      adaptive: m = currently masked count, t = 0-based step, minimum
      ceil(m / (T - t)); "exceeds tau" is strict (c > tau); accepted
      positions take their argmax token and are never re-masked;
  R7  confidence is top-1 softmax probability of the temperature-scaled
      logits z = (h . W_v) / theta; argmax ties go to the lowest index;
  R8  the block's first step attends to the full prefix, later steps to the
      pruned prefix; attention is bidirectional over [prefix ; block] with
      softmax scale 1/sqrt(d) and GQA head group floor(h Hkv / Hq);
  R13 keep pools (selection variants beyond the paper's two modality pools):
      positions are grouped into pools, each with its own keep count, and
      each pool keeps its top positions as in R4.  'modality' is the paper's
      keep (text pool, image pool); 'per_image' gives every image its own
      pool at r_img (which positions form an image is an input;
      image_pool_ids numbers maximal image runs); 'global' is one pool
      over the whole prefix at one ratio r (the paper's "global keep ratio
      r = 0.5" sentence read as a budget for the whole prefix);
  R14 residual chain (optional): the block LM head reads h = H + O, the
      step's own hidden state plus the last layer's attention output with
      its heads concatenated (Hq d = D), so the attention output reaches
      the confidences; off by default (h is then an independent input);
  R15 the full forward pass of a block's first step recomputes the prefix:
      every prefix position attends to every prefix position of its
      sequence (no causal mask, the prefix being one clean context), with
      scale 1/sqrt(d) and GQA group floor(h Hkv / Hq); the prefix does not
      attend to the block being decoded.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

TEXT = 0
IMAGE = 1
UNMASK_ADAPTIVE = 0
UNMASK_FIXED = 1


def _np(x):
    """numpy view of a numpy array, list or torch tensor (copied to host)."""
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if str(x.dtype) in ("torch.bfloat16", "torch.float16"):
            x = x.float()
        x = x.numpy()
    return np.asarray(x)


def _f64(x):
    """Exact fp64 copy of a numpy array or a torch tensor (bf16 ok)."""
    return np.asarray(_np(x), dtype=np.float64)


# --------------------------------------------------------------------------
# Sparse Prefix Retention: key-norm importance (paper: definition of I-bar_i)
# --------------------------------------------------------------------------
def key_norm_importance(K):
    """Mean-normalised key-norm importance I_i of every prefix position.

    Paper, Sparse Prefix Retention paragraph: I_i = ||k_i||_2 divided by
    (1/L) sum_j ||k_j||_2, L = number of prefix positions.  Readings R2, R3.

    K: [NL, L, Hkv, d] keys of one sequence's prefix.  Returns I [L] (fp64).
    """
    K = _f64(K)
    NL, L = K.shape[0], K.shape[1]
    if L == 0:
        return np.zeros(0)
    flat = K.reshape(NL, L, -1)
    norm_per_layer = np.sqrt(np.sum(flat * flat, axis=2))     # [NL, L]
    key_norm = norm_per_layer.mean(axis=0)                    # [L]
    mean_norm = key_norm.sum() / L
    if mean_norm == 0.0:
        return np.zeros(L)
    return key_norm / mean_norm


# --------------------------------------------------------------------------
# Top-1 softmax confidence (paper: c_i = max_v p_theta(v | x_t))
# --------------------------------------------------------------------------
def lm_confidence(h, W, theta=None, rows=None, chunk=64, want_logits=False):
    """Top-1 softmax confidence and greedy token of LM-head rows.

    Paper, Sparse Prefix Retention paragraph (c_i, the top-1 softmax
    confidence) and Non-uniform Token Unmasking paragraph (c_n = p(x0_hat^n),
    x0_hat the predicted token).  Reading R7: logits z_v = (h . W_v) / theta.

    h: [M, D]; W: [V, D]; theta: [M] or None (= 1); rows: optional subset of
    row indices.  Returns (c [m], argmax [m] int64, z [m, V] or None).
    """
    h = _f64(h)
    W = _f64(W)
    M = h.shape[0]
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    th = np.ones(M) if theta is None else _f64(theta)
    c = np.empty(len(rows))
    am = np.empty(len(rows), dtype=np.int64)
    zs = [] if want_logits else None
    for a in range(0, len(rows), chunk):
        r = rows[a:a + chunk]
        z = (h[r] @ W.T) / th[r][:, None]                      # [m, V] logits
        p = np.exp(z - z.max(axis=1, keepdims=True))
        p = p / p.sum(axis=1, keepdims=True)                   # softmax
        c[a:a + chunk] = p.max(axis=1)
        am[a:a + chunk] = np.argmax(z, axis=1)                 # first max wins
        if want_logits:
            zs.append(z)
    z_all = np.concatenate(zs, axis=0) if want_logits and zs else None
    return c, am, z_all


# --------------------------------------------------------------------------
# Composite score and modality-aware keep (paper: Sparse Prefix Retention)
# --------------------------------------------------------------------------
def composite_score(importance, confidence, alpha=0.5):
    """s_i blending key-norm importance and confidence.  Reading R1."""
    return alpha * _f64(importance) + (1.0 - alpha) * _f64(confidence)


def keep_count(n, r):
    """floor(r * n) for the decimal keep ratio r (reading R4)."""
    return math.floor(Fraction(repr(float(r))) * int(n))


def select_kept(score, modality, r_text, r_img):
    """Kept prefix positions, ascending (readings R4, R5).

    Paper, Sparse Prefix Retention paragraph: separate keep ratios for text
    and image; within each modality the top floor(r n) positions by s_i are
    retained and the rest evicted.
    """
    s = _f64(score)
    mod = _np(modality).astype(np.int64)
    kept = []
    for tag, r in ((TEXT, r_text), (IMAGE, r_img)):
        pos = [int(i) for i in np.nonzero(mod == tag)[0]]
        k = keep_count(len(pos), r)
        ranked = sorted(pos, key=lambda i: (-s[i], i))
        kept += ranked[:k]
    return np.array(sorted(kept), dtype=np.int64)


def select_kept_pools(score, pool, keep):
    """Kept prefix positions, ascending, when every position belongs to a
    keep pool (reading R13): pool p retains its keep[p] highest-scoring
    members, ties by ascending index (R4).

    Paper, Sparse Prefix Retention paragraph: within each group the top
    positions by s_i are retained and the rest evicted.
    """
    s = _f64(score)
    pid = _np(pool).astype(np.int64)
    kept = []
    for p, k in enumerate(keep):
        members = [int(i) for i in np.nonzero(pid == p)[0]]
        if not 0 <= int(k) <= len(members):
            raise ValueError(f"pool {p}: keep {k} of {len(members)}")
        ranked = sorted(members, key=lambda i: (-s[i], i))
        kept += ranked[:int(k)]
    return np.array(sorted(kept), dtype=np.int64)


def image_pool_ids(modality):
    """Pool id of every position for the 'per_image' policy (reading R13):
    0 for text, 1 + j for the j-th maximal run of image positions."""
    mod = _np(modality).astype(np.int64) != 0
    ids = np.zeros(len(mod), dtype=np.int64)
    run = 0
    for i in range(len(mod)):
        if mod[i]:
            if i == 0 or not mod[i - 1]:
                run += 1
            ids[i] = run
    return ids


def pool_keep_counts(pool_sizes, policy, r_text=1.0, r_img=0.8, r=0.5):
    """Keep count of every pool (reading R13), pool_sizes[p] = members of
    pool p: 'modality' and 'per_image' keep floor(r_text n) of pool 0 (text)
    and floor(r_img n) of every other pool; 'global' has the single pool 0
    and keeps floor(r n) of it."""
    if policy == "global":
        if len(pool_sizes) != 1:
            raise ValueError("the global policy has one pool")
        return [keep_count(pool_sizes[0], r)]
    if policy not in ("modality", "per_image"):
        raise ValueError(policy)
    return [keep_count(n, r_text if p == 0 else r_img) for p, n in enumerate(pool_sizes)]


def compact(K, kept):
    """Pruned cache: the kept rows of every layer, in kept order.

    K: [NL, L, Hkv, d]; kept: ascending indices.  Returns [NL, k, Hkv, d]
    (fp64, exact copies of the stored values).
    """
    return _f64(K)[:, _np(kept).astype(np.int64)]


# --------------------------------------------------------------------------
# Bidirectional in-block attention over [prefix ; block]  (reading R8)
# --------------------------------------------------------------------------
def block_attention(Q, Kp, Vp, Kb, Vb, layers=None):
    """Attention of the block's queries over the (pruned) prefix plus the
    block's own keys, every layer, every query head, no causal mask.

    Paper, Sparse Prefix Retention paragraph: every step after the first
    attends to the pruned prefix; the block itself attends bidirectionally
    (block diffusion setting, BDLM paragraph of the training section).

    Q: [NL, LB, Hq, d]; Kp, Vp: [NL, k, Hkv, d]; Kb, Vb: [NL, LB, Hkv, d].
    Returns O [NL, LB, Hq, d] (fp64).
    """
    Q, Kp, Vp, Kb, Vb = (_f64(x) for x in (Q, Kp, Vp, Kb, Vb))
    NL, LB, Hq, d = Q.shape
    Hkv = Kb.shape[2]
    O = np.zeros((NL, LB, Hq, d))
    for l in (range(NL) if layers is None else layers):
        for h in range(Hq):
            g = (h * Hkv) // Hq
            keys = np.concatenate([Kp[l, :, g, :], Kb[l, :, g, :]], axis=0)
            vals = np.concatenate([Vp[l, :, g, :], Vb[l, :, g, :]], axis=0)
            scores = (Q[l, :, h, :] @ keys.T) / math.sqrt(d)    # [LB, k+LB]
            p = np.exp(scores - scores.max(axis=1, keepdims=True))
            p = p / p.sum(axis=1, keepdims=True)
            O[l, :, h, :] = p @ vals
    return O


def prefix_attention(Q, K, V, rows=None):
    """Self-attention of the prefix over itself in the full forward pass of
    a block's first step (reading R15): every prefix position attends to
    every prefix position, no causal mask.

    Paper, Sparse Prefix Retention paragraph: the first step of each block
    performs a full forward pass, which yields the logits and the complete
    KV cache of the prefix.

    Q: [NL, n, Hq, d]; K, V: [NL, n, Hkv, d]; rows: optional subset of the
    query positions.  Returns O [NL, m, Hq, d] (fp64), m = len(rows) or n.
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    NL, n, Hq, d = Q.shape
    Hkv = K.shape[2]
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.zeros((NL, len(rows), Hq, d))
    for l in range(NL):
        for h in range(Hq):
            g = (h * Hkv) // Hq
            scores = (Q[l, rows, h, :] @ K[l, :, g, :].T) / math.sqrt(d)   # [m, n]
            p = np.exp(scores - scores.max(axis=1, keepdims=True))
            p = p / p.sum(axis=1, keepdims=True)
            O[l, :, h, :] = p @ V[l, :, g, :]
    return O


# --------------------------------------------------------------------------
# Non-uniform token unmasking (paper: Non-uniform Token Unmasking)  R6
# --------------------------------------------------------------------------
def _ceil_div(a, b):
    return -(-a // b)


def unmask_step(conf, argmax, mask, tokens, t, T, tau, mode=UNMASK_ADAPTIVE):
    """One unmask decision for one block.

    Adaptive: accept every masked position whose confidence exceeds tau; if
    fewer than ceil(m / (T - t)) qualify, accept that many, the most
    confident first.  Fixed: accept ceil(LB / T) per step, most confident
    first.  The threshold comparison and the ranking are taken on fp32
    confidences (the precision the library computes them in).

    Returns (mask', tokens', accepted [LB] bool).
    """
    conf32 = _f64(conf).astype(np.float32)
    tau32 = np.float32(tau)
    mask = _np(mask).astype(bool).copy()
    tokens = _np(tokens).astype(np.int64).copy()
    argmax = _np(argmax)
    LB = mask.shape[0]
    masked = [j for j in range(LB) if mask[j]]
    m = len(masked)
    by_conf = sorted(masked, key=lambda j: (-float(conf32[j]), j))
    if m == 0:
        chosen = []
    elif mode == UNMASK_FIXED:
        chosen = by_conf[:min(m, _ceil_div(LB, T))]
    else:
        k_min = m if T - t <= 1 else _ceil_div(m, T - t)
        chosen = [j for j in masked if conf32[j] > tau32]
        if len(chosen) < k_min:
            chosen = by_conf[:k_min]
    accepted = np.zeros(LB, dtype=bool)
    for j in chosen:
        accepted[j] = True
        mask[j] = False
        tokens[j] = int(argmax[j])
    return mask, tokens, accepted


# --------------------------------------------------------------------------
# One block, end to end
# --------------------------------------------------------------------------
def residual_hidden(h, O):
    """h + O of the last layer, heads concatenated (reading R14).

    h: [LB, D]; O: [NL, LB, Hq, d] with Hq d = D.  Returns [LB, D] (fp64).
    """
    O = _f64(O)
    NL, LB, Hq, d = O.shape
    return _f64(h) + O[NL - 1].reshape(LB, Hq * d)


def decode_block(prefix, steps, W, *, LB, T, tau, r_text, r_img, alpha=0.5,
                 mode=UNMASK_ADAPTIVE, residual=False):
    """Decode one block of LB masked tokens in at most T steps.

    Paper, SPRINT paragraphs: the block's first step is a full forward pass
    (logits of every prefix position and its complete KV cache); each prefix
    position is scored and the prefix cache pruned per modality once; every
    step attends, predicts and unmasks.

    prefix: dict K, V [NL][n][Hkv][d], H [n][D], theta [n], modality [n].
    steps:  callable t -> dict Q, Kb, Vb, h, theta (the step's inputs).
    residual: the LM head reads h + O of the last layer (reading R14).
    Returns a dict with the kept set, scores and the per-step trajectory.
    """
    c_pre, am_pre, _ = lm_confidence(prefix["H"], W, prefix["theta"])
    importance = key_norm_importance(prefix["K"])
    score = composite_score(importance, c_pre, alpha)
    kept = select_kept(score, prefix["modality"], r_text, r_img)
    Kp = compact(prefix["K"], kept)
    Vp = compact(prefix["V"], kept)

    mask = np.ones(LB, dtype=bool)
    tokens = np.full(LB, -1, dtype=np.int64)
    traj = []
    for t in range(T):
        if not mask.any():
            break
        x = steps(t)
        if t == 0:
            O = block_attention(x["Q"], prefix["K"], prefix["V"], x["Kb"], x["Vb"])
        else:
            O = block_attention(x["Q"], Kp, Vp, x["Kb"], x["Vb"])
        h = residual_hidden(x["h"], O) if residual else x["h"]
        conf, am, _ = lm_confidence(h, W, x["theta"])
        mask, tokens, acc = unmask_step(conf, am, mask, tokens, t, T, tau, mode)
        traj.append({"t": t, "O": O, "conf": conf, "argmax": am,
                     "accepted": acc, "mask": mask.copy(),
                     "tokens": tokens.copy()})
    return {"importance": importance, "prefix_conf": c_pre,
            "prefix_argmax": am_pre, "score": score, "kept": kept,
            "steps": traj, "tokens": tokens}
