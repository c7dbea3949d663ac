"""Pins of the CPU oracle against what the paper and mathematics fix.

None of these checks retypes the oracle's formula: each uses a hand-worked
value (tests/golden, each with its citation), a closed form, an invariant,
a special case that reduces to a library routine, or a brute force written
as a different computation on tiny inputs.  The last section plants
mistakes in copies of the oracle's functions and shows a pin catches each.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import sprint_oracle as orc

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- key norm
def check_importance_golden(fn):
    for name in ("keynorm_hand.json", "keynorm_layers_hand.json"):
        g = load(name)
        got = fn(np.array(g["K"]))
        np.testing.assert_allclose(got, g["expected_importance"], rtol=0, atol=1e-15)


def check_importance_invariants(fn):
    rng = np.random.default_rng(1)
    K = rng.normal(size=(3, 37, 2, 8)) * rng.lognormal(0, 0.5, size=(1, 37, 1, 1))
    I = fn(K)
    assert abs(I.mean() - 1.0) < 1e-12                      # mean(I) = 1
    np.testing.assert_allclose(fn(7.5 * K), I, rtol=1e-13)  # scale invariance
    perm = rng.permutation(37)
    np.testing.assert_allclose(fn(K[:, perm]), I[perm], rtol=1e-13)
    # Flipping signs or permuting the feature axis inside a position's key
    # leaves every norm, hence I, unchanged.
    np.testing.assert_allclose(fn(-K), I, rtol=1e-13)
    np.testing.assert_allclose(fn(K[..., ::-1]), I, rtol=1e-13)


def test_importance_golden():
    check_importance_golden(orc.key_norm_importance)


def test_importance_invariants():
    check_importance_invariants(orc.key_norm_importance)


def test_importance_layer_average_closed_form():
    # Each (layer, position) key is e * a unit vector spread over the heads,
    # so its norm is exactly e; I must be mean_l(e) / mean_i(mean_l(e)).
    rng = np.random.default_rng(2)
    NL, L, Hkv, d = 4, 9, 3, 5
    e = rng.uniform(0.5, 3.0, size=(NL, L))
    unit = rng.normal(size=(NL, L, Hkv, d))
    unit /= np.sqrt((unit ** 2).sum(axis=(2, 3), keepdims=True))
    K = unit * e[:, :, None, None]
    u = e.mean(axis=0)
    np.testing.assert_allclose(orc.key_norm_importance(K), u * L / u.sum(), rtol=1e-12)


def test_importance_degenerate():
    assert orc.key_norm_importance(np.zeros((2, 0, 1, 4))).shape == (0,)
    np.testing.assert_array_equal(orc.key_norm_importance(np.zeros((2, 5, 1, 4))), 0.0)
    # one position: I = 1 whatever its norm
    np.testing.assert_allclose(orc.key_norm_importance(np.full((1, 1, 2, 3), 4.0)), [1.0])


# -------------------------------------------------------------- confidence
def brute_confidence(h, W, theta):
    """Softmax written the textbook way with explicit loops: p_v = e^{z_v} /
    sum_u e^{z_u}, no max-subtraction; argmax by first strict improvement.
    Also returns the loop-computed logits z."""
    out_c, out_a, out_z = [], [], []
    for i in range(len(h)):
        z = []
        for v in range(len(W)):
            acc = 0.0
            for k in range(len(h[i])):
                acc += float(h[i][k]) * float(W[v][k])
            z.append(acc / float(theta[i]))
        den = sum(math.exp(x) for x in z)
        p = [math.exp(x) / den for x in z]
        best = 0
        for v in range(1, len(z)):
            if z[v] > z[best]:
                best = v
        out_c.append(max(p))
        out_a.append(best)
        out_z.append(z)
    return np.array(out_c), np.array(out_a), np.array(out_z)


def check_confidence_golden(fn):
    for case in load("confidence_hand.json")["cases"]:
        c, am, z = fn(np.array(case["h"]), np.array(case["W"]), np.array(case["theta"]),
                      want_logits=True)
        np.testing.assert_allclose(c, case["expected_c"], rtol=1e-14)
        np.testing.assert_array_equal(am, case["expected_argmax"])
        np.testing.assert_allclose(z, case["expected_logits"], rtol=1e-14, atol=1e-15)


def check_confidence_brute(fn):
    rng = np.random.default_rng(3)
    M, D, V = 5, 7, 11          # all different, so a transposed operand fails
    h = rng.normal(size=(M, D))
    W = rng.normal(size=(V, D)) * 0.7
    theta = rng.uniform(0.5, 4.0, size=M)
    c, am, z = fn(h, W, theta, want_logits=True)
    bc, ba, bz = brute_confidence(h, W, theta)
    np.testing.assert_allclose(c, bc, rtol=1e-12)
    np.testing.assert_array_equal(am, ba)
    np.testing.assert_allclose(z, bz, rtol=1e-12, atol=1e-14)


def test_confidence_golden():
    check_confidence_golden(orc.lm_confidence)


def test_confidence_brute_force():
    check_confidence_brute(orc.lm_confidence)


def test_confidence_closed_forms():
    rng = np.random.default_rng(4)
    # all logits equal: c = 1/V exactly, argmax 0
    V, D = 13, 4
    c, am, _ = orc.lm_confidence(np.zeros((3, D)), rng.normal(size=(V, D)))
    np.testing.assert_allclose(c, 1.0 / V, rtol=1e-15)
    np.testing.assert_array_equal(am, 0)
    # V = 2: c = sigmoid(|z1 - z0|)
    h = rng.normal(size=(6, 3))
    W = rng.normal(size=(2, 3))
    theta = rng.uniform(0.5, 4, size=6)
    z = (h @ W.T) / theta[:, None]
    c, am, _ = orc.lm_confidence(h, W, theta)
    np.testing.assert_allclose(c, scipy.special.expit(np.abs(z[:, 1] - z[:, 0])), rtol=1e-13)
    np.testing.assert_array_equal(am, (z[:, 1] > z[:, 0]).astype(int))
    # one dominant logit (+50 over V-1 zeros): c = 1 / (1 + (V-1) e^-50)
    V = 9
    W = np.zeros((V, 1))
    W[5, 0] = 50.0
    c, am, _ = orc.lm_confidence(np.ones((1, 1)), W)
    assert abs(c[0] - 1.0 / (1.0 + (V - 1) * math.exp(-50.0))) < 1e-15
    assert am[0] == 5
    # temperature: theta -> large flattens to 1/V; h, theta scaled together cancel
    h = rng.normal(size=(4, 5))
    W = rng.normal(size=(7, 5))
    c_hot, _, _ = orc.lm_confidence(h, W, np.full(4, 1e9))
    np.testing.assert_allclose(c_hot, 1 / 7, rtol=1e-6)
    c1, a1, _ = orc.lm_confidence(h, W, np.full(4, 1.0))
    c3, a3, _ = orc.lm_confidence(3 * h, W, np.full(4, 3.0))
    np.testing.assert_allclose(c1, c3, rtol=1e-13)
    np.testing.assert_array_equal(a1, a3)
    # confidence equals scipy's softmax maximum
    z = (h @ W.T)
    np.testing.assert_allclose(c1, scipy.special.softmax(z, axis=1).max(axis=1), rtol=1e-13)


def test_confidence_rows_subset_and_logits():
    rng = np.random.default_rng(5)
    h = rng.normal(size=(9, 4))
    W = rng.normal(size=(6, 4))
    th = rng.uniform(0.5, 4, size=9)
    c, am, z = orc.lm_confidence(h, W, th, want_logits=True, chunk=4)
    cs, ams, _ = orc.lm_confidence(h, W, th, rows=[7, 2])
    np.testing.assert_allclose(cs, c[[7, 2]], rtol=1e-14)
    np.testing.assert_array_equal(ams, am[[7, 2]])
    # logits of a row subset are those rows of the full logits, and chunking
    # does not change them
    _, _, zs = orc.lm_confidence(h, W, th, rows=[7, 2], want_logits=True, chunk=1)
    np.testing.assert_allclose(zs, z[[7, 2]], rtol=1e-14, atol=1e-15)


# ------------------------------------------------------------ keep / select
def brute_kept(s, modality, r_text, r_img, counts):
    """Rank definition: i survives iff fewer than k_mu positions of its
    modality beat it (higher s, or equal s at a lower index)."""
    kept = []
    for i in range(len(s)):
        mu = modality[i]
        beaten_by = sum(1 for j in range(len(s)) if modality[j] == mu and
                        (s[j] > s[i] or (s[j] == s[i] and j < i)))
        if beaten_by < counts[mu]:
            kept.append(i)
    return kept


def check_select_golden(score_fn, select_fn):
    g = load("select_hand.json")
    s = score_fn(np.array(g["importance"]), np.array(g["confidence"]), g["alpha"])
    np.testing.assert_allclose(s, g["expected_score"], rtol=0, atol=1e-15)
    kept = select_fn(s, np.array(g["modality"]), g["r_text"], g["r_img"])
    assert list(kept) == g["expected_kept"]
    g = load("select_modality_hand.json")
    for case in g["cases"]:
        kept = select_fn(np.array(g["score"]), np.array(g["modality"]),
                         case["r_text"], case["r_img"])
        assert list(kept) == case["expected_kept"], case


def check_select_brute(select_fn):
    rng = np.random.default_rng(6)
    for trial in range(200):
        n = int(rng.integers(0, 14))
        modality = rng.integers(0, 2, size=n)
        # coarse values so that ties are frequent
        s = rng.integers(0, 5, size=n) / 4.0
        r_text, r_img = rng.choice([0.0, 0.25, 0.5, 0.8, 1.0], size=2)
        counts = {0: math.floor(r_text * (modality == 0).sum() + 1e-9),
                  1: math.floor(r_img * (modality == 1).sum() + 1e-9)}
        kept = select_fn(s, modality, float(r_text), float(r_img))
        assert list(kept) == brute_kept(s, modality, r_text, r_img, counts)


def test_select_golden():
    check_select_golden(orc.composite_score, orc.select_kept)


def test_select_brute_force():
    check_select_brute(orc.select_kept)


def test_keep_count_table():
    # floor(r n) worked by hand, including a product that binary floating
    # point rounds below the integer (0.29 * 100 = 28.999... in doubles)
    table = [(1024, 0.8, 819), (3072, 0.8, 2457), (64, 0.8, 51), (100, 0.29, 29),
             (1024, 1.0, 1024), (1024, 0.0, 0), (3, 0.5, 1), (0, 0.8, 0),
             (16384, 0.8, 13107), (7, 0.999, 6)]
    for n, r, k in table:
        assert orc.keep_count(n, r) == k, (n, r)


def check_select_alpha_extremes(score_fn):
    """alpha = 1 ranks by key-norm importance alone, alpha = 0 by confidence
    alone (the two ends of the blend)."""
    rng = np.random.default_rng(7)
    n = 40
    I = rng.uniform(0.2, 2.0, size=n)
    c = rng.uniform(0.0, 1.0, size=n)
    mod = np.zeros(n, dtype=int)
    k = orc.keep_count(n, 0.25)
    kept1 = orc.select_kept(score_fn(I, c, 1.0), mod, 0.25, 1.0)
    assert list(kept1) == sorted(np.argsort(-I, kind="stable")[:k])
    kept0 = orc.select_kept(score_fn(I, c, 0.0), mod, 0.25, 1.0)
    assert list(kept0) == sorted(np.argsort(-c, kind="stable")[:k])
    assert len(kept1) == k == 10


def test_select_alpha_extremes_and_counts():
    check_select_alpha_extremes(orc.composite_score)
    rng = np.random.default_rng(7)
    n = 40
    I = rng.uniform(0.2, 2.0, size=n)
    c = rng.uniform(0.0, 1.0, size=n)
    # r = 1 keeps everything in order; r = 0 keeps nothing
    s = orc.composite_score(I, c)
    mod = rng.integers(0, 2, size=n)
    assert list(orc.select_kept(s, mod, 1.0, 1.0)) == list(range(n))
    assert len(orc.select_kept(s, mod, 0.0, 0.0)) == 0
    # modalities are independent pools
    s2 = s.copy()
    s2[mod == 1] = rng.uniform(size=(mod == 1).sum())
    k_a = set(orc.select_kept(s, mod, 0.5, 0.5)) & set(np.nonzero(mod == 0)[0])
    k_b = set(orc.select_kept(s2, mod, 0.5, 0.5)) & set(np.nonzero(mod == 0)[0])
    assert k_a == k_b


def brute_kept_pools(s, pool, keep):
    """Rank definition per pool: i survives iff fewer than keep[p] members
    of its pool p beat it (higher s, or equal s at a lower index)."""
    return [i for i in range(len(s))
            if sum(1 for j in range(len(s)) if pool[j] == pool[i] and
                   (s[j] > s[i] or (s[j] == s[i] and j < i))) < keep[pool[i]]]


def check_pools_golden(fn):
    g = load("select_pools_hand.json")
    for case in g["cases"]:
        kept = fn(np.array(g["score"]), np.array(g["pool"]), case["keep"])
        assert list(kept) == case["expected_kept"], case


def check_pools_brute(fn):
    rng = np.random.default_rng(16)
    for trial in range(300):
        n = int(rng.integers(0, 16))
        P = int(rng.integers(1, 5))
        pool = rng.integers(0, P, size=n)
        s = rng.integers(0, 4, size=n) / 3.0  # coarse: frequent ties
        keep = [int(rng.integers(0, (pool == p).sum() + 1)) for p in range(P)]
        assert list(fn(s, pool, keep)) == brute_kept_pools(s, pool, keep), (s, pool, keep)


def test_select_pools_golden_and_brute_force():
    check_pools_golden(orc.select_kept_pools)
    check_pools_brute(orc.select_kept_pools)


def test_select_pools_special_cases():
    rng = np.random.default_rng(17)
    n = 50
    s = rng.uniform(size=n)
    pool = rng.integers(0, 3, size=n)
    sizes = [int((pool == p).sum()) for p in range(3)]
    assert list(orc.select_kept_pools(s, pool, sizes)) == list(range(n))   # keep all
    assert len(orc.select_kept_pools(s, pool, [0, 0, 0])) == 0             # keep none
    # one pool at half: exactly the floor(n/2) largest scores
    kept = orc.select_kept_pools(s, np.zeros(n, int), [n // 2])
    assert sorted(kept) == sorted(np.argsort(-s, kind="stable")[:n // 2])
    # pools are independent: rescoring one pool leaves the others' keeps
    s2 = s.copy()
    s2[pool == 1] = rng.uniform(size=sizes[1])
    keep = [3, 4, 5]
    a = set(orc.select_kept_pools(s, pool, keep)) - set(np.nonzero(pool == 1)[0])
    b = set(orc.select_kept_pools(s2, pool, keep)) - set(np.nonzero(pool == 1)[0])
    assert a == b
    with pytest.raises(ValueError):
        orc.select_kept_pools(s, pool, [sizes[0] + 1, 0, 0])
    # the two modality pools with floor(r n) counts are the paper's keep
    mod = rng.integers(0, 2, size=n)
    counts = orc.pool_keep_counts([int((mod == 0).sum()), int((mod == 1).sum())], "modality",
                                  r_text=0.5, r_img=0.8)
    assert list(orc.select_kept_pools(s, mod, counts)) == list(
        orc.select_kept(s, mod, 0.5, 0.8))


def test_pool_ids_and_counts_golden():
    g = load("select_pools_hand.json")
    runs = g["image_runs"]
    assert list(orc.image_pool_ids(np.array(runs["modality"]))) == runs["expected_pool"]
    assert list(orc.image_pool_ids(np.zeros(5, int))) == [0] * 5
    assert list(orc.image_pool_ids(np.ones(3, int))) == [1, 1, 1]
    c = g["counts"]
    assert orc.pool_keep_counts(c["sizes"], "per_image", c["r_text"], c["r_img"]) == \
        c["expected_per_image"]
    for n, r, k in c["global"]:
        assert orc.pool_keep_counts([n], "global", r=r) == [k]


def test_residual_hidden_closed_forms():
    """h + O of the last layer: O = 0 gives h; h = 0 gives the last layer's
    heads laid side by side; earlier layers do not matter; a hand case."""
    rng = np.random.default_rng(18)
    NL, LB, Hq, d = 3, 4, 2, 3
    h = rng.normal(size=(LB, Hq * d))
    O = rng.normal(size=(NL, LB, Hq, d))
    np.testing.assert_array_equal(orc.residual_hidden(h, np.zeros_like(O)), h)
    z = orc.residual_hidden(np.zeros_like(h), O)
    for j in range(LB):
        np.testing.assert_array_equal(z[j], np.concatenate([O[NL - 1, j, 0], O[NL - 1, j, 1]]))
    O2 = O.copy()
    O2[:NL - 1] = 7.0
    np.testing.assert_array_equal(orc.residual_hidden(h, O2), orc.residual_hidden(h, O))
    hand = orc.residual_hidden(np.array([[1.0, 2.0, 3.0, 4.0]]),
                               np.array([[[[10.0, 20.0], [30.0, 40.0]]]]))
    np.testing.assert_array_equal(hand, [[11.0, 22.0, 33.0, 44.0]])


def test_compact_identity_and_gather():
    rng = np.random.default_rng(8)
    K = rng.normal(size=(2, 10, 3, 4))
    np.testing.assert_array_equal(orc.compact(K, np.arange(10)), K)
    idx = np.array([1, 4, 9])
    got = orc.compact(K, idx)
    for j, i in enumerate(idx):
        np.testing.assert_array_equal(got[:, j], K[:, i])
    assert orc.compact(K, np.zeros(0, dtype=int)).shape == (2, 0, 3, 4)


# --------------------------------------------------------------- attention
def brute_attention(Q, Kp, Vp, Kb, Vb):
    """Loops over layer, query head, block row; GQA by explicit head groups;
    softmax as e^x / sum e^x without max-subtraction."""
    NL, LB, Hq, d = Q.shape
    Hkv = Kb.shape[2]
    group = Hq // Hkv
    O = np.zeros(Q.shape)
    for l in range(NL):
        for h in range(Hq):
            g = h // group
            keys = [Kp[l, i, g] for i in range(Kp.shape[1])] + [Kb[l, j, g] for j in range(LB)]
            vals = [Vp[l, i, g] for i in range(Vp.shape[1])] + [Vb[l, j, g] for j in range(LB)]
            for r in range(LB):
                w = [math.exp(sum(Q[l, r, h, x] * k[x] for x in range(d)) / math.sqrt(d))
                     for k in keys]
                tot = sum(w)
                for x in range(d):
                    O[l, r, h, x] = sum(w[i] * vals[i][x] for i in range(len(w))) / tot
    return O


def check_attention_brute(fn):
    rng = np.random.default_rng(9)
    NL, LB, Hq, Hkv, d, k = 2, 3, 4, 2, 5, 6
    Q = rng.normal(size=(NL, LB, Hq, d))
    Kp, Vp = rng.normal(size=(2, NL, k, Hkv, d))
    Kb, Vb = rng.normal(size=(2, NL, LB, Hkv, d))
    np.testing.assert_allclose(fn(Q, Kp, Vp, Kb, Vb), brute_attention(Q, Kp, Vp, Kb, Vb),
                               rtol=1e-12, atol=1e-13)


def brute_prefix_attention(Q, K, V):
    """Loops over layer, query head, query position and key position; GQA
    by explicit head groups; softmax as e^x / sum e^x."""
    NL, n, Hq, d = Q.shape
    group = Hq // K.shape[2]
    O = np.zeros(Q.shape)
    for l in range(NL):
        for h in range(Hq):
            g = h // group
            for r in range(n):
                w = [math.exp(sum(Q[l, r, h, x] * K[l, j, g, x] for x in range(d)) / math.sqrt(d))
                     for j in range(n)]
                tot = sum(w)
                for x in range(d):
                    O[l, r, h, x] = sum(w[j] * V[l, j, g, x] for j in range(n)) / tot
    return O


def check_prefix_attention(fn):
    rng = np.random.default_rng(19)
    NL, n, Hq, Hkv, d = 2, 7, 4, 2, 5
    Q = rng.normal(size=(NL, n, Hq, d))
    K, V = rng.normal(size=(2, NL, n, Hkv, d)) * rng.lognormal(0, 0.5, size=(1, 1, n, 1, 1))
    np.testing.assert_allclose(fn(Q, K, V), brute_prefix_attention(Q, K, V), rtol=1e-12,
                               atol=1e-13)
    # bidirectional: permuting the prefix positions permutes the outputs (a
    # causal mask would break this)
    perm = rng.permutation(n)
    np.testing.assert_allclose(fn(Q[:, perm], K[:, perm], V[:, perm]), fn(Q, K, V)[:, perm],
                               rtol=1e-12, atol=1e-13)


def test_prefix_attention_brute_force_and_bidirectional():
    check_prefix_attention(orc.prefix_attention)


def test_prefix_attention_special_cases():
    rng = np.random.default_rng(20)
    NL, Hq, Hkv, d = 2, 4, 2, 6
    # one position: o = v
    Q = rng.normal(size=(NL, 1, Hq, d))
    K, V = rng.normal(size=(2, NL, 1, Hkv, d))
    O = orc.prefix_attention(Q, K, V)
    for h in range(Hq):
        np.testing.assert_allclose(O[:, 0, h], V[:, 0, h // 2], rtol=1e-15)
    # identical keys: every query gets the mean of the values
    n = 9
    Q = rng.normal(size=(NL, n, Hq, d))
    K = np.broadcast_to(rng.normal(size=d), (NL, n, Hkv, d)).copy()
    V = rng.normal(size=(NL, n, Hkv, d))
    O = orc.prefix_attention(Q, K, V)
    for h in range(Hq):
        np.testing.assert_allclose(O[:, :, h], np.broadcast_to(V[:, :, h // 2].mean(axis=1)[:, None],
                                                                (NL, n, d)), rtol=1e-12)
    # the prefix's own attention equals the block attention with the keys
    # split anywhere into a "prefix" part and a "block" part (both pinned
    # separately), for any subset of query rows
    n = 11
    Q = rng.normal(size=(NL, n, Hq, d))
    K, V = rng.normal(size=(2, NL, n, Hkv, d))
    rows = [0, 4, 10, 7]
    for split in (0, 3, n - 1, n):
        want = orc.block_attention(Q[:, rows], K[:, :split], V[:, :split], K[:, split:],
                                   V[:, split:])
        np.testing.assert_allclose(orc.prefix_attention(Q, K, V, rows=rows), want, rtol=1e-12,
                                   atol=1e-13)
    # GQA equals multi-head attention with every KV head repeated per group
    rep = lambda a: np.repeat(a, Hq // Hkv, axis=2)  # noqa: E731
    np.testing.assert_allclose(orc.prefix_attention(Q, K, V),
                               orc.prefix_attention(Q, rep(K), rep(V)), rtol=1e-13)


def test_prefix_attention_planted_mistakes():
    def causal(Q, K, V):
        Q, K, V = (np.asarray(a, float) for a in (Q, K, V))
        NL, n, Hq, d = Q.shape
        O = np.zeros(Q.shape)
        for i in range(n):
            O[:, i] = orc.prefix_attention(Q[:, :i + 1], K[:, :i + 1], V[:, :i + 1])[:, i]
        return O

    def no_scale(Q, K, V):
        return orc.prefix_attention(np.asarray(Q) * math.sqrt(np.asarray(Q).shape[-1]), K, V)

    def modulo_group(Q, K, V):
        Q = np.asarray(Q)
        Hq, Hkv = Q.shape[2], np.asarray(K).shape[2]
        order = [(h % Hkv) * (Hq // Hkv) + h // Hkv for h in range(Hq)]
        return orc.prefix_attention(Q[:, :, order], K, V)[:, :, np.argsort(order)]

    def softmax_over_queries(Q, K, V):
        Q, K, V = (np.asarray(a, float) for a in (Q, K, V))
        NL, n, Hq, d = Q.shape
        O = np.zeros(Q.shape)
        for l in range(NL):
            for h in range(Hq):
                g = h * K.shape[2] // Hq
                s = Q[l, :, h] @ K[l, :, g].T / math.sqrt(d)
                p = np.exp(s - s.max(axis=0, keepdims=True))
                p = p / p.sum(axis=0, keepdims=True)
                O[l, :, h] = p @ V[l, :, g]
        return O
    for bad in (causal, no_scale, modulo_group, softmax_over_queries):
        _fails(check_prefix_attention, bad)


def test_attention_brute_force():
    check_attention_brute(orc.block_attention)


def test_attention_special_cases():
    rng = np.random.default_rng(10)
    NL, Hq, Hkv, d = 1, 2, 1, 4
    # a single key (no prefix, block of 1): o = v
    Q = rng.normal(size=(NL, 1, Hq, d))
    Kb, Vb = rng.normal(size=(2, NL, 1, Hkv, d))
    empty = np.zeros((NL, 0, Hkv, d))
    O = orc.block_attention(Q, empty, empty, Kb, Vb)
    np.testing.assert_allclose(O[0, 0, 0], Vb[0, 0, 0], rtol=1e-15)
    np.testing.assert_allclose(O[0, 0, 1], Vb[0, 0, 0], rtol=1e-15)
    # identical keys: o = mean of the values
    LB, k = 3, 5
    Q = rng.normal(size=(NL, LB, Hq, d))
    key = rng.normal(size=d)
    Kp = np.broadcast_to(key, (NL, k, Hkv, d)).copy()
    Kb = np.broadcast_to(key, (NL, LB, Hkv, d)).copy()
    Vp = rng.normal(size=(NL, k, Hkv, d))
    Vb = rng.normal(size=(NL, LB, Hkv, d))
    O = orc.block_attention(Q, Kp, Vp, Kb, Vb)
    mean_v = np.concatenate([Vp[0, :, 0], Vb[0, :, 0]]).mean(axis=0)
    for r in range(LB):
        for h in range(Hq):
            np.testing.assert_allclose(O[0, r, h], mean_v, rtol=1e-12)
    # zero query: uniform weights whatever the keys
    Kp = rng.normal(size=(NL, k, Hkv, d))
    O = orc.block_attention(np.zeros((NL, LB, Hq, d)), Kp, Vp, Kb, Vb)
    np.testing.assert_allclose(O[0, 1, 0], mean_v, rtol=1e-12)
    # bidirectional, no mask: permuting key/value rows changes nothing
    perm = rng.permutation(k)
    np.testing.assert_allclose(orc.block_attention(Q, Kp[:, perm], Vp[:, perm], Kb, Vb),
                               orc.block_attention(Q, Kp, Vp, Kb, Vb), rtol=1e-12)


def test_attention_gqa_equals_replicated_mha():
    rng = np.random.default_rng(11)
    NL, LB, Hq, Hkv, d, k = 2, 4, 6, 2, 8, 7
    Q = rng.normal(size=(NL, LB, Hq, d))
    Kp, Vp = rng.normal(size=(2, NL, k, Hkv, d))
    Kb, Vb = rng.normal(size=(2, NL, LB, Hkv, d))
    rep = lambda x: np.repeat(x, Hq // Hkv, axis=2)   # head h uses group h // 3
    np.testing.assert_allclose(orc.block_attention(Q, Kp, Vp, Kb, Vb),
                               orc.block_attention(Q, rep(Kp), rep(Vp), rep(Kb), rep(Vb)),
                               rtol=1e-13)


# ------------------------------------------------------------------ unmask
def check_unmask_golden(fn):
    for case in load("unmask_hand.json")["cases"]:
        mode = orc.UNMASK_FIXED if case["mode"] == "fixed" else orc.UNMASK_ADAPTIVE
        LB = len(case["conf"])
        argmax = np.arange(100, 100 + LB)
        tokens = np.full(LB, -1)
        mask, tok, acc = fn(case["conf"], argmax, case["mask"], tokens,
                            case["t"], case["T"], case["tau"], mode)
        assert sorted(np.nonzero(acc)[0].tolist()) == case["expected_accepted"], case
        for j in case["expected_accepted"]:
            assert tok[j] == 100 + j and not mask[j]


def check_unmask_termination(fn):
    rng = np.random.default_rng(12)
    for trial in range(300):
        LB = int(rng.integers(1, 40))
        T = int(rng.integers(1, 10))
        tau = float(rng.choice([0.5, 0.9, 0.95, 1.0, 2.0]))
        mask = np.ones(LB, dtype=bool)
        tokens = np.full(LB, -1)
        m_prev = LB
        for t in range(T):
            conf = rng.uniform(size=LB)
            mask_new, tokens, acc = fn(conf, np.arange(LB), mask, tokens, t, T, tau)
            assert not (acc & ~mask).any()              # only masked positions
            assert not (mask_new & ~mask).any()         # never re-masked
            m = int(mask_new.sum())
            # at least ceil(m_prev/(T-t)) accepted each step
            assert m_prev - m >= -(-m_prev // (T - t))
            assert m <= m_prev * (T - t - 1) / (T - t) + 1e-9
            mask, m_prev = mask_new, m
        assert m_prev == 0                               # terminates within T


def test_unmask_golden():
    check_unmask_golden(orc.unmask_step)


def test_unmask_terminates():
    check_unmask_termination(orc.unmask_step)


def test_unmask_threshold_extremes_and_fixed():
    rng = np.random.default_rng(13)
    LB, T = 32, 8
    conf = rng.uniform(0.1, 0.8, size=LB)
    # tau >= 1: exactly ceil(m/(T-t)) per step
    mask = np.ones(LB, dtype=bool)
    tokens = np.full(LB, -1)
    for t in range(T):
        m = int(mask.sum())
        mask, tokens, acc = orc.unmask_step(conf, np.arange(LB), mask, tokens, t, T, 1.0)
        assert acc.sum() == -(-m // (T - t))
    # tau below every confidence: everything at t = 0
    mask, tokens, acc = orc.unmask_step(conf, np.arange(LB), np.ones(LB, bool),
                                        np.full(LB, -1), 0, T, 0.05)
    assert acc.all() and not mask.any()
    # fixed schedule: ceil(LB/T) per step, most confident first
    mask = np.ones(LB, dtype=bool)
    tokens = np.full(LB, -1)
    for t in range(T):
        mask, tokens, acc = orc.unmask_step(conf, np.arange(LB), mask, tokens, t, T,
                                            0.0, orc.UNMASK_FIXED)
        assert acc.sum() == 4
    assert not mask.any()
    _, _, acc = orc.unmask_step(conf, np.arange(LB), np.ones(LB, bool), np.full(LB, -1),
                                0, T, 0.0, orc.UNMASK_FIXED)
    assert set(np.nonzero(acc)[0]) == set(np.argsort(-conf)[:4])


# ---------------------------------------------------------- whole block
def test_decode_block_tiny_terminates_and_r1_keeps_all():
    import torch  # noqa: F401  (workload generator draws with torch)
    from workload import WORKLOADS, prefix_inputs, step_inputs, lm_head_weight
    w = WORKLOADS["tiny-256"]
    pre = prefix_inputs(w)
    W = lm_head_weight(w)
    steps = lambda t: step_inputs(w, 0, 0, t)
    out = orc.decode_block(pre, steps, W, LB=w.LB, T=w.T, tau=w.tau,
                           r_text=w.r_text, r_img=w.r_img)
    assert len(out["steps"]) <= w.T
    assert not out["steps"][-1]["mask"].any()
    assert (out["tokens"] >= 0).all() and (out["tokens"] < w.V).all()
    assert len(out["kept"]) == 192 + 51
    out1 = orc.decode_block(pre, steps, W, LB=w.LB, T=w.T, tau=w.tau, r_text=1.0, r_img=1.0)
    assert list(out1["kept"]) == list(range(256))
    # steps after the first see the full prefix when r = 1
    if len(out1["steps"]) > 1:
        x = steps(1)
        np.testing.assert_array_equal(
            out1["steps"][1]["O"],
            orc.block_attention(x["Q"], pre["K"], pre["V"], x["Kb"], x["Vb"]))


# --------------------------------------------- planted mistakes are caught
def _fails(check, fn, *extra):
    with pytest.raises(AssertionError):
        check(fn, *extra)


def test_planted_mistakes_are_caught():
    # key norm: normaliser per modality / missing sqrt / sum over layers
    def no_sqrt(K):
        K = np.asarray(K, float)
        u = (K.reshape(K.shape[0], K.shape[1], -1) ** 2).sum(-1).mean(0)
        return u / u.mean()

    def first_layer_only(K):
        return orc.key_norm_importance(np.asarray(K)[:1])

    def max_normalised(K):
        I = orc.key_norm_importance(K)
        return I / I.max()
    for bad in (no_sqrt, first_layer_only, max_normalised):
        with pytest.raises(AssertionError):
            check_importance_golden(bad)

    # confidence: temperature dropped / multiplied / transposed W / last argmax
    def no_temp(h, W, th, **kw):
        return orc.lm_confidence(h, W, None, **kw)

    def mul_temp(h, W, th, **kw):
        return orc.lm_confidence(h, W, 1.0 / np.asarray(th), **kw)

    def last_argmax(h, W, th, **kw):
        c, am, z = orc.lm_confidence(h, W, th, want_logits=True)
        am = z.shape[1] - 1 - np.argmax(z[:, ::-1], axis=1)
        return c, am, z
    # logits offset by their maximum: c and argmax are blind to the shift,
    # the hand-worked logits are not
    def shifted_logits(h, W, th, **kw):
        c, am, z = orc.lm_confidence(h, W, th, want_logits=True)
        return c, am, z - z.max(axis=1, keepdims=True)

    # logits left without the temperature while c keeps it
    def logits_no_temp(h, W, th, **kw):
        c, am, _ = orc.lm_confidence(h, W, th)
        _, _, z = orc.lm_confidence(h, W, None, want_logits=True)
        return c, am, z
    _fails(check_confidence_brute, no_temp)
    _fails(check_confidence_brute, mul_temp)
    _fails(check_confidence_golden, last_argmax)
    _fails(check_confidence_golden, shifted_logits)
    _fails(check_confidence_brute, shifted_logits)
    _fails(check_confidence_golden, logits_no_temp)

    # selection: ties to the higher index / one pooled ranking / ceil for floor
    def ties_high(s, mod, rt, ri):
        s = np.asarray(s, float)
        mod = np.asarray(mod)
        kept = []
        for tag, r in ((0, rt), (1, ri)):
            pos = list(np.nonzero(mod == tag)[0])
            k = orc.keep_count(len(pos), r)
            kept += sorted(pos, key=lambda i: (-s[i], -i))[:k]
        return np.array(sorted(kept))

    def pooled(s, mod, rt, ri):
        mod = np.asarray(mod)
        k = orc.keep_count((mod == 0).sum(), rt) + orc.keep_count((mod == 1).sum(), ri)
        return np.array(sorted(sorted(range(len(s)), key=lambda i: (-s[i], i))[:k]))

    def ceil_count(s, mod, rt, ri):
        s = np.asarray(s, float)
        mod = np.asarray(mod)
        kept = []
        for tag, r in ((0, rt), (1, ri)):
            pos = list(np.nonzero(mod == tag)[0])
            k = math.ceil(r * len(pos) - 1e-9)
            kept += sorted(pos, key=lambda i: (-s[i], i))[:k]
        return np.array(sorted(kept))
    for bad in (ties_high, pooled, ceil_count):
        with pytest.raises(AssertionError):
            check_select_golden(orc.composite_score, bad)
            check_select_brute(bad)
    # keep pools: pool ids ignored / ties to the higher index / one too many
    def pools_ignored(s, pool, keep):
        return np.array(sorted(sorted(range(len(s)), key=lambda i: (-s[i], i))[:sum(keep)]))

    def pools_ties_high(s, pool, keep):
        s, pool = np.asarray(s, float), np.asarray(pool)
        kept = []
        for p, k in enumerate(keep):
            kept += sorted(np.nonzero(pool == p)[0], key=lambda i: (-s[i], -i))[:k]
        return np.array(sorted(kept))

    def pools_one_more(s, pool, keep):
        s, pool = np.asarray(s, float), np.asarray(pool)
        kept = []
        for p, k in enumerate(keep):
            kept += sorted(np.nonzero(pool == p)[0], key=lambda i: (-s[i], i))[:k + 1]
        return np.array(sorted(kept))
    for bad in (pools_ignored, pools_ties_high, pools_one_more):
        _fails(check_pools_golden, bad)
        _fails(check_pools_brute, bad)

    # the blend with its weights swapped agrees at alpha = 0.5; the alpha = 1
    # pin (pure key-norm order) catches it
    _fails(check_select_alpha_extremes, lambda I, c, a: a * c + (1 - a) * I)

    # attention: missing 1/sqrt(d) / wrong GQA group / block keys dropped
    def no_scale(Q, Kp, Vp, Kb, Vb):
        d = np.asarray(Q).shape[-1]
        return orc.block_attention(np.asarray(Q) * math.sqrt(d), Kp, Vp, Kb, Vb)

    def modulo_group(Q, Kp, Vp, Kb, Vb):
        Q = np.asarray(Q)
        Hq, Hkv = Q.shape[2], np.asarray(Kb).shape[2]
        order = [(h % Hkv) * (Hq // Hkv) + h // Hkv for h in range(Hq)]
        inv = np.argsort(order)
        return orc.block_attention(Q[:, :, order], Kp, Vp, Kb, Vb)[:, :, inv]

    def prefix_only(Q, Kp, Vp, Kb, Vb):
        Kb = np.asarray(Kb)
        return orc.block_attention(Q, Kp, Vp, Kb[:, :0], np.asarray(Vb)[:, :0])
    for bad in (no_scale, modulo_group, prefix_only):
        _fails(check_attention_brute, bad)

    # unmask: >= for >, 1-based step, no minimum
    def ge_tau(conf, am, mask, tok, t, T, tau, mode=0):
        return orc.unmask_step(np.nextafter(np.asarray(conf, np.float32), np.float32(2)),
                               am, mask, tok, t, T, tau, mode)

    def one_based(conf, am, mask, tok, t, T, tau, mode=0):
        return orc.unmask_step(conf, am, mask, tok, t + 1, T, tau, mode)

    def no_minimum(conf, am, mask, tok, t, T, tau, mode=0):
        return orc.unmask_step(conf, am, mask, tok, 0, 10 ** 9, tau, mode)
    _fails(check_unmask_golden, one_based)
    _fails(check_unmask_termination, no_minimum)
    # the >= variant is caught by a confidence exactly at tau
    conf = np.full(4, np.float32(0.9))
    _, _, acc = ge_tau(conf, np.arange(4), np.ones(4, bool), np.full(4, -1), 0, 4, 0.9)
    _, _, acc_ok = orc.unmask_step(conf, np.arange(4), np.ones(4, bool), np.full(4, -1), 0, 4, 0.9)
    assert acc.sum() == 4 and acc_ok.sum() == 1
