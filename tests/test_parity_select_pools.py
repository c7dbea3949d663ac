"""GPU parity of sprint_score_prune_pools (kept set with a keep count per
pool) against the oracle, and against sprint_score_prune when the pools are
the two modalities."""
import numpy as np
import pytest
import torch

from oracle import sprint_oracle as orc
from tests import gpu_cases as gc
from workload import WORKLOADS, prefix_inputs, random_confidences, small_workload

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sp():
    from kv_cache_pruning_step_b300 import sprint
    return sprint


def keep_table(sp, pools_host, n_pools, policy, r_text, r_img, r=0.5):
    """[S][n_pools] keep counts from the library's floor(r n)."""
    keep = []
    for pl in pools_host:
        sizes = np.bincount(pl, minlength=n_pools)[:n_pools]
        if policy == "global":
            keep.append([sp.sprint_keep_count(int(sizes[0]), r)] + [0] * (n_pools - 1))
        else:
            keep.append([sp.sprint_keep_count(int(n), r_text if p == 0 else r_img)
                         for p, n in enumerate(sizes)])
    return keep


def run_pools(sp, w, prefixes, confs, pools, n_pools, keep):
    cat = gc.concat_prefixes(prefixes)
    lens = [p["modality"].numel() for p in prefixes]
    koff = [0]
    for k in keep:
        koff.append(koff[-1] + sum(k))
    kept_off = torch.tensor(koff, dtype=torch.int32, device=DEV)
    pool = torch.cat([torch.as_tensor(p, dtype=torch.uint8) for p in pools]).to(DEV)
    keep_t = torch.tensor(keep, dtype=torch.int32, device=DEV).reshape(-1)
    conf = torch.cat(confs).to(DEV)
    status = sp.new_status(DEV)
    kept, score = sp.sprint_score_prune_pools(cat["K"], cat["off"], sum(lens), w.NL, w.Hkv, w.d,
                                              conf, pool, n_pools, keep_t, w.alpha, kept_off,
                                              koff[-1], want_score=True, status=status)
    torch.cuda.synchronize()
    return kept.cpu().numpy(), score.cpu().numpy(), koff, cat["off_host"], status.item()


def check_against_oracle(w, prefixes, confs, pools, keep, kept, score, koff, off, what):
    for s, p in enumerate(prefixes):
        sc = score[off[s]:off[s + 1]]
        # decisions on the GPU's own fp32 scores: exact
        want = orc.select_kept_pools(sc, pools[s], keep[s])
        assert kept[koff[s]:koff[s + 1]].tolist() == want.tolist(), f"{what} seq {s}"
        # the scores themselves against the oracle's fp64 scores
        if len(sc):
            so = orc.composite_score(orc.key_norm_importance(p["K"]), confs[s].numpy(),
                                     w.alpha)
            assert np.abs(sc - so).max() <= gc.SCORE_EXCUSE, f"{what} seq {s} scores"


@pytest.mark.parametrize("name", ["tiny-256", "prefix-4k", "prefix-32k", "batch-16x8k"])
def test_modality_pools_equal_score_prune(sp, name):
    """Pools = modalities with floor(r n) keeps: the same kept set and scores,
    bit for bit, as the two-modality selection."""
    w = WORKLOADS[name]
    prefixes = [prefix_inputs(w, seq=s, device=DEV) for s in range(min(w.S, 16))]
    confs = [random_confidences(p["modality"].numel(), seed=50 + s) for s, p in
             enumerate(prefixes)]
    pools = [p["modality"].cpu().numpy().astype(np.int64) for p in prefixes]
    keep = keep_table(sp, pools, 2, "modality", w.r_text, w.r_img)
    kept, score, koff, off, st = run_pools(sp, w, prefixes, confs, pools, 2, keep)
    assert st == 0
    cat = gc.concat_prefixes(prefixes)
    kept_off = torch.tensor(koff, dtype=torch.int32, device=DEV)
    status = sp.new_status(DEV)
    k2, s2 = sp.sprint_score_prune(cat["K"], cat["off"], off[-1], w.NL, w.Hkv, w.d,
                                   torch.cat(confs).to(DEV), cat["modality"], w.alpha, w.r_text,
                                   w.r_img, kept_off, koff[-1], want_score=True, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert np.array_equal(kept, k2.cpu().numpy())
    assert np.array_equal(score, s2.cpu().numpy())


@pytest.mark.parametrize("name", ["prefix-32k", "batch-16x8k"])
def test_per_image_pools(sp, name):
    """Text plus one pool per image (16 images of 1024 at 32K; up to 32
    images of 256 per sequence in the batch), every image at r_img."""
    w = WORKLOADS[name]
    prefixes = [prefix_inputs(w, seq=s, device=DEV) for s in range(min(w.S, 16))]
    confs = [random_confidences(p["modality"].numel(), seed=70 + s) for s, p in
             enumerate(prefixes)]
    pools = [p["image"].cpu().numpy().astype(np.int64) for p in prefixes]
    n_pools = int(max(pl.max() for pl in pools)) + 1
    keep = keep_table(sp, pools, n_pools, "per_image", w.r_text, w.r_img)
    kept, score, koff, off, st = run_pools(sp, w, prefixes, confs, pools, n_pools, keep)
    assert st == 0
    check_against_oracle(w, prefixes, confs, pools, keep, kept, score, koff, off, name)
    # every image keeps floor(r_img * its size) of its own positions
    for s in range(len(prefixes)):
        ks = kept[koff[s]:koff[s + 1]]
        got = np.bincount(pools[s][ks], minlength=n_pools)[:n_pools]
        assert got.tolist() == keep[s]


@pytest.mark.parametrize("r", [0.5, 0.25])
def test_global_pool(sp, r):
    """One pool over the whole prefix: floor(r n) positions, both modalities
    competing (the 'global keep ratio' reading)."""
    w = WORKLOADS["prefix-4k"]
    pre = prefix_inputs(w, device=DEV)
    n = pre["modality"].numel()
    conf = random_confidences(n, seed=90)
    pools = [np.zeros(n, np.int64)]
    keep = [[sp.sprint_keep_count(n, r)]]
    kept, score, koff, off, st = run_pools(sp, w, [pre], [conf], pools, 1, keep)
    assert st == 0 and len(kept) == n * r
    check_against_oracle(w, [pre], [conf], pools, keep, kept, score, koff, off, f"global {r}")


def test_ragged_random_pools_and_ties(sp):
    """Ragged sequences (0 to 2051 positions), 5 pools with random keep
    counts; one sequence with every score equal (ties everywhere: the lowest
    positions of each pool are kept)."""
    lens = [0, 1, 129, 700, 2051, 333]
    prefixes, confs, pools, keep = [], [], [], []
    g = np.random.default_rng(5)
    for s, n in enumerate(lens):
        w = small_workload(dtype="bf16", NL=2, Hq=4, Hkv=2, d=64, n=n, n_img=n // 2,
                           seed=110 + s)
        p = prefix_inputs(w, seq=s, device=DEV)
        c = random_confidences(n, seed=120 + s)
        if s == 5:  # identical keys and confidences: all scores equal
            p["K"][:] = 0.5
            c[:] = 0.25
        prefixes.append(p)
        confs.append(c)
        pl = g.integers(0, 5, size=n)
        pools.append(pl)
        sizes = np.bincount(pl, minlength=5)
        keep.append([int(g.integers(0, sz + 1)) for sz in sizes])
    kept, score, koff, off, st = run_pools(sp, w, prefixes, confs, pools, 5, keep)
    assert st == 0
    check_against_oracle(w, prefixes, confs, pools, keep, kept, score, koff, off, "ragged")
    ks = kept[koff[5]:koff[6]]
    for p in range(5):
        members = np.nonzero(pools[5] == p)[0]
        assert np.array_equal(ks[pools[5][ks] == p], members[:keep[5][p]])


def test_ragged_pools_in_clusters(sp):
    """Sequences long enough on average for clusters of 4 CTAs per
    sequence, among them sequences shorter than one CTA's slice (empty
    slices in their clusters) and one with every score equal: pool sizes,
    key ranges, ties and the compaction's cross-CTA offsets must hold."""
    lens = [0, 3, 40000, 9000, 1, 20000]
    prefixes, confs, pools, keep = [], [], [], []
    g = np.random.default_rng(9)
    for s, n in enumerate(lens):
        w = small_workload(dtype="bf16", NL=2, Hq=4, Hkv=2, d=64, n=n, n_img=n // 2,
                           seed=140 + s)
        p = prefix_inputs(w, seq=s, device=DEV)
        c = random_confidences(n, seed=150 + s)
        if s == 5:  # identical keys and confidences: all scores equal
            p["K"][:] = 0.5
            c[:] = 0.25
        prefixes.append(p)
        confs.append(c)
        pl = g.integers(0, 7, size=n)
        pools.append(pl)
        sizes = np.bincount(pl, minlength=7)
        keep.append([int(g.integers(0, sz + 1)) for sz in sizes])
    kept, score, koff, off, st = run_pools(sp, w, prefixes, confs, pools, 7, keep)
    assert st == 0
    check_against_oracle(w, prefixes, confs, pools, keep, kept, score, koff, off, "clusters")
    ks = kept[koff[5]:koff[6]]
    for p in range(7):
        members = np.nonzero(pools[5] == p)[0]
        assert np.array_equal(ks[pools[5][ks] == p], members[:keep[5][p]])


def test_bad_counts_and_pool_ids_reported(sp):
    w = small_workload(dtype="bf16", NL=1, Hq=4, Hkv=2, d=64, n=300, n_img=100, seed=3)
    pre = prefix_inputs(w, device=DEV)
    conf = random_confidences(300, seed=4)
    pl = np.zeros(300, np.int64)
    pl[::3] = 1
    # a keep count above its pool's size
    _, _, _, _, st = run_pools(sp, w, [pre], [conf], [pl], 2, [[10, 101]])
    assert st & sp.STATUS_KEPT_MISMATCH
    # a pool id >= n_pools
    bad = pl.copy()
    bad[7] = 4
    _, _, _, _, st = run_pools(sp, w, [pre], [conf], [bad], 2, [[10, 10]])
    assert st & sp.STATUS_BAD_INDEX


@pytest.mark.parametrize("selection,name", [("per_image", "prefix-4k"), ("global", "prefix-4k"),
                                            ("per_image", "tiny-256")])
def test_decoder_selection_variants(sp, selection, name):
    """BlockDecoder with per-image or whole-prefix pools: the kept set is the
    oracle's on the decoder's own scores, and the native driver and the
    call-per-step path decode the same block."""
    from kv_cache_pruning_step_b300 import BlockDecoder
    from workload import lm_head_weight, step_inputs
    w = WORKLOADS[name]
    W = lm_head_weight(w, device=DEV)
    pre = prefix_inputs(w, device=DEV)
    mod = pre["modality"].cpu().numpy()
    img = pre["image"].cpu().numpy().astype(np.int64)
    counts = [(int((mod == 0).sum()), int((mod != 0).sum()))]
    sizes = [np.bincount(img).tolist()]
    steps = []
    for t in range(w.T):
        x = step_inputs(w, 0, 0, t, device=DEV)
        steps.append({"Q": x["Q"][None].contiguous(), "Kb": x["Kb"][None].contiguous(),
                      "Vb": x["Vb"][None].contiguous(), "h": x["h"], "theta": x["theta"]})

    def make():
        return BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                            r_text=w.r_text, r_img=w.r_img, alpha=w.alpha,
                            modality_counts=counts, selection=selection, r_global=0.5,
                            pool_sizes=sizes)
    a, b = make(), make()
    ra = a.decode(pre, lambda t: steps[t])
    rb = b.decode_stepwise(pre, lambda t: steps[t])
    torch.cuda.synchronize()
    assert a.status.item() == 0 and b.status.item() == 0
    assert ra.steps == rb.steps and torch.equal(ra.tokens, rb.tokens)
    pool = img if selection == "per_image" else np.zeros_like(img)
    keep = orc.pool_keep_counts(np.bincount(pool).tolist(), selection, w.r_text, w.r_img, 0.5)
    want = orc.select_kept_pools(a.score.cpu().numpy(), pool, keep)
    assert a.kept_idx.cpu().numpy().tolist() == want.tolist()
    assert a.total_kept == sum(keep)


def test_key_norms_then_select_pools_equals_score_prune_pools(sp):
    """sprint_key_norms followed by sprint_select_kept_pools gives
    sprint_score_prune_pools' kept set and scores bit for bit."""
    lens = [0, 3, 40000, 9000, 1, 700]
    prefixes, confs, pools, keep = [], [], [], []
    g = np.random.default_rng(13)
    for s, n in enumerate(lens):
        w = small_workload(dtype="bf16", NL=2, Hq=4, Hkv=2, d=64, n=n, n_img=n // 2,
                           seed=170 + s)
        prefixes.append(prefix_inputs(w, seq=s, device=DEV))
        confs.append(random_confidences(n, seed=180 + s))
        pl = g.integers(0, 5, size=n)
        pools.append(pl)
        sizes = np.bincount(pl, minlength=5)
        keep.append([int(g.integers(0, sz + 1)) for sz in sizes])
    kept, score, koff, off, st = run_pools(sp, w, prefixes, confs, pools, 5, keep)
    assert st == 0
    cat = gc.concat_prefixes(prefixes)
    n = sum(lens)
    pool = torch.cat([torch.as_tensor(p, dtype=torch.uint8) for p in pools]).to(DEV)
    keep_t = torch.tensor(keep, dtype=torch.int32, device=DEV).reshape(-1)
    kept_off = torch.tensor(koff, dtype=torch.int32, device=DEV)
    status = sp.new_status(DEV)
    u = sp.sprint_key_norms(cat["K"], cat["off"], n, w.NL, w.Hkv, w.d, status=status)
    kept2, score2 = sp.sprint_select_kept_pools(u, cat["off"], n, torch.cat(confs).to(DEV), pool,
                                                5, keep_t, w.alpha, kept_off, koff[-1],
                                                want_score=True, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert np.array_equal(kept, kept2.cpu().numpy())
    assert np.array_equal(score, score2.cpu().numpy())
