"""GPU parity of sprint_score_prune and sprint_compact_kv against the oracle.

Stage-wise: the confidences fed to the scorer are seeded stand-ins from the
workload generator, so the selection is checked on its own inputs."""
import numpy as np
import pytest
import torch

from oracle import sprint_oracle as orc
from tests import gpu_cases as gc
from workload import (WORKLOADS, prefix_inputs, random_confidences, small_workload)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sp():
    from kv_cache_pruning_step_b300 import sprint
    return sprint


def run_score_prune(sp, w, prefixes, confs, r_text, r_img, alpha=0.5):
    cat = gc.concat_prefixes(prefixes)
    conf = torch.cat(confs).to(DEV)
    kept_host, kept_off = gc.kept_offsets([p["modality"] for p in prefixes], r_text, r_img, DEV)
    status = sp.new_status(DEV)
    kept_idx, score = sp.sprint_score_prune(
        cat["K"], cat["off"], cat["off_host"][-1], w.NL, w.Hkv, w.d, conf, cat["modality"],
        alpha, r_text, r_img, kept_off, kept_host[-1], want_score=True, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return cat, conf, kept_host, kept_off, kept_idx, score, status


def check_sequences(w, prefixes, confs, cat, kept_host, kept_idx, score, r_text, r_img, alpha=0.5):
    kept_idx = kept_idx.cpu().numpy()
    score = score.cpu().numpy()
    excused = 0
    for s, p in enumerate(prefixes):
        a, b = cat["off_host"][s], cat["off_host"][s + 1]
        imp = orc.key_norm_importance(p["K"])
        s_o = orc.composite_score(imp, confs[s].cpu().numpy().astype(np.float32), alpha)
        np.testing.assert_allclose(score[a:b], s_o, rtol=0, atol=gc.SCORE_EXCUSE / 2)
        _, nd = gc.check_kept(kept_idx[kept_host[s]:kept_host[s + 1]], s_o,
                              p["modality"].cpu().numpy(), r_text, r_img, f"seq {s}")
        excused += nd
    return excused


def test_tiny_fp32(sp):
    w = WORKLOADS["tiny-256"]
    pre = prefix_inputs(w, device=DEV)
    conf = random_confidences(256, 1, device=DEV)
    cat, conf_d, kh, ko, kept, score, _ = run_score_prune(sp, w, [pre], [conf], w.r_text, w.r_img)
    assert kept.numel() == 192 + 51
    check_sequences(w, [pre], [conf], cat, kh, kept, score, w.r_text, w.r_img)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("r_text,r_img", [(1.0, 0.8), (1.0, 1.0), (0.5, 0.29), (0.0, 0.8),
                                          (0.75, 0.0)])
def test_fuzz_ragged_sequences(sp, dtype, r_text, r_img):
    shapes = [(97, 33), (1, 0), (300, 300), (513, 1), (40, 12), (0, 0), (9000, 4500)]
    prefixes, confs = [], []
    for s, (n, n_img) in enumerate(shapes):
        w = small_workload(dtype=dtype, NL=3, Hkv=2, d=64, n=n, n_img=n_img, seed=20 + s)
        p = prefix_inputs(w, seq=s, device=DEV)
        # interleave the modalities with a seeded permutation
        g = torch.Generator().manual_seed(s)
        p["modality"] = p["modality"][torch.randperm(n, generator=g)].to(DEV)
        prefixes.append(p)
        confs.append(random_confidences(n, 100 + s, device=DEV))
    cat, conf_d, kh, ko, kept, score, _ = run_score_prune(sp, w, prefixes, confs, r_text, r_img)
    check_sequences(w, prefixes, confs, cat, kh, kept, score, r_text, r_img)


def _ragged_prefixes(shapes, NL, Hkv, d, dtype, seed0):
    prefixes, confs = [], []
    for s, (n, n_img) in enumerate(shapes):
        w = small_workload(dtype=dtype, NL=NL, Hkv=Hkv, d=d, n=n, n_img=n_img, seed=seed0 + s)
        p = prefix_inputs(w, seq=s, device=DEV)
        g = torch.Generator().manual_seed(seed0 + s)
        p["modality"] = p["modality"][torch.randperm(n, generator=g)].to(DEV)
        prefixes.append(p)
        confs.append(random_confidences(n, seed0 + 50 + s, device=DEV))
    return w, prefixes, confs


@pytest.mark.parametrize("shapes", [
    # average lengths that give clusters of 2, 4 and 8 CTAs per sequence, with
    # empty sequences, sequences shorter than the cluster, and slices that
    # end mid-warp
    [(5000, 1234), (4000, 0), (0, 0), (5, 5)],
    [(15000, 7001), (7, 3)],
    [(40000, 20000), (5, 2), (100, 0)],
])
@pytest.mark.parametrize("r_text,r_img", [(1.0, 0.8), (0.5, 0.29)])
def test_cluster_sizes_ragged(sp, shapes, r_text, r_img):
    w, prefixes, confs = _ragged_prefixes(shapes, 2, 1, 8, "f32", 300)
    cat, conf_d, kh, ko, kept, score, _ = run_score_prune(sp, w, prefixes, confs, r_text, r_img)
    check_sequences(w, prefixes, confs, cat, kh, kept, score, r_text, r_img)


def test_long_sequence_keys_in_workspace(sp):
    """A sequence whose slice of the cluster exceeds what shared memory
    stages (more than 8 x 16384 positions) keeps its keys in the workspace;
    a short sequence in the same call is staged."""
    shapes = [(140000, 70001), (300, 100)]
    w, prefixes, confs = _ragged_prefixes(shapes, 1, 1, 8, "f32", 400)
    for r_text, r_img in ((1.0, 0.8), (0.37, 0.61)):
        cat, conf_d, kh, ko, kept, score, _ = run_score_prune(sp, w, prefixes, confs, r_text,
                                                              r_img)
        check_sequences(w, prefixes, confs, cat, kh, kept, score, r_text, r_img)


def test_ties_go_to_lower_index(sp):
    w = small_workload(dtype="f32", NL=2, Hkv=2, d=64, n=64, n_img=0, seed=3)
    p = prefix_inputs(w, device=DEV)
    conf = random_confidences(64, 5, device=DEV)
    # positions 10..19 become exact copies of position 5: identical scores
    for i in range(10, 20):
        p["K"][:, i] = p["K"][:, 5]
        conf[i] = conf[5]
    # keep exactly half; the copies straddle the threshold in several r
    for r in (0.1, 0.25, 0.5, 0.8):
        cat, conf_d, kh, ko, kept, score, _ = run_score_prune(sp, w, [p], [conf], r, 1.0)
        s_np = score.cpu().numpy()
        assert len(set(s_np[[5] + list(range(10, 20))].tolist())) == 1
        kept_o = orc.select_kept(s_np.astype(np.float64), p["modality"].cpu().numpy(), r, 1.0)
        assert kept.cpu().numpy().tolist() == kept_o.tolist()


def test_alpha_extremes(sp):
    w = small_workload(dtype="f32", NL=2, Hkv=2, d=64, n=200, n_img=80, seed=4)
    p = prefix_inputs(w, device=DEV)
    conf = random_confidences(200, 6, device=DEV)
    for alpha in (0.0, 1.0, 0.3):
        cat, conf_d, kh, ko, kept, score, _ = run_score_prune(sp, w, [p], [conf], 0.6, 0.4, alpha)
        check_sequences(w, [p], [conf], cat, kh, kept, score, 0.6, 0.4, alpha)


def test_kept_offsets_mismatch_reports_status(sp):
    w = small_workload(dtype="f32", n=50, n_img=10)
    p = prefix_inputs(w, device=DEV)
    conf = random_confidences(50, 1, device=DEV)
    cat = gc.concat_prefixes([p])
    kept_off = torch.tensor([0, 7], dtype=torch.int32, device=DEV)
    kept_idx = torch.full((7,), -5, dtype=torch.int32, device=DEV)
    status = sp.new_status(DEV)
    sp.sprint_score_prune(cat["K"], cat["off"], 50, w.NL, w.Hkv, w.d, conf, cat["modality"],
                          0.5, 1.0, 0.8, kept_off, 7, kept_idx=kept_idx, status=status)
    torch.cuda.synchronize()
    assert status.item() & sp.STATUS_KEPT_MISMATCH
    assert (kept_idx == -5).all()


@pytest.mark.parametrize("name", ["prefix-4k", "prefix-32k", "batch-16x8k"])
def test_full_size_workloads(sp, name):
    w = WORKLOADS[name]
    prefixes = [prefix_inputs(w, seq=s, device=DEV) for s in range(w.S)]
    confs = [random_confidences(p["modality"].numel(), 7 + s, device=DEV)
             for s, p in enumerate(prefixes)]
    cat, conf_d, kh, ko, kept, score, _ = run_score_prune(sp, w, prefixes, confs, w.r_text, w.r_img)
    # the oracle's key norms at full size, sequence by sequence
    excused = check_sequences(w, prefixes, confs, cat, kh, kept, score, w.r_text, w.r_img)
    assert excused <= 4
    # r = 1 keeps every position, ascending
    cat, conf_d, kh, ko, kept1, _, _ = run_score_prune(sp, w, prefixes, confs, 1.0, 1.0)
    got = kept1.cpu().numpy()
    for s in range(w.S):
        n = cat["off_host"][s + 1] - cat["off_host"][s]
        assert got[kh[s]:kh[s + 1]].tolist() == list(range(n))


@pytest.mark.parametrize("name,dtype", [("tiny-256", None), ("prefix-32k", None),
                                        ("batch-16x8k", None)])
def test_compaction_is_an_exact_gather(sp, name, dtype):
    w = WORKLOADS[name]
    prefixes = [prefix_inputs(w, seq=s, device=DEV) for s in range(w.S)]
    confs = [random_confidences(p["modality"].numel(), 9 + s, device=DEV)
             for s, p in enumerate(prefixes)]
    cat, conf_d, kh, ko, kept, score, _ = run_score_prune(sp, w, prefixes, confs, w.r_text, w.r_img)
    status = sp.new_status(DEV)
    Kp, Vp = sp.sprint_compact_kv(cat["K"], cat["V"], cat["off"], cat["off_host"][-1], w.NL,
                                  w.Hkv, w.d, kept, ko, kh[-1], status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kept_np = kept.cpu().numpy()
    row = w.NL * w.Hkv * w.d
    for s, p in enumerate(prefixes):
        k_s = kh[s + 1] - kh[s]
        idx = kept_np[kh[s]:kh[s + 1]]
        for src, dst in ((p["K"], Kp), (p["V"], Vp)):
            want = orc.compact(src, idx)
            got = gc.host(dst[kh[s] * row:kh[s + 1] * row].view(w.NL, k_s, w.Hkv, w.d))
            np.testing.assert_array_equal(got, want)


def test_compaction_identity_and_bad_index(sp):
    w = small_workload(dtype="bf16", NL=3, Hkv=2, d=64, n=77, n_img=20)
    p = prefix_inputs(w, device=DEV)
    cat = gc.concat_prefixes([p])
    idx = torch.arange(77, dtype=torch.int32, device=DEV)
    off = torch.tensor([0, 77], dtype=torch.int32, device=DEV)
    status = sp.new_status(DEV)
    Kp, Vp = sp.sprint_compact_kv(cat["K"], cat["V"], cat["off"], 77, w.NL, w.Hkv, w.d, idx, off,
                                  77, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(Kp, cat["K"]) and torch.equal(Vp, cat["V"])
    idx[3] = 77  # outside the prefix: reported, row skipped
    Kp.zero_()
    sp.sprint_compact_kv(cat["K"], cat["V"], cat["off"], 77, w.NL, w.Hkv, w.d, idx, off, 77,
                         Kp=Kp, Vp=Vp, status=status)
    torch.cuda.synchronize()
    assert status.item() & sp.STATUS_BAD_INDEX


@pytest.mark.parametrize("dtype,shapes", [
    ("bf16", [(4096, 3072)]),
    ("f32", [(5000, 1234), (4000, 0), (0, 0), (5, 5)]),
    ("bf16", [(40000, 20000), (5, 2), (100, 0)]),
])
def test_key_norms_then_select_equals_score_prune(sp, dtype, shapes):
    """sprint_key_norms followed by sprint_select_kept (the split the
    decoder overlaps with the prefix LM head) gives sprint_score_prune's
    kept set and scores bit for bit, and the key norms are the oracle's."""
    w, prefixes, confs = _ragged_prefixes(shapes, 2, 2, 64, dtype, 500)
    r_text, r_img = 1.0, 0.8
    cat, conf, kh, ko, kept, score, _ = run_score_prune(sp, w, prefixes, confs, r_text, r_img)
    n = cat["off_host"][-1]
    status = sp.new_status(DEV)
    u = sp.sprint_key_norms(cat["K"], cat["off"], n, w.NL, w.Hkv, w.d, status=status)
    kept2, score2 = sp.sprint_select_kept(u, cat["off"], n, conf, cat["modality"], 0.5, r_text,
                                          r_img, ko, kh[-1], want_score=True, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(kept, kept2)
    assert torch.equal(score, score2)
    for s, p in enumerate(prefixes):
        a, b = cat["off_host"][s], cat["off_host"][s + 1]
        if b > a:  # u over its mean is the oracle's importance
            us = u[a:b].cpu().numpy().astype(np.float64)
            np.testing.assert_allclose(us / us.mean(), orc.key_norm_importance(p["K"]),
                                       rtol=1e-5)
