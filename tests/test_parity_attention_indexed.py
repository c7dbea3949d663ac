"""GPU parity of sprint_block_attn_indexed: attention over the kept rows of
the full cache read through the kept indices.

It must equal sprint_compact_kv followed by sprint_block_attn bit for bit
(same keys in the same order, same kernels' arithmetic), and the oracle's
attention over the oracle's compacted cache within the attention tolerance.
"""
import numpy as np
import pytest
import torch

from oracle import sprint_oracle as orc
from tests import gpu_cases as gc
from workload import WORKLOADS, prefix_inputs, small_workload, step_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sp():
    from kv_cache_pruning_step_b300 import sprint
    return sprint


def random_kept(lens, frac, seed, sort=True):
    """Seeded kept sets: for sequence s, round(frac * n_s) distinct local
    indices (ascending unless sort=False), plus the CSR offsets."""
    g = torch.Generator().manual_seed(seed)
    sets, off = [], [0]
    for n in lens:
        k = int(round(frac * n))
        idx = torch.randperm(n, generator=g)[:k]
        if sort:
            idx = idx.sort().values
        sets.append(idx.to(torch.int32))
        off.append(off[-1] + k)
    return sets, off


def both_paths(sp, w, prefixes, steps, kept_sets, kept_off):
    """(O from compact + attention, O from indexed attention, status)."""
    cat = gc.concat_prefixes(prefixes)
    lens = [p["modality"].numel() for p in prefixes]
    Q = torch.stack([x["Q"] for x in steps]).contiguous()
    Kb = torch.stack([x["Kb"] for x in steps]).contiguous()
    Vb = torch.stack([x["Vb"] for x in steps]).contiguous()
    idx = (torch.cat(kept_sets) if kept_sets else torch.empty(0, dtype=torch.int32)).to(DEV)
    koff = torch.tensor(kept_off, dtype=torch.int32, device=DEV)
    total_kept, max_kept = kept_off[-1], max([b - a for a, b in zip(kept_off, kept_off[1:])])
    status = sp.new_status(DEV)
    Kp, Vp = sp.sprint_compact_kv(cat["K"], cat["V"], cat["off"], sum(lens), w.NL, w.Hkv, w.d,
                                  idx, koff, total_kept, status=status)
    O_c = sp.sprint_block_attn(Q, Kp, Vp, koff, max_kept, total_kept, Kb, Vb, status=status)
    status_i = sp.new_status(DEV)
    O_i = sp.sprint_block_attn_indexed(Q, cat["K"], cat["V"], cat["off"], sum(lens), idx, koff,
                                       max_kept, total_kept, Kb, Vb, status=status_i)
    torch.cuda.synchronize()
    assert status.item() == 0
    return O_c, O_i, status_i.item()


def check_oracle(w, prefixes, steps, kept_sets, O, picks, layers=None, what=""):
    for s in picks:
        p, x, kept = prefixes[s], steps[s], kept_sets[s].numpy()
        want = orc.block_attention(x["Q"], orc.compact(p["K"], kept), orc.compact(p["V"], kept),
                                   x["Kb"], x["Vb"], layers=layers)
        sel = list(range(w.NL)) if layers is None else layers
        gc.assert_close(gc.host(O[s])[sel], want[sel], w.torch_dtype, f"{what} seq {s}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("Hq,Hkv,d,LB", [(4, 2, 64, 32), (16, 4, 128, 32), (8, 8, 64, 16),
                                         (6, 2, 128, 7), (2, 1, 64, 1)])
def test_indexed_equals_compacted_ragged(sp, dtype, Hq, Hkv, d, LB):
    lens = [0, 1, 129, 700, 2051]
    prefixes, steps = [], []
    for s, n in enumerate(lens):
        w = small_workload(dtype=dtype, NL=2, Hq=Hq, Hkv=Hkv, d=d, LB=LB, n=n, n_img=n // 3,
                           seed=40 + s)
        prefixes.append(prefix_inputs(w, seq=s, device=DEV))
        steps.append(step_inputs(w, s, 0, 3, device=DEV))
    kept_sets, kept_off = random_kept(lens, 0.8, seed=7)
    O_c, O_i, st = both_paths(sp, w, prefixes, steps, kept_sets, kept_off)
    assert st == 0
    assert torch.equal(O_c, O_i)
    check_oracle(w, prefixes, steps, kept_sets, O_i, picks=range(len(lens)),
                 what=f"{dtype} {Hq}/{Hkv}/{d}/{LB}")


@pytest.mark.parametrize("frac", [0.0, 0.3, 1.0])
def test_indexed_keep_fractions(sp, frac):
    """Nothing kept (block keys only), a sparse set spanning several tiles, and
    everything kept (r = 1: equals attention over the full prefix)."""
    lens = [300, 1000]
    prefixes, steps = [], []
    for s, n in enumerate(lens):
        w = small_workload(dtype="bf16", NL=3, Hq=16, Hkv=4, d=128, LB=32, n=n, n_img=n // 2,
                           seed=90 + s)
        prefixes.append(prefix_inputs(w, seq=s, device=DEV))
        steps.append(step_inputs(w, s, 0, 1, device=DEV))
    kept_sets, kept_off = random_kept(lens, frac, seed=8)
    O_c, O_i, st = both_paths(sp, w, prefixes, steps, kept_sets, kept_off)
    assert st == 0 and torch.equal(O_c, O_i)
    check_oracle(w, prefixes, steps, kept_sets, O_i, picks=[0, 1], what=f"frac {frac}")
    if frac == 1.0:
        cat = gc.concat_prefixes(prefixes)
        O_full = sp.sprint_block_attn(torch.stack([x["Q"] for x in steps]).contiguous(),
                                      cat["K"], cat["V"], cat["off"], max(lens), sum(lens),
                                      torch.stack([x["Kb"] for x in steps]).contiguous(),
                                      torch.stack([x["Vb"] for x in steps]).contiguous())
        assert torch.equal(O_full, O_i)


def test_indexed_any_order_and_repeats(sp):
    """The keys are taken in the order the indices give, repeats included."""
    w = small_workload(dtype="bf16", NL=2, Hq=8, Hkv=2, d=128, LB=16, n=900, n_img=300, seed=5)
    pre = prefix_inputs(w, device=DEV)
    x = step_inputs(w, 0, 0, 2, device=DEV)
    g = torch.Generator().manual_seed(3)
    idx = torch.randint(0, 900, (700,), generator=g).to(torch.int32)  # unsorted, repeats
    O_c, O_i, st = both_paths(sp, w, [pre], [x], [idx], [0, 700])
    assert st == 0 and torch.equal(O_c, O_i)
    check_oracle(w, [pre], [x], [idx], O_i, picks=[0], what="unsorted")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_indexed_bad_index_reported_and_read_as_zeros(sp, dtype):
    """An index outside [0, n_s) sets SPRINT_STATUS_BAD_INDEX and that key
    and value are read as zeros (the kernels check every index before use)."""
    w = small_workload(dtype=dtype, NL=2, Hq=4, Hkv=2, d=64, LB=8, n=200, n_img=50, seed=6)
    pre = prefix_inputs(w, device=DEV)
    x = step_inputs(w, 0, 0, 1, device=DEV)
    idx = torch.arange(0, 200, 2, dtype=torch.int32)
    idx[10] = 200       # one past the prefix
    idx[57] = -3
    cat = gc.concat_prefixes([pre])
    koff = torch.tensor([0, 100], dtype=torch.int32, device=DEV)
    status = sp.new_status(DEV)
    O = sp.sprint_block_attn_indexed(x["Q"][None].contiguous(), cat["K"], cat["V"], cat["off"],
                                     200, idx.to(DEV), koff, 100, 100,
                                     x["Kb"][None].contiguous(), x["Vb"][None].contiguous(),
                                     status=status)
    torch.cuda.synchronize()
    assert status.item() & sp.STATUS_BAD_INDEX
    safe = idx.clone()
    safe[10] = safe[57] = 0
    Kp = orc.compact(pre["K"], safe.numpy())
    Vp = orc.compact(pre["V"], safe.numpy())
    Kp[:, [10, 57]] = 0.0
    Vp[:, [10, 57]] = 0.0
    want = orc.block_attention(x["Q"], Kp, Vp, x["Kb"], x["Vb"])
    gc.assert_close(gc.host(O[0]), want, w.torch_dtype, "bad index as zeros")


def test_indexed_many_short_sequences_two_stage_ring(sp):
    """300 short sequences: the bf16 kernel runs a 2-stage ring, where each
    gathered tile is signalled as soon as its copies land."""
    g = torch.Generator().manual_seed(12)
    lens = torch.randint(0, 201, (300,), generator=g).tolist()
    prefixes, steps = [], []
    for s, n in enumerate(lens):
        w = small_workload(dtype="bf16", NL=1, Hq=8, Hkv=2, d=128, LB=16, n=n, n_img=n // 4,
                           seed=900 + s)
        prefixes.append(prefix_inputs(w, seq=s, device=DEV))
        steps.append(step_inputs(w, s, 0, 1, device=DEV))
    kept_sets, kept_off = random_kept(lens, 0.7, seed=9)
    O_c, O_i, st = both_paths(sp, w, prefixes, steps, kept_sets, kept_off)
    assert st == 0 and torch.equal(O_c, O_i)
    check_oracle(w, prefixes, steps, kept_sets, O_i, picks=[0, 1, 150, 299], what="many")


@pytest.mark.parametrize("name", ["prefix-4k", "prefix-32k"])
def test_indexed_full_size(sp, name):
    """Full-size caches with the workload's keep counts (all text, 80% of the
    image rows): bit-identical to the compacted path, oracle on sampled layers."""
    w = WORKLOADS[name]
    pre = prefix_inputs(w, device=DEV)
    x = step_inputs(w, 0, 0, 1, device=DEV)
    mod = pre["modality"].cpu().numpy() != 0
    g = np.random.default_rng(21)
    img = np.flatnonzero(mod)
    keep_img = g.choice(img, size=orc.keep_count(len(img), w.r_img), replace=False)
    kept = np.sort(np.concatenate([np.flatnonzero(~mod), keep_img])).astype(np.int32)
    kept_t = torch.from_numpy(kept)
    O_c, O_i, st = both_paths(sp, w, [pre], [x], [kept_t], [0, len(kept)])
    assert st == 0 and torch.equal(O_c, O_i)
    check_oracle(w, [pre], [x], [kept_t], O_i, picks=[0], layers=[0, w.NL - 1], what=name)
